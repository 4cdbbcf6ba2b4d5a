// Host orchestrator and C ABI of the LoPA branch-verification library.
//
// One context owns the static KV cache, the per-branch Pre-Write scratch, activations
// and the decoding state (in device memory), and two captured CUDA graphs:
//   start graph : the block-start forward of a fresh all-[MASK] block (1 branch), whose
//                 logit summary seeds the first LoPA iteration;
//   step graph  : one LoPA iteration - decide (anchor + lookahead branches), the
//                 isolated verification forward of all 1+k branches, select (branch
//                 confidence, winner, logit reuse), Commit-Winner of the winner's K/V,
//                 finalize.
// Every graph reads the block position from device memory, so one capture serves the
// whole decode ("Decoding-efficiency revolution" blog, section 5.2: without CUDA graphs
// kernel-launch overhead dominates).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace lopa;

namespace {

thread_local std::string g_init_error;

}  // namespace

namespace lopa {
void set_global_error(const char* msg) { g_init_error = msg ? msg : ""; }

// Programmatic dependent launch is on unless LOPA_NO_PDL is set (a debugging switch).
bool pdl_enabled() {
  static const bool on = getenv("LOPA_NO_PDL") == nullptr;
  return on;
}

cudaError_t set_uniform_carveout() {
  cudaError_t e;
  if ((e = gemm_set_carveout()) != cudaSuccess) return e;
  if ((e = attention_set_carveout()) != cudaSuccess) return e;
  if ((e = pointwise_set_carveout()) != cudaSuccess) return e;
  return decide_set_carveout();
}
}  // namespace lopa

namespace {

struct Plan {
  int nb = 0, Bq = 0, T = 0, tok_box = 0, kv_to_cache = 0;
  bool lm = false;
  const int* tok = nullptr;
  int* am_out = nullptr;
  float* mp_out = nullptr;
  std::vector<GemmLaunch> qkv, o, gu, dn;
  std::vector<AttnLaunch> attn;
  GemmLaunch lmh;
};

}  // namespace

struct lopa_ctx {
  lopa_model_config mc{};
  lopa_decode_config dc{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int num_sms = 0;
  int ccap[kMaxClusterSplits + 1] = {};  // resident clusters of 1, 2, 4 q/k/v-GEMM CTAs
  // borrowed weights
  const bf16 *embed = nullptr, *final_norm = nullptr;
  std::vector<const bf16*> attn_norm, mlp_norm;
  // owned tile-major copies: q/k/v stacked, output, gate/up stacked, down (per layer), and
  // the LM head: bf16, or E4M3 codes with one float32 scale per row (w8)
  bool w8 = false;
  std::vector<const void*> wqkv, wo, wgu, wd;
  const void* lm_head = nullptr;
  std::vector<const float*> sqkv, so, sgu, sd;
  const float* slm = nullptr;
  // owned device memory
  std::vector<void*> allocs;
  bf16 *kc = nullptr, *vc = nullptr, *ks = nullptr, *vs = nullptr;
  float* x = nullptr;
  bf16* n = nullptr;
  float* part = nullptr;  // split-K partial sums [split][T][d] of the O and down projections
  size_t part_floats = 0;
  float* xws = nullptr;   // q/k/v split-K exchange workspace
  size_t xws_floats = 0;
  bf16 *q = nullptr, *attn = nullptr, *hm = nullptr;
  float *pm = nullptr, *ps = nullptr;
  int* pi = nullptr;
  int nvt = 0, part_ld = 0;
  float *cos_t = nullptr, *sin_t = nullptr;
  int *branch_tok = nullptr, *valid = nullptr, *am_b = nullptr, *tok_rows = nullptr;
  float* mp_b = nullptr;
  int* out_tokens = nullptr;
  DevState* st = nullptr;
  int Tmax = 0, nbmax = 0, qkv_rows = 0;
  int nslots = 0;  // branch rows the block buffers hold: nbmax, at least 2 (a merged pass)
  // K cache [L][max_seq][Hk*dh], K scratch [L][nslots*B][Hk*dh]; values transposed:
  // V^T cache [L][Hk*dh][vt_ld], V^T scratch [L][Hk*dh][nslots*B].
  size_t cache_layer = 0, scr_layer = 0, vt_cache_layer = 0;
  int vt_ld = 0;
  // graphs
  // step_plans[nb]: verification forward of nb branches (nb = 1..1+k; step_plan is the
  // full one); merged_plan: [completing branch ; blank next block] with block-causal
  // attention; start_plan: the block-start forward of a fresh block.
  std::vector<Plan> step_plans;
  Plan& step_plan() { return step_plans.back(); }
  Plan merged_plan, start_plan;
  Plan prefill_plan;  // the prompt forward of the last prompt length (rebuilt when it changes)
  std::vector<cudaGraphExec_t> step_execs;
  cudaGraphExec_t merged_exec = nullptr, start_exec = nullptr;
  int cur_nb = 0;  // branch count of the graph being captured
  // lopa_time_forward: forward-only graphs (0 block start, 1 verification), built lazily
  Plan time_start_plan;
  const Plan* fwd_plan = nullptr;
  cudaGraphExec_t fwd_exec[2] = {nullptr, nullptr};
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  lopa_step_result* h_res = nullptr;  // pinned
  int* h_next = nullptr;              // pinned: {n_valid, final_w} of the last decide
  // host-side view of the decode
  // block_fresh: the current block has no logits yet (needs its block-start forward);
  // in_block: it has had at least one iteration; next_nv / next_final: the branches the
  // last decide built for the coming iteration (valid when !block_fresh).
  bool prefilled = false, block_fresh = true, in_block = false;
  int next_nv = 0, next_final = -1;
  int P = 0, P0 = 0;
  std::string err;
};

namespace {

int fail(lopa_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c)
    c->err = buf;
  else
    g_init_error = buf;
  return code;
}

#define CK(call)                                                                        \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(ctx, LOPA_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                                  \
  } while (0)

template <typename T>
int dalloc(lopa_ctx* ctx, T** p, size_t count) {
  void* v = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 256);
  if (cudaMalloc(&v, bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(ctx, LOPA_ERR_OOM, "cudaMalloc of %zu bytes failed", bytes);
  }
  ctx->allocs.push_back(v);
  *p = static_cast<T*>(v);
  return 0;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int round16(int v) { return (v + 15) / 16 * 16; }

// Split-K factor that fills the GPU with roughly one CTA per SM.
int pick_splits(int tiles, int k_blocks, int num_sms) {
  int s = num_sms / std::max(tiles, 1);
  s = std::min(s, std::max(k_blocks / 2, 1));
  s = std::min(s, 16);  // the consumers read every split: keep that bounded
  return std::max(s, 1);
}

// Tiling of a split-K projection over T token rows: weight tiles (128 rows) per CTA and the
// split count.  Two tiles per CTA halve the activation traffic from L2 per weight byte (the
// token tile is loaded once for both); the split count then fills the SMs.
void proj_tiling(int nrows, int K, int T, int num_sms, int* na, int* splits) {
  const int tok_box = std::min(256, round16(T));
  const int zt = (T + tok_box - 1) / tok_box;
  *na = nrows < 256 ? 1 : 2;
  const int tiles = ((nrows + *na * 128 - 1) / (*na * 128)) * zt;
  *splits = pick_splits(tiles, K / 64, num_sms);
}

// Floats of split-K partials a forward over T rows needs (output and down projections).
size_t partial_floats(const lopa_ctx* ctx, int T) {
  const lopa_model_config& m = ctx->mc;
  const int Ks[2] = {m.n_heads * m.head_dim, m.ffn};
  size_t need = 0;
  for (int i = 0; i < 2; ++i) {
    int na, splits;
    proj_tiling(m.d_model, Ks[i], T, ctx->num_sms, &na, &splits);
    need = std::max(need, (size_t)splits * T * m.d_model);
  }
  return need;
}

// Tiling of the clustered q/k/v GEMM over T token rows: na weight tiles (128 rows each)
// per CTA and cs K-splits per output tile, the splits of a tile forming one cluster.
// Picks the most CTAs that are resident at once (all tiles in one wave), then the larger
// na (fewer activation re-reads), then the smaller cluster (less exchange).  When no
// choice fits one wave, na = 2 and cs = 1.
int qkv_box(int T) { return std::min(256, round16(T)); }

void qkv_tiling(const lopa_ctx* ctx, int nrows, int K, int T, int* na, int* cs) {
  const int tok_box = qkv_box(T);
  const int zt = (T + tok_box - 1) / tok_box;
  int best = 0;
  *na = 2;
  *cs = 1;
  for (int n = 2; n >= 1; --n) {
    const int tiles = ((nrows + n * 128 - 1) / (n * 128)) * zt;
    for (int c = 1; c <= kMaxClusterSplits; c *= 2) {
      if (c > 1 && c > K / 64 / 2) break;
      if (tiles > ctx->ccap[c]) continue;
      if (tiles * c > best) {
        best = tiles * c;
        *na = n;
        *cs = c;
      }
    }
  }
}

int build_plan(lopa_ctx* ctx, Plan& p, int nb, int Bq, int kv_to_cache, bool lm, const int* tok,
               int* am_out, float* mp_out, bool causal = false) {
  const lopa_model_config& m = ctx->mc;
  const int L = m.n_layers, d = m.d_model, H = m.n_heads, dh = m.head_dim, F = m.ffn;
  p.nb = nb;
  p.Bq = Bq;
  p.T = nb * Bq;
  p.tok_box = std::min(256, round16(p.T));
  p.kv_to_cache = kv_to_cache;
  p.lm = lm;
  p.tok = tok;
  p.am_out = am_out;
  p.mp_out = mp_out;
  p.qkv.resize(L);
  p.attn.resize(L);
  p.o.resize(L);
  p.gu.resize(L);
  p.dn.resize(L);
  auto plan = [&](GemmLaunch& G, int mode, const void* act, int K, const void* w,
                  const float* wscale, int nrows, const char* what) -> int {
    int na = 2, splits = 1;
    if (mode == GEMM_QKV) {
      qkv_tiling(ctx, nrows, K, p.T, &na, &splits);
    } else if (mode == GEMM_RED_ADD) {
      proj_tiling(nrows, K, p.T, ctx->num_sms, &na, &splits);
      while (splits > 1 && (size_t)splits * p.T * nrows > ctx->part_floats) --splits;
    }
    const char* e = plan_gemm(&G, mode, act, ctx->Tmax, p.T, w, nrows, K, na, splits,
                              mode == GEMM_QKV ? qkv_box(p.T) : p.tok_box,
                              ctx->num_sms, /*w_packed=*/true, wscale);
    if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s GEMM: %s", what, e);
    if (mode == GEMM_RED_ADD) {
      if ((size_t)G.args.splits * p.T * nrows > ctx->part_floats)
        return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s GEMM: partial buffer too small", what);
      G.args.out_f32 = ctx->part;
      G.args.ldo = nrows;
      G.args.atomic = 0;
      G.args.split_stride = (size_t)p.T * nrows;
    }
    G.args.err = &ctx->st->err;
    return 0;
  };
  for (int l = 0; l < L; ++l) {
    int r;
    auto sc = [&](const std::vector<const float*>& v) { return ctx->w8 ? v[l] : nullptr; };
    if ((r = plan(p.qkv[l], GEMM_QKV, ctx->n, d, ctx->wqkv[l], sc(ctx->sqkv), ctx->qkv_rows, "qkv")))
      return r;
    GemmArgs& qa = p.qkv[l].args;
    qa.q = ctx->q;
    bf16* kcl = ctx->kc + (size_t)l * ctx->cache_layer;
    bf16* vcl = ctx->vc + (size_t)l * ctx->vt_cache_layer;
    bf16* ksl = ctx->ks + (size_t)l * ctx->scr_layer;
    bf16* vsl = ctx->vs + (size_t)l * ctx->scr_layer;
    qa.kdst = kv_to_cache ? kcl : ksl;
    qa.vdst = kv_to_cache ? vcl : vsl;
    qa.ldv = kv_to_cache ? ctx->vt_ld : ctx->nslots * ctx->dc.block;
    qa.cos_t = ctx->cos_t;
    qa.sin_t = ctx->sin_t;
    qa.dP = &ctx->st->P;
    qa.H = H;
    qa.Hk = m.n_kv_heads;
    qa.dh = dh;
    qa.Bq = Bq;
    qa.kv_to_cache = kv_to_cache;
    qa.pos_linear = causal ? 1 : 0;
    qa.xws = ctx->xws;
    if (qkv_exchange_floats(p.qkv[l].grid.x, qa.splits, p.qkv[l].grid.z, qa.nbox) > ctx->xws_floats)
      return fail(ctx, LOPA_ERR_UNSUPPORTED, "q/k/v exchange workspace too small");
    AttnArgs aa = {};
    aa.q = ctx->q;
    aa.out = ctx->attn;
    aa.kc = kcl;
    aa.vtc = vcl;
    aa.kb = ksl;
    aa.vtb = vsl;
    aa.dP = &ctx->st->P;
    aa.pk_add = kv_to_cache ? p.T : 0;
    aa.ldvc = ctx->vt_ld;
    aa.ldvb = ctx->nslots * ctx->dc.block;
    aa.Bq = Bq;
    aa.Bk = kv_to_cache ? 0 : Bq;
    aa.Bk_stride = Bq;
    aa.nbq = nb;
    aa.causal = causal ? 1 : 0;
    aa.H = H;
    aa.Hk = m.n_kv_heads;
    aa.err = &ctx->st->err;
    const char* ea = plan_attention(&p.attn[l], aa, dh, m.max_seq, ctx->vt_ld);
    if (ea[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", ea);
    if ((r = plan(p.o[l], GEMM_RED_ADD, ctx->attn, H * dh, ctx->wo[l], sc(ctx->so), d, "o"))) return r;
    if ((r = plan(p.gu[l], GEMM_SWIGLU, ctx->n, d, ctx->wgu[l], sc(ctx->sgu), 2 * F, "gate/up")))
      return r;
    p.gu[l].args.out_bf16 = ctx->hm;
    p.gu[l].args.ldh = F;
    if ((r = plan(p.dn[l], GEMM_RED_ADD, ctx->hm, F, ctx->wd[l], sc(ctx->sd), d, "down"))) return r;
  }
  if (lm) {
    const int na = p.T > 128 ? 2 : 1;
    const char* e = plan_gemm(&p.lmh, GEMM_LMSTATS, ctx->n, ctx->Tmax, p.T, ctx->lm_head, m.vocab,
                              d, na, 1, 0, ctx->num_sms, /*w_packed=*/true, ctx->w8 ? ctx->slm : nullptr);
    if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "lm-head GEMM: %s", e);
    GemmArgs& a = p.lmh.args;
    a.V = m.vocab;
    a.mask_id = m.mask_id;
    a.scale = m.logit_scale;
    a.part_m = ctx->pm;
    a.part_s = ctx->ps;
    a.part_i = ctx->pi;
    a.part_ld = ctx->part_ld;
    a.err = &ctx->st->err;
  }
  return 0;
}

// Enqueues one forward of plan p on the context stream (also used inside capture).
int enqueue_forward(lopa_ctx* ctx, const Plan& p) {
  const lopa_model_config& m = ctx->mc;
  const int L = m.n_layers, d = m.d_model;
  cudaStream_t s = ctx->stream;
  CK(launch_embed_norm(p.tok, p.T, ctx->embed, ctx->attn_norm[0], ctx->x, ctx->n, d, m.rms_eps,
                       m.vocab, &ctx->st->err, s));
  for (int l = 0; l < L; ++l) {
    CK(launch_gemm(p.qkv[l], s));  // q, k, v + RoPE; K/V Pre-Write
    CK(launch_attention(p.attn[l], s));
    CK(launch_gemm(p.o[l], s));  // split-K partials of attn . Wo^T
    CK(launch_residual_norm(ctx->x, ctx->part, p.o[l].args.splits, p.o[l].args.split_stride,
                            ctx->mlp_norm[l], ctx->n, p.T, d, m.rms_eps, s));
    CK(launch_gemm(p.gu[l], s));
    CK(launch_gemm(p.dn[l], s));  // split-K partials of h . Wd^T
    CK(launch_residual_norm(ctx->x, ctx->part, p.dn[l].args.splits, p.dn[l].args.split_stride,
                            l + 1 < L ? ctx->attn_norm[l + 1] : ctx->final_norm, ctx->n, p.T, d,
                            m.rms_eps, s));
  }
  if (p.lm) {
    CK(launch_gemm(p.lmh, s));
    CK(launch_lm_merge(ctx->pm, ctx->ps, ctx->pi, ctx->nvt, ctx->part_ld, p.T, p.am_out, p.mp_out,
                       s));
  }
  return 0;
}

// One LoPA iteration after its decide: the verification forward of plan p (nb branches),
// select, Commit-Winner, finalize (with next-block logits for the merged plan), then the
// decide of the coming iteration, whose branch count and completion flag the host reads
// back with the step result.
int enqueue_iteration(lopa_ctx* ctx, const Plan& p, int nb_select, bool merged) {
  const int B = ctx->dc.block, mask = ctx->mc.mask_id;
  cudaStream_t s = ctx->stream;
  int r = enqueue_forward(ctx, p);
  if (r) return r;
  CK(launch_select(ctx->st, B, nb_select, mask, ctx->branch_tok, ctx->valid, ctx->am_b, ctx->mp_b, s));
  KvStrides kv;
  kv.k_cache = ctx->cache_layer;
  kv.k_scr = ctx->scr_layer;
  kv.v_cache = ctx->vt_cache_layer;
  kv.v_scr = ctx->scr_layer;
  kv.ld_cache = ctx->vt_ld;
  kv.ld_scr = ctx->nslots * B;
  CK(launch_commit_kv(ctx->st, ctx->ks, ctx->vs, ctx->kc, ctx->vc, ctx->mc.n_layers, B,
                      ctx->mc.n_kv_heads * ctx->mc.head_dim, kv, s));
  CK(launch_finalize(ctx->st, B, mask, ctx->out_tokens, merged ? ctx->am_b + B : nullptr,
                     merged ? ctx->mp_b + B : nullptr, s));
  CK(launch_decide(ctx->st, B, ctx->dc.k, ctx->dc.tau, mask, ctx->branch_tok, ctx->valid, s));
  return 0;
}

int step_fn(lopa_ctx* ctx) {
  return enqueue_iteration(ctx, ctx->step_plans[ctx->cur_nb], ctx->cur_nb, false);
}
int merged_fn(lopa_ctx* ctx) { return enqueue_iteration(ctx, ctx->merged_plan, 1, true); }

int capture(lopa_ctx* ctx, int (*fn)(lopa_ctx*), cudaGraphExec_t* exec) {
  cudaGraph_t g = nullptr;
  CK(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
  int r = fn(ctx);
  cudaError_t e = cudaStreamEndCapture(ctx->stream, &g);
  if (r) {
    if (g) cudaGraphDestroy(g);
    return r;
  }
  if (e != cudaSuccess) return fail(ctx, LOPA_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
  e = cudaGraphInstantiate(exec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess)
    return fail(ctx, LOPA_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  return 0;
}

int start_fn(lopa_ctx* ctx) {
  int r = enqueue_forward(ctx, ctx->start_plan);
  if (r) return r;
  CK(launch_decide(ctx->st, ctx->dc.block, ctx->dc.k, ctx->dc.tau, ctx->mc.mask_id, ctx->branch_tok,
                   ctx->valid, ctx->stream));
  return 0;
}

int check_device_error(lopa_ctx* ctx) {
  int e = 0;
  CK(cudaMemcpyAsync(&e, &ctx->st->err, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  if (e) return fail(ctx, LOPA_ERR_DEVICE_TIMEOUT, "device-side wait gave up (code %d)", e);
  return 0;
}

int validate(const lopa_model_config* c, const lopa_decode_config* d) {
  lopa_ctx* ctx = nullptr;
  if (!c || !d) return fail(ctx, LOPA_ERR_INVALID_ARG, "null config");
  if (c->n_layers < 1 || c->d_model < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->vocab < 2 ||
      c->ffn < 1 || c->max_seq < 1)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "model dimensions must be positive");
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128");
  if (c->n_heads % c->n_kv_heads) return fail(ctx, LOPA_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (c->d_model % 128 || c->ffn % 128 || ((c->n_heads + 2 * c->n_kv_heads) * c->head_dim) % 128 ||
      (c->n_heads * c->head_dim) % 64)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "d_model, ffn and q/k/v rows must be multiples of 128");
  if (c->d_model > 4096) return fail(ctx, LOPA_ERR_UNSUPPORTED, "d_model must be <= 4096");
  if (c->mask_id < 0 || c->mask_id >= c->vocab) return fail(ctx, LOPA_ERR_INVALID_ARG, "mask_id out of range");
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f) || !std::isfinite(c->logit_scale))
    return fail(ctx, LOPA_ERR_INVALID_ARG, "bad rms_eps / rope_base / logit_scale");
  if (d->block < 16 || d->block > LOPA_MAX_BLOCK || d->block % 16)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "block must be 16..%d and a multiple of 16", LOPA_MAX_BLOCK);
  if (d->k < 0 || d->k >= LOPA_MAX_BRANCHES) return fail(ctx, LOPA_ERR_INVALID_ARG, "k must be 0..%d", LOPA_MAX_BRANCHES - 1);
  if (d->max_prompt < 1 || d->max_prompt + d->block > c->max_seq)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "need 1 <= max_prompt and max_prompt + block <= max_seq");
  if (!std::isfinite(d->tau)) return fail(ctx, LOPA_ERR_INVALID_ARG, "tau must be finite");
  if (c->weight_format != LOPA_WEIGHTS_BF16 && c->weight_format != LOPA_WEIGHTS_E4M3)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "unknown weight_format %d", c->weight_format);
  return 0;
}

int init_impl(lopa_ctx* ctx, const lopa_weights* w) {
  const lopa_model_config& m = ctx->mc;
  const int L = m.n_layers, d = m.d_model, H = m.n_heads, Hk = m.n_kv_heads, dh = m.head_dim;
  const int F = m.ffn, V = m.vocab, B = ctx->dc.block;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev));
  int major = 0, minor = 0;
  CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  CK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (major != 10) return fail(ctx, LOPA_ERR_UNSUPPORTED, "needs an sm_10x GPU (found sm_%d%d)", major, minor);
  CK(gemm_set_smem_limits());
  CK(attention_set_smem_limits());
  ctx->w8 = m.weight_format == LOPA_WEIGHTS_E4M3;
  for (int c = 1; c <= kMaxClusterSplits; c *= 2)
    ctx->ccap[c] = gemm_cluster_capacity(GEMM_QKV, c, (size_t)gemm_max_smem(), ctx->w8);
  if (ctx->ccap[1] < 1) return fail(ctx, LOPA_ERR_UNSUPPORTED, "projection GEMM cannot be resident");
  if (!ctx->stream) {
    CK(cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking));
    ctx->own_stream = true;
  }
  // weights
  if (!aligned16(w->embed) || !aligned16(w->lm_head) || !aligned16(w->final_norm) || !w->attn_norm ||
      !w->wq || !w->wk || !w->wv || !w->wo || !w->mlp_norm || !w->wg || !w->wu || !w->wd)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
  ctx->embed = static_cast<const bf16*>(w->embed);
  ctx->final_norm = static_cast<const bf16*>(w->final_norm);
  for (int l = 0; l < L; ++l) {
    const void* ps[9] = {w->attn_norm[l], w->wq[l], w->wk[l], w->wv[l], w->wo[l],
                         w->mlp_norm[l],  w->wg[l], w->wu[l], w->wd[l]};
    for (const void* p : ps)
      if (!aligned16(p)) return fail(ctx, LOPA_ERR_INVALID_ARG, "layer %d weight pointer null or unaligned", l);
    ctx->attn_norm.push_back(static_cast<const bf16*>(w->attn_norm[l]));
    ctx->mlp_norm.push_back(static_cast<const bf16*>(w->mlp_norm[l]));
  }
  // buffers
  ctx->nbmax = ctx->dc.k + 1;
  ctx->nslots = std::max(ctx->nbmax, 2);
  ctx->Tmax = std::max(ctx->nslots * B, ctx->dc.max_prompt);
  ctx->qkv_rows = (H + 2 * Hk) * dh;
  ctx->cache_layer = (size_t)m.max_seq * Hk * dh;
  ctx->vt_ld = (m.max_seq + 63) / 64 * 64;
  ctx->vt_cache_layer = (size_t)Hk * dh * ctx->vt_ld;
  ctx->scr_layer = (size_t)ctx->nslots * B * Hk * dh;
  ctx->nvt = (V + 255) / 256;
  ctx->part_ld = ctx->nslots * B;
  ctx->part_floats = std::max(partial_floats(ctx, ctx->nslots * B),
                              std::max(partial_floats(ctx, B), partial_floats(ctx, ctx->dc.max_prompt)));
  const size_t T = ctx->Tmax;
  {
    // q/k/v exchange workspace: the largest any forward needs (1..nslots branch slots of one
    // block, or the prompt).
    auto need = [&](int T2) {
      int na, cs;
      qkv_tiling(ctx, ctx->qkv_rows, d, T2, &na, &cs);
      const int nbox = qkv_box(T2);
      const int gx = (ctx->qkv_rows + na * 128 - 1) / (na * 128);
      return qkv_exchange_floats(gx, cs, (T2 + nbox - 1) / nbox, nbox);
    };
    ctx->xws_floats = need(ctx->dc.max_prompt);
    for (int nb = 1; nb <= ctx->nslots; ++nb) ctx->xws_floats = std::max(ctx->xws_floats, need(nb * B));
  }
  int r;
  if ((r = dalloc(ctx, &ctx->kc, ctx->cache_layer * L)) || (r = dalloc(ctx, &ctx->vc, ctx->vt_cache_layer * L)) ||
      (r = dalloc(ctx, &ctx->ks, ctx->scr_layer * L)) || (r = dalloc(ctx, &ctx->vs, ctx->scr_layer * L)) ||
      (r = dalloc(ctx, &ctx->x, T * d)) || (r = dalloc(ctx, &ctx->n, T * d)) ||
      (r = dalloc(ctx, &ctx->part, ctx->part_floats)) || (r = dalloc(ctx, &ctx->q, T * H * dh)) ||
      (r = dalloc(ctx, &ctx->xws, ctx->xws_floats)) ||
      (r = dalloc(ctx, &ctx->attn, T * H * dh)) || (r = dalloc(ctx, &ctx->hm, T * F)) ||
      (r = dalloc(ctx, &ctx->pm, (size_t)ctx->nvt * ctx->part_ld)) ||
      (r = dalloc(ctx, &ctx->ps, (size_t)ctx->nvt * ctx->part_ld)) ||
      (r = dalloc(ctx, &ctx->pi, (size_t)ctx->nvt * ctx->part_ld)) ||
      (r = dalloc(ctx, &ctx->cos_t, (size_t)m.max_seq * dh / 2)) ||
      (r = dalloc(ctx, &ctx->sin_t, (size_t)m.max_seq * dh / 2)) ||
      (r = dalloc(ctx, &ctx->branch_tok, (size_t)ctx->nslots * B)) ||
      (r = dalloc(ctx, &ctx->valid, (size_t)LOPA_MAX_BRANCHES)) ||
      (r = dalloc(ctx, &ctx->am_b, (size_t)ctx->nslots * B)) ||
      (r = dalloc(ctx, &ctx->mp_b, (size_t)ctx->nslots * B)) ||
      (r = dalloc(ctx, &ctx->tok_rows, T)) || (r = dalloc(ctx, &ctx->out_tokens, (size_t)m.max_seq)) ||
      (r = dalloc(ctx, &ctx->st, 1)))
    return r;
  cudaStream_t s = ctx->stream;
  CK(cudaMemsetAsync(ctx->kc, 0, ctx->cache_layer * L * sizeof(bf16), s));
  CK(cudaMemsetAsync(ctx->vc, 0, ctx->vt_cache_layer * L * sizeof(bf16), s));
  CK(cudaMemsetAsync(ctx->ks, 0, ctx->scr_layer * L * sizeof(bf16), s));
  CK(cudaMemsetAsync(ctx->vs, 0, ctx->scr_layer * L * sizeof(bf16), s));
  CK(cudaMemsetAsync(ctx->st, 0, sizeof(DevState), s));
  CK(cudaMemsetAsync(ctx->out_tokens, 0, (size_t)m.max_seq * sizeof(int), s));
  CK(launch_rope_table(ctx->cos_t, ctx->sin_t, m.max_seq, dh, (double)m.rope_base, s));
  CK(launch_state_reset(ctx->st, 0, B, m.mask_id, s));
  // Owned tile-major copies of the projection weights and the LM head: every 16 KB
  // (32 KB for the LM head) tile the GEMMs stream becomes one contiguous HBM run; q, k and
  // v (and gate and up) are stacked into the one matrix their GEMM streams.
  // E4M3 weight stream: per-row scales, then the codes in the same tile-major layout
  // (rows past the end of the last tile have code 0 and scale 1).
  auto pack = [&](std::vector<const void*>& dst, std::vector<const float*>& dscale, PackSources src,
                  int K, int tile_rows) -> int {
    int rows = 0;
    for (int i = 0; i < PackSources::kMax; ++i) rows += src.rows[i];
    const size_t elems = packed_elems(rows, K, tile_rows);
    int rr;
    if (ctx->w8) {
      const int rows_pad = (int)(elems / K);
      uint8_t* p = nullptr;
      float* sp = nullptr;
      if ((rr = dalloc(ctx, &p, elems)) || (rr = dalloc(ctx, &sp, (size_t)rows_pad))) return rr;
      CK(launch_row_scales(src, K, sp, rows_pad, s));
      CK(launch_pack_e4m3(src, sp, p, K, tile_rows, false, rows_pad, s));
      dst.push_back(p);
      dscale.push_back(sp);
      return 0;
    }
    bf16* p = nullptr;
    if ((rr = dalloc(ctx, &p, elems))) return rr;
    CK(launch_pack_tiles(src, p, K, tile_rows, s));
    dst.push_back(p);
    return 0;
  };
  auto src = [](const void* a, int ra, const void* b = nullptr, int rb = 0, const void* c = nullptr,
                int rc = 0) {
    PackSources ps = {{static_cast<const bf16*>(a), static_cast<const bf16*>(b),
                       static_cast<const bf16*>(c)},
                      {ra, rb, rc}};
    return ps;
  };
  for (int l = 0; l < L; ++l) {
    if ((r = pack(ctx->wqkv, ctx->sqkv, src(w->wq[l], H * dh, w->wk[l], Hk * dh, w->wv[l], Hk * dh), d, 128)) ||
        (r = pack(ctx->wo, ctx->so, src(w->wo[l], d), H * dh, 128)) ||
        (r = pack(ctx->wgu, ctx->sgu, src(w->wg[l], F, w->wu[l], F), d, 128)) ||
        (r = pack(ctx->wd, ctx->sd, src(w->wd[l], d), F, 128)))
      return r;
  }
  {
    std::vector<const void*> lm;
    std::vector<const float*> slm;
    if ((r = pack(lm, slm, src(w->lm_head, V), d, 256))) return r;
    ctx->lm_head = lm[0];
    ctx->slm = ctx->w8 ? slm[0] : nullptr;
  }
  CK(cudaEventCreate(&ctx->ev0));
  CK(cudaEventCreate(&ctx->ev1));
  CK(cudaMallocHost(&ctx->h_res, sizeof(lopa_step_result)));
  CK(cudaMallocHost(&ctx->h_next, 2 * sizeof(int)));
  // plans and graphs
  ctx->step_plans.resize(ctx->nbmax + 1);
  for (int nb = 1; nb <= ctx->nbmax; ++nb)
    if ((r = build_plan(ctx, ctx->step_plans[nb], nb, B, 0, true, ctx->branch_tok, ctx->am_b, ctx->mp_b)))
      return r;
  if ((r = build_plan(ctx, ctx->merged_plan, 2, B, 0, true, ctx->branch_tok, ctx->am_b, ctx->mp_b,
                      /*causal=*/true)))
    return r;
  if ((r = build_plan(ctx, ctx->start_plan, 1, B, 0, true, ctx->st->tok, ctx->st->am, ctx->st->mp)))
    return r;
  CK(cudaStreamSynchronize(s));
  ctx->step_execs.assign(ctx->nbmax + 1, nullptr);
  for (int nb = 1; nb <= ctx->nbmax; ++nb) {
    ctx->cur_nb = nb;
    if ((r = capture(ctx, step_fn, &ctx->step_execs[nb]))) return r;
  }
  if ((r = capture(ctx, merged_fn, &ctx->merged_exec))) return r;
  if ((r = capture(ctx, start_fn, &ctx->start_exec))) return r;
  return 0;
}

void destroy(lopa_ctx* ctx) {
  if (!ctx) return;
  if (ctx->stream) cudaStreamSynchronize(ctx->stream);
  for (auto e : ctx->step_execs)
    if (e) cudaGraphExecDestroy(e);
  if (ctx->merged_exec) cudaGraphExecDestroy(ctx->merged_exec);
  for (auto e : ctx->fwd_exec)
    if (e) cudaGraphExecDestroy(e);
  if (ctx->start_exec) cudaGraphExecDestroy(ctx->start_exec);
  if (ctx->ev0) cudaEventDestroy(ctx->ev0);
  if (ctx->ev1) cudaEventDestroy(ctx->ev1);
  if (ctx->h_res) cudaFreeHost(ctx->h_res);
  if (ctx->h_next) cudaFreeHost(ctx->h_next);
  for (void* p : ctx->allocs) cudaFree(p);
  if (ctx->own_stream) cudaStreamDestroy(ctx->stream);
  delete ctx;
}

// Reads back the branch count and completion flag of the last decide (synchronises).
int read_next(lopa_ctx* ctx) {
  static_assert(offsetof(DevState, final_w) == offsetof(DevState, n_valid) + sizeof(int),
                "n_valid and final_w are adjacent");
  CK(cudaMemcpyAsync(ctx->h_next, &ctx->st->n_valid, 2 * sizeof(int), cudaMemcpyDeviceToHost,
                     ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  ctx->next_nv = ctx->h_next[0];
  ctx->next_final = ctx->h_next[1];
  if (ctx->next_nv < 1 || ctx->next_nv > ctx->nbmax || ctx->next_final < -1 || ctx->next_final > 1)
    return fail(ctx, LOPA_ERR_BAD_STATE, "decide produced %d branches (final %d)", ctx->next_nv,
                ctx->next_final);
  return 0;
}

// Runs one iteration (plus the block-start forward when the block has no logits yet).
// The branches were built by the decide at the end of the previous graph; the host picks
// the forward that evaluates them: only the valid branches (nb = 1 + lookaheads); or, when
// the iteration completes the block, only the completing branch - together with the next
// block's block-start rows (block-causal attention) when a next block fits.
int step_impl(lopa_ctx* ctx, lopa_step_result* out, bool allow_merge) {
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "lopa_step before lopa_prefill");
  const int B = ctx->dc.block;
  if (ctx->P + B > ctx->mc.max_seq)
    return fail(ctx, LOPA_ERR_BAD_STATE, "KV cache full: next block would end at %d > max_seq %d",
                ctx->P + B, ctx->mc.max_seq);
  int fwd = 0, r;
  if (ctx->block_fresh) {
    CK(cudaGraphLaunch(ctx->start_exec, ctx->stream));  // block-start forward + decide
    if ((r = read_next(ctx))) return r;
    fwd = 1;
  }
  const bool merge = ctx->next_final >= 0 && allow_merge && ctx->P + 2 * B <= ctx->mc.max_seq;
  cudaGraphExec_t g = merge ? ctx->merged_exec
                            : ctx->step_execs[ctx->next_final >= 0 ? 1 : ctx->next_nv];
  CK(cudaGraphLaunch(g, ctx->stream));
  CK(cudaMemcpyAsync(ctx->h_res, &ctx->st->res, sizeof(lopa_step_result), cudaMemcpyDeviceToHost,
                     ctx->stream));
  if ((r = read_next(ctx))) return r;
  lopa_step_result& res = *ctx->h_res;
  res.forwards = 1 + fwd;
  if (res.device_error)
    return fail(ctx, LOPA_ERR_DEVICE_TIMEOUT, "device-side wait gave up (code %d)", res.device_error);
  ctx->in_block = res.block_done == 0;
  if (res.block_done) {
    ctx->P += B;
    ctx->block_fresh = !merge;  // a merged iteration leaves the next block's logits ready
  } else {
    ctx->block_fresh = false;
  }
  if (out) *out = res;
  return 0;
}

}  // namespace

extern "C" {

int lopa_version(void) { return 200; }

#ifdef LOPA_TIMELINE
// Timeline builds only: every instrumented kernel launched from now on appends its per-CTA
// records to buf (device memory: a 16-byte header {count, capacity, 0, 0}, then capacity
// records of lopa::tl::Rec); NULL stops recording.
int lopa_timeline_set_buffer(void* buf) {
  unsigned* p = static_cast<unsigned*>(buf);
  cudaError_t e = timeline_set_buffer_gemm(p);
  if (e == cudaSuccess) e = timeline_set_buffer_attention(p);
  if (e == cudaSuccess) e = timeline_set_buffer_pointwise(p);
  if (e == cudaSuccess) e = timeline_set_buffer_decide(p);
  return e == cudaSuccess ? 0 : LOPA_ERR_CUDA;
}
#endif

const char* lopa_last_error(const lopa_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_init_error.c_str();
}

int lopa_init_model(const lopa_model_config* cfg, const lopa_weights* w, const lopa_decode_config* dcfg,
                    void* stream, lopa_ctx** out) {
  if (!out) return fail(nullptr, LOPA_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (!w) return fail(nullptr, LOPA_ERR_INVALID_ARG, "weights are null");
  int r = validate(cfg, dcfg);
  if (r) return r;
  lopa_ctx* ctx = new lopa_ctx();
  ctx->mc = *cfg;
  ctx->dc = *dcfg;
  ctx->stream = static_cast<cudaStream_t>(stream);
  r = init_impl(ctx, w);
  if (r) {
    g_init_error = ctx->err;
    destroy(ctx);
    return r;
  }
  *out = ctx;
  return 0;
}

void lopa_free(lopa_ctx* ctx) { destroy(ctx); }

int lopa_prefill(lopa_ctx* ctx, const int32_t* prompt, int n) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (!prompt || n < 1 || n > ctx->dc.max_prompt)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "prompt length %d outside [1, %d]", n, ctx->dc.max_prompt);
  for (int i = 0; i < n; ++i)
    if (prompt[i] < 0 || prompt[i] >= ctx->mc.vocab)
      return fail(ctx, LOPA_ERR_INVALID_ARG, "prompt token %d at %d out of range", prompt[i], i);
  cudaStream_t s = ctx->stream;
  CK(cudaMemcpyAsync(ctx->tok_rows, prompt, sizeof(int) * n, cudaMemcpyHostToDevice, s));
  CK(launch_state_reset(ctx->st, 0, ctx->dc.block, ctx->mc.mask_id, s));
  int r;
  if (ctx->prefill_plan.T != n) {
    ctx->prefill_plan = Plan();
    if ((r = build_plan(ctx, ctx->prefill_plan, 1, n, 1, false, ctx->tok_rows, nullptr, nullptr))) {
      ctx->prefill_plan = Plan();
      return r;
    }
  }
  if ((r = enqueue_forward(ctx, ctx->prefill_plan))) return r;
  CK(launch_state_reset(ctx->st, n, ctx->dc.block, ctx->mc.mask_id, s));
  if ((r = check_device_error(ctx))) return r;
  ctx->prefilled = true;
  ctx->block_fresh = true;
  ctx->in_block = false;
  ctx->P = ctx->P0 = n;
  return 0;
}

int lopa_step(lopa_ctx* ctx, lopa_step_result* out) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  return step_impl(ctx, out, /*allow_merge=*/true);
}

int lopa_decode(lopa_ctx* ctx, int gen_len, int32_t* out_tokens, lopa_stats* out) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "lopa_decode before lopa_prefill");
  const int B = ctx->dc.block;
  if (gen_len < 0 || gen_len % B) return fail(ctx, LOPA_ERR_INVALID_ARG, "gen_len must be a multiple of %d", B);
  if (ctx->in_block) return fail(ctx, LOPA_ERR_BAD_STATE, "a block is in progress; finish it with lopa_step");
  if (ctx->P + gen_len > ctx->mc.max_seq)
    return fail(ctx, LOPA_ERR_BAD_STATE, "decode would end at %d > max_seq %d", ctx->P + gen_len, ctx->mc.max_seq);
  const int start = ctx->P - ctx->P0;
  lopa_stats st{};
  CK(cudaEventRecord(ctx->ev0, ctx->stream));
  for (int b = 0; b < gen_len / B; ++b) {
    int iters = 0;
    // The last block of this decode does not start the block after it.
    const bool allow_merge = b + 1 < gen_len / B;
    while (true) {
      lopa_step_result r;
      int rc = step_impl(ctx, &r, allow_merge);
      if (rc) return rc;
      st.forwards += r.forwards;
      st.steps += 1;
      if (r.block_done) break;
      if (++iters > B) return fail(ctx, LOPA_ERR_BAD_STATE, "block did not finish within %d iterations", B);
    }
    st.blocks += 1;
    st.tokens += B;
  }
  CK(cudaEventRecord(ctx->ev1, ctx->stream));
  CK(cudaEventSynchronize(ctx->ev1));
  float ms = 0.f;
  CK(cudaEventElapsedTime(&ms, ctx->ev0, ctx->ev1));
  st.seconds = ms * 1e-3;
  if (out_tokens && gen_len > 0) {
    CK(cudaMemcpyAsync(out_tokens, ctx->out_tokens + start, sizeof(int) * gen_len,
                       cudaMemcpyDeviceToHost, ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
  }
  if (out) *out = st;
  return 0;
}

int lopa_rewind(lopa_ctx* ctx, int pos) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "rewind before lopa_prefill");
  const int B = ctx->dc.block;
  const int committed = ctx->P;
  if (pos < ctx->P0 || pos > committed || (pos - ctx->P0) % B)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "rewind position %d must be in [%d, %d] on a block boundary",
                pos, ctx->P0, committed);
  CK(launch_state_reset(ctx->st, pos, B, ctx->mc.mask_id, ctx->stream));
  // state_reset sets P0 = pos too; put the prompt length back.
  CK(cudaMemcpyAsync(&ctx->st->P0, &ctx->P0, sizeof(int), cudaMemcpyHostToDevice, ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  ctx->P = pos;
  ctx->block_fresh = true;
  ctx->in_block = false;
  return 0;
}

int lopa_time_gemm(lopa_ctx* ctx, int kind, int iters, float* avg_ms) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (kind < 0 || kind > 4 || iters < 1 || !avg_ms) return fail(ctx, LOPA_ERR_INVALID_ARG, "bad kind/iters");
  const Plan& p = ctx->step_plan();
  const int L = ctx->mc.n_layers;
  cudaStream_t s = ctx->stream;
  // The launches are captured into a graph (as in the decoding step), so host launch
  // cost does not enter the timing; layers are cycled so no weight stays in L2.
  cudaGraph_t g = nullptr;
  cudaGraphExec_t ge = nullptr;
  CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  cudaError_t ce = cudaSuccess;
  for (int i = 0; i < iters && ce == cudaSuccess; ++i) {
    const int l = i % L;
    const GemmLaunch& G = kind == 0 ? p.qkv[l] : kind == 1 ? p.o[l] : kind == 2 ? p.gu[l]
                        : kind == 3 ? p.dn[l] : p.lmh;
    ce = launch_gemm(G, s);
  }
  cudaError_t ee = cudaStreamEndCapture(s, &g);
  if (ce != cudaSuccess || ee != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return fail(ctx, LOPA_ERR_CUDA, "capture of timed GEMMs failed: %s",
                cudaGetErrorString(ce != cudaSuccess ? ce : ee));
  }
  ce = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (ce != cudaSuccess) return fail(ctx, LOPA_ERR_CUDA, "instantiate: %s", cudaGetErrorString(ce));
  float ms = 0.f;
  ce = cudaGraphLaunch(ge, s);  // warm-up
  if (ce == cudaSuccess) ce = cudaEventRecord(ctx->ev0, s);
  if (ce == cudaSuccess) ce = cudaGraphLaunch(ge, s);
  if (ce == cudaSuccess) ce = cudaEventRecord(ctx->ev1, s);
  if (ce == cudaSuccess) ce = cudaEventSynchronize(ctx->ev1);
  if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, ctx->ev0, ctx->ev1);
  cudaGraphExecDestroy(ge);
  if (ce != cudaSuccess) return fail(ctx, LOPA_ERR_CUDA, "timed GEMMs: %s", cudaGetErrorString(ce));
  *avg_ms = ms / iters;
  return check_device_error(ctx);
}

int lopa_time_forward(lopa_ctx* ctx, int kind, int iters, float* median_ms, float* mean_ms) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if ((kind != 0 && kind != 1) || iters < 1 || iters > 10000 || !median_ms)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "bad kind/iters");
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "time_forward before lopa_prefill");
  if (ctx->P + ctx->dc.block > ctx->mc.max_seq)
    return fail(ctx, LOPA_ERR_BAD_STATE, "no room for a block at prefix %d (max_seq %d)", ctx->P,
                ctx->mc.max_seq);
  cudaStream_t s = ctx->stream;
  if (!ctx->fwd_exec[kind]) {
    // Forward-only graphs.  The block-start one writes its logit summary to the branch
    // buffers (not the block state), so neither changes the decoding state.
    Plan& p = kind == 1 ? ctx->step_plan() : ctx->time_start_plan;
    int r;
    if (kind == 0 && (r = build_plan(ctx, p, 1, ctx->dc.block, 0, true, ctx->st->tok, ctx->am_b,
                                     ctx->mp_b)))
      return r;
    ctx->fwd_plan = &p;
    if ((r = capture(ctx, [](lopa_ctx* c) { return enqueue_forward(c, *c->fwd_plan); },
                     &ctx->fwd_exec[kind])))
      return r;
  }
  std::vector<cudaEvent_t> ev(iters + 1, nullptr);
  cudaError_t ce = cudaSuccess;
  for (auto& e : ev)
    if (ce == cudaSuccess) ce = cudaEventCreate(&e);
  if (ce == cudaSuccess) ce = cudaGraphLaunch(ctx->fwd_exec[kind], s);  // warm-up
  if (ce == cudaSuccess) ce = cudaEventRecord(ev[0], s);
  for (int i = 0; i < iters && ce == cudaSuccess; ++i) {
    ce = cudaGraphLaunch(ctx->fwd_exec[kind], s);
    if (ce == cudaSuccess) ce = cudaEventRecord(ev[i + 1], s);
  }
  if (ce == cudaSuccess) ce = cudaEventSynchronize(ev[iters]);
  std::vector<float> ms(iters, 0.f);
  for (int i = 0; i < iters && ce == cudaSuccess; ++i) ce = cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]);
  for (auto e : ev)
    if (e) cudaEventDestroy(e);
  if (ce != cudaSuccess) return fail(ctx, LOPA_ERR_CUDA, "timed forward: %s", cudaGetErrorString(ce));
  double sum = 0;
  for (float v : ms) sum += v;
  std::sort(ms.begin(), ms.end());
  *median_ms = ms[iters / 2];
  if (mean_ms) *mean_ms = (float)(sum / iters);
  return check_device_error(ctx);
}

int lopa_get_block_state(lopa_ctx* ctx, int32_t* tok, int32_t* am, float* mp, int* prefix_len) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  const int B = ctx->dc.block;
  cudaStream_t s = ctx->stream;
  if (tok) CK(cudaMemcpyAsync(tok, ctx->st->tok, sizeof(int) * B, cudaMemcpyDeviceToHost, s));
  if (am) CK(cudaMemcpyAsync(am, ctx->st->am, sizeof(int) * B, cudaMemcpyDeviceToHost, s));
  if (mp) CK(cudaMemcpyAsync(mp, ctx->st->mp, sizeof(float) * B, cudaMemcpyDeviceToHost, s));
  if (prefix_len) CK(cudaMemcpyAsync(prefix_len, &ctx->st->P, sizeof(int), cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  return 0;
}

int lopa_set_block_state(lopa_ctx* ctx, const int32_t* tok, const int32_t* am, const float* mp) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "set_block_state before lopa_prefill");
  if (!tok || !am || !mp) return fail(ctx, LOPA_ERR_INVALID_ARG, "null state array");
  const int B = ctx->dc.block;
  bool any_mask = false;
  for (int i = 0; i < B; ++i) {
    if (tok[i] < 0 || tok[i] >= ctx->mc.vocab || am[i] < 0 || am[i] >= ctx->mc.vocab)
      return fail(ctx, LOPA_ERR_INVALID_ARG, "token out of range at %d", i);
    any_mask |= tok[i] == ctx->mc.mask_id;
  }
  if (!any_mask) return fail(ctx, LOPA_ERR_INVALID_ARG, "state must have at least one [MASK]");
  if (ctx->P + B > ctx->mc.max_seq) return fail(ctx, LOPA_ERR_BAD_STATE, "KV cache full");
  cudaStream_t s = ctx->stream;
  CK(cudaMemcpyAsync(ctx->st->tok, tok, sizeof(int) * B, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(ctx->st->am, am, sizeof(int) * B, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(ctx->st->mp, mp, sizeof(float) * B, cudaMemcpyHostToDevice, s));
  CK(launch_decide(ctx->st, B, ctx->dc.k, ctx->dc.tau, ctx->mc.mask_id, ctx->branch_tok, ctx->valid, s));
  int r = read_next(ctx);
  if (r) return r;
  ctx->block_fresh = false;
  ctx->in_block = true;
  return 0;
}

int lopa_verify_forward(lopa_ctx* ctx, const int32_t* branch_tok, int nb, int32_t* am, float* mp,
                        float* hidden) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (!ctx->prefilled) return fail(ctx, LOPA_ERR_BAD_STATE, "verify_forward before lopa_prefill");
  if (!branch_tok || nb < 1 || nb > ctx->nbmax)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "nb must be 1..%d", ctx->nbmax);
  const int B = ctx->dc.block, T = nb * B, d = ctx->mc.d_model;
  if (ctx->P + B > ctx->mc.max_seq) return fail(ctx, LOPA_ERR_BAD_STATE, "KV cache full");
  for (int i = 0; i < T; ++i)
    if (branch_tok[i] < 0 || branch_tok[i] >= ctx->mc.vocab)
      return fail(ctx, LOPA_ERR_INVALID_ARG, "branch token out of range at %d", i);
  cudaStream_t s = ctx->stream;
  CK(cudaMemcpyAsync(ctx->tok_rows, branch_tok, sizeof(int) * T, cudaMemcpyHostToDevice, s));
  Plan p;
  int r = build_plan(ctx, p, nb, B, 0, true, ctx->tok_rows, ctx->am_b, ctx->mp_b);
  if (r) return r;
  if ((r = enqueue_forward(ctx, p))) return r;
  if (am) CK(cudaMemcpyAsync(am, ctx->am_b, sizeof(int) * T, cudaMemcpyDeviceToHost, s));
  if (mp) CK(cudaMemcpyAsync(mp, ctx->mp_b, sizeof(float) * T, cudaMemcpyDeviceToHost, s));
  if (hidden) CK(cudaMemcpyAsync(hidden, ctx->x, sizeof(float) * T * d, cudaMemcpyDeviceToHost, s));
  return check_device_error(ctx);
}

int lopa_read_kv(lopa_ctx* ctx, int layer, int pos0, int n, uint16_t* k, uint16_t* v) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (layer < 0 || layer >= ctx->mc.n_layers || pos0 < 0 || n < 0 || pos0 + n > ctx->mc.max_seq)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "layer/position range out of bounds");
  const size_t row = (size_t)ctx->mc.n_kv_heads * ctx->mc.head_dim;
  cudaStream_t s = ctx->stream;
  if (k && n > 0)
    CK(cudaMemcpyAsync(k, ctx->kc + (size_t)layer * ctx->cache_layer + (size_t)pos0 * row,
                       n * row * 2, cudaMemcpyDeviceToHost, s));
  std::vector<uint16_t> vt(v && n > 0 ? row * n : 0);
  if (!vt.empty())
    CK(cudaMemcpy2DAsync(vt.data(), (size_t)n * 2,
                         ctx->vc + (size_t)layer * ctx->vt_cache_layer + pos0,
                         (size_t)ctx->vt_ld * 2, (size_t)n * 2, row, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  for (size_t r = 0; r < vt.size() / (n > 0 ? n : 1) && !vt.empty(); ++r)
    for (int c = 0; c < n; ++c) v[(size_t)c * row + r] = vt[r * n + c];
  return 0;
}

int lopa_debug_set_device_error(lopa_ctx* ctx, int code) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  CK(cudaMemcpyAsync(&ctx->st->err, &code, sizeof(int), cudaMemcpyHostToDevice, ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  return 0;
}

int lopa_read_branch_kv(lopa_ctx* ctx, int layer, int branch, uint16_t* k, uint16_t* v) {
  if (!ctx) return fail(nullptr, LOPA_ERR_INVALID_ARG, "ctx is null");
  if (layer < 0 || layer >= ctx->mc.n_layers || branch < 0 || branch >= ctx->nbmax)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "layer/branch out of range");
  const size_t row = (size_t)ctx->mc.n_kv_heads * ctx->mc.head_dim;
  const int B = ctx->dc.block;
  const size_t off = (size_t)layer * ctx->scr_layer;
  cudaStream_t s = ctx->stream;
  if (k) CK(cudaMemcpyAsync(k, ctx->ks + off + (size_t)branch * B * row, B * row * 2,
                            cudaMemcpyDeviceToHost, s));
  std::vector<uint16_t> vt(v ? row * B : 0);
  if (v)
    CK(cudaMemcpy2DAsync(vt.data(), (size_t)B * 2, ctx->vs + off + (size_t)branch * B,
                         (size_t)ctx->nslots * B * 2, (size_t)B * 2, row, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (v)
    for (size_t r = 0; r < row; ++r)
      for (int c = 0; c < B; ++c) v[(size_t)c * row + r] = vt[r * B + c];
  return 0;
}

// ---------------------------------------------------------------- kernel-level calls

int lopa_linear_accumulate(const void* x, const void* w, float* y, int T, int N, int K, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(x) || !aligned16(w) || !y) return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (T < 1 || N < 128 || N % 128 || K < 64 || K % 64)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "need T >= 1, N % 128 == 0, K % 64 == 0");
  CK(gemm_set_smem_limits());
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int tok_box = std::min(256, round16(T));
  const int na = N >= 256 ? 2 : 1;
  const int tiles = ((N + na * 128 - 1) / (na * 128)) * ((T + tok_box - 1) / tok_box);
  GemmLaunch G;
  const char* e = plan_gemm(&G, GEMM_RED_ADD, x, T, T, w, N, K, na, pick_splits(tiles, K / 64, sms),
                            tok_box, sms);
  if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", e);
  G.args.out_f32 = y;
  G.args.ldo = N;
  G.args.atomic = 1;
  cudaError_t se = cudaSuccess;
  G.args.err = call_status_word(&se);
  CK(se);
  G.args.wait_ns = call_wait_limit_ns();
  CK(launch_gemm(G, static_cast<cudaStream_t>(stream)));
  return 0;
}

int lopa_swiglu(const void* x, const void* w, void* h, int T, int F, int K, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(x) || !aligned16(w) || !aligned16(h))
    return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (T < 1 || F < 128 || F % 128 || K < 64 || K % 64)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "need T >= 1, F % 128 == 0, K % 64 == 0");
  CK(gemm_set_smem_limits());
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  GemmLaunch G;
  const char* e = plan_gemm(&G, GEMM_SWIGLU, x, T, T, w, 2 * F, K, 2, 1, std::min(256, round16(T)), sms);
  if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", e);
  G.args.out_bf16 = static_cast<bf16*>(h);
  G.args.ldh = F;
  cudaError_t se = cudaSuccess;
  G.args.err = call_status_word(&se);
  CK(se);
  G.args.wait_ns = call_wait_limit_ns();
  CK(launch_gemm(G, static_cast<cudaStream_t>(stream)));
  return 0;
}

int lopa_quantize_e4m3(const void* w, int rows, int K, uint8_t* codes, float* scales, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(w) || !aligned16(codes) || !scales) return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (rows < 1 || K < 64 || K % 64) return fail(ctx, LOPA_ERR_INVALID_ARG, "need rows >= 1 and K % 64 == 0");
  PackSources src = {{static_cast<const bf16*>(w), nullptr, nullptr}, {rows, 0, 0}};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(launch_row_scales(src, K, scales, rows, s));
  CK(launch_pack_e4m3(src, scales, codes, K, 128, true, rows, s));
  return 0;
}

int lopa_linear_accumulate_e4m3(const void* x, const uint8_t* codes, const float* scales, float* y,
                                int T, int N, int K, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(x) || !aligned16(codes) || !scales || !y)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (T < 1 || N < 128 || N % 128 || K < 64 || K % 64)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "need T >= 1, N % 128 == 0, K % 64 == 0");
  CK(gemm_set_smem_limits());
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int tok_box = std::min(256, round16(T));
  const int na = N >= 256 ? 2 : 1;
  const int tiles = ((N + na * 128 - 1) / (na * 128)) * ((T + tok_box - 1) / tok_box);
  GemmLaunch G;
  const char* e = plan_gemm(&G, GEMM_RED_ADD, x, T, T, codes, N, K, na, pick_splits(tiles, K / 64, sms),
                            tok_box, sms, false, scales);
  if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", e);
  G.args.out_f32 = y;
  G.args.ldo = N;
  G.args.atomic = 1;
  cudaError_t se = cudaSuccess;
  G.args.err = call_status_word(&se);
  CK(se);
  G.args.wait_ns = call_wait_limit_ns();
  CK(launch_gemm(G, static_cast<cudaStream_t>(stream)));
  return 0;
}

size_t lopa_lmhead_workspace_bytes(int rows, int vocab) {
  if (rows < 1 || vocab < 1) return 0;
  return (size_t)((vocab + 255) / 256) * rows * 12 + 256;
}

int lopa_lmhead_argmax(const void* hidden, const void* lm_head, int rows, int d_model, int vocab,
                       float logit_scale, int mask_id, void* workspace, size_t workspace_bytes,
                       int32_t* argmax_out, float* maxp_out, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(hidden) || !aligned16(lm_head) || !aligned16(workspace) || !argmax_out || !maxp_out)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (rows < 1 || vocab < 2 || d_model < 64 || d_model % 64 || mask_id < 0 || mask_id >= vocab)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "bad shape");
  if (workspace_bytes < lopa_lmhead_workspace_bytes(rows, vocab))
    return fail(ctx, LOPA_ERR_INVALID_ARG, "workspace too small");
  CK(gemm_set_smem_limits());
  const int nvt = (vocab + 255) / 256;
  float* pm = static_cast<float*>(workspace);
  float* ps = pm + (size_t)nvt * rows;
  int* pi = reinterpret_cast<int*>(ps + (size_t)nvt * rows);
  GemmLaunch G;
  const char* e = plan_gemm(&G, GEMM_LMSTATS, hidden, rows, rows, lm_head, vocab, d_model,
                            rows > 128 ? 2 : 1, 1, 0, 0);
  if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", e);
  GemmArgs& a = G.args;
  a.V = vocab;
  a.mask_id = mask_id;
  a.scale = logit_scale;
  a.part_m = pm;
  a.part_s = ps;
  a.part_i = pi;
  a.part_ld = rows;
  cudaError_t se = cudaSuccess;
  a.err = call_status_word(&se);
  CK(se);
  a.wait_ns = call_wait_limit_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(launch_gemm(G, s));
  CK(launch_lm_merge(pm, ps, pi, nvt, rows, rows, argmax_out, maxp_out, s));
  return 0;
}

int lopa_branch_attention(const void* q, const void* k_prefix, const void* vt_prefix,
                          int prefix_len, int ld_vt_prefix, const void* k_block,
                          const void* vt_block, int n_branches, int block, int n_heads,
                          int n_kv_heads, int head_dim, void* out, void* stream) {
  lopa_ctx* ctx = nullptr;
  if (!aligned16(q) || !aligned16(k_block) || !aligned16(vt_block) || !aligned16(out))
    return fail(ctx, LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (prefix_len < 0 || (prefix_len > 0 && (!aligned16(k_prefix) || !aligned16(vt_prefix) ||
                                            ld_vt_prefix < prefix_len || ld_vt_prefix % 8)))
    return fail(ctx, LOPA_ERR_INVALID_ARG, "bad prefix (ld_vt_prefix must be >= prefix_len and a multiple of 8)");
  if (n_branches < 1 || block < 16 || block > 4096 || block % 16 || n_heads < 1 ||
      n_kv_heads < 1 || n_heads % n_kv_heads)
    return fail(ctx, LOPA_ERR_INVALID_ARG, "bad shape");
  if (head_dim != 32 && head_dim != 64 && head_dim != 128)
    return fail(ctx, LOPA_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128");
  AttnArgs a = {};
  a.q = static_cast<const bf16*>(q);
  a.out = static_cast<bf16*>(out);
  a.kc = static_cast<const bf16*>(k_prefix);
  a.vtc = static_cast<const bf16*>(vt_prefix);
  a.kb = static_cast<const bf16*>(k_block);
  a.vtb = static_cast<const bf16*>(vt_block);
  a.dP = nullptr;
  a.pk_add = prefix_len;
  a.ldvc = prefix_len > 0 ? ld_vt_prefix : 8;
  a.ldvb = n_branches * block;
  a.Bq = block;
  a.Bk = block;
  a.Bk_stride = block;
  a.nbq = n_branches;
  a.H = n_heads;
  a.Hk = n_kv_heads;
  cudaError_t se = cudaSuccess;
  a.err = call_status_word(&se);
  CK(se);
  a.wait_ns = call_wait_limit_ns();
  AttnLaunch L;
  const char* e = plan_attention(&L, a, head_dim, prefix_len, prefix_len);
  if (e[0]) return fail(ctx, LOPA_ERR_UNSUPPORTED, "%s", e);
  CK(attention_set_smem_limits());
  CK(launch_attention(L, static_cast<cudaStream_t>(stream)));
  return 0;
}

}  // extern "C"
