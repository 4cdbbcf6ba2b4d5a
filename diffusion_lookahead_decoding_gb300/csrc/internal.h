// Host-side interfaces between the translation units of the LoPA library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lopa.h"

namespace lopa {

typedef __nv_bfloat16 bf16;

// Sets the message lopa_last_error(NULL) returns (failures of context-free calls).
void set_global_error(const char* msg);

#ifdef LOPA_TIMELINE
cudaError_t timeline_set_buffer_gemm(unsigned* p);
cudaError_t timeline_set_buffer_attention(unsigned* p);
cudaError_t timeline_set_buffer_pointwise(unsigned* p);
cudaError_t timeline_set_buffer_decide(unsigned* p);
#endif

// ------------------------------------------------------------------ file-scope device words
constexpr int kMaxDevices = 64;
// Per-device cache of a file-scope __device__ variable's address, keyed by the context.
struct SymbolCache {
  unsigned long long ctx_id[kMaxDevices] = {};
  void* addr[kMaxDevices] = {};
};
// Identifier of the current CUDA context (0 if unknown).
unsigned long long current_context_id();
// Device address of `sym` in the current context (looked up again when the context changes).
cudaError_t symbol_address(const void* sym, SymbolCache& cache, void** out);
// Error word of the kernel-level entry points on the current device.
int* call_status_word(cudaError_t* e);
// Wait limit of the kernel-level entry points (0 = the default), see lopa_set_wait_limit_ns.
unsigned long long call_wait_limit_ns();
// Reads (asynchronously, into *code) and clears the error word of lopa_lmhead_argmax_static.
cudaError_t lmhead_static_take_status(cudaStream_t s, int* code);

// Launches `kern` with programmatic stream serialization (the kernels call pdl_wait
// before reading their predecessor's outputs) and, when cluster.x > 0, as thread-block
// clusters of `cluster` CTAs.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster.x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  return launch_pdl_cluster(kern, grid, block, smem, s, dim3(0, 0, 0), args...);
}

// ------------------------------------------------------------------ GEMM (tcgen05)
enum GemmMode : int {
  GEMM_RED_ADD = 0,  // out_f32[t][n] += sum_k act[t][k] * w[n][k]   (weights on M, tokens on N)
  GEMM_SWIGLU = 1,   // out_bf16[t][f] = silu(gate) * up             (weights on M, tokens on N)
  GEMM_LMSTATS = 2,  // per (vocab tile, token): max, sum exp, argmax  (tokens on M, vocab on N)
  GEMM_QKV = 3,      // q/k/v projection + RoPE + bf16 Pre-Write; split-K summed in a cluster
};

// Modes whose K-splits form one thread-block cluster and are summed through distributed
// shared memory; such a cluster has 1, 2 or 4 CTAs.
inline bool gemm_mode_clustered(int mode) { return mode == GEMM_QKV; }
constexpr int kMaxClusterSplits = 4;
// Floats of the QKV exchange workspace a launch with grid (gx, splits, gz) and token box
// nbox needs: per (tile, token block) two rounds x splits regions of nbox x 128 floats.
inline size_t qkv_exchange_floats(int gx, int splits, int gz, int nbox) {
  return (size_t)gx * gz * 2 * splits * nbox * 128;
}

struct GemmArgs {
  int mode;
  int na;            // A tiles (128 rows each) per CTA: 1 or 2
  int nbox;          // rows of the B tile = MMA N (16..256, multiple of 16)
  int a_rows;        // rows of the A tensor (tiles at or beyond are skipped)
  int k_blocks;      // K / 64
  int splits;        // split-K factor (grid.y); the cluster size in the clustered modes
  int w_stages, x_stages;  // depth of the weight and activation smem rings
  uint32_t a_tile_bytes, w_slot_bytes, x_slot_bytes;
  int T;             // valid token rows
  int F;             // SWIGLU: row offset of the up half in [2F][K]
  int V, mask_id;    // LMSTATS
  float scale;       // LMSTATS logit scale
  float* out_f32;    int ldo;
  int atomic;        // RED_ADD: 1 = atomicAdd into out_f32, 0 = store partial of split y
  size_t split_stride;  // RED_ADD partials: elements between splits
  bf16* out_bf16;    int ldh;
  float* part_m; float* part_s; int* part_i; int part_ld;
  // QKV: A rows are [H q heads | Hk k heads | Hk v heads] x dh.  Token row t is position
  // t % Bq of its branch, at absolute position *dP + t % Bq.  q -> group-major
  // [Hk][T][H/Hk][dh]; k -> kdst [row][Hk][dh]; v -> transposed vdst [Hk*dh][ldv] at
  // column row; row = t, or with kv_to_cache the cache position *dP + t % Bq.
  bf16* q; bf16* kdst; bf16* vdst; int ldv;
  const float* cos_t; const float* sin_t;  // [positions][dh/2]
  const int* dP;
  int H, Hk, dh, Bq, kv_to_cache;
  int pos_linear;    // QKV: token row t sits at position *dP + t (consecutive blocks), not
                     // *dP + t % Bq (parallel branches of one block)
  float* xws;        // QKV: split-K exchange workspace (see qkv_exchange_floats)
  int* err;
  int w_packed;      // weight operand in tile-major layout (see launch_pack_tiles)
  int w8;            // weights are E4M3 codes with one float32 scale per weight row
  const float* wscale;  // E4M3: scale per weight row ([a_rows]; LM head: padded to 256 rows)
  int f_stages;      // E4M3: depth of the staging ring of codes
  uint32_t f_slot_bytes;
  int zt;            // token boxes (LM head: token groups); grid.x = tiles x zt with the box
                     // index fastest, so the CTAs sharing a weight tile run side by side
  unsigned long long wait_ns;  // limit of every device-side wait (0 = the 2 s default)
};

struct GemmLaunch {
  CUtensorMap mapA, mapB;
  GemmArgs args;
  dim3 grid;
  size_t smem;
};

// Encodes a 2-D bf16 tensor map over a row-major [rows][cols] matrix (row pitch ld
// elements, 0 = cols) with a box of box_rows x 64 columns and 128-byte swizzle; reads
// outside [rows][cols] return zeros.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, char* errbuf, size_t errlen, uint64_t ld = 0);

// Fills `L` for one GEMM.  Returns an empty string on success, else a reason.  With
// w_packed the weight is in the tile-major layout written by launch_pack_tiles (tiles of
// 128 rows, 256 for the LM head); otherwise it is row-major [n_rows_w][K].  With w_scale
// the weight holds E4M3 codes (one byte per element, same layouts) and w_scale one float32
// scale per weight row.
const char* plan_gemm(GemmLaunch* L, int mode, const void* act, int act_rows_alloc, int T,
                      const void* w, int n_rows_w, int K, int na, int splits, int tok_box,
                      int num_sms, bool w_packed = false, const float* w_scale = nullptr);

// Tile-major weight packing: up to three row-major [rows_i][K] matrices, stacked by rows,
// -> [ceil(rows/tile_rows)][K/64][tile_rows][64] (rows = the sum of rows_i).
struct PackSources {
  static constexpr int kMax = 3;
  const bf16* ptr[kMax];
  int rows[kMax];  // 0 for unused entries
};
size_t packed_elems(int rows, int K, int tile_rows);
cudaError_t launch_pack_tiles(const PackSources& src, bf16* dst, int K, int tile_rows,
                              cudaStream_t s);
// E4M3 weight stream: scale[r] = max|row r| / 448 (float32; 1 for a zero row) for rows
// [0, rows_out) of the stacked sources (rows past their end are zero), and the codes
// E4M3(w / scale) packed tile-major ([tiles][K/64][tile_rows][64] bytes) or row-major
// ([rows_out][K] bytes).
cudaError_t launch_row_scales(const PackSources& src, int K, float* scale, int rows_out,
                              cudaStream_t s);
cudaError_t launch_pack_e4m3(const PackSources& src, const float* scale, uint8_t* dst, int K,
                             int tile_rows, bool row_major, int rows_out, cudaStream_t s);
// Gives every kernel of the library the same (maximal) shared-memory carveout, so that
// consecutive kernels never make an SM change its L1/shared split.
cudaError_t set_uniform_carveout();
cudaError_t gemm_set_carveout();
cudaError_t attention_set_carveout();
cudaError_t pointwise_set_carveout();
cudaError_t decide_set_carveout();
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t s);
cudaError_t gemm_set_smem_limits();
// Clusters of `cs` GEMM CTAs (with `smem` bytes of dynamic shared memory each) that can
// be resident at once; 0 if such clusters cannot be launched.
int gemm_cluster_capacity(int mode, int cs, size_t smem, bool w8 = false);
int gemm_max_smem();

// ------------------------------------------------------------------ attention
// Layouts: q [Hk][nbq*Bq][G][dh] (group-major rows), out [nbq*Bq][H*dh], keys row-major
// [pos][Hk][dh], values transposed [Hk*dh][positions].
struct AttnArgs {
  const bf16* q;
  bf16* out;
  const bf16* kc;      // prefix keys   [*][Hk][dh]
  const bf16* vtc;     // prefix values [Hk*dh][ldvc]
  const bf16* kb;      // block keys    [nbq][Bk_stride][Hk][dh]
  const bf16* vtb;     // block values  [Hk*dh][nbq*Bk_stride]
  const int* dP;       // device prefix length (may be null -> 0)
  int pk_add;          // prefix keys = *dP + pk_add
  int ldvc, ldvb;      // row lengths of vtc and vtb (multiples of 8)
  int causal;          // 0: branch b sees its own block keys; 1: blocks 0..b (consecutive
                       // blocks of one sequence, e.g. a finished block and the next one)
  int Bq, Bk, Bk_stride, nbq, H, Hk;
  int* err;            // device error word (bounded waits), may be null
  unsigned long long wait_ns;  // limit of every device-side wait (0 = the 2 s default)
};
struct AttnLaunch {
  CUtensorMap maps[5];  // head_dim 128: q, prefix K, prefix V^T, block K, block V^T
  AttnArgs args;
  int dh;
  dim3 grid;
};
// Fills `L` (tensor maps over kc with kc_rows positions and vtc with vtc_cols positions;
// reads beyond are zeros).  Returns an empty string on success, else a reason.
const char* plan_attention(AttnLaunch* L, const AttnArgs& a, int dh, int kc_rows, int vtc_cols);
cudaError_t launch_attention(const AttnLaunch& L, cudaStream_t s);
cudaError_t attention_set_smem_limits();

// ------------------------------------------------------------------ pointwise
// Token ids outside [0, V) (possible only after a device-side wait gave up and left garbage
// in the state) read row 0 and record DEV_BAD_INDEX in *err.
cudaError_t launch_embed_norm(const int* tok, int T, const bf16* E, const bf16* g, float* x,
                              bf16* n, int d, float eps, int V, int* err, cudaStream_t s);
// x[t] += sum over splits of part[s][t] (split order); n[t] = bf16(rmsnorm(x[t]) * g).
cudaError_t launch_residual_norm(float* x, const float* part, int nsplit, size_t split_stride,
                                 const bf16* g, bf16* n, int T, int d, float eps, cudaStream_t s);
cudaError_t launch_lm_merge(const float* pm, const float* ps, const int* pi, int nvt,
                            int part_ld, int T, int* am, float* mp, cudaStream_t s);
cudaError_t launch_rope_table(float* cos_t, float* sin_t, int S, int dh, double base,
                              cudaStream_t s);

// ------------------------------------------------------------------ decision / commit
// Decoding state kept in device memory so that one captured graph serves every
// iteration and every block position.
struct DevState {
  int P;            // committed prefix length = absolute position of the current block
  int P0;           // prompt length
  int winner;       // winner of the last iteration
  int block_done;   // 1 when the last iteration completed the block
  int err;          // device error word (DeviceError)
  int n_valid;      // 1 + number of lookahead branches built by the last decide
  int final_w;      // the last decide's iteration completes the block with this branch
                    // (its tokens in slot 0, a blank block in slot 1), else -1
  int pad;
  int tok[LOPA_MAX_BLOCK];   // current block tokens ([MASK] where unfilled)
  int am[LOPA_MAX_BLOCK];    // greedy token of the logits that produced `tok`
  float mp[LOPA_MAX_BLOCK];  // its probability
  int cand[LOPA_MAX_BRANCHES];  // lookahead candidate of branch b+1 (-1 if none)
  lopa_step_result res;
};

// branch_tok holds max(k + 1, 2) blocks of B tokens: a completing iteration writes its
// winner to block 0 and a blank block to block 1 whatever k is.
cudaError_t launch_decide(void* st, int B, int k, float tau, int mask_id, int* branch_tok,
                          int* valid, cudaStream_t s);
cudaError_t launch_select(void* st, int B, int nb, int mask_id, const int* branch_tok,
                          const int* valid, const int* am_b, const float* mp_b,
                          cudaStream_t s);
// Per-layer strides (elements) of the K cache / scratch ([pos][Hk*dh] rows) and of the
// transposed V cache / scratch ([Hk*dh][ld] rows), and the V^T row lengths.
struct KvStrides {
  size_t k_cache, k_scr, v_cache, v_scr;
  int ld_cache, ld_scr;
};
cudaError_t launch_commit_kv(const void* st, const bf16* ks, const bf16* vts, bf16* kc,
                             bf16* vtc, int L, int B, int row_elems, const KvStrides& kv,
                             cudaStream_t s);
cudaError_t launch_finalize(void* st, int B, int mask_id, int* out_tokens, const int* am_next,
                            const float* mp_next, cudaStream_t s);
cudaError_t launch_state_reset(void* st, int P, int B, int mask_id, cudaStream_t s);

}  // namespace lopa
