/*
 * lopa.h - C ABI of the GB300 (sm_103a) LoPA branch-verification library.
 *
 * LoPA (Lookahead Parallel Decoding, arXiv 2512.16229) decodes a diffusion LM block by
 * block.  In every iteration it keeps the anchor branch (standard confidence-driven
 * greedy fill), adds k lookahead branches (each fills one more of the k most confident
 * masked positions), verifies all 1+k branches in ONE forward pass with attention
 * isolated per branch, scores each branch by the mean max-probability of its remaining
 * masked positions, keeps the winner and reuses the winner's logits for the next fill.
 * Sources: "SJTU x Huawei Xiaoyi release LoPA: 7B diffusion LM, 1000+ tokens/s single
 * sample" - sections "Core design of LoPA" (the iteration) and "LoPA-Dist" (static KV
 * cache with the two-phase Pre-Write / Commit-Winner-Cache update).
 *
 * Conventions for every call:
 *   - Return 0 (LOPA_OK) on success or a negative LOPA_ERR_* code, with a message in
 *     lopa_last_error().  Argument and state errors (INVALID_ARG, BAD_STATE,
 *     UNSUPPORTED) are detected before any work is enqueued and leave the decoding state
 *     as it was.  A device timeout (or a non-sticky CUDA error) in the middle of an
 *     iteration or a decode can leave the block state and the cache beyond the committed
 *     prefix partly updated: lopa_rewind (or lopa_prefill) brings the context back to a
 *     block boundary.  A sticky CUDA error (a device fault) leaves the CUDA context, and
 *     with it the lopa_ctx, unusable.  No call aborts the process or traps the device:
 *     device-side waits are bounded and report LOPA_ERR_DEVICE_TIMEOUT.
 *   - "device" pointers are CUDA global-memory pointers on the current device;
 *     "host" pointers are ordinary CPU memory.  bf16 = IEEE bfloat16 stored as
 *     16-bit words.  All matrices are row-major.
 *   - Work is enqueued on the caller's CUDA stream (a cudaStream_t passed as void*;
 *     NULL = legacy default stream).  Calls that return results to host memory
 *     synchronize that stream before returning.
 *   - A lopa_ctx is not thread-safe; use one per thread or serialize calls.
 */
#ifndef LOPA_H
#define LOPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LOPA_MAX_BRANCHES 16 /* 1 anchor + up to 15 lookahead branches */
#define LOPA_MAX_BLOCK 64    /* block length B */

enum {
  LOPA_OK = 0,
  LOPA_ERR_INVALID_ARG = -1,    /* bad pointer, size, shape or config */
  LOPA_ERR_BAD_STATE = -2,      /* call out of order (e.g. step before prefill) or cache full */
  LOPA_ERR_CUDA = -3,           /* a CUDA runtime call failed */
  LOPA_ERR_OOM = -4,            /* device allocation failed */
  LOPA_ERR_DEVICE_TIMEOUT = -5, /* a bounded device-side wait gave up */
  LOPA_ERR_UNSUPPORTED = -6     /* shape outside what the kernels implement */
};

typedef struct lopa_ctx lopa_ctx; /* opaque; owned by the library */

/* Decoder-only transformer of the Qwen2.5 family (pre-norm RMSNorm, RoPE with the
 * rotate-half convention, grouped-query attention, SwiGLU MLP, untied LM head).
 * Kernel limits: head_dim in {32, 64, 128}; d_model, n_heads*head_dim and ffn
 * multiples of 64; (n_heads + 2*n_kv_heads)*head_dim, d_model and ffn multiples of
 * 128; d_model <= 4096; n_heads a multiple of n_kv_heads. */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int mask_id;       /* token id of [MASK]; it is never predicted */
  int max_seq;       /* capacity of the static KV cache in tokens (prompt + output) */
  float rope_base;   /* RoPE theta base */
  float rms_eps;     /* RMSNorm epsilon */
  float logit_scale; /* logits = logit_scale * (final_hidden . lm_head_row) */
  int weight_format; /* LOPA_WEIGHTS_BF16 (0) or LOPA_WEIGHTS_E4M3 (1), see below */
} lopa_model_config;

/* Format of the weights the GEMMs stream (lopa_model_config.weight_format).  The caller
 * always passes bf16 matrices; with LOPA_WEIGHTS_E4M3, lopa_init_model quantises every
 * projection matrix and the LM head on the GPU, per output row r: scale s_r = max|W_r| /
 * 448 and codes E4M3(W_r / s_r) (the 8-bit float with 4 exponent bits, bias 7, and 3
 * fraction bits; round to nearest even, saturating at +-448; both quotients in float32;
 * an all-zero row gets s_r = 1), and the forward uses codes * s_r as the weight: half the
 * weight bytes per forward.  Activations, the embedding table and the norm gains stay
 * bf16, the arithmetic bf16 x bf16 -> fp32.  ("Decoding-efficiency revolution" blog,
 * section 4.1 and the LoPA announcement's "LoPA-Dist" section name quantisation as part of
 * the system without fixing a format; this per-channel E4M3 weight stream is this
 * library's reading.) */
#define LOPA_WEIGHTS_BF16 0
#define LOPA_WEIGHTS_E4M3 1

/* Device pointers (bf16), every matrix in the nn.Linear layout [out_features][in_features],
 * row-major, 16-byte aligned.  Per-layer entries are HOST arrays of n_layers device
 * pointers; the arrays themselves are copied at init and need not outlive the call.
 * lopa_init_model copies the projection matrices and lm_head into context-owned tile-major
 * copies (the layout the GEMMs stream; q, k and v are stacked into one matrix, gate and up
 * into another) - bf16, or E4M3 codes plus per-row scales with LOPA_WEIGHTS_E4M3; the
 * embedding and the norm gains stay borrowed and must outlive the context.  The caller may
 * free the projection matrices and lm_head after init. */
typedef struct {
  const void* embed;              /* [vocab][d_model] */
  const void* lm_head;            /* [vocab][d_model] */
  const void* final_norm;         /* [d_model] */
  const void* const* attn_norm;   /* [L] -> [d_model] */
  const void* const* wq;          /* [L] -> [H*dh][d_model], rows head-major */
  const void* const* wk;          /* [L] -> [Hk*dh][d_model] */
  const void* const* wv;          /* [L] -> [Hk*dh][d_model] */
  const void* const* wo;          /* [L] -> [d_model][H*dh] */
  const void* const* mlp_norm;    /* [L] -> [d_model] */
  const void* const* wg;          /* [L] -> [ffn][d_model] (gate) */
  const void* const* wu;          /* [L] -> [ffn][d_model] (up) */
  const void* const* wd;          /* [L] -> [d_model][ffn] */
} lopa_weights;

typedef struct {
  int block;      /* block length B, 16 <= B <= LOPA_MAX_BLOCK, multiple of 16 */
  int k;          /* lookahead branches, 0 <= k < LOPA_MAX_BRANCHES */
  float tau;      /* confidence threshold of the anchor fill (fill when maxp >= tau) */
  int max_prompt; /* longest prompt lopa_prefill will accept */
} lopa_decode_config;

/* Outcome of one LoPA iteration (one verification forward). */
typedef struct {
  int winner;            /* winning branch, 0 = anchor */
  int n_filled;          /* positions filled by this iteration (anchor fills + lookahead fill of the winner) */
  int block_done;        /* 1 when the block has no [MASK] left; it is then committed */
  int n_valid_branches;  /* 1 + min(k, masked positions left after the anchor fill) */
  int forwards;          /* forward passes run by this call (1, or 2 when a block-start forward ran) */
  int prefix_len;        /* committed prefix length P when the iteration ran */
  int device_error;      /* 0, or a device-side error code */
  float conf[LOPA_MAX_BRANCHES]; /* branch confidences; -inf for invalid branches, and for
                                    every branch but the winner in a completing iteration */
  int filled_pos[LOPA_MAX_BLOCK]; /* first n_filled entries: positions in the block, ascending */
  int filled_tok[LOPA_MAX_BLOCK]; /* tokens written at those positions */
} lopa_step_result;

typedef struct {
  long long tokens;   /* generated tokens */
  long long forwards; /* forward passes: one per iteration, plus the first block's start
                         forward (later blocks start inside the completing iteration's
                         pass); prefill excluded */
  long long steps;    /* LoPA iterations */
  long long blocks;   /* completed blocks */
  double seconds;     /* device time of the decode (CUDA events), prefill excluded */
} lopa_stats;

/* Validates the configs, copies the projection weights into tile-major owned copies,
 * records the borrowed embedding / norm pointers, allocates the static KV cache (K as
 * [L][max_seq][Hk][dh], V transposed as [L][Hk*dh][positions]), the per-branch Pre-Write
 * scratch, activations and state, precomputes RoPE tables and captures the iteration
 * into CUDA graphs.  stream: cudaStream_t to enqueue on (borrowed).  *out receives the
 * context.  Weight memory: about the size of the projection weights plus lm_head (half of it
 * with LOPA_WEIGHTS_E4M3). */
int lopa_init_model(const lopa_model_config* cfg, const lopa_weights* w,
                    const lopa_decode_config* dcfg, void* stream, lopa_ctx** out);

/* Runs the prompt (host int32 ids, n tokens, 1 <= n <= max_prompt) as one block that
 * attends bidirectionally within itself, writes its K/V into cache[0:n), and resets the
 * decoding state to an empty first output block at position n.  Synchronizes. */
int lopa_prefill(lopa_ctx* ctx, const int32_t* prompt, int n);

/* One LoPA iteration on the current block (running the block-start forward first when
 * the block is fresh): anchor fill, lookahead branches, one isolated verification
 * forward over the valid branches, confidences, winner, Commit-Winner of the winner's
 * K/V, logit reuse.  An iteration that completes the block (nothing masked after the
 * anchor fill, or one position that lookahead branch 1 fills) has its winner fixed before
 * the forward (confidence 1.0, lowest index): only that branch is evaluated, and when the
 * next block fits in max_seq its all-[MASK] start rows run in the same pass
 * (block-causal attention), so the next block starts with its logits in place.  out
 * (host, may be NULL) receives the outcome.  Synchronizes.  BAD_STATE before prefill or
 * when the next block would exceed max_seq. */
int lopa_step(lopa_ctx* ctx, lopa_step_result* out);

/* Decodes gen_len tokens (a multiple of the block length) from a block boundary:
 * for each block, the block-start forward then iterations until no [MASK] is left (the
 * last block of the call does not start the block after it).
 * out_tokens: host int32[gen_len] (may be NULL); out: host stats (may be NULL). */
int lopa_decode(lopa_ctx* ctx, int gen_len, int32_t* out_tokens, lopa_stats* out);

/* Discards everything decoded after absolute position pos (prompt_len <= pos <= the
 * committed prefix, pos - prompt_len a multiple of the block length): the cache beyond
 * pos counts as empty and the state becomes a fresh block at pos.  The prompt's K/V
 * stay, so a new decode of the same prompt needs no second prefill. */
int lopa_rewind(lopa_ctx* ctx, int pos);

/* Message of the last failed call on ctx (or of the last failed init when ctx is NULL). */
const char* lopa_last_error(const lopa_ctx* ctx);

/* Frees everything the context owns (including the weight copies; not the borrowed
 * embedding / norm gains or the stream). */
void lopa_free(lopa_ctx* ctx);

/* ---- inspection (used by parity tests) ---------------------------------------- */

/* Copies the current block state to host: tok[B] (int32, [MASK] where unfilled),
 * am[B] / mp[B] = greedy token and its probability from the logits that produced the
 * state (the reused logits), *prefix_len = committed prefix P.  Any output may be NULL. */
int lopa_get_block_state(lopa_ctx* ctx, int32_t* tok, int32_t* am, float* mp, int* prefix_len);

/* Overwrites the current block's tok/am/mp (host arrays of B entries) so that the next
 * lopa_step starts from that state (no block-start forward). */
int lopa_set_block_state(lopa_ctx* ctx, const int32_t* tok, const int32_t* am, const float* mp);

/* Runs one verification forward of nb branches (host int32 [nb][B], 1 <= nb <= 1+k)
 * for the current block position without changing the state or the cache.  Outputs
 * (host, each may be NULL): am/mp [nb][B]; hidden [nb][B][d_model] fp32 = residual
 * stream after the last layer (before the final norm). */
int lopa_verify_forward(lopa_ctx* ctx, const int32_t* branch_tok, int nb, int32_t* am,
                        float* mp, float* hidden);

/* Copies cache K and V for layer, positions [pos0, pos0+n) to host as bf16 words
 * [n][Hk][dh] each (either may be NULL). */
int lopa_read_kv(lopa_ctx* ctx, int layer, int pos0, int n, uint16_t* k, uint16_t* v);

/* Copies the Pre-Write scratch K and V of one branch (the block K/V its last
 * verification forward produced) for layer to host as bf16 words [B][Hk][dh] each. */
int lopa_read_branch_kv(lopa_ctx* ctx, int layer, int branch, uint16_t* k, uint16_t* v);

/* Test hook (diagnostics): writes `code` into the context's device error word, as a
 * device-side wait that gave up would.  The next lopa_step / lopa_decode then returns
 * LOPA_ERR_DEVICE_TIMEOUT; lopa_rewind (or lopa_prefill) clears the word.  Synchronizes. */
int lopa_debug_set_device_error(lopa_ctx* ctx, int code);

/* ---- kernel-level entry points (device pointers, caller's stream) -------------- */
/* These calls only enqueue work and return; argument errors are returned at once.  Their
 * bounded device-side waits record a wait that gave up in a device word of the library
 * (one per device; nothing is allocated), which lopa_kernel_status reads. */

/* Synchronizes `stream` and reports whether a device-side wait of a kernel-level call
 * (including lopa_lmhead_argmax_static) gave up since the last lopa_kernel_status on this
 * device: LOPA_ERR_DEVICE_TIMEOUT (code in lopa_last_error(NULL); the outputs of that call
 * are not valid) or LOPA_OK.  Clears the record.  Allocates nothing. */
int lopa_kernel_status(void* stream);

/* Test hook: every device-side wait of the kernel-level calls launched after this call
 * gives up after `ns` nanoseconds instead of the default 2 s (0 restores the default).
 * A wait that gives up stops its kernel cleanly: the kernel waits (with the default bound)
 * for the copies and tensor-core operations it started, frees its tensor memory and
 * returns.  Context calls (lopa_step, ...) always use the default. */
int lopa_set_wait_limit_ns(unsigned long long ns);

/* y[T][N] += x[T][K] . w[N][K]^T with bf16 inputs and fp32 accumulation on the
 * tcgen05 tensor cores (the projection kernel of the verification forward).
 * T >= 1, N multiple of 128, K multiple of 64; x, w 16-byte aligned; y fp32.  The
 * update is applied with atomic adds, so y must not be written concurrently by others. */
int lopa_linear_accumulate(const void* x, const void* w, float* y, int T, int N, int K,
                           void* stream);

/* Gate/up projection with the SwiGLU activation, the first half of the MLP of every layer
 * of the verification forward (Dream-7B follows the Qwen2.5 architecture; the branch rows
 * of all branches share one matmul: "Decoding-efficiency revolution" blog, section 3.3):
 *   h[t][f] = bf16( silu(g) * u ),  g = x[t] . w[f],  u = x[t] . w[F + f],
 *   silu(g) = g / (1 + exp(-g)), sums in fp32 on the tcgen05 tensor cores.
 * x [T][K] bf16, w [2F][K] bf16 (the F gate rows, then the F up rows; row-major),
 * h [T][F] bf16 (written); all device pointers, 16-byte aligned.  T >= 1, F a multiple of
 * 128, K a multiple of 64. */
int lopa_swiglu(const void* x, const void* w, void* h, int T, int F, int K, void* stream);

/* Per-row E4M3 quantisation as lopa_init_model does it for LOPA_WEIGHTS_E4M3:
 * w [rows][K] bf16 (device, 16-byte aligned), K a multiple of 64 -> codes [rows][K] bytes
 * (device, 16-byte aligned), scales [rows] float32 (device).  The weight row r is then
 * codes[r] * scales[r]. */
int lopa_quantize_e4m3(const void* w, int rows, int K, uint8_t* codes, float* scales, void* stream);

/* lopa_linear_accumulate with an E4M3 weight: y[T][N] += x[T][K] . (diag(scales) codes)^T,
 * codes [N][K] bytes and scales [N] as lopa_quantize_e4m3 writes them (device, 16-byte
 * aligned codes); the codes are widened to bf16 on chip and the scale is applied to the
 * fp32 sum.  Same limits as lopa_linear_accumulate. */
int lopa_linear_accumulate_e4m3(const void* x, const uint8_t* codes, const float* scales, float* y,
                                int T, int N, int K, void* stream);

/* Bytes of device workspace lopa_lmhead_argmax needs for `rows` rows. */
size_t lopa_lmhead_workspace_bytes(int rows, int vocab);

/* Fused LM head + online softmax ("SJTU x Huawei Xiaoyi release LoPA", section "Core
 * design of LoPA": logits of the verification pass are reused, so only their greedy
 * token and confidence are kept).  For each row r of hidden [rows][d_model] (bf16):
 * z = logit_scale * hidden_r . lm_head^T over vocab (mask_id excluded);
 * argmax_out[r] = argmax z (lowest id on ties), maxp_out[r] = 1 / sum exp(z - max z).
 * Full-vocabulary logits are never written.  workspace: device buffer of at least
 * lopa_lmhead_workspace_bytes(rows, vocab) bytes. */
int lopa_lmhead_argmax(const void* hidden, const void* lm_head, int rows, int d_model,
                       int vocab, float logit_scale, int mask_id, void* workspace,
                       size_t workspace_bytes, int32_t* argmax_out, float* maxp_out,
                       void* stream);

/* lopa_lmhead_argmax for callers that cannot allocate device memory.  (The paper has no
 * counterpart; this is a deployment convenience.)  Code running under a caller-owned
 * memory pool, in a loop that must never enter an allocator, or in a host that hands out
 * only fixed buffers cannot provide the workspace lopa_lmhead_argmax needs.  This call
 * computes the same result with its workspace in a fixed 4 MiB array inside the
 * library's device memory, held on every GPU that loads the library until exit; it
 * allocates nothing and calls no allocating routine.
 *   - rows * ceil(vocab / 256) * 12 must be <= 4 MiB (e.g. 256 rows at vocab 152064);
 *     larger requests return LOPA_ERR_INVALID_ARG with a message in lopa_last_error(NULL).
 *   - The first call on a device (with that device current) looks up the array's device
 *     address; make that first call before any stream capture that includes this call.
 *   - All calls on a device share the array: calls that can overlap on the GPU (e.g. on
 *     different streams without ordering) race and must be avoided.  Nothing in the array
 *     needs clearing between calls.
 *   - A device-side wait that gives up is recorded in a second fixed word beside the array
 *     and reported by lopa_kernel_status.
 *   - The addresses are looked up again if the device's context changes (e.g. after
 *     cudaDeviceReset); that call, too, should come before any stream capture.
 * Other arguments, layouts and results are those of lopa_lmhead_argmax. */
int lopa_lmhead_argmax_static(const void* hidden, const void* lm_head, int rows, int d_model,
                              int vocab, float logit_scale, int mask_id, int32_t* argmax_out,
                              float* maxp_out, void* stream);

/* Branch-isolated attention (same passage, "attention isolated between branches"):
 * for branch b, query row (i, h) attends to the shared prefix keys [0, prefix_len)
 * and to its own block keys [0, block) only, bidirectionally, with softmax scale
 * 1/sqrt(head_dim) and grouped-query heads (head h uses KV head g = h / G, G =
 * n_heads / n_kv_heads).  Layouts are the ones the verification forward keeps on the
 * GPU (all bf16, 16-byte aligned):
 *   q          [n_kv_heads][n_branches*block][G][head_dim]  (query (t, h) at
 *              [h / G][t][h % G], t = b*block + i)
 *   k_prefix   [prefix_len][n_kv_heads][head_dim]
 *   vt_prefix  [n_kv_heads*head_dim][ld_vt_prefix]  values transposed: V[p][g][d] at
 *              row g*head_dim + d, column p; ld_vt_prefix >= prefix_len, multiple of 8
 *   k_block    [n_branches][block][n_kv_heads][head_dim]
 *   vt_block   [n_kv_heads*head_dim][n_branches*block]  (V of branch b position i at
 *              column b*block + i)
 *   out        [n_branches*block][n_heads*head_dim]
 * head_dim in {32, 64, 128}; block a multiple of 16, <= 4096.  prefix_len may be 0
 * (k_prefix / vt_prefix then unused).  head_dim 128 runs on the tcgen05 tensor cores. */
int lopa_branch_attention(const void* q, const void* k_prefix, const void* vt_prefix,
                          int prefix_len, int ld_vt_prefix, const void* k_block,
                          const void* vt_block, int n_branches, int block, int n_heads,
                          int n_kv_heads, int head_dim, void* out, void* stream);

/* Diagnostics: launches the verification-step GEMM of one kind (0 = q/k/v, 1 = output
 * projection, 2 = gate/up + SwiGLU, 3 = down, 4 = LM head) `iters` times on the
 * context stream, cycling over the layers' weights, and writes the mean launch time
 * in milliseconds (CUDA events) to *avg_ms.  The decoding state is not changed; the
 * activation buffers hold garbage afterwards until the next forward rewrites them. */
int lopa_time_gemm(lopa_ctx* ctx, int kind, int iters, float* avg_ms);

/* Verification-step latency: launches the captured forward of one kind (1 = the
 * (1+k)-branch verification forward of a LoPA iteration, steps a3-a8 over the current
 * branch tokens; 0 = the block-start forward of the current block) `iters` times back to
 * back (1 <= iters <= 10000) on the context stream, each bracketed by CUDA events, and
 * writes the median (and, if mean_ms is not NULL, the mean) per-launch milliseconds.
 * Needs a prefilled context with room for a block at the current prefix (else
 * LOPA_ERR_BAD_STATE).  The forwards write only activations, the Pre-Write scratch and
 * the per-branch logit summaries: the decoding state is unchanged. */
int lopa_time_forward(lopa_ctx* ctx, int kind, int iters, float* median_ms, float* mean_ms);

/* Library version (major*10000 + minor*100 + patch). */
int lopa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LOPA_H */
