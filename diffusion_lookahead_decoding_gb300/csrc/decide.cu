// Decision and commit kernels of one LoPA iteration ("SJTU x Huawei Xiaoyi release
// LoPA", sections "Core design of LoPA" and "LoPA-Dist"):
//   decide   : anchor fill (confidence-driven greedy, threshold tau, at least one fill)
//              and the k lookahead branches (one extra fill each, at the k most
//              confident positions still masked);
//   select   : branch confidence = mean max-probability over the branch's remaining
//              masked positions, winner = highest confidence (ties -> lowest branch),
//              then the winner's tokens and logit summary become the state (logit reuse);
//   commit   : Commit-Winner-Cache - copy the winner's pre-written block K/V from the
//              branch scratch into the static cache;
//   finalize : when the block has no [MASK] left, emit it and advance the prefix.
// Blocks are at most 64 positions, so each decision runs in one CTA.
#include "common.cuh"
#include "internal.h"
#include "timeline.cuh"

namespace lopa {

LOPA_TL_UNIT(decide)

namespace {

constexpr unsigned kFull = 0xffffffffu;

// (value, index) pair reduced to the larger value, the lower index on equal values; -1
// marks an empty slot.  Every lane of the warp gets the result.
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, v, o);
    const int oi = __shfl_xor_sync(kFull, idx, o);
    const bool take = oi >= 0 && (idx < 0 || ov > v || (ov == v && oi < idx));
    v = take ? ov : v;
    idx = take ? oi : idx;
  }
}

__global__ void decide_kernel(DevState* st, int B, int k, float tau, int mask_id,
                              int* __restrict__ branch_tok, int* __restrict__ valid) {
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  __shared__ float s_mp[LOPA_MAX_BLOCK];
  __shared__ int s_rem[LOPA_MAX_BLOCK];
  __shared__ int s_cand[LOPA_MAX_BRANCHES];
  __shared__ float s_bv[LOPA_MAX_BLOCK / 32];
  __shared__ int s_bi[LOPA_MAX_BLOCK / 32];
  const int i = threadIdx.x;  // blockDim.x == LOPA_MAX_BLOCK (two warps)
  const int lane = i & 31, wid = i >> 5;
  const int nb = k + 1;
  const int tok = i < B ? st->tok[i] : 0;
  const int am = i < B ? st->am[i] : 0;
  const float mp = i < B ? st->mp[i] : 0.f;
  const bool masked = i < B && tok == mask_id;
  bool fill = masked && mp >= tau;
  s_mp[i] = mp;
  if (i < LOPA_MAX_BRANCHES) s_cand[i] = -1;
  const int any_fill = __syncthreads_or(fill);
  if (!any_fill) {
    // Fill the single most confident masked position (lowest position on ties): a warp
    // (max, lowest index) reduction per warp, then the two warps' winners.
    float v = masked ? mp : -INFINITY;
    int idx = masked ? i : -1;
    warp_argmax(v, idx);
    if (lane == 0) {
      s_bv[wid] = v;
      s_bi[wid] = idx;
    }
    __syncthreads();
    v = s_bv[lane & 1];
    idx = s_bi[lane & 1];
    if (lane >= 2) idx = -1;
    warp_argmax(v, idx);
    fill = (i == idx);
  }
  const int anchor = fill ? am : tok;
  const bool rem = masked && !fill;
  s_rem[i] = rem;
  const int nrem = __syncthreads_count(rem);
  const int nl = nrem < k ? nrem : k;
  if (rem) {
    // Rank among the remaining positions: more confident first, then lower position.
    int rank = 0;
    for (int j = 0; j < B; ++j)
      if (s_rem[j] && (s_mp[j] > mp || (s_mp[j] == mp && j < i))) ++rank;
    if (rank < nl) s_cand[rank] = i;
  }
  __syncthreads();
  // The iteration completes the block when no position stays masked after the anchor
  // fill (the anchor completes it) or exactly one does and lookahead branch 1 fills it.
  // A completing branch has confidence 1.0 and every other branch less (its mean covers
  // at least one masked position), so the lowest completing branch wins whatever the
  // forward returns: final_w.  Only it is evaluated: its tokens go to slot 0, and slot 1
  // becomes a blank block for a block-start forward merged into the same pass.
  const int final_w = nrem == 0 ? 0 : (nrem == 1 && nl >= 1 ? 1 : -1);
  if (i < B) {
    if (final_w >= 0) {
      const bool extra = final_w == 1 && s_cand[0] == i;
      branch_tok[i] = extra ? am : anchor;
      branch_tok[B + i] = mask_id;
    } else {
      for (int b = 0; b < nb; ++b) {
        const bool extra = b >= 1 && s_cand[b - 1] == i;
        branch_tok[b * B + i] = extra ? am : anchor;
      }
    }
  }
  if (i < nb) valid[i] = final_w >= 0 ? i == 0 : (i == 0) || (i - 1 < nl);
  if (i < LOPA_MAX_BRANCHES) st->cand[i] = s_cand[i];
  if (i == 0) {
    st->n_valid = 1 + nl;
    st->final_w = final_w;
  }
  TL_END(tl::DECIDE);
}

// One warp per branch (blockDim.x == 32 * LOPA_MAX_BRANCHES).
__global__ void select_kernel(DevState* st, int B, int nb, int mask_id,
                              const int* __restrict__ branch_tok, const int* __restrict__ valid,
                              const int* __restrict__ am_b, const float* __restrict__ mp_b) {
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  __shared__ float s_conf[LOPA_MAX_BRANCHES];
  __shared__ int s_w;
  __shared__ int s_old[LOPA_MAX_BLOCK];
  __shared__ int s_new[LOPA_MAX_BLOCK];
  const int i = threadIdx.x;
  const int lane = i & 31, b = i >> 5;
  if (b < nb) {
    // Branch confidence: mean maxp over the branch's masked positions (lane j holds
    // positions j and j + 32), summed by a fixed shuffle tree; no masked position -> 1.0.
    float sum = 0.f;
    int cnt = 0;
    for (int j = lane; j < B; j += 32) {
      if (branch_tok[b * B + j] == mask_id) {
        sum += mp_b[b * B + j];
        ++cnt;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(kFull, sum, o);
      cnt += __shfl_xor_sync(kFull, cnt, o);
    }
    if (lane == 0) s_conf[b] = valid[b] ? (cnt ? sum / (float)cnt : 1.0f) : -INFINITY;
  }
  if (i < B) s_old[i] = st->tok[i];
  __syncthreads();
  if (b == 0) {
    // Winner: highest confidence, lowest branch on ties.
    float v = lane < nb ? s_conf[lane] : -INFINITY;
    int idx = lane < nb ? lane : -1;
    warp_argmax(v, idx);
    if (lane == 0) s_w = idx;
  }
  __syncthreads();
  const int w = s_w;
  if (i < B) {
    const int nt = branch_tok[w * B + i];
    s_new[i] = nt;
    st->tok[i] = nt;
    st->am[i] = am_b[w * B + i];
    st->mp[i] = mp_b[w * B + i];
  }
  __syncthreads();
  // Positions this iteration filled, in ascending order: a ballot per warp, each filled
  // position's slot = the filled positions before it (popcounts).
  __shared__ unsigned s_bal[LOPA_MAX_BLOCK / 32];
  const bool filled = i < B && s_old[i] == mask_id && s_new[i] != mask_id;
  const unsigned bal = __ballot_sync(kFull, filled);
  if (lane == 0 && b < LOPA_MAX_BLOCK / 32) s_bal[b] = bal;
  const int any_masked = __syncthreads_or(i < B && s_new[i] == mask_id);
  lopa_step_result& r = st->res;
  if (filled) {
    const int slot = (b == 1 ? __popc(s_bal[0]) : 0) + __popc(bal & ((1u << lane) - 1u));
    r.filled_pos[slot] = i;
    r.filled_tok[slot] = s_new[i];
  }
  // In a completing iteration only the winner (slot 0) was evaluated: it is reported
  // under its branch index, every other branch as -inf.
  const int fw = st->final_w;
  if (i < LOPA_MAX_BRANCHES)
    r.conf[i] = fw >= 0 ? (i == fw ? s_conf[0] : -INFINITY) : (i < nb ? s_conf[i] : -INFINITY);
  if (i == 0) {
    const int done = !any_masked;
    r.winner = fw >= 0 ? fw : w;
    r.n_filled = __popc(s_bal[0]) + (B > 32 ? __popc(s_bal[1]) : 0);
    r.block_done = done;
    r.n_valid_branches = st->n_valid;
    r.prefix_len = st->P;
    r.device_error = st->err;
    r.forwards = 1;
    st->winner = w;
    st->block_done = done;
  }
  TL_END(tl::SELECT);
}

// grid: (L, 2 [K, V], chunks); copies B rows of row_elems bf16 of the winner's branch.
// Commit-Winner: copies the winner branch's block K ([B][row_elems] rows) and V^T
// (columns [w*B, w*B+B) of each of the row_elems rows) from the Pre-Write scratch into the
// static cache at the block position P.  blockIdx.y: 0 = K, 1 = V^T.
__global__ void commit_kv_kernel(const DevState* st, const bf16* __restrict__ ks,
                                 const bf16* __restrict__ vts, bf16* __restrict__ kc,
                                 bf16* __restrict__ vtc, int B, int row_elems, KvStrides kv) {
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  const int l = blockIdx.x;
  const int w = st->winner;
  const int P = st->P;
  if (blockIdx.y == 0) {
    const bf16* src = ks + (size_t)l * kv.k_scr + (size_t)w * B * row_elems;
    bf16* dst = kc + (size_t)l * kv.k_cache + (size_t)P * row_elems;
    const int n16 = B * row_elems / 8;
    for (int e = blockIdx.z * blockDim.x + threadIdx.x; e < n16; e += gridDim.z * blockDim.x)
      reinterpret_cast<uint4*>(dst)[e] = reinterpret_cast<const uint4*>(src)[e];
  } else {
    const bf16* src = vts + (size_t)l * kv.v_scr + (size_t)w * B;
    bf16* dst = vtc + (size_t)l * kv.v_cache + P;
    const int n = B * row_elems;
    for (int e = blockIdx.z * blockDim.x + threadIdx.x; e < n; e += gridDim.z * blockDim.x) {
      const int r = e / B, c = e - r * B;
      dst[(size_t)r * kv.ld_cache + c] = src[(size_t)r * kv.ld_scr + c];
    }
  }
  TL_END(tl::COMMIT);
}

// With am_next / mp_next (the logit summary of a block-start forward run in the same
// pass) a finished block is followed by the next block with its first logits in place.
__global__ void finalize_kernel(DevState* st, int B, int mask_id, int* __restrict__ out_tokens,
                                const int* __restrict__ am_next, const float* __restrict__ mp_next) {
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  const int i = threadIdx.x;
  const int P = st->P, P0 = st->P0;
  const int done = st->block_done;
  __syncthreads();
  if (done) {
    if (i < B) {
      out_tokens[P - P0 + i] = st->tok[i];
      st->tok[i] = mask_id;
      if (am_next) {
        st->am[i] = am_next[i];
        st->mp[i] = mp_next[i];
      }
    }
    if (i == 0) st->P = P + B;
  }
  TL_END(tl::FINALIZE);
}

__global__ void state_reset_kernel(DevState* st, int P, int B, int mask_id) {
  const int i = threadIdx.x;
  if (i < LOPA_MAX_BLOCK) {
    st->tok[i] = i < B ? mask_id : 0;
    st->am[i] = 0;
    st->mp[i] = 0.f;
  }
  if (i < LOPA_MAX_BRANCHES) st->cand[i] = -1;
  if (i == 0) {
    st->P = P;
    st->P0 = P;
    st->winner = 0;
    st->block_done = 0;
    st->err = 0;
    st->n_valid = 0;
    st->final_w = -1;
  }
}

}  // namespace

cudaError_t decide_set_carveout() {
  const int c = cudaSharedmemCarveoutMaxShared;
  const void* ks[] = {(const void*)decide_kernel, (const void*)select_kernel,
                      (const void*)commit_kv_kernel, (const void*)finalize_kernel};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decide(void* st, int B, int k, float tau, int mask_id, int* branch_tok,
                          int* valid, cudaStream_t s) {
  return launch_pdl(decide_kernel, dim3(1), dim3(LOPA_MAX_BLOCK), 0, s, static_cast<DevState*>(st),
                    B, k, tau, mask_id, branch_tok, valid);
}

cudaError_t launch_select(void* st, int B, int nb, int mask_id, const int* branch_tok,
                          const int* valid, const int* am_b, const float* mp_b,
                          cudaStream_t s) {
  return launch_pdl(select_kernel, dim3(1), dim3(32 * LOPA_MAX_BRANCHES), 0, s,
                    static_cast<DevState*>(st), B, nb, mask_id, branch_tok, valid, am_b, mp_b);
}

cudaError_t launch_commit_kv(const void* st, const bf16* ks, const bf16* vts, bf16* kc,
                             bf16* vtc, int L, int B, int row_elems, const KvStrides& kv,
                             cudaStream_t s) {
  const int n = B * row_elems;
  const int chunks = (n + 255) / 256 < 16 ? (n + 255) / 256 : 16;
  return launch_pdl(commit_kv_kernel, dim3(L, 2, chunks), dim3(256), 0, s,
                    static_cast<const DevState*>(st), ks, vts, kc, vtc, B, row_elems, kv);
}

cudaError_t launch_finalize(void* st, int B, int mask_id, int* out_tokens, const int* am_next,
                            const float* mp_next, cudaStream_t s) {
  return launch_pdl(finalize_kernel, dim3(1), dim3(LOPA_MAX_BLOCK), 0, s,
                    static_cast<DevState*>(st), B, mask_id, out_tokens, am_next, mp_next);
}

cudaError_t launch_state_reset(void* st, int P, int B, int mask_id, cudaStream_t s) {
  state_reset_kernel<<<1, LOPA_MAX_BLOCK, 0, s>>>(static_cast<DevState*>(st), P, B, mask_id);
  return cudaGetLastError();
}

}  // namespace lopa
