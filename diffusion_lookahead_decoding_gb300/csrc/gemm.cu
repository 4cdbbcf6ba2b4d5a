// Branch-batched projection GEMMs on the sm_103a tensor cores (tcgen05 + TMEM, TMA-fed).
//
// Every projection of the verification forward multiplies the (1+k)*B token rows of
// all branches by one weight matrix ("Decoding-efficiency revolution" blog, section
// 3.3: all branch forwards share one matmul).  The weight stream is the cost, so each
// CTA owns a slab of weight rows and streams it once through TMA -> shared memory ->
// tcgen05.mma, with the whole token tile (up to 256 rows) on the MMA's other side:
//
//   RED_ADD : D[w_row][tok] = W . X^T over a K-split; the epilogue stores the split's
//             fp32 partial [split][T][N] (summed in a fixed order by the consumer) or,
//             for the standalone call, adds it atomically into an fp32 [T][N] output.
//   SWIGLU  : two accumulators (gate rows f, up rows F+f) and an epilogue that writes
//             bf16 silu(gate)*up for the down projection.
//   LMSTATS : tokens on M (two 128-row tiles), 256 vocab rows on N; the epilogue keeps
//             per (vocab tile, token) the max logit, its id and sum exp(z - max), so
//             full-vocabulary logits never reach memory.
//
// Weights and activations travel in two separate shared-memory rings: the weight ring
// is deeper (weights come from HBM, activations from L2), so more weight bytes are in
// flight per SM.  Roles in a CTA of 224 threads: warp 0 streams weights (before waiting
// on the previous kernel, since weights never depend on it), warp 6 streams activations,
// warp 1 allocates TMEM and issues the MMAs, warps 2..5 run the epilogue (each reads its
// 32 TMEM lanes).  All waits are bounded (see common.cuh).
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

constexpr int kThreads = 224;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxStages = 8;

struct SmemTail {
  uint64_t wfull[kMaxStages], wempty[kMaxStages];
  uint64_t xfull[kMaxStages], xempty[kMaxStages];
  uint64_t accf;
  uint32_t tmem_addr;
  int abort;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = smem + (size_t)a.w_stages * a.w_slot_bytes;
  SmemTail* tail = reinterpret_cast<SmemTail*>(xring + (size_t)a.x_stages * a.x_slot_bytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int SW = a.w_stages, SX = a.x_stages;
  // The weight operand is A (128-row tiles) except for the LM head, where it is B.
  constexpr bool kWeightIsA = MODE != GEMM_LMSTATS;

  // Tile coordinates.
  int a_row[2];
  bool a_ok[2];
  int b_row;
  if (MODE == GEMM_RED_ADD) {
    a_row[0] = blockIdx.x * a.na * 128;
    a_row[1] = a_row[0] + 128;
    b_row = blockIdx.z * a.nbox;
    a_ok[0] = a_row[0] < a.a_rows;
    a_ok[1] = a.na > 1 && a_row[1] < a.a_rows;
  } else if (MODE == GEMM_SWIGLU) {
    a_row[0] = blockIdx.x * 128;
    a_row[1] = a.F + blockIdx.x * 128;
    b_row = blockIdx.z * a.nbox;
    a_ok[0] = a_ok[1] = true;
  } else {
    a_row[0] = blockIdx.z * a.na * 128;
    a_row[1] = a_row[0] + 128;
    b_row = blockIdx.x * a.nbox;
    a_ok[0] = a_row[0] < a.T;
    a_ok[1] = a.na > 1 && a_row[1] < a.T;
  }
  const int kb0 = (int)(((long long)blockIdx.y * a.k_blocks) / a.splits);
  const int kb1 = (int)(((long long)(blockIdx.y + 1) * a.k_blocks) / a.splits);
  const int nk = kb1 - kb0;
  const uint32_t ncols = a.na == 2 ? 512u : 256u;
  const uint32_t a_bytes = (a_ok[0] ? a.a_tile_bytes : 0u) + (a_ok[1] ? a.a_tile_bytes : 0u);
  const uint32_t b_bytes = a.nbox * 128u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(smem_u32(&tail->wfull[s]), 1);
      mbar_init(smem_u32(&tail->wempty[s]), 1);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(smem_u32(&tail->xfull[s]), 1);
      mbar_init(smem_u32(&tail->xempty[s]), 1);
    }
    mbar_init(smem_u32(&tail->accf), 1);
    tail->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tail->tmem_addr), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_addr;
  volatile int* abort = &tail->abort;
  pdl_trigger();

  if (warp == 0 || warp == 6) {
    // Producers: warp 0 streams the weight operand, warp 6 the activation operand.
    const bool weights = warp == 0;
    if (lane == 0) {
      if (!weights) pdl_wait();  // activations are written by the previous kernel
      const int S = weights ? SW : SX;
      uint8_t* ring = weights ? wring : xring;
      const uint32_t slot = weights ? a.w_slot_bytes : a.x_slot_bytes;
      uint64_t* full = weights ? tail->wfull : tail->xfull;
      uint64_t* empty = weights ? tail->wempty : tail->xempty;
      const bool is_a = weights == kWeightIsA;
      const uint64_t pol = weights ? policy_evict_first() : policy_evict_last();
      const uint32_t bytes = is_a ? a_bytes : b_bytes;
      for (int it = 0; it < nk; ++it) {
        const int s = it % S;
        if (it >= S && !mbar_wait_bounded(smem_u32(&empty[s]), ((uint32_t)(it / S) & 1u) ^ 1u,
                                          abort, a.err, DEV_TIMEOUT_PRODUCER))
          break;
        const uint32_t fb = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + (size_t)s * slot);
        const int kx = (kb0 + it) * 64;
        mbar_arrive_expect_tx(fb, bytes);
        if (is_a) {
          if (a_ok[0]) tma_load_2d(dst, &mapA, fb, kx, a_row[0], pol);
          if (a_ok[1]) tma_load_2d(dst + a.a_tile_bytes, &mapA, fb, kx, a_row[1], pol);
        } else {
          tma_load_2d(dst, &mapB, fb, kx, b_row, pol);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, a.nbox);
      bool ok = true;
      for (int it = 0; it < nk; ++it) {
        const int sw = it % SW, sx = it % SX;
        if (!mbar_wait_bounded(smem_u32(&tail->wfull[sw]), (uint32_t)(it / SW) & 1u, abort, a.err,
                               DEV_TIMEOUT_MMA) ||
            !mbar_wait_bounded(smem_u32(&tail->xfull[sx]), (uint32_t)(it / SX) & 1u, abort, a.err,
                               DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ws = smem_u32(wring + (size_t)sw * a.w_slot_bytes);
        const uint32_t xs = smem_u32(xring + (size_t)sx * a.x_slot_bytes);
        const uint32_t abase = kWeightIsA ? ws : xs;
        const uint64_t bdesc = sw128_desc(kWeightIsA ? xs : ws);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (!a_ok[i]) continue;
            const uint64_t adesc = sw128_desc(abase + i * a.a_tile_bytes);
            mma_bf16(tmem + (uint32_t)(i * 256), adesc + 2 * kk, bdesc + 2 * kk, idesc,
                     (it | kk) != 0);
          }
        }
        mma_commit(smem_u32(&tail->wempty[sw]));
        mma_commit(smem_u32(&tail->xempty[sx]));
      }
      if (ok) mma_commit(smem_u32(&tail->accf));
    }
  } else {
    // Epilogue warps 2..5: warp w may only touch TMEM lanes 32*(w%4) .. +31.  The
    // outputs may still be read by the previous kernel until it completes.
    pdl_wait();
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    if (nk > 0 && mbar_wait_bounded(smem_u32(&tail->accf), 0, abort, a.err, DEV_TIMEOUT_EPILOGUE)) {
      tc_fence_after();
      if (MODE == GEMM_RED_ADD) {
        for (int i = 0; i < 2; ++i) {
          if (!a_ok[i]) continue;
          const int n = a_row[i] + r;
          for (int c = 0; c < a.nbox; c += 16) {
            float v[16];
            tmem_ld16(lane_base + (uint32_t)(i * 256 + c), v);
            if (a.atomic) {
              for (int j = 0; j < 16; ++j) {
                const int t = b_row + c + j;
                if (t < a.T) atomicAdd(a.out_f32 + (size_t)t * a.ldo + n, v[j]);
              }
            } else {
              // Plain stores of this split's partial sums; a warp writes 128 contiguous
              // bytes per token.  The consumer kernel adds the splits in a fixed order.
              float* base = a.out_f32 + (size_t)blockIdx.y * a.split_stride + n;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int t = b_row + c + j;
                if (t < a.T) base[(size_t)t * a.ldo] = v[j];
              }
            }
          }
        }
      } else if (MODE == GEMM_SWIGLU) {
        const int f = a_row[0] + r;
        for (int c = 0; c < a.nbox; c += 16) {
          float g[16], u[16];
          tmem_ld16(lane_base + (uint32_t)c, g);
          tmem_ld16(lane_base + (uint32_t)(256 + c), u);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = b_row + c + j;
            const float h = g[j] / (1.0f + __expf(-g[j])) * u[j];
            if (t < a.T) a.out_bf16[(size_t)t * a.ldh + f] = __float2bfloat16_rn(h);
          }
        }
      } else {
        const int vt = blockIdx.x;
        for (int i = 0; i < 2; ++i) {
          if (!a_ok[i]) continue;
          const int t = a_row[i] + r;
          float m = -INFINITY, ssum = 0.f;
          int idx = 0;
          for (int c = 0; c < a.nbox; c += 16) {
            float v[16];
            __syncwarp();
            tmem_ld16(lane_base + (uint32_t)(i * 256 + c), v);
            float cm = -INFINITY;
            int ci = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int id = b_row + c + j;
              v[j] = (id < a.V && id != a.mask_id) ? v[j] * a.scale : -INFINITY;
              if (v[j] > cm) { cm = v[j]; ci = id; }  // strict: lowest id wins ties
            }
            if (cm != -INFINITY) {
              const float nm = fmaxf(m, cm);
              float acc = (m == -INFINITY) ? 0.f : ssum * __expf(m - nm);
#pragma unroll
              for (int j = 0; j < 16; ++j) acc += __expf(v[j] - nm);
              if (cm > m) idx = ci;
              m = nm;
              ssum = acc;
            }
          }
          if (t < a.T) {
            const size_t o = (size_t)vt * a.part_ld + t;
            a.part_m[o] = m;
            a.part_s[o] = ssum;
            a.part_i[o] = idx;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

uint32_t round1k(uint32_t v) { return (v + 1023) & ~1023u; }

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, char* errbuf, size_t errlen) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0) {
    snprintf(errbuf, errlen, "tensor map base/stride not 16-byte aligned");
    return false;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled failed (%d) rows=%llu cols=%llu box=%u", (int)r,
             (unsigned long long)rows, (unsigned long long)cols, box_rows);
    return false;
  }
  return true;
}

int gemm_max_smem() { return kMaxSmem; }

cudaError_t gemm_set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemm_kernel<GEMM_RED_ADD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemm_kernel<GEMM_SWIGLU>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(gemm_kernel<GEMM_LMSTATS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMaxSmem);
}

// act: [act_rows_alloc][K] bf16 activations (T valid rows); w: [n_rows_w][K] bf16.
const char* plan_gemm(GemmLaunch* L, int mode, const void* act, int act_rows_alloc, int T,
                      const void* w, int n_rows_w, int K, int na, int splits, int tok_box,
                      int num_sms) {
  static thread_local char err[256];
  memset(L, 0, sizeof(*L));
  GemmArgs& a = L->args;
  if (K % 64 != 0 || K <= 0) return "GEMM K must be a positive multiple of 64";
  if (T <= 0) return "GEMM needs at least one token row";
  a.mode = mode;
  a.k_blocks = K / 64;
  a.T = T;
  a.a_tile_bytes = 128 * 128;  // 128 rows x 64 bf16
  if (mode == GEMM_LMSTATS) {
    a.na = na;
    a.nbox = 256;
    a.a_rows = T;
    a.splits = 1;
    if (!make_tmap_bf16(&L->mapA, act, act_rows_alloc, K, 128, err, sizeof(err))) return err;
    if (!make_tmap_bf16(&L->mapB, w, n_rows_w, K, 256, err, sizeof(err))) return err;
    L->grid = dim3((n_rows_w + 255) / 256, 1, (T + na * 128 - 1) / (na * 128));
    a.w_slot_bytes = round1k(a.nbox * 128);
    a.x_slot_bytes = round1k(a.na * a.a_tile_bytes);
  } else {
    if (tok_box < 16 || tok_box > 256 || tok_box % 16 != 0) return "token box must be 16..256, multiple of 16";
    if (n_rows_w % 128 != 0) return "GEMM N must be a multiple of 128";
    a.na = (mode == GEMM_SWIGLU) ? 2 : na;
    a.F = n_rows_w / 2;
    a.nbox = tok_box;
    a.a_rows = n_rows_w;
    a.splits = (mode == GEMM_SWIGLU) ? 1 : splits;
    if (a.splits < 1) a.splits = 1;
    if (a.splits > a.k_blocks) a.splits = a.k_blocks;
    if (!make_tmap_bf16(&L->mapA, w, n_rows_w, K, 128, err, sizeof(err))) return err;
    if (!make_tmap_bf16(&L->mapB, act, act_rows_alloc, K, tok_box, err, sizeof(err))) return err;
    const int gx = (mode == GEMM_SWIGLU) ? (n_rows_w / 2) / 128 : (n_rows_w + a.na * 128 - 1) / (a.na * 128);
    L->grid = dim3(gx, a.splits, (T + tok_box - 1) / tok_box);
    a.w_slot_bytes = round1k(a.na * a.a_tile_bytes);
    a.x_slot_bytes = round1k(a.nbox * 128);
  }
  (void)num_sms;
  // Activations come from L2 (short latency): 3 slots, more when they are small.  The
  // weight ring takes the rest of shared memory.
  const int budget = kMaxSmem - 1024 - (int)sizeof(SmemTail) - 64;
  a.x_stages = a.x_slot_bytes <= 8192 ? 6 : 3;
  a.w_stages = (budget - a.x_stages * (int)a.x_slot_bytes) / (int)a.w_slot_bytes;
  if (a.w_stages > kMaxStages) a.w_stages = kMaxStages;
  if (a.w_stages < 2) return "GEMM tile does not fit in shared memory";
  L->smem = 1024 + (size_t)a.w_stages * a.w_slot_bytes + (size_t)a.x_stages * a.x_slot_bytes +
            sizeof(SmemTail) + 64;
  return "";
}

cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t s) {
  switch (L.args.mode) {
    case GEMM_RED_ADD:
      return launch_pdl(gemm_kernel<GEMM_RED_ADD>, L.grid, dim3(kThreads), L.smem, s, L.mapA,
                        L.mapB, L.args);
    case GEMM_SWIGLU:
      return launch_pdl(gemm_kernel<GEMM_SWIGLU>, L.grid, dim3(kThreads), L.smem, s, L.mapA,
                        L.mapB, L.args);
    default:
      return launch_pdl(gemm_kernel<GEMM_LMSTATS>, L.grid, dim3(kThreads), L.smem, s, L.mapA,
                        L.mapB, L.args);
  }
}

}  // namespace lopa
