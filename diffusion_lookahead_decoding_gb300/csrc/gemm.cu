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
//   QKV     : the q/k/v projection.  The K-splits of one output tile form a thread-block
//             cluster; each CTA writes its fp32 partial tile to an L2 exchange region and
//             CTA r of the cluster sums token slice r over all splits (fixed split order),
//             applies RoPE to q/k and writes bf16 q, K and V (the Pre-Write).  Only the
//             cluster's CTAs read these partials, right after they are written.
//   SWIGLU  : two accumulators (gate rows f, up rows F+f) and an epilogue that writes
//             bf16 silu(gate)*up for the down projection.
//   LMSTATS : tokens on M (two 128-row tiles), 256 vocab rows on N; the epilogue keeps
//             per (vocab tile, token) the max logit, its id and sum exp(z - max), so
//             full-vocabulary logits never reach memory.
//
// Weights and activations travel in two separate shared-memory rings: the weight ring
// is deeper (weights come from HBM, activations from L2), so more weight bytes are in
// flight per SM.  Roles in a CTA of 352 threads: warp 0 streams weights (before waiting
// on the previous kernel, since weights never depend on it), warp 10 streams
// activations, warp 1 allocates TMEM and issues the MMAs, warps 2..9 run the epilogue
// (two warps per TMEM lane quarter, splitting the columns).  Split-K partials are stored
// straight from the TMEM registers (a warp's lanes are 32 consecutive output features: one
// 128-byte line per store); the SwiGLU output is staged in the freed rings so that its bf16
// rows leave as 16-byte stores.  All waits are bounded.
//
// E4M3 weight stream (template flag F8): the weight TMA brings 8-bit codes (half the HBM
// bytes) into a staging ring; eight converter warps widen each stage to bf16 in the
// 128-byte-swizzled K-major layout the MMA reads (exactly: every E4M3 value is a bf16
// value) and hand the slot to the MMA warp; the epilogue multiplies each weight row's
// accumulator by that row's float32 scale.  The MMA itself stays bf16 x bf16 -> fp32.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "timeline.cuh"

namespace lopa {

LOPA_TL_UNIT(gemm)

namespace {

constexpr int kEpiWarps = 8;
constexpr int kThreads = (3 + kEpiWarps) * 32;  // W producer, MMA, 8 epilogue warps, X producer
// E4M3 stream: 8 converter warps (codes -> bf16) after the 11 warps above.  The q/k/v kernel
// adds none: its register-heavy exchange epilogue would spill, so there the 8 epilogue warps
// convert during the main loop instead (measured faster for q/k/v, slower for the others,
// whose epilogue warps then also compete for issue slots with the MMA and producer warps).
template <int MODE>
__host__ __device__ constexpr int conv_threads() { return (MODE == GEMM_QKV ? 0 : 8) * 32; }
template <int MODE, bool F8>
__host__ __device__ constexpr int threads_of() { return kThreads + (F8 ? conv_threads<MODE>() : 0); }
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxStages = 8;

// Barrier among the eight epilogue warps only (named barrier 3, 256 threads).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

struct SmemTail {
  uint64_t wfull[kMaxStages], wempty[kMaxStages];
  uint64_t xfull[kMaxStages], xempty[kMaxStages];
  uint64_t ffull[kMaxStages], fempty[kMaxStages];  // E4M3 stream: staging ring of codes
  uint64_t accf;
  uint64_t cfull;  // clustered mode: every split's partial tile is in the exchange workspace
  uint64_t drain;  // after a wait gave up: completion of every MMA this CTA issued
  uint32_t tmem_addr;
  int abort;
  int w_issued, x_issued;  // TMA loads issued into the weight / activation ring
  int mma_issued;          // 1 once the MMA warp issued an MMA
  unsigned long long tl_tw;  // timeline builds: when the accumulator was complete
};

// E4M3 -> bf16, two codes per 32-bit pair.  Each 16-bit lane gets the code's sign in bit
// 15 and its 7 magnitude bits in bits 4..10: the exponent field e and fraction m land in
// the low exponent bits and the top fraction bits of a bf16, which then reads
// 2^(e-127) * 1.m (e >= 1) or 2^-126 * 0.m (e = 0).  The code's value is 2^(e-7) * 1.m or
// 2^-6 * 0.m, so one exact multiplication by 2^120 finishes the conversion for normal and
// subnormal codes alike.
__device__ __forceinline__ uint32_t bf16x2_times_2p120(uint32_t bits) {
  __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&bits);
  const uint32_t k2p120 = 0x7B807B80u;  // bf16 2^120 in both lanes
  h = __hmul2(h, *reinterpret_cast<const __nv_bfloat162*>(&k2p120));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Four codes (bytes of w, lowest byte = lowest column) -> two bf16 pairs.  The byte
// permutations place the magnitudes in the low bytes of the lanes and the signs in the
// high bytes; magnitude * 16 + sign assembles a lane (the fields do not overlap).
__device__ __forceinline__ uint2 e4m3x4_to_bf16(uint32_t w) {
  const uint32_t m = w & 0x7F7F7F7Fu, s = w & 0x80808080u;
  const uint32_t lo = __byte_perm(m, 0u, 0x4140) * 16u + __byte_perm(s, 0u, 0x1404);
  const uint32_t hi = __byte_perm(m, 0u, 0x4342) * 16u + __byte_perm(s, 0u, 0x3424);
  return make_uint2(bf16x2_times_2p120(lo), bf16x2_times_2p120(hi));
}

template <int MODE, bool F8>
__global__ void __launch_bounds__(threads_of<MODE, F8>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TL_DECL;
  TL_START();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = smem + (size_t)a.w_stages * a.w_slot_bytes;
  uint8_t* fring = xring + (size_t)a.x_stages * a.x_slot_bytes;
  SmemTail* tail = reinterpret_cast<SmemTail*>(fring + (F8 ? (size_t)a.f_stages * a.f_slot_bytes : 0));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int SW = a.w_stages, SX = a.x_stages, SF = F8 ? a.f_stages : 1;
  constexpr bool kEpiConverts = conv_threads<MODE>() == 0;  // E4M3: epilogue warps convert
  constexpr int kConvAll = kEpiConverts ? kEpiWarps * 32 : conv_threads<MODE>();  // converting threads
  // The weight operand is A (128-row tiles) except for the LM head, where it is B.
  constexpr bool kWeightIsA = MODE != GEMM_LMSTATS;

  // Tile coordinates.  The token box (LM head: token group) is the fastest-varying index of
  // blockIdx.x: the zt CTAs that stream the same weight tile are launched together, so the
  // tile crosses HBM once and the other CTAs' reads hit L2.
  const int zt = a.zt > 0 ? a.zt : 1;
  const int bx = blockIdx.x / zt, bz = blockIdx.x - bx * zt;
  int a_row[2];
  bool a_ok[2];
  int b_row;
  constexpr bool kCluster = MODE == GEMM_QKV;
  if (MODE == GEMM_RED_ADD || kCluster) {
    a_row[0] = bx * a.na * 128;
    a_row[1] = a_row[0] + 128;
    b_row = bz * a.nbox;
    a_ok[0] = a_row[0] < a.a_rows;
    a_ok[1] = a.na > 1 && a_row[1] < a.a_rows;
  } else if (MODE == GEMM_SWIGLU) {
    a_row[0] = bx * 128;
    a_row[1] = a.F + bx * 128;
    b_row = bz * a.nbox;
    a_ok[0] = a_ok[1] = true;
  } else {
    a_row[0] = bz * a.na * 128;
    a_row[1] = a_row[0] + 128;
    b_row = bx * a.nbox;
    a_ok[0] = a_row[0] < a.T;
    a_ok[1] = a.na > 1 && a_row[1] < a.T;
  }
  const int kb0 = (int)(((long long)blockIdx.y * a.k_blocks) / a.splits);
  const int kb1 = (int)(((long long)(blockIdx.y + 1) * a.k_blocks) / a.splits);
  const int nk = kb1 - kb0;
  const uint32_t ncols = a.na == 2 ? 512u : 256u;
  const uint32_t a_bytes = (a_ok[0] ? a.a_tile_bytes : 0u) + (a_ok[1] ? a.a_tile_bytes : 0u);
  const uint32_t b_bytes = a.nbox * 128u;
  const uint64_t lim = wait_limit(a.wait_ns);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(smem_u32(&tail->wfull[s]), F8 ? kConvAll / 32 : 1);
      mbar_init(smem_u32(&tail->wempty[s]), 1);
    }
    for (int s = 0; F8 && s < SF; ++s) {
      mbar_init(smem_u32(&tail->ffull[s]), 1);
      mbar_init(smem_u32(&tail->fempty[s]), kConvAll / 32);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(smem_u32(&tail->xfull[s]), 1);
      mbar_init(smem_u32(&tail->xempty[s]), 1);
    }
    mbar_init(smem_u32(&tail->accf), 1);
    mbar_init(smem_u32(&tail->drain), 1);
    if (kCluster) mbar_init(smem_u32(&tail->cfull), a.splits);
    tail->abort = 0;
    tail->w_issued = tail->x_issued = 0;
    tail->mma_issued = 0;
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
  if (kCluster) cluster_arrive_relaxed();  // this CTA's mbarriers are initialised
  const uint32_t tmem = tail->tmem_addr;
  volatile int* abort = &tail->abort;
  pdl_trigger();

  // E4M3 stream, converters (the extra converter warps, or in the q/k/v kernel the epilogue
  // warps during the main loop): stage `it` of codes (rows of 64
  // bytes, tile after tile) becomes the bf16 operand in converted slot it % SW, 128-byte
  // swizzled: row r, 16-byte chunk c at r * 128 + ((c ^ (r & 7)) << 4).  Item e = (row,
  // 16-code part): one 16-byte load and two 16-byte stores (chunks 2 * part and
  // 2 * part + 1).  A thread loads all its items of a stage before converting; each warp
  // then fences its stores for the async proxy and one lane signals the MMA warp and the
  // producer (barrier counts = converting warps).  ct: 0 .. kConvAll - 1.
  auto convert_stages = [&](int ct) {
    constexpr int kItems = (256 * 4 + kConvAll - 1) / kConvAll;  // per thread, largest stage
    const int rows = kWeightIsA ? ((a_ok[0] ? 128 : 0) + (a_ok[1] ? 128 : 0)) : a.nbox;
    for (int it = 0; it < nk; ++it) {
      const int s = it % SF, sw = it % SW;
      if (!mbar_wait_bounded(smem_u32(&tail->ffull[s]), (uint32_t)(it / SF) & 1u, abort, a.err,
                             DEV_TIMEOUT_CONVERT, lim))
        break;
      if (it >= SW && !mbar_wait_bounded(smem_u32(&tail->wempty[sw]), ((uint32_t)(it / SW) & 1u) ^ 1u,
                                         abort, a.err, DEV_TIMEOUT_CONVERT, lim))
        break;
      const uint8_t* src = fring + (size_t)s * a.f_slot_bytes;
      uint8_t* dst = wring + (size_t)sw * a.w_slot_bytes;
      uint4 v[kItems];
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int e = ct + j * kConvAll;
        if (e < rows * 4) v[j] = *reinterpret_cast<const uint4*>(src + (e >> 2) * 64 + (e & 3) * 16);
      }
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int e = ct + j * kConvAll;
        if (e >= rows * 4) continue;
        const int row = e >> 2, part = e & 3;
        const uint2 p0 = e4m3x4_to_bf16(v[j].x), p1 = e4m3x4_to_bf16(v[j].y);
        const uint2 p2 = e4m3x4_to_bf16(v[j].z), p3 = e4m3x4_to_bf16(v[j].w);
        uint8_t* rb = dst + row * 128;
        const int sw7 = row & 7;
        *reinterpret_cast<uint4*>(rb + (((2 * part) ^ sw7) << 4)) = make_uint4(p0.x, p0.y, p1.x, p1.y);
        *reinterpret_cast<uint4*>(rb + (((2 * part + 1) ^ sw7) << 4)) = make_uint4(p2.x, p2.y, p3.x, p3.y);
      }
      fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&tail->wfull[sw]));
        mbar_arrive(smem_u32(&tail->fempty[s]));
      }
    }
  };

  if (warp == 0 || warp == 2 + kEpiWarps) {
    // Producers: warp 0 streams the weight operand, the last warp the activation operand.
    const bool weights = warp == 0;
    if (lane == 0) {
      if (!weights) pdl_wait();  // activations are written by the previous kernel
      // E4M3: the weight loads fill the staging ring with codes (one byte per element).
      const bool codes = F8 && weights;
      const int S = codes ? SF : weights ? SW : SX;
      uint8_t* ring = codes ? fring : weights ? wring : xring;
      const uint32_t slot = codes ? a.f_slot_bytes : weights ? a.w_slot_bytes : a.x_slot_bytes;
      uint64_t* full = codes ? tail->ffull : weights ? tail->wfull : tail->xfull;
      uint64_t* empty = codes ? tail->fempty : weights ? tail->wempty : tail->xempty;
      const bool is_a = weights == kWeightIsA;
      const uint64_t pol = weights ? policy_evict_first() : policy_evict_last();
      const uint32_t bytes = (is_a ? a_bytes : b_bytes) >> (codes ? 1 : 0);
      const uint32_t tile_bytes = a.a_tile_bytes >> (codes ? 1 : 0);
      int issued = 0;
      for (int it = 0; it < nk; ++it) {
        const int s = it % S;
        if (it >= S && !mbar_wait_bounded(smem_u32(&empty[s]), ((uint32_t)(it / S) & 1u) ^ 1u,
                                          abort, a.err, DEV_TIMEOUT_PRODUCER, lim))
          break;
        const uint32_t fb = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(ring + (size_t)s * slot);
        const int kb = kb0 + it;
        const bool packed = weights && a.w_packed;
        // Row-major: (x = k offset, y = row).  Tile-major: tile (row / tile_rows, kb) is
        // one contiguous box at y = (tile * k_blocks + kb) * tile_rows, x = 0.
        const int kx = packed ? 0 : kb * 64;
        mbar_arrive_expect_tx(fb, bytes);
        if (is_a) {
          const int y0 = packed ? ((a_row[0] >> 7) * a.k_blocks + kb) * 128 : a_row[0];
          const int y1 = packed ? ((a_row[1] >> 7) * a.k_blocks + kb) * 128 : a_row[1];
          if (a_ok[0]) tma_load_2d(dst, &mapA, fb, kx, y0, pol);
          if (a_ok[1]) tma_load_2d(dst + tile_bytes, &mapA, fb, kx, y1, pol);
        } else {
          const int y = packed ? ((b_row / a.nbox) * a.k_blocks + kb) * a.nbox : b_row;
          tma_load_2d(dst, &mapB, fb, kx, y, pol);
        }
        ++issued;
      }
      if (weights)
        tail->w_issued = issued;
      else
        tail->x_issued = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, a.nbox);
      bool ok = true;
      for (int it = 0; it < nk; ++it) {
        const int sw = it % SW, sx = it % SX;
        if (!mbar_wait_bounded(smem_u32(&tail->wfull[sw]), (uint32_t)(it / SW) & 1u, abort, a.err,
                               DEV_TIMEOUT_MMA, lim) ||
            !mbar_wait_bounded(smem_u32(&tail->xfull[sx]), (uint32_t)(it / SX) & 1u, abort, a.err,
                               DEV_TIMEOUT_MMA, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tail->mma_issued = 1;
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
  } else if (F8 && warp >= 3 + kEpiWarps) {
    convert_stages((int)threadIdx.x - kThreads);
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // Epilogue warps 2..9: warp w may only touch TMEM lanes 32*(w%4) .. +31, so each
    // lane quarter has two warps; they take alternate 16-column chunks.  The outputs may
    // still be read by the previous kernel until it completes.  In the E4M3 q/k/v kernel they
    // first convert the weight stream.
    if (F8 && kEpiConverts) convert_stages((int)threadIdx.x - 64);
    pdl_wait();
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int te = threadIdx.x - 64;  // 0..255 over the epilogue warps
    const int nchunk = a.nbox / 16;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    // E4M3 stream: the scale of the weight row of this thread's TMEM lane in accumulator i
    // (weights on M); 1 for bf16 weights.
    auto row_scale = [&](int i) { return F8 ? __ldg(a.wscale + a_row[i] + r) : 1.0f; };
    // Every epilogue thread waits for the accumulator (bounded); the warp-wide TMEM reads
    // then follow one decision for all eight warps, taken after a barrier from the shared
    // abort flag (set by any wait of the CTA that gave up).
    auto accum_ready = [&]() {
      mbar_wait_bounded(smem_u32(&tail->accf), 0, abort, a.err, DEV_TIMEOUT_EPILOGUE, lim);
      if (te == 0) TL_STAMP(tail->tl_tw);
      epilogue_sync();
      return *abort == 0;
    };
    if (kCluster) {
      // Split-K sum inside the cluster, through L2.  Per 128-row accumulator ("round"):
      // every CTA writes its fp32 partial tile [token][128 columns] straight from TMEM to
      // its region of the exchange workspace (coalesced: a warp covers a 128-byte row
      // segment) and signals all peers' cfull (release, cluster scope); CTA `rank` then
      // sums tokens [tlo, tlo + ntok) of the tile over the splits in split order with
      // 16-byte L2 loads.  Regions are per round, so nothing is overwritten while read.
      const bool ok = nk > 0 && accum_ready();
      tc_fence_after();
      const int S = a.splits;
      const int rank = (int)cluster_ctarank();
      const int tlo = rank * a.nbox / S, ntok = (rank + 1) * a.nbox / S - tlo;
      const uint32_t cfull = smem_u32(&tail->cfull);
      const int P = a.dP ? *a.dP : 0;
      // Exchange region of split c, round i for this cluster (tile x, token block z).
      auto region = [&](int i, int c) {
        return a.xws + ((((size_t)bz * (gridDim.x / zt) + bx) * 2 + i) * S + c) *
                           (size_t)a.nbox * 128;
      };
      cluster_wait();  // every peer's mbarriers are initialised
      int round = 0;
      for (int i = 0; i < 2; ++i) {
        if (!a_ok[i]) continue;  // the same for every CTA of the cluster
        if (ok) {
          float* mine = region(i, rank);
          const float sc = row_scale(i);
          for (int ci = half; ci < nchunk; ci += 2) {
            float v[16];
            tmem_ld16(lane_base + (uint32_t)(i * 256 + ci * 16), v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              __stcg(mine + (size_t)(ci * 16 + j) * 128 + r, F8 ? v[j] * sc : v[j]);
          }
          __threadfence();
        }
        epilogue_sync();
        if (te == 0)
          for (int c = 0; c < S; ++c) mbar_arrive_cluster(mapa_shared(cfull, (uint32_t)c));
        if (mbar_wait_cluster_bounded(cfull, (uint32_t)round & 1u, abort, a.err,
                                      DEV_TIMEOUT_CLUSTER, lim)) {
          const float* src[kMaxClusterSplits];
#pragma unroll
          for (int c = 0; c < kMaxClusterSplits; ++c) src[c] = region(i, c < S ? c : 0);
          const int dh = a.dh, hdh = dh >> 1, per_head = dh >> 3;
          const int G = a.H / a.Hk;
          const int head0 = a_row[i] / dh;  // first head of this 128-row tile
          const int vfirst = a.H + a.Hk;    // first value head
          constexpr int kStep = kEpiWarps * 32;
          // (1) q and k.  Work item e: token tlo + e/16, columns j..j+3 of a head and their
          // rotation partners j+dh/2..+3.  Two items per pass keep 4*S loads in flight.
          const int nitem = head0 < vfirst ? ntok * 16 : 0;
          for (int e0 = te; e0 < nitem; e0 += 2 * kStep) {
            float4 v[2][2][kMaxClusterSplits];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = e0 + h * kStep;
              const int tt = tlo + (e >> 4), u = e & 15;
              const int hd = u / per_head, j = (u - hd * per_head) * 4;
              const int off = tt * 128 + hd * dh + j;
              if (e < nitem && head0 + hd < vfirst) {
#pragma unroll
                for (int c = 0; c < kMaxClusterSplits; ++c)
                  if (c < S) {
                    v[h][0][c] = __ldcg(reinterpret_cast<const float4*>(src[c] + off));
                    v[h][1][c] = __ldcg(reinterpret_cast<const float4*>(src[c] + off + hdh));
                  }
              }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = e0 + h * kStep;
              const int tt = tlo + (e >> 4), u = e & 15;
              const int t = b_row + tt;
              const int hd = u / per_head, j = (u - hd * per_head) * 4;
              const int head = head0 + hd;
              if (e >= nitem || t >= a.T || head >= vfirst) continue;
              float4 x1 = v[h][0][0], x2 = v[h][1][0];
#pragma unroll
              for (int c = 1; c < kMaxClusterSplits; ++c)
                if (c < S) {
                  x1.x += v[h][0][c].x; x1.y += v[h][0][c].y; x1.z += v[h][0][c].z; x1.w += v[h][0][c].w;
                  x2.x += v[h][1][c].x; x2.y += v[h][1][c].y; x2.z += v[h][1][c].z; x2.w += v[h][1][c].w;
                }
              // RoPE, rotate-half form, at absolute position P + bi.
              const int bi = a.pos_linear ? t : t % a.Bq;
              const float4 cs = *reinterpret_cast<const float4*>(a.cos_t + (size_t)(P + bi) * hdh + j);
              const float4 sn = *reinterpret_cast<const float4*>(a.sin_t + (size_t)(P + bi) * hdh + j);
              const float4 y1 = make_float4(x1.x * cs.x - x2.x * sn.x, x1.y * cs.y - x2.y * sn.y,
                                            x1.z * cs.z - x2.z * sn.z, x1.w * cs.w - x2.w * sn.w);
              const float4 y2 = make_float4(x2.x * cs.x + x1.x * sn.x, x2.y * cs.y + x1.y * sn.y,
                                            x2.z * cs.z + x1.z * sn.z, x2.w * cs.w + x1.w * sn.w);
              // q: group-major [Hk][T][G][dh]; k: [row][Hk][dh], row = cache position or t.
              const size_t kv_row = a.kv_to_cache ? (size_t)(P + bi) : (size_t)t;
              bf16* dst = head < a.H
                              ? a.q + (((size_t)(head / G) * a.T + t) * G + head % G) * dh
                              : a.kdst + (kv_row * a.Hk + (head - a.H)) * dh;
              store4_bf16(dst + j, y1.x, y1.y, y1.z, y1.w);
              store4_bf16(dst + j + hdh, y2.x, y2.y, y2.z, y2.w);
            }
          }
          // (2) v, stored transposed: V^T[(head - vfirst) * dh + d][column], column = cache
          // position or t.  Work item: 4 columns of the tile x 8 consecutive tokens, so the
          // stores are 16-byte runs along the position axis.
          const int vcol0 = max(vfirst * dh - a_row[i], 0);
          if (vcol0 < 128) {
            const int nf4 = (128 - vcol0) / 4, ntg = (ntok + 7) / 8;
            for (int e = te; e < nf4 * ntg; e += kStep) {
              const int f = vcol0 + (e % nf4) * 4, tt0 = tlo + (e / nf4) * 8;
              float4 acc[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tt0 + k >= tlo + ntok) continue;
                const int off = (tt0 + k) * 128 + f;
                float4 w[kMaxClusterSplits];
#pragma unroll
                for (int c = 0; c < kMaxClusterSplits; ++c)
                  if (c < S) w[c] = __ldcg(reinterpret_cast<const float4*>(src[c] + off));
                acc[k] = w[0];
#pragma unroll
                for (int c = 1; c < kMaxClusterSplits; ++c)
                  if (c < S) {
                    acc[k].x += w[c].x; acc[k].y += w[c].y; acc[k].z += w[c].z; acc[k].w += w[c].w;
                  }
              }
              const int vrow = a_row[i] + f - vfirst * dh;  // (value head) * dh + d
              const int t0 = b_row + tt0;
              const int col0 = a.kv_to_cache ? P + t0 % a.Bq : t0;
              const bool whole = tt0 + 8 <= tlo + ntok && t0 + 8 <= a.T && (col0 & 7) == 0 &&
                                 (!a.kv_to_cache || t0 % a.Bq + 8 <= a.Bq);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                bf16* vr = a.vdst + (size_t)(vrow + q4) * a.ldv;
                float x[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  x[k] = q4 == 0 ? acc[k].x : q4 == 1 ? acc[k].y : q4 == 2 ? acc[k].z : acc[k].w;
                if (whole) {
                  uint4 o;
                  __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
                  for (int k = 0; k < 4; ++k) h2[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
                  *reinterpret_cast<uint4*>(vr + col0) = o;
                } else {
#pragma unroll
                  for (int k = 0; k < 8; ++k) {
                    const int t = t0 + k;
                    if (tt0 + k >= tlo + ntok || t >= a.T) continue;
                    vr[a.kv_to_cache ? P + t % a.Bq : t] = __float2bfloat16_rn(x[k]);
                  }
                }
              }
            }
          }
        }
        ++round;
      }
    } else if (nk > 0 && accum_ready()) {
      tc_fence_after();
      float* stage = reinterpret_cast<float*>(smem);
      if (MODE == GEMM_RED_ADD) {
        for (int i = 0; i < 2; ++i) {
          if (!a_ok[i]) continue;
          if (a.atomic) {  // standalone accumulate: fp32 atomics into out_f32
            const int n = a_row[i] + r;
            const float sc = row_scale(i);
            for (int ci = half; ci < nchunk; ci += 2) {
              float v[16];
              tmem_ld16(lane_base + (uint32_t)(i * 256 + ci * 16), v);
              for (int j = 0; j < 16; ++j) {
                const int t = b_row + ci * 16 + j;
                if (t < a.T) atomicAdd(a.out_f32 + (size_t)t * a.ldo + n, F8 ? v[j] * sc : v[j]);
              }
            }
            continue;
          }
          // This split's partial sums, stored straight from the TMEM registers: a warp's
          // lanes are 32 consecutive output features, so every store instruction writes one
          // whole 128-byte line of a token's row.  The consumer adds the splits in a fixed
          // order.
          const float sc = row_scale(i);
          float* base = a.out_f32 + (size_t)blockIdx.y * a.split_stride + a_row[i] + r;
          for (int ci = half; ci < nchunk; ci += 2) {
            float v[16];
            tmem_ld16(lane_base + (uint32_t)(i * 256 + ci * 16), v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = b_row + ci * 16 + j;
              if (t < a.T) base[(size_t)t * a.ldo] = F8 ? v[j] * sc : v[j];
            }
          }
        }
      } else if (MODE == GEMM_SWIGLU) {
        const float sg = row_scale(0), su = row_scale(1);
        for (int ci = half; ci < nchunk; ci += 2) {
          float g[16], u[16];
          tmem_ld16x2(lane_base + (uint32_t)(ci * 16), lane_base + (uint32_t)(256 + ci * 16), g, u);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (F8) {
              g[j] *= sg;
              u[j] *= su;
            }
            stage[(ci * 16 + j) * 128 + r] = __fdividef(g[j], 1.0f + __expf(-g[j])) * u[j];
          }
        }
        epilogue_sync();
        bf16* base = a.out_bf16 + a_row[0];
        for (int e = te; e < a.nbox * 16; e += kEpiWarps * 32) {
          const int tt = e >> 4, c8 = (e & 15) * 8;
          if (b_row + tt < a.T) {
            const float4 x0 = *reinterpret_cast<const float4*>(stage + tt * 128 + c8);
            const float4 x1 = *reinterpret_cast<const float4*>(stage + tt * 128 + c8 + 4);
            uint4 o;
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&o);
            h2[0] = __floats2bfloat162_rn(x0.x, x0.y);
            h2[1] = __floats2bfloat162_rn(x0.z, x0.w);
            h2[2] = __floats2bfloat162_rn(x1.x, x1.y);
            h2[3] = __floats2bfloat162_rn(x1.z, x1.w);
            *reinterpret_cast<uint4*>(base + (size_t)(b_row + tt) * a.ldh + c8) = o;
          }
        }
      } else {
        // Each warp pair (same lane quarter) scans alternate 16-column chunks of the
        // 256-row vocabulary tile; the two running (max, sum exp, argmax) states of a
        // token are merged through shared memory.
        const int vt = bx;
        float* xm = stage;
        float* xs = stage + 128;
        int* xi = reinterpret_cast<int*>(stage + 256);
        for (int i = 0; i < 2; ++i) {
          if (!a_ok[i]) continue;
          const int t = a_row[i] + r;
          float m = -INFINITY, ssum = 0.f;
          int idx = 0x7fffffff;
          for (int ci = half; ci < nchunk; ci += 2) {
            float v[16];
            __syncwarp();
            tmem_ld16(lane_base + (uint32_t)(i * 256 + ci * 16), v);
            float cm = -INFINITY;
            int cidx = 0;
            float ws[16];  // E4M3 stream: scales of these 16 vocabulary rows (same for the warp)
            if (F8) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int id = b_row + ci * 16 + j;
                ws[j] = id < a.V ? __ldg(a.wscale + id) : 0.f;
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int id = b_row + ci * 16 + j;
              if (F8) v[j] *= ws[j];
              v[j] = (id < a.V && id != a.mask_id) ? v[j] * a.scale : -INFINITY;
              if (v[j] > cm) { cm = v[j]; cidx = id; }  // strict: lowest id wins ties
            }
            if (cm != -INFINITY) {
              const float nm = fmaxf(m, cm);
              float acc = (m == -INFINITY) ? 0.f : ssum * __expf(m - nm);
#pragma unroll
              for (int j = 0; j < 16; ++j) acc += __expf(v[j] - nm);
              if (cm > m) idx = cidx;
              m = nm;
              ssum = acc;
            }
          }
          if (half == 1) {
            xm[r] = m;
            xs[r] = ssum;
            xi[r] = idx;
          }
          epilogue_sync();
          if (half == 0) {
            const float m1 = xm[r], s1 = xs[r];
            const int i1 = xi[r];
            if (m1 != -INFINITY) {
              if (m == -INFINITY) {
                m = m1; ssum = s1; idx = i1;
              } else {
                const float nm = fmaxf(m, m1);
                ssum = ssum * __expf(m - nm) + s1 * __expf(m1 - nm);
                idx = m > m1 ? idx : (m1 > m ? i1 : min(idx, i1));
                m = nm;
              }
            }
            if (t < a.T) {
              const size_t o = (size_t)vt * a.part_ld + t;
              a.part_m[o] = m;
              a.part_s[o] = ssum;
              a.part_i[o] = m == -INFINITY ? 0 : idx;
            }
          }
          epilogue_sync();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort) {
    // A bounded wait gave up in this CTA.  Before its shared memory and TMEM are released,
    // wait (bounded) for every TMA copy it issued and every MMA it started.
    if (lane == 0 && (warp == 0 || warp == 2 + kEpiWarps)) {
      const bool weights = warp == 0;
      const int S = weights ? (F8 ? SF : SW) : SX;
      const int n = weights ? tail->w_issued : tail->x_issued;
      uint64_t* full = weights ? (F8 ? tail->ffull : tail->wfull) : tail->xfull;
      for (int s = 0; s < S && s < n; ++s) {
        const int last = s + ((n - 1 - s) / S) * S;  // the last load issued into slot s
        mbar_wait_drain(smem_u32(&full[s]), (uint32_t)(last / S) & 1u);
      }
    } else if (lane == 0 && warp == 1 && tail->mma_issued) {
      mma_commit(smem_u32(&tail->drain));
      mbar_wait_drain(smem_u32(&tail->drain), 0);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (kCluster) {
    // No CTA leaves while a peer may still signal its mbarriers: the epilogue warps closed
    // the start phase of the cluster barrier, the other warps close it here; then the whole
    // cluster meets once more.  Every wait before this point is bounded.
    if (warp < 2 || warp >= 2 + kEpiWarps) cluster_wait();  // producers, MMA, converters
    cluster_arrive_release();
    cluster_wait();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
#ifdef LOPA_TIMELINE
  if (threadIdx.x == 0) tl_tw = tail->tl_tw;
#endif
  TL_END(tl::GEMM + MODE);
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

// Smallest ring size that can hold a staged output tile of nbox tokens x 128 columns.
uint32_t stage_bytes(int mode, int nbox) {
  return mode == GEMM_LMSTATS ? 384 * 4 : (uint32_t)nbox * 128 * 4;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, char* errbuf, size_t errlen, uint64_t ld) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  if (ld == 0) ld = cols;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0 || ld < cols) {
    snprintf(errbuf, errlen, "tensor map base/stride not 16-byte aligned");
    return false;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
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

// 2-D tensor map over a row-major [rows][cols] byte matrix (E4M3 codes) with a box of
// box_rows x 64 bytes, no swizzle (the converter warps read it row by row); reads outside
// [rows][cols] return zeros.
bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows, char* errbuf, size_t errlen) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || cols % 16 != 0) {
    snprintf(errbuf, errlen, "E4M3 tensor map base/stride not 16-byte aligned");
    return false;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled (u8) failed (%d) rows=%llu cols=%llu box=%u",
             (int)r, (unsigned long long)rows, (unsigned long long)cols, box_rows);
    return false;
  }
  return true;
}

int gemm_max_smem() { return kMaxSmem; }

template <int MODE, bool F8>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(gemm_kernel<MODE, F8>);
}

// Indexed by [E4M3 stream][mode].
const void* const kKernels[2][4] = {
    {kernel_ptr<GEMM_RED_ADD, false>(), kernel_ptr<GEMM_SWIGLU, false>(),
     kernel_ptr<GEMM_LMSTATS, false>(), kernel_ptr<GEMM_QKV, false>()},
    {kernel_ptr<GEMM_RED_ADD, true>(), kernel_ptr<GEMM_SWIGLU, true>(),
     kernel_ptr<GEMM_LMSTATS, true>(), kernel_ptr<GEMM_QKV, true>()}};

cudaError_t gemm_set_smem_limits() {
  for (const void* k : kKernels[0]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  for (const void* k : kKernels[1]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  return set_uniform_carveout();
}

cudaError_t gemm_set_carveout() {
  for (const auto& row : kKernels)
    for (const void* k : row) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int gemm_cluster_capacity(int mode, int cs, size_t smem, bool w8) {
  if (mode < 0 || mode > GEMM_QKV || cs < 1 || cs > kMaxClusterSplits) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, (unsigned)cs, 1);
  cfg.blockDim = dim3(w8 ? threads_of<GEMM_QKV, true>() : kThreads);
  if (mode != GEMM_QKV) cfg.blockDim = dim3(w8 ? threads_of<GEMM_RED_ADD, true>() : kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)cs;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kKernels[w8 ? 1 : 0][mode], &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// act: [act_rows_alloc][K] bf16 activations (T valid rows); w: [n_rows_w][K] bf16.
const char* plan_gemm(GemmLaunch* L, int mode, const void* act, int act_rows_alloc, int T,
                      const void* w, int n_rows_w, int K, int na, int splits, int tok_box,
                      int num_sms, bool w_packed, const float* w_scale) {
  static thread_local char err[256];
  const bool w8 = w_scale != nullptr;
  // Packed weights are viewed as [tiles * K/64 * tile_rows][64]: one box = one tile.
  auto weight_map = [&](CUtensorMap* map, int tile_rows) {
    const uint64_t tiles = (uint64_t)(n_rows_w + tile_rows - 1) / tile_rows;
    if (w8)
      return w_packed ? make_tmap_u8(map, w, tiles * (K / 64) * tile_rows, 64, tile_rows, err, sizeof(err))
                      : make_tmap_u8(map, w, n_rows_w, K, tile_rows, err, sizeof(err));
    if (!w_packed) return make_tmap_bf16(map, w, n_rows_w, K, tile_rows, err, sizeof(err));
    return make_tmap_bf16(map, w, tiles * (K / 64) * tile_rows, 64, tile_rows, err, sizeof(err));
  };
  memset(L, 0, sizeof(*L));
  GemmArgs& a = L->args;
  if (K % 64 != 0 || K <= 0) return "GEMM K must be a positive multiple of 64";
  if (T <= 0) return "GEMM needs at least one token row";
  a.mode = mode;
  a.w8 = w8 ? 1 : 0;
  a.wscale = w_scale;
  a.w_packed = w_packed ? 1 : 0;
  a.k_blocks = K / 64;
  a.T = T;
  a.a_tile_bytes = 128 * 128;  // 128 rows x 64 bf16
  if (mode == GEMM_LMSTATS) {
    a.na = na;
    a.nbox = 256;
    a.a_rows = T;
    a.splits = 1;
    if (!make_tmap_bf16(&L->mapA, act, act_rows_alloc, K, 128, err, sizeof(err))) return err;
    if (!weight_map(&L->mapB, 256)) return err;
    a.zt = (T + na * 128 - 1) / (na * 128);
    L->grid = dim3((n_rows_w + 255) / 256 * a.zt, 1, 1);
    a.w_slot_bytes = round1k(a.nbox * 128);
    a.x_slot_bytes = round1k(a.na * a.a_tile_bytes);
  } else {
    if (tok_box < 16 || tok_box > 256 || tok_box % 16 != 0) return "token box must be 16..256, multiple of 16";
    if (n_rows_w % 128 != 0) return "GEMM N must be a multiple of 128";
    a.na = (mode == GEMM_SWIGLU) ? 2 : na;
    if (a.na != 1 && a.na != 2) return "GEMM tiles per CTA must be 1 or 2";
    a.F = n_rows_w / 2;
    a.nbox = tok_box;
    a.a_rows = n_rows_w;
    a.splits = (mode == GEMM_SWIGLU) ? 1 : splits;
    if (a.splits < 1) a.splits = 1;
    if (gemm_mode_clustered(mode)) {
      // The K-splits of a tile are one cluster: 1, 2 or 4 CTAs, each with >= 1 K block.
      if ((a.splits & (a.splits - 1)) != 0 || a.splits > kMaxClusterSplits ||
          a.splits > a.k_blocks)
        return "cluster split count must be 1, 2 or 4 and at most K/64";
    } else if (a.splits > a.k_blocks) {
      a.splits = a.k_blocks;
    }
    if (!weight_map(&L->mapA, 128)) return err;
    if (!make_tmap_bf16(&L->mapB, act, act_rows_alloc, K, tok_box, err, sizeof(err))) return err;
    const int gx = (mode == GEMM_SWIGLU) ? (n_rows_w / 2) / 128 : (n_rows_w + a.na * 128 - 1) / (a.na * 128);
    a.zt = (T + tok_box - 1) / tok_box;
    L->grid = dim3(gx * a.zt, a.splits, 1);
    a.w_slot_bytes = round1k(a.na * a.a_tile_bytes);
    a.x_slot_bytes = round1k(a.nbox * 128);
  }
  (void)num_sms;
  // Activations come from L2 (short latency): 3 slots, more when they are small.  The
  // weight ring takes the rest of shared memory.  E4M3 stream: two converted bf16 slots
  // and the rest as the staging ring of codes (the bytes in flight from HBM).
  const int budget = kMaxSmem - 1024 - (int)sizeof(SmemTail) - 64;
  a.x_stages = a.x_slot_bytes <= 8192 ? 6 : 3;
  if (w8) {
    a.f_slot_bytes = a.w_slot_bytes / 2;  // one byte per element instead of two (1 KB multiple)
    a.w_stages = 2;
    a.f_stages = (budget - a.x_stages * (int)a.x_slot_bytes - a.w_stages * (int)a.w_slot_bytes) /
                 (int)a.f_slot_bytes;
    if (a.f_stages > kMaxStages) a.f_stages = kMaxStages;
    if (a.f_stages < 2) return "GEMM tile does not fit in shared memory";
  } else {
    a.w_stages = (budget - a.x_stages * (int)a.x_slot_bytes) / (int)a.w_slot_bytes;
    if (a.w_stages > kMaxStages) a.w_stages = kMaxStages;
    if (a.w_stages < 2) return "GEMM tile does not fit in shared memory";
  }
  const size_t rings = (size_t)a.w_stages * a.w_slot_bytes + (size_t)a.x_stages * a.x_slot_bytes +
                       (size_t)a.f_stages * a.f_slot_bytes;
  if (rings < stage_bytes(mode, a.nbox)) return "GEMM output tile does not fit in the staging area";
  L->smem = 1024 + rings + sizeof(SmemTail) + 64;
  return "";
}

template <bool F8>
cudaError_t launch_gemm_t(const GemmLaunch& L, cudaStream_t s) {
  switch (L.args.mode) {
    case GEMM_RED_ADD:
      return launch_pdl(gemm_kernel<GEMM_RED_ADD, F8>, L.grid, dim3(threads_of<GEMM_RED_ADD, F8>()),
                        L.smem, s, L.mapA, L.mapB, L.args);
    case GEMM_SWIGLU:
      return launch_pdl(gemm_kernel<GEMM_SWIGLU, F8>, L.grid, dim3(threads_of<GEMM_SWIGLU, F8>()),
                        L.smem, s, L.mapA, L.mapB, L.args);
    case GEMM_LMSTATS:
      return launch_pdl(gemm_kernel<GEMM_LMSTATS, F8>, L.grid, dim3(threads_of<GEMM_LMSTATS, F8>()),
                        L.smem, s, L.mapA, L.mapB, L.args);
    case GEMM_QKV:
      return launch_pdl_cluster(gemm_kernel<GEMM_QKV, F8>, L.grid, dim3(threads_of<GEMM_QKV, F8>()),
                                L.smem, s, dim3(1, L.args.splits, 1), L.mapA, L.mapB, L.args);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t s) {
  return L.args.w8 ? launch_gemm_t<true>(L, s) : launch_gemm_t<false>(L, s);
}

}  // namespace lopa
