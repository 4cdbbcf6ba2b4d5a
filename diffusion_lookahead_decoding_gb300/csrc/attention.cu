// Branch-isolated attention for the verification forward.
//
// "SJTU x Huawei Xiaoyi release LoPA", section "Core design of LoPA": all candidate
// branches are verified in one forward because attention is isolated between branches.
// Query (b, i, h) attends to the committed prefix keys [0, P) - shared by every branch -
// and to the keys of its own branch's block only, bidirectionally inside the block
// ("Decoding-efficiency revolution" blog, section 3.3: a branch sees the prompt and its
// own tokens, never another branch's).
//
// Layouts (written by the q/k/v projection epilogue):
//   q      [Hk][T][G][dh]   group-major: the rows of KV head g are (token t, head-in-group
//                           hg) pairs, t = b * Bq + i, so one K/V tile serves every query
//                           head of the group (grouped-query attention);
//   K      [pos][Hk][dh]    prefix cache; block keys [nb][Bk_stride][Hk][dh];
//   V^T    [Hk*dh][ld]      values stored transposed (position innermost), so a V tile is
//                           a K-major operand of P V;
//   out    [T][H*dh].
// Key tiles run over the prefix first, then over the block keys of the branches that a
// CTA's rows belong to, with a per-row branch mask.
//
// head_dim 128 runs on the 5th-generation tensor cores (tcgen05): a CTA owns 128 query
// rows (= TMEM lanes).  The softmax warps load Q into TMEM; one warp streams K / V^T tiles
// of 128 keys with TMA; one warp issues S = Q K^T (Q from TMEM) into a double-buffered TMEM
// tile and O += P V into a TMEM accumulator, with P read from TMEM as well: the softmax
// warps (one thread per row and key half) read S, compute P as a bf16 head and a bf16 tail
// (two MMAs keep P's fp32 accuracy), write it over S, and rescale O in TMEM only when a
// row's running maximum grows by more than 2^8 (the result is unchanged: O and the
// normaliser share the same reference).  Shared memory holds only the K / V^T ring.
// Eight softmax warps: two per TMEM lane quarter, each on half of the 128 keys.  A row
// tile's CTA walks its key tiles in sequence, so with a prefix of 4 or more key tiles
// the two CTAs of a cluster pair split the tiles and rank 0 merges the two softmax states
// (reference maximum, sum, O) through distributed shared memory; pairs are launched only
// when a prefix can reach that length and the pairs fit the SMs in one wave.
// head_dim 32 and 64 run on bf16 mma.sync with the same layouts.
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "timeline.cuh"

namespace lopa {

LOPA_TL_UNIT(attention)

namespace {

constexpr int kKeyTile = 64;

// Key-tile schedule shared by both kernels (KT keys per tile: 128 on the tensor-core path,
// 64 on mma.sync): prefix tiles [0, n_pre), then block-key tiles covering the scratch
// columns [kb_lo, kb_end) of the branches in [b_lo, b_hi].
struct KeySched {
  int Pk, n_pre, kb_lo, n_br;
};

template <int KT>
__device__ __forceinline__ KeySched key_sched(const AttnArgs& a, int b_lo, int b_hi) {
  KeySched k;
  k.Pk = a.pk_add + (a.dP ? *a.dP : 0);
  k.n_pre = (k.Pk + KT - 1) / KT;
  k.kb_lo = (a.causal ? 0 : b_lo) * a.Bk_stride;
  const int kb_end = b_hi * a.Bk_stride + a.Bk;
  k.n_br = a.Bk > 0 ? (kb_end - k.kb_lo + KT - 1) / KT : 0;
  return k;
}

// Key columns [lo, hi) of tile j (tile-local) that a row of branch br may see: the
// committed prefix, or the br-th branch's own block keys (with `causal`, the keys of
// blocks 0..br).
template <int KT>
__device__ __forceinline__ void visible_range(const AttnArgs& a, const KeySched& k, int j, int br,
                                              int& lo, int& hi) {
  if (j < k.n_pre) {
    lo = 0;
    hi = k.Pk - j * KT;
    return;
  }
  const int col0 = k.kb_lo + (j - k.n_pre) * KT;
  lo = (a.causal ? 0 : br * a.Bk_stride) - col0;
  hi = br * a.Bk_stride + a.Bk - col0;
}

// 2^x on the special-function unit (ex2.approx: relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// ================================================================ tcgen05 path (dh = 128)
constexpr int kTcRows = 128;
constexpr int kTcKeys = 128;     // keys per tile (the N of S = Q K^T)
constexpr int kTcStages = 3;     // K / V^T ring depth
constexpr int kTcSoftWarps = 8;  // two per TMEM lane quarter, each on half the keys
constexpr int kTcThreads = (2 + kTcSoftWarps) * 32;  // warp 0 TMA, warp 1 MMA, softmax
constexpr uint32_t kTcAtom = 128 * 64 * 2;  // one 128-byte-swizzled atom: 128 rows x 64 bf16
constexpr uint32_t kTcKBytes = 2 * kTcAtom;  // K tile: 128 keys x (two 64-wide halves of dh)
constexpr uint32_t kTcVBytes = 2 * kTcAtom;  // V^T tile: 128 (dh) x (two 64-key halves)
constexpr uint32_t kTcStageBytes = kTcKBytes + kTcVBytes;
constexpr uint32_t kTcOffTail = kTcStages * kTcStageBytes;
// TMEM columns: Q (bf16, two per column) [0, 64); S / P buffer b at 128 + 128 b (S as 128
// fp32 columns, overwritten in place by P); O (fp32) [384, 512).
constexpr uint32_t kTmQ = 0, kTmS = 128, kTmO = 384, kTmCols = 512;
constexpr float kLazyRescale = 8.0f;  // log2 units
// Split keys: a CTA pair (cluster of 2 along z) shares a row tile; when the prefix spans at
// least this many key tiles (512 keys), rank 0 takes the first half of the tiles and rank 1 the rest,
// and rank 0 merges the two softmax states through distributed shared memory.
constexpr int kSplitMinTiles = 4;
// Merge stash (in the freed K / V^T ring): O as [128 columns][128 rows] fp32, then the
// rows' reference maxima and sums.
constexpr int kExM = 128 * kTcRows, kExL = kExM + kTcRows;

struct TcTail {
  uint64_t qfull;
  uint64_t kvfull[kTcStages], kvempty[kTcStages];
  uint64_t sfull[2], pfull[2], pempty[2];
  uint64_t odone;
  uint64_t drain;  // after a wait gave up: completion of every MMA this CTA issued
  int kv_issued;   // K / V^T stages loaded by TMA
  int mma_issued;  // 1 once an MMA was issued
  float xmax[2][2][kTcRows];  // [buffer][key half][row]: half-row maxima
  float xsum[2][kTcRows];     // [key half][row]: half-row sums of P
  uint32_t tmem;
  int abort;
};
constexpr size_t kTcSmem = 1024 + kTcOffTail + sizeof(TcTail);

// The q map is not read by the kernel (the softmax warps load Q rows into TMEM); it is
// the valid stand-in address of the maps a launch does not use.
struct TcMaps {
  CUtensorMap q, kc, vtc, kb, vtb;
};

// Stores 8 / 16 32-bit words into consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
               "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// Loads 64 consecutive fp32 TMEM columns of this thread's lane (two 32x32b.x32 loads,
// one wait; threading the registers through the wait keeps every use after it).
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, float (&v)[64]) {
  uint32_t x[32], y[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
                 "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]),
                 "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]),
                 "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]),
                 "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
               : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(y[0]), "=r"(y[1]), "=r"(y[2]), "=r"(y[3]), "=r"(y[4]), "=r"(y[5]), "=r"(y[6]),
                 "=r"(y[7]), "=r"(y[8]), "=r"(y[9]), "=r"(y[10]), "=r"(y[11]), "=r"(y[12]), "=r"(y[13]),
                 "=r"(y[14]), "=r"(y[15]), "=r"(y[16]), "=r"(y[17]), "=r"(y[18]), "=r"(y[19]),
                 "=r"(y[20]), "=r"(y[21]), "=r"(y[22]), "=r"(y[23]), "=r"(y[24]), "=r"(y[25]),
                 "=r"(y[26]), "=r"(y[27]), "=r"(y[28]), "=r"(y[29]), "=r"(y[30]), "=r"(y[31])
               : "r"(ta + 32u));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5]), "+r"(x[6]),
                 "+r"(x[7]), "+r"(x[8]), "+r"(x[9]), "+r"(x[10]), "+r"(x[11]), "+r"(x[12]), "+r"(x[13]),
                 "+r"(x[14]), "+r"(x[15]), "+r"(x[16]), "+r"(x[17]), "+r"(x[18]), "+r"(x[19]),
                 "+r"(x[20]), "+r"(x[21]), "+r"(x[22]), "+r"(x[23]), "+r"(x[24]), "+r"(x[25]),
                 "+r"(x[26]), "+r"(x[27]), "+r"(x[28]), "+r"(x[29]), "+r"(x[30]), "+r"(x[31]),
                 "+r"(y[0]), "+r"(y[1]), "+r"(y[2]), "+r"(y[3]), "+r"(y[4]), "+r"(y[5]), "+r"(y[6]),
                 "+r"(y[7]), "+r"(y[8]), "+r"(y[9]), "+r"(y[10]), "+r"(y[11]), "+r"(y[12]), "+r"(y[13]),
                 "+r"(y[14]), "+r"(y[15]), "+r"(y[16]), "+r"(y[17]), "+r"(y[18]), "+r"(y[19]),
                 "+r"(y[20]), "+r"(y[21]), "+r"(y[22]), "+r"(y[23]), "+r"(y[24]), "+r"(y[25]),
                 "+r"(y[26]), "+r"(y[27]), "+r"(y[28]), "+r"(y[29]), "+r"(y[30]), "+r"(y[31])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(x[i]);
    v[32 + i] = __uint_as_float(y[i]);
  }
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T: A's 128 rows are the TMEM lanes, its K bf16
// values two per 32-bit column (element 2c in the low half of column c).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcMaps m, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TL_DECL;
  TL_START();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  TcTail* tail = reinterpret_cast<TcTail*>(smem + kTcOffTail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.H / a.Hk;
  const int T = a.nbq * a.Bq;
  const int rows = T * G;  // query rows of this KV head
  const int g = blockIdx.y;
  const int R0 = blockIdx.x * kTcRows;
  const int b_lo = (R0 / G) / a.Bq;
  const int b_hi = (min(R0 + kTcRows, rows) - 1) / G / a.Bq;
  // The key schedule depends on the committed prefix length *dP only, which kernels of
  // earlier, completed launches wrote, so it is read before the wait on the previous kernel.
  // Key tiles [j0, j0 + nl) of this CTA (both CTAs of a pair compute the same `split`); the
  // second CTA of a pair has nothing to do unless the keys are split and leaves at once.
  const KeySched ks = key_sched<kTcKeys>(a, b_lo, b_hi);
  const int n = ks.n_pre + ks.n_br;
  const int rank = gridDim.z > 1 ? (int)blockIdx.z : 0;
  const bool split = gridDim.z > 1 && ks.n_pre >= kSplitMinTiles;
  const int hsplit = split ? min(ks.n_pre, n / 2) : n;
  const int j0 = (split && rank == 1) ? hsplit : 0;
  const int nl = split ? (rank == 0 ? hsplit : n - hsplit) : (rank == 0 ? n : 0);
  if (rank == 1 && nl == 0) {
    pdl_trigger();
    TL_END(tl::ATTN_TC);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&tail->qfull), kTcSoftWarps * 32);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(smem_u32(&tail->kvfull[s]), 1);
      mbar_init(smem_u32(&tail->kvempty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&tail->sfull[s]), 1);
      mbar_init(smem_u32(&tail->pfull[s]), kTcSoftWarps * 32);
      mbar_init(smem_u32(&tail->pempty[s]), 1);
    }
    mbar_init(smem_u32(&tail->odone), 1);
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort = 0;
    tail->kv_issued = 0;
    tail->mma_issued = 0;
    fence_mbar_init();
    tma_prefetch_desc(&m.kc);
    tma_prefetch_desc(&m.vtc);
    tma_prefetch_desc(&m.kb);
    tma_prefetch_desc(&m.vtb);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tail->tmem), kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem;
  volatile int* abort = &tail->abort;
  pdl_trigger();
  pdl_wait();  // q and the block keys come from the previous kernel; out may be read by it
  TL_WAITED();
  const uint64_t lim = wait_limit(a.wait_ns);

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int issued = 0;
      for (int jl = 0; jl < nl; ++jl) {
        const int j = j0 + jl;  // key tile; ring slots and phases count local tiles
        const int s = jl % kTcStages;
        if (jl >= kTcStages &&
            !mbar_wait_bounded(smem_u32(&tail->kvempty[s]), (uint32_t)(jl / kTcStages - 1) & 1u,
                               abort, a.err, DEV_TIMEOUT_PRODUCER, lim))
          break;
        const uint32_t fb = smem_u32(&tail->kvfull[s]);
        const uint32_t kdst = smem_u32(smem + s * kTcStageBytes);
        const uint32_t vdst = kdst + kTcKBytes;
        mbar_arrive_expect_tx(fb, kTcStageBytes);
        const bool pre = j < ks.n_pre;
        const CUtensorMap* km = pre ? &m.kc : &m.kb;
        const CUtensorMap* vm = pre ? &m.vtc : &m.vtb;
        const int k0 = pre ? j * kTcKeys : ks.kb_lo + (j - ks.n_pre) * kTcKeys;
        tma_load_2d(kdst, km, fb, g * 128, k0, keep);
        tma_load_2d(kdst + kTcAtom, km, fb, g * 128 + 64, k0, keep);
        tma_load_2d(vdst, vm, fb, k0, g * 128, keep);
        tma_load_2d(vdst + kTcAtom, vm, fb, k0 + 64, g * 128, keep);
        ++issued;
      }
      tail->kv_issued = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S_{j+1} = Q K_{j+1}^T is issued before O += P_j V_j, into the buffer that
      // P_{j-1} V_{j-1} has finished reading.
      const uint32_t idesc_s = idesc_bf16(128, kTcKeys);
      const uint32_t idesc_o = idesc_bf16(128, 128);
      bool ok = mbar_wait_bounded(smem_u32(&tail->qfull), 0, abort, a.err, DEV_TIMEOUT_MMA, lim);
      auto issue_s = [&](int j) {
        const int s = j % kTcStages, sb = j & 1;
        ok = ok && mbar_wait_bounded(smem_u32(&tail->kvfull[s]), (uint32_t)(j / kTcStages) & 1u,
                                     abort, a.err, DEV_TIMEOUT_MMA, lim);
        ok = ok && (j < 2 || mbar_wait_bounded(smem_u32(&tail->pempty[sb]),
                                               (uint32_t)((j >> 1) - 1) & 1u, abort, a.err,
                                               DEV_TIMEOUT_MMA, lim));
        if (!ok) return;
        tc_fence_after();
        tail->mma_issued = 1;
        const uint32_t kbase = smem_u32(smem + s * kTcStageBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = sw128_desc(kbase + (kk >> 2) * kTcAtom) + 2 * (kk & 3);
          mma_bf16_ts(tmem + kTmS + 128u * sb, tmem + kTmQ + 8u * kk, bd, idesc_s, kk > 0);
        }
        mma_commit(smem_u32(&tail->sfull[sb]));
      };
      if (ok && nl > 0) {
        tc_fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < nl; ++i) {
        if (i + 1 < nl) issue_s(i + 1);
        const int pb = i & 1, si = i % kTcStages;
        ok = ok && mbar_wait_bounded(smem_u32(&tail->pfull[pb]), (uint32_t)(i >> 1) & 1u, abort,
                                     a.err, DEV_TIMEOUT_MMA, lim);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vbase = smem_u32(smem + si * kTcStageBytes + kTcKBytes);
        const uint32_t pcol = tmem + kTmS + 128u * pb;
        // Keys [16c, 16c + 16): half hh = c / 4 of the tile, P head columns 64 hh + 8 mq
        // and tail columns 64 hh + 32 + 8 mq (mq = c % 4), V^T atom hh at key offset 16 mq.
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int hh = c >> 2, mq = c & 3;
          const uint64_t bd = sw128_desc(vbase + hh * kTcAtom) + 2 * mq;
          mma_bf16_ts(tmem + kTmO, pcol + 64u * hh + 8u * mq, bd, idesc_o, (i | c) != 0);
          mma_bf16_ts(tmem + kTmO, pcol + 64u * hh + 32u + 8u * mq, bd, idesc_o, 1u);
        }
        mma_commit(smem_u32(&tail->kvempty[si]));
        mma_commit(smem_u32(&tail->pempty[pb]));
      }
      if (ok) mma_commit(smem_u32(&tail->odone));
    }
  } else {
    // Softmax + epilogue.  Warp w serves TMEM lane quarter q = w % 4 (query rows
    // 32q..32q+31, one per lane) and key half h: S columns [64h, 64h+64) and O columns
    // [64h, 64h+64); the two warps of a quarter exchange their half-row maxima through
    // shared memory (named barrier 1 + q).  tcgen05.ld/st are warp-wide, so every decision
    // guarding one is made uniform across the warp.
    constexpr unsigned kAll = 0xffffffffu;
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int R = R0 + r;
    const bool row_ok = R < rows;
    const int t = row_ok ? R / G : 0;
    const int hg = row_ok ? R - t * G : 0;
    const int br = t / a.Bq;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t o_base = lane_base + kTmO + (uint32_t)(h * 64);
    const float sl2 = 1.4426950408889634f / sqrtf(128.0f);  // log2(e) / sqrt(dh)
    // Q row R, columns [64h, 64h + 64), into TMEM (bf16 pairs; rows past the end as 0).
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((size_t)g * rows + R) * 128 + h * 64);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 v = row_ok ? qrow[c * 4 + e] : make_uint4(0, 0, 0, 0);
          w[4 * e] = v.x;
          w[4 * e + 1] = v.y;
          w[4 * e + 2] = v.z;
          w[4 * e + 3] = v.w;
        }
        tmem_st16u(lane_base + kTmQ + (uint32_t)(h * 32 + c * 16), w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&tail->qfull));
    }
    // Both warps of a quarter pass the same number of pair barriers: after a failed
    // (bounded) wait a warp keeps iterating with its waits and TMEM accesses skipped
    // (`ok` stays warp-uniform), so its partner is never left at a barrier.
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory"); };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      ok = ok && __all_sync(kAll, mbar_wait_bounded(smem_u32(bar), parity, abort, a.err,
                                                    DEV_TIMEOUT_EPILOGUE, lim));
    };
    for (int jl = 0; jl < nl; ++jl) {
      const int j = j0 + jl;  // key tile (masks); buffers and phases count local tiles
      const int sb = jl & 1;
      const uint32_t s_col = lane_base + kTmS + 128u * sb + (uint32_t)(h * 64);
      wait_all(&tail->sfull[sb], (uint32_t)(jl >> 1) & 1u);
      float sv[64];
      if (ok) {
        tc_fence_after();
        tmem_ld32x2(s_col, sv);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = -INFINITY;
      }
      // Mask only where the tile is not wholly visible (the last prefix tile, block keys).
      if (j >= ks.n_pre - 1) {
        int vlo, vhi;
        visible_range<kTcKeys>(a, ks, j, br, vlo, vhi);
        vlo -= h * 64;
        vhi -= h * 64;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < vlo || c >= vhi) sv[c] = -INFINITY;
      }
      float m0 = sv[0], m1 = sv[1], m2 = sv[2], m3 = sv[3];
#pragma unroll
      for (int c = 4; c < 60; c += 8) {
        m0 = fmax3(m0, sv[c], sv[c + 1]);
        m1 = fmax3(m1, sv[c + 2], sv[c + 3]);
        m2 = fmax3(m2, sv[c + 4], sv[c + 5]);
        m3 = fmax3(m3, sv[c + 6], sv[c + 7]);
      }
      m0 = fmax3(m0, sv[60], sv[61]);
      m1 = fmax3(m1, sv[62], sv[63]);
      const float hm = fmax3(m0, m1, fmaxf(m2, m3));
      tail->xmax[sb][h][r] = hm;
      pair_sync();
      const float mx = fmaxf(hm, tail->xmax[sb][h ^ 1][r]) * sl2;  // row max, log2 units
      // Lazy rescale: a row moves its reference maximum only when the tile maximum
      // exceeds it by more than 2^8 (also at its first visible key).  O then holds
      // P_0..P_{j-1} V relative to the old reference and is rescaled once P_{j-1} V has
      // landed; the warp rescales together, rows that keep their reference with alpha = 1.
      const bool need = mx > m_ref + kLazyRescale;
      const bool need_o = need && m_ref != -INFINITY;  // only for jl >= 1
      const float alpha = need_o ? exp2f(m_ref - mx) : 1.f;
      if (ok && __any_sync(kAll, need_o)) {
        wait_all(&tail->pempty[(jl - 1) & 1], (uint32_t)((jl - 1) >> 1) & 1u);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 64; c += 32) {
            float u[16], w[16];
            tmem_ld16x2(o_base + c, o_base + c + 16, u, w);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              u[e] *= alpha;
              w[e] *= alpha;
            }
            tmem_st16(o_base + c, u);
            tmem_st16(o_base + c + 16, w);
          }
        }
      }
      if (need_o) l *= alpha;
      if (need) m_ref = mx;
      // P = 2^(s * sl2 - m_ref) (masked s = -inf gives 0) as a bf16 head and a bf16 tail
      // (two MMAs keep P's fp32 accuracy), written over this warp's own S columns: keys
      // 64h + 16mq + [0, 16) go to head columns 8mq + [0, 8) and tail columns
      // 32 + 8mq + [0, 8) of the half.  Pairs of keys use the packed two-lane FMA / add.
      const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
      const float2 sl2x2 = make_float2(sl2, sl2), nmx2 = make_float2(nm, nm);
      float2 l2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int mq = 0; mq < 4; ++mq) {
        uint32_t hw[8], tw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = mq * 16 + 2 * e;
          const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), sl2x2, nmx2);
          const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          l2 = __fadd2_rn(l2, p);
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p.x, p.y);
          const float2 tl = __ffma2_rn(__bfloat1622float2(h2), make_float2(-1.f, -1.f), p);
          const __nv_bfloat162 t2 = __floats2bfloat162_rn(tl.x, tl.y);
          hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
          tw[e] = *reinterpret_cast<const uint32_t*>(&t2);
        }
        if (ok) {
          tmem_st8u(s_col + 8u * mq, hw);
          tmem_st8u(s_col + 32u + 8u * mq, tw);
        }
      }
      l += l2.x + l2.y;
      tmem_st_wait();  // also covers the O rescale's stores
      tc_fence_before();
      mbar_arrive(smem_u32(&tail->pfull[sb]));
    }
    // Epilogue: out row = O / l in bf16 (a row that saw no key is written as zeros); l is
    // the sum of the two half-row sums, which share the row's reference maximum.
    const bool got = ok && nl > 0 &&
                     mbar_wait_bounded(smem_u32(&tail->odone), 0, abort, a.err, DEV_TIMEOUT_EPILOGUE,
                                       lim);
    const bool have_o = __all_sync(kAll, got);
    tc_fence_after();
    tail->xsum[h][r] = l;
    pair_sync();
    const float lt = l + tail->xsum[h ^ 1][r];
    if (split) {
      // Stash this CTA's softmax state for the merge after the role branches: O (relative to
      // the row's reference maximum m_ref) as ex[column][row] fp32, then m_ref and the row sum.
      // The K / V^T ring is free: every MMA has completed (odone).
      float* ex = reinterpret_cast<float*>(smem);
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        float u[16], w[16];
        if (have_o) {
          tmem_ld16x2(o_base + c, o_base + c + 16, u, w);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = w[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          ex[(h * 64 + c + e) * kTcRows + r] = u[e];
          ex[(h * 64 + c + 16 + e) * kTcRows + r] = w[e];
        }
      }
      if (h == 0) {
        ex[kExM + r] = have_o ? m_ref : -INFINITY;
        ex[kExL + r] = have_o ? lt : 0.f;
      }
    }
    const float inv = lt > 0.f ? 1.0f / lt : 0.f;
    bf16* orow = a.out + ((size_t)t * a.H + g * G + hg) * 128 + h * 64;
#pragma unroll
    for (int c = 0; c < 64 && !split && rank == 0; c += 32) {
      float u[16], w[16];
      if (have_o) {
        tmem_ld16x2(o_base + c, o_base + c + 16, u, w);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) u[e] = w[e] = 0.f;
      }
      uint4 o4[4];
      uint32_t* ow = reinterpret_cast<uint32_t*>(o4);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 v0 = __floats2bfloat162_rn(u[2 * e] * inv, u[2 * e + 1] * inv);
        const __nv_bfloat162 v1 = __floats2bfloat162_rn(w[2 * e] * inv, w[2 * e + 1] * inv);
        ow[e] = *reinterpret_cast<const uint32_t*>(&v0);
        ow[8 + e] = *reinterpret_cast<const uint32_t*>(&v1);
      }
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 4; ++e) reinterpret_cast<uint4*>(orow + c)[e] = o4[e];
      }
    }
  }
  if (split) {
    // Both CTAs of the pair have stashed their state (every wait before this point is
    // bounded, so both arrive); rank 0 merges the two halves of the keys and writes the
    // output; the second barrier keeps rank 1's shared memory alive until it is read.
    cluster_arrive_release();
    cluster_wait();
    if (rank == 0 && warp >= 2) {
      const int q = warp & 3, h = (warp - 2) >> 2;
      const int r = q * 32 + lane;
      const int R = R0 + r;
      if (R < rows) {
        const int t = R / G, hg = R - t * G;
        const float* mine = reinterpret_cast<const float*>(smem);
        const uint32_t peer = mapa_shared(smem_u32(smem), 1u);
        const float m0 = mine[kExM + r], l0 = mine[kExL + r];
        const float m1 = ld_dsmem_f32(peer + 4u * (uint32_t)(kExM + r));
        const float l1 = ld_dsmem_f32(peer + 4u * (uint32_t)(kExL + r));
        const float mm = fmaxf(m0, m1);
        const float a0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mm);
        const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mm);
        const float lt = l0 * a0 + l1 * a1;
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        bf16* orow = a.out + ((size_t)t * a.H + g * G + hg) * 128 + h * 64;
#pragma unroll 2
        for (int c = 0; c < 64; c += 8) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int idx = (h * 64 + c + e) * kTcRows + r;
            o[e] = (mine[idx] * a0 + ld_dsmem_f32(peer + 4u * (uint32_t)idx) * a1) * inv;
          }
          uint4 o4;
          uint32_t* ow = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
            ow[e] = *reinterpret_cast<const uint32_t*>(&v);
          }
          *reinterpret_cast<uint4*>(orow + c) = o4;
        }
      }
    }
    cluster_arrive_release();
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (*abort) {
    // A bounded wait gave up in this CTA: wait (bounded) for the K / V^T copies and the
    // MMAs it started before its shared memory and TMEM are released.
    if (lane == 0 && warp == 0) {
      const int nl = tail->kv_issued;
      for (int s = 0; s < kTcStages && s < nl; ++s) {
        const int last = s + ((nl - 1 - s) / kTcStages) * kTcStages;
        mbar_wait_drain(smem_u32(&tail->kvfull[s]), (uint32_t)(last / kTcStages) & 1u);
      }
    } else if (lane == 0 && warp == 1 && tail->mma_issued) {
      mma_commit(smem_u32(&tail->drain));
      mbar_wait_drain(smem_u32(&tail->drain), 0);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
  TL_END(tl::ATTN_TC);
}

// ================================================================ mma.sync path (dh 32, 64)
constexpr int kRowsPerCta = 64;
constexpr int kThreads = 256;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte async copy; bytes < 16 zero-fills the rest (bytes = 0: a zero chunk).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Barrier among the 128 threads of one key group (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int kg) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + kg) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// One CTA serves 64 query rows of one (branch, KV head).  Its 8 warps form two key groups
// of 4 row-warps; key tiles alternate between the groups, each group double-buffers its
// K and V^T tiles with cp.async, and the two partial softmax states are merged at the end.
template <int DH>
__global__ void __launch_bounds__(kThreads) attn_mma_kernel(const AttnArgs a) {
  constexpr int KP = DH + 8;        // K tile row pitch (elements)
  constexpr int VP = kKeyTile + 8;  // V^T tile row pitch
  constexpr int KT = kKeyTile * KP, VT = DH * VP;
  constexpr int CH = DH / 8;        // 16-byte chunks per key row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sm = reinterpret_cast<bf16*>(smem_raw);
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kg = warp >> 2, rw = warp & 3, gtid = threadIdx.x & 127;
  const int grp = lane >> 2, tig = lane & 3;
  const int b = blockIdx.z, g = blockIdx.y;
  const int G = a.H / a.Hk;
  const int T = a.nbq * a.Bq;
  const int rows = a.Bq * G;  // rows of this (branch, KV head)
  const KeySched ks = key_sched<kKeyTile>(a, b, b);
  const int ntiles = ks.n_pre + ks.n_br;
  const int my_tiles = ntiles > kg ? (ntiles - kg + 1) / 2 : 0;
  const float sl2 = 1.4426950408889634f / sqrtf((float)DH);  // log2(e) / sqrt(dh)
  // This key group's buffers: K of buffer j, then V^T of buffer j.
  auto Kb = [&](int j) { return sm + (kg * 2 + j) * (KT + VT); };
  auto Vb = [&](int j) { return sm + (kg * 2 + j) * (KT + VT) + KT; };

  auto load_tile = [&](int tile, int buf) {
    const bool pre = tile < ks.n_pre;
    const int base = pre ? tile * kKeyTile : ks.kb_lo + (tile - ks.n_pre) * kKeyTile;
    const int lim = pre ? ks.Pk : b * a.Bk_stride + a.Bk;  // first invisible column
    for (int c = gtid; c < kKeyTile * CH; c += 128) {
      const int key = c / CH, col = (c - key * CH) * 8;
      const int kk = base + key;
      const bf16* src = pre ? a.kc + ((size_t)kk * a.Hk + g) * DH + col
                            : a.kb + ((size_t)kk * a.Hk + g) * DH + col;
      const bool in = kk < lim;
      cp_async16(smem_u32(Kb(buf) + key * KP + col), in ? src : a.kb, in ? 16 : 0);
    }
    for (int c = gtid; c < DH * (kKeyTile / 8); c += 128) {
      const int d = c >> 3, k8 = (c & 7) * 8;
      const int kk = base + k8;
      const int nv = min(max(lim - kk, 0), 8);
      const bf16* src = pre ? a.vtc + (size_t)(g * DH + d) * a.ldvc + kk
                            : a.vtb + (size_t)(g * DH + d) * a.ldvb + kk;
      cp_async16(smem_u32(Vb(buf) + d * VP + k8), nv > 0 ? src : a.kb, nv * 2);
    }
    cp_async_commit();
  };

  // Q fragments for rows row0+grp and row0+grp+8 (clamped; stores are predicated).
  const int row0 = blockIdx.x * kRowsPerCta + rw * 16;
  uint32_t qa[DH / 16][4];
  {
    const bf16* qrow[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      int r = row0 + grp + h2 * 8;
      r = r < rows ? r : rows - 1;
      qrow[h2] = a.q + ((size_t)g * T * G + (size_t)b * a.Bq * G + r) * DH;
    }
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc) {
      qa[kc][0] = *reinterpret_cast<const uint32_t*>(qrow[0] + kc * 16 + 2 * tig);
      qa[kc][1] = *reinterpret_cast<const uint32_t*>(qrow[1] + kc * 16 + 2 * tig);
      qa[kc][2] = *reinterpret_cast<const uint32_t*>(qrow[0] + kc * 16 + 8 + 2 * tig);
      qa[kc][3] = *reinterpret_cast<const uint32_t*>(qrow[1] + kc * 16 + 8 + 2 * tig);
    }
  }

  float o[DH / 8][4];
#pragma unroll
  for (int j = 0; j < DH / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};

  if (my_tiles > 0) load_tile(kg, 0);
  for (int it = 0; it < my_tiles; ++it) {
    const int tile = kg + 2 * it, buf = it & 1;
    if (it + 1 < my_tiles) {
      load_tile(tile + 2, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    group_sync(kg);
    const bf16* Ks = Kb(buf);
    const bf16* Vs = Vb(buf);

    // S = Q K^T; one ldmatrix.x4 fetches the B fragments of two 8-key groups.
    float s[8][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) s[ng][0] = s[ng][1] = s[ng][2] = s[ng][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int mi = lane >> 3;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(Ks + (np * 16 + (mi >> 1) * 8 + (lane & 7)) * KP + kc * 16 + (mi & 1) * 8),
                b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[kc], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[kc], b2, b3);
      }
    }
    int vlo, vhi;
    visible_range<kKeyTile>(a, ks, tile, b, vlo, vhi);
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = ng * 8 + 2 * tig + (e & 1);
        const float v = (c >= vlo && c < vhi) ? s[ng][e] * sl2 : -INFINITY;
        s[ng][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    }
    float alpha[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      tmax[h2] = fmaxf(tmax[h2], __shfl_xor_sync(0xffffffffu, tmax[h2], 1));
      tmax[h2] = fmaxf(tmax[h2], __shfl_xor_sync(0xffffffffu, tmax[h2], 2));
      const float mnew = fmaxf(mrow[h2], tmax[h2]);
      alpha[h2] = mnew == -INFINITY ? 1.f : exp2f(mrow[h2] - mnew);
      mrow[h2] = mnew;
      lrow[h2] *= alpha[h2];
    }
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) {
      o[j][0] *= alpha[0]; o[j][1] *= alpha[0];
      o[j][2] *= alpha[1]; o[j][3] *= alpha[1];
    }
    // P = head + tail, both bf16 (16 significant bits): P V keeps fp32-level accuracy.
    uint32_t pa[4][4], pl[4][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        p[e] = s[ng][e] == -INFINITY ? 0.f : exp2f(s[ng][e] - mrow[e >> 1]);
      lrow[0] += p[0] + p[1];
      lrow[1] += p[2] + p[3];
      const int kc2 = ng >> 1, hi = ng & 1;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      pa[kc2][hi * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
      pa[kc2][hi * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      pl[kc2][hi * 2 + 0] = pack_bf16(p[0] - f01.x, p[1] - f01.y);
      pl[kc2][hi * 2 + 1] = pack_bf16(p[2] - f23.x, p[3] - f23.y);
    }
    // O += P V, 16 keys at a time; V^T rows are (dh) with keys contiguous, so the B
    // fragments come from non-transposing ldmatrix.
#pragma unroll
    for (int kc2 = 0; kc2 < 4; ++kc2) {
      uint32_t vf[DH / 16][4];
#pragma unroll
      for (int dg = 0; dg < DH / 16; ++dg) {
        const int mi = lane >> 3;
        ldsm_x4(smem_u32(Vs + (dg * 16 + (mi >> 1) * 8 + (lane & 7)) * VP + kc2 * 16 + (mi & 1) * 8),
                vf[dg][0], vf[dg][1], vf[dg][2], vf[dg][3]);
      }
#pragma unroll
      for (int dg = 0; dg < DH / 16; ++dg) {
        mma_bf16_16816(o[2 * dg], pa[kc2], vf[dg][0], vf[dg][1]);
        mma_bf16_16816(o[2 * dg + 1], pa[kc2], vf[dg][2], vf[dg][3]);
      }
#pragma unroll
      for (int dg = 0; dg < DH / 16; ++dg) {
        mma_bf16_16816(o[2 * dg], pl[kc2], vf[dg][0], vf[dg][1]);
        mma_bf16_16816(o[2 * dg + 1], pl[kc2], vf[dg][2], vf[dg][3]);
      }
    }
    group_sync(kg);  // this buffer is refilled two tiles later
  }

  // Merge the two key groups' softmax states: group 1 hands its state over in smem.
  __syncthreads();
  float* xch = reinterpret_cast<float*>(smem_raw);
  constexpr int PER = DH / 2 + 4;  // floats per lane: o fragments + m[2] + l[2]
  float* mine = xch + ((size_t)rw * 32 + lane) * PER;
  if (kg == 1) {
#pragma unroll
    for (int j = 0; j < DH / 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) mine[j * 4 + e] = o[j][e];
    mine[DH / 2 + 0] = mrow[0];
    mine[DH / 2 + 1] = mrow[1];
    mine[DH / 2 + 2] = lrow[0];
    mine[DH / 2 + 3] = lrow[1];
  }
  __syncthreads();
  if (kg == 1) return;
  float sc0[2], sc1[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const float m1 = mine[DH / 2 + h2];
    const float m = fmaxf(mrow[h2], m1);
    sc0[h2] = mrow[h2] == -INFINITY ? 0.f : exp2f(mrow[h2] - m);
    sc1[h2] = m1 == -INFINITY ? 0.f : exp2f(m1 - m);
    float l = lrow[h2] * sc0[h2] + mine[DH / 2 + 2 + h2] * sc1[h2];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    lrow[h2] = l > 0.f ? 1.0f / l : 0.f;
  }
  // Stage the CTA's 64 x DH output tile in shared memory (behind the exchange area), then
  // write whole rows with 16-byte stores.
  bf16* ostage = reinterpret_cast<bf16*>(smem_raw + (size_t)4 * 32 * PER * sizeof(float));
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int rr = rw * 16 + grp + h2 * 8;
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) {
      const float v0 = (o[j][2 * h2] * sc0[h2] + mine[j * 4 + 2 * h2] * sc1[h2]) * lrow[h2];
      const float v1 = (o[j][2 * h2 + 1] * sc0[h2] + mine[j * 4 + 2 * h2 + 1] * sc1[h2]) * lrow[h2];
      *reinterpret_cast<uint32_t*>(ostage + rr * DH + j * 8 + 2 * tig) = pack_bf16(v0, v1);
    }
  }
  group_sync(0);
  for (int c = gtid; c < kRowsPerCta * CH; c += 128) {
    const int rr = c / CH, col = (c - rr * CH) * 8;
    const int r = blockIdx.x * kRowsPerCta + rr;
    if (r >= rows) continue;
    const int i = r / G, hg = r - i * G;
    bf16* orow = a.out + ((size_t)(b * a.Bq + i) * a.H + g * G + hg) * DH;
    *reinterpret_cast<uint4*>(orow + col) = *reinterpret_cast<const uint4*>(ostage + rr * DH + col);
  }
  TL_END(tl::ATTN_MMA);
}

template <int DH>
constexpr size_t attn_mma_smem() {
  return (size_t)4 * (kKeyTile * (DH + 8) + DH * (kKeyTile + 8)) * sizeof(bf16);
}

}  // namespace

cudaError_t attention_set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn_mma_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_mma_smem<32>())) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_mma_smem<64>())) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kTcSmem);
}

cudaError_t attention_set_carveout() {
  const void* ks[] = {(const void*)attn_mma_kernel<32>, (const void*)attn_mma_kernel<64>,
                      (const void*)attn_tc_kernel};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

const char* plan_attention(AttnLaunch* L, const AttnArgs& a, int dh, int kc_rows, int vtc_cols) {
  static thread_local char err[256];
  memset(L, 0, sizeof(*L));
  L->args = a;
  L->dh = dh;
  const int G = a.H / a.Hk;
  const int T = a.nbq * a.Bq;
  if (a.H % a.Hk || T < 1) return "attention: bad head grouping or empty batch";
  if (a.Bk > a.Bk_stride || (a.Bk > 0 && a.Bk_stride % 8)) return "attention: block stride must be a multiple of 8";
  if (a.causal && a.Bk != a.Bk_stride) return "attention: block-causal keys must be contiguous";
  if (a.ldvc % 8 || a.ldvb % 8 || (a.Bk > 0 && a.ldvb < a.nbq * a.Bk_stride))
    return "attention: V^T row lengths must be multiples of 8 covering every branch";
  if (dh == 32 || dh == 64) {
    L->grid = dim3((a.Bq * G + kRowsPerCta - 1) / kRowsPerCta, a.Hk, a.nbq);
    return "";
  }
  if (dh != 128) return "attention: head_dim must be 32, 64 or 128";
  static_assert(sizeof(TcMaps) == 5 * sizeof(CUtensorMap), "tensor map pack");
  CUtensorMap* maps = &L->maps[0];
  const int kbr = a.nbq * a.Bk_stride;
  // With no prefix or no block keys the corresponding maps are never used: point them
  // at the query array so that every map is valid.
  if (!make_tmap_bf16(&maps[0], a.q, (uint64_t)a.Hk * T * G, 128, 128, err, sizeof(err)) ||
      !make_tmap_bf16(&maps[1], kc_rows > 0 ? (const void*)a.kc : (const void*)a.q,
                      kc_rows > 0 ? kc_rows : T, kc_rows > 0 ? (uint64_t)a.Hk * 128 : 128, kTcKeys,
                      err, sizeof(err)) ||
      !make_tmap_bf16(&maps[2], vtc_cols > 0 ? (const void*)a.vtc : (const void*)a.q,
                      vtc_cols > 0 ? (uint64_t)a.Hk * 128 : T, vtc_cols > 0 ? vtc_cols : 128, 128,
                      err, sizeof(err), vtc_cols > 0 ? (uint64_t)a.ldvc : 0) ||
      !make_tmap_bf16(&maps[3], a.Bk > 0 ? (const void*)a.kb : (const void*)a.q,
                      a.Bk > 0 ? kbr : T, a.Bk > 0 ? (uint64_t)a.Hk * 128 : 128, kTcKeys, err,
                      sizeof(err)) ||
      !make_tmap_bf16(&maps[4], a.Bk > 0 ? (const void*)a.vtb : (const void*)a.q,
                      a.Bk > 0 ? (uint64_t)a.Hk * 128 : T, a.Bk > 0 ? kbr : 128, 128, err,
                      sizeof(err), a.Bk > 0 ? (uint64_t)a.ldvb : 0))
    return err;
  // z: the CTA pair of a row tile, when a prefix can reach the split threshold (kc_rows is
  // the most prefix keys the launch can see) and the pairs fit the SMs in one wave
  // (otherwise the row tiles alone fill the GPU and the keys are not split).
  const unsigned tiles = (unsigned)((T * G + kTcRows - 1) / kTcRows) * (unsigned)a.Hk;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 0;
  }
  const bool may_split = (max(kc_rows, a.pk_add) + kTcKeys - 1) / kTcKeys >= kSplitMinTiles;
  L->grid = dim3((T * G + kTcRows - 1) / kTcRows, a.Hk,
                 may_split && 2 * tiles <= (unsigned)sms ? 2 : 1);
  return "";
}

cudaError_t launch_attention(const AttnLaunch& L, cudaStream_t s) {
  switch (L.dh) {
    case 32:
      return launch_pdl(attn_mma_kernel<32>, L.grid, dim3(kThreads), attn_mma_smem<32>(), s, L.args);
    case 64:
      return launch_pdl(attn_mma_kernel<64>, L.grid, dim3(kThreads), attn_mma_smem<64>(), s, L.args);
    case 128: {
      TcMaps m;
      memcpy(&m, L.maps, sizeof(m));
      return launch_pdl_cluster(attn_tc_kernel, L.grid, dim3(kTcThreads), kTcSmem, s,
                                dim3(1, 1, L.grid.z), m, L.args);
    }
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace lopa
