// Branch-isolated attention for the verification forward.
//
// "SJTU x Huawei Xiaoyi release LoPA", section "Core design of LoPA": all candidate
// branches are verified in one forward because attention is isolated between branches.
// Query (b, i, h) attends to the committed prefix keys [0, P) - shared by every branch -
// and to the keys of its own branch's block only, bidirectionally inside the block
// ("Decoding-efficiency revolution" blog, section 3.3: a branch sees the prompt and its
// own tokens, never another branch's).
//
// One CTA serves 64 query rows of one (branch, KV head): the rows are the (position,
// head-in-group) pairs that share KV head g, so every K/V tile in shared memory serves all
// query heads of the group (grouped-query attention).  Its 8 warps form two key groups of
// 4 row-warps; key tiles of 64 alternate between the groups, each group double-buffers
// its tiles with cp.async, and the two partial softmax states are merged at the end.
// S = Q K^T and P V run on bf16 mma.sync with an fp32 online softmax; P enters P V as a
// bf16 head plus a bf16 tail, which keeps its fp32 accuracy.
#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

constexpr int kRowsPerCta = 64;
constexpr int kKeyTile = 64;
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

template <int DH>
__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnArgs a) {
  constexpr int PITCH = DH + 8;  // bf16/f16 elements per smem row (breaks bank conflicts)
  constexpr int TILE = kKeyTile * PITCH;
  constexpr int CH = DH / 8;     // 16-byte chunks per key row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* sm = reinterpret_cast<bf16*>(smem_raw);

  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kg = warp >> 2, rw = warp & 3, gtid = threadIdx.x & 127;
  const int grp = lane >> 2, tig = lane & 3;
  const int b = blockIdx.z, g = blockIdx.y;
  const int G = a.H / a.Hk;
  const int rows = a.Bq * G;
  const int Pk = a.pk_add + (a.dP ? *a.dP : 0);
  const int nkeys = Pk + a.Bk;
  const int ntiles = (nkeys + kKeyTile - 1) / kKeyTile;
  const int my_tiles = ntiles > kg ? (ntiles - kg + 1) / 2 : 0;
  const float sl2 = 1.4426950408889634f / sqrtf((float)DH);  // log2(e) / sqrt(dh)
  // This key group's buffers: K of buffer j at (4kg + 2j) tiles, V right after it.
  auto Kb = [&](int j) { return sm + (kg * 4 + 2 * j) * TILE; };
  auto Vb = [&](int j) { return sm + (kg * 4 + 2 * j + 1) * TILE; };

  auto load_tile = [&](int tile, int buf) {
    for (int c = gtid; c < kKeyTile * CH; c += 128) {
      const int key = c / CH, col = (c - key * CH) * 8;
      const int kk = tile * kKeyTile + key;
      const bf16 *ks = a.kb, *vs = a.vb;
      int bytes = 0;
      if (kk < Pk) {
        const size_t off = ((size_t)kk * a.Hk + g) * DH + col;
        ks = a.kc + off;
        vs = a.vc + off;
        bytes = 16;
      } else if (kk < nkeys) {
        const size_t off = (((size_t)b * a.Bk_stride + (kk - Pk)) * a.Hk + g) * DH + col;
        ks = a.kb + off;
        vs = a.vb + off;
        bytes = 16;
      }
      cp_async16(smem_u32(Kb(buf) + key * PITCH + col), ks, bytes);  // bytes 0 -> zeros
      cp_async16(smem_u32(Vb(buf) + key * PITCH + col), vs, bytes);
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
      const int i = r / G, hg = r - i * G;
      qrow[h2] = a.q + ((size_t)(b * a.Bq + i) * a.H + g * G + hg) * DH;
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
    const int kt = tile * kKeyTile;

    float s[8][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) s[ng][0] = s[ng][1] = s[ng][2] = s[ng][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc) {
#pragma unroll
      for (int ng = 0; ng < 8; ++ng) {
        const bf16* kp = Ks + (ng * 8 + grp) * PITCH + kc * 16 + 2 * tig;
        mma_bf16_16816(s[ng], qa[kc], *reinterpret_cast<const uint32_t*>(kp),
                       *reinterpret_cast<const uint32_t*>(kp + 8));
      }
    }
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kt + ng * 8 + 2 * tig + (e & 1);
        const float v = key < nkeys ? s[ng][e] * sl2 : -INFINITY;
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
      alpha[h2] = exp2f(mrow[h2] - mnew);  // 0 on the first tile (mrow = -inf)
      mrow[h2] = mnew;
      lrow[h2] *= alpha[h2];
    }
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) {
      o[j][0] *= alpha[0]; o[j][1] *= alpha[0];
      o[j][2] *= alpha[1]; o[j][3] *= alpha[1];
    }
    // P = hi + lo with both parts bf16 (16 significant bits): P V keeps fp32-level
    // accuracy, so the bf16 rounding of the attention output matches an exact softmax.
    uint32_t pa[4][4], pl[4][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) {
      const float p0 = exp2f(s[ng][0] - mrow[0]), p1 = exp2f(s[ng][1] - mrow[0]);
      const float p2 = exp2f(s[ng][2] - mrow[1]), p3 = exp2f(s[ng][3] - mrow[1]);
      lrow[0] += p0 + p1;
      lrow[1] += p2 + p3;
      const int kc2 = ng >> 1, hi = ng & 1;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      pa[kc2][hi * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
      pa[kc2][hi * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      pl[kc2][hi * 2 + 0] = pack_bf16(p0 - f01.x, p1 - f01.y);
      pl[kc2][hi * 2 + 1] = pack_bf16(p2 - f23.x, p3 - f23.y);
    }
#pragma unroll
    for (int kc2 = 0; kc2 < 4; ++kc2) {
#pragma unroll
      for (int dg = 0; dg < DH / 16; ++dg) {
        const int mi = lane >> 3;
        const int key = kc2 * 16 + (mi & 1) * 8 + (lane & 7);
        const int col = dg * 16 + (mi >> 1) * 8;
        const uint32_t addr = smem_u32(Vs + key * PITCH + col);
        uint32_t r0, r1, r2, r3;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                     : "r"(addr));
        mma_bf16_16816(o[2 * dg], pa[kc2], r0, r1);
        mma_bf16_16816(o[2 * dg + 1], pa[kc2], r2, r3);
        mma_bf16_16816(o[2 * dg], pl[kc2], r0, r1);
        mma_bf16_16816(o[2 * dg + 1], pl[kc2], r2, r3);
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
    lrow[h2] = 1.0f / l;
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
}

template <int DH>
constexpr size_t attn_smem() {
  return (size_t)8 * kKeyTile * (DH + 8) * sizeof(bf16);
}

}  // namespace

cudaError_t attention_set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_smem<32>())) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_smem<64>())) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem<128>());
}

cudaError_t attention_set_carveout() {
  cudaError_t e;
  const int c = cudaSharedmemCarveoutMaxShared;
  if ((e = cudaFuncSetAttribute(attn_kernel<32>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                c)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                c)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
}

cudaError_t launch_attention(const AttnArgs& a, int dh, cudaStream_t s) {
  const int rows = a.Bq * (a.H / a.Hk);
  dim3 grid((rows + kRowsPerCta - 1) / kRowsPerCta, a.Hk, a.nbq);
  switch (dh) {
    case 32: return launch_pdl(attn_kernel<32>, grid, dim3(kThreads), attn_smem<32>(), s, a);
    case 64: return launch_pdl(attn_kernel<64>, grid, dim3(kThreads), attn_smem<64>(), s, a);
    case 128: return launch_pdl(attn_kernel<128>, grid, dim3(kThreads), attn_smem<128>(), s, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lopa
