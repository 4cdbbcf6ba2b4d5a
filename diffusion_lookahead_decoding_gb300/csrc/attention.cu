// Branch-isolated attention for the verification forward.
//
// "SJTU x Huawei Xiaoyi release LoPA", section "Core design of LoPA": all candidate
// branches are verified in one forward because attention is isolated between branches.
// Query (b, i, h) attends to the committed prefix keys [0, P) - shared by every branch -
// and to the keys of its own branch's block only, bidirectionally inside the block
// ("Decoding-efficiency revolution" blog, section 3.3: a branch sees the prompt and its
// own tokens, never another branch's).
//
// One CTA = 4 warps = 64 query rows of one (branch, KV head): the rows are the
// (position, head-in-group) pairs that share KV head g, so one K/V tile in shared memory
// serves every query head of the group (grouped-query attention).  Keys stream in tiles
// of 64 from the prefix cache then from the branch's block scratch; S = Q K^T and O = P V
// run on bf16 mma.sync tensor-core instructions with an fp32 online softmax.
#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

constexpr int kRowsPerCta = 64;
constexpr int kKeyTile = 64;

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
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

template <int DH>
__global__ void __launch_bounds__(128) attn_kernel(const AttnArgs a) {
  constexpr int PITCH = DH + 8;  // bf16 elements per smem row (breaks bank conflicts)
  __shared__ __align__(16) bf16 Ks[kKeyTile * PITCH];
  __shared__ __align__(16) bf16 Vs[kKeyTile * PITCH];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int b = blockIdx.z, g = blockIdx.y;
  const int G = a.H / a.Hk;
  const int rows = a.Bq * G;
  const int Pk = a.pk_add + (a.dP ? *a.dP : 0);
  const int nkeys = Pk + a.Bk;
  const float sl2 = 1.4426950408889634f / sqrtf((float)DH);  // log2(e) / sqrt(dh)

  // Q fragments for rows row0+grp and row0+grp+8 (clamped; stores are predicated).
  const int row0 = blockIdx.x * kRowsPerCta + warp * 16;
  const bf16* qrow[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    int r = row0 + grp + h2 * 8;
    r = r < rows ? r : rows - 1;
    const int i = r / G, hg = r - i * G;
    qrow[h2] = a.q + ((size_t)(b * a.Bq + i) * a.H + g * G + hg) * DH;
  }
  uint32_t qa[DH / 16][4];
#pragma unroll
  for (int kc = 0; kc < DH / 16; ++kc) {
    qa[kc][0] = *reinterpret_cast<const uint32_t*>(qrow[0] + kc * 16 + 2 * tig);
    qa[kc][1] = *reinterpret_cast<const uint32_t*>(qrow[1] + kc * 16 + 2 * tig);
    qa[kc][2] = *reinterpret_cast<const uint32_t*>(qrow[0] + kc * 16 + 8 + 2 * tig);
    qa[kc][3] = *reinterpret_cast<const uint32_t*>(qrow[1] + kc * 16 + 8 + 2 * tig);
  }

  float o[DH / 8][4];
#pragma unroll
  for (int j = 0; j < DH / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};

  for (int kt = 0; kt < nkeys; kt += kKeyTile) {
    __syncthreads();
    constexpr int CH = DH / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < kKeyTile * CH; c += 128) {
      const int key = c / CH, col = (c - key * CH) * 8;
      const int kk = kt + key;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (kk < Pk) {
        const size_t off = ((size_t)kk * a.Hk + g) * DH + col;
        kv = *reinterpret_cast<const uint4*>(a.kc + off);
        vv = *reinterpret_cast<const uint4*>(a.vc + off);
      } else if (kk < nkeys) {
        const size_t off = (((size_t)b * a.Bk_stride + (kk - Pk)) * a.Hk + g) * DH + col;
        kv = *reinterpret_cast<const uint4*>(a.kb + off);
        vv = *reinterpret_cast<const uint4*>(a.vb + off);
      }
      *reinterpret_cast<uint4*>(&Ks[key * PITCH + col]) = kv;
      *reinterpret_cast<uint4*>(&Vs[key * PITCH + col]) = vv;
    }
    __syncthreads();

    // S = Q K^T for 16 rows x 64 keys per warp.
    float s[8][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) s[ng][0] = s[ng][1] = s[ng][2] = s[ng][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc) {
#pragma unroll
      for (int ng = 0; ng < 8; ++ng) {
        const bf16* kp = &Ks[(ng * 8 + grp) * PITCH + kc * 16 + 2 * tig];
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kp);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kp + 8);
        mma16816(s[ng], qa[kc], b0, b1);
      }
    }
    // Scale to log2 units, mask keys past the end, online softmax update.
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
    uint32_t pa[4][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng) {
      const float p0 = exp2f(s[ng][0] - mrow[0]), p1 = exp2f(s[ng][1] - mrow[0]);
      const float p2 = exp2f(s[ng][2] - mrow[1]), p3 = exp2f(s[ng][3] - mrow[1]);
      lrow[0] += p0 + p1;
      lrow[1] += p2 + p3;
      const int kc2 = ng >> 1, hi = ng & 1;
      pa[kc2][hi * 2 + 0] = pack_bf16(p0, p1);
      pa[kc2][hi * 2 + 1] = pack_bf16(p2, p3);
    }
    // O += P V: B fragments of V (keys x dh) via ldmatrix.trans.
#pragma unroll
    for (int kc2 = 0; kc2 < 4; ++kc2) {
#pragma unroll
      for (int dg = 0; dg < DH / 16; ++dg) {
        const int mi = lane >> 3;
        const int key = kc2 * 16 + (mi & 1) * 8 + (lane & 7);
        const int col = dg * 16 + (mi >> 1) * 8;
        const uint32_t addr = smem_u32(&Vs[key * PITCH + col]);
        uint32_t r0, r1, r2, r3;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                     : "r"(addr));
        mma16816(o[2 * dg], pa[kc2], r0, r1);
        mma16816(o[2 * dg + 1], pa[kc2], r2, r3);
      }
    }
  }

  // Normalise and store bf16.
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    float l = lrow[h2];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    lrow[h2] = 1.0f / l;
  }
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = row0 + grp + h2 * 8;
    if (r >= rows) continue;
    const int i = r / G, hg = r - i * G;
    bf16* orow = a.out + ((size_t)(b * a.Bq + i) * a.H + g * G + hg) * DH;
#pragma unroll
    for (int j = 0; j < DH / 8; ++j) {
      const uint32_t v = pack_bf16(o[j][2 * h2] * lrow[h2], o[j][2 * h2 + 1] * lrow[h2]);
      *reinterpret_cast<uint32_t*>(orow + j * 8 + 2 * tig) = v;
    }
  }
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, int dh, cudaStream_t s) {
  const int rows = a.Bq * (a.H / a.Hk);
  dim3 grid((rows + kRowsPerCta - 1) / kRowsPerCta, a.Hk, a.nbq);
  switch (dh) {
    case 32: attn_kernel<32><<<grid, 128, 0, s>>>(a); break;
    case 64: attn_kernel<64><<<grid, 128, 0, s>>>(a); break;
    case 128: attn_kernel<128><<<grid, 128, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace lopa
