// Memory-bound kernels of the verification forward: embedding + RMSNorm, RMSNorm,
// RoPE + K/V Pre-Write, the LM-head partial merge, and the RoPE table.
#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

__device__ __forceinline__ void load8(const bf16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ void store8(bf16* p, const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}

// x[t] = E[tok[t]] (fp32), n[t] = bf16(x * rsqrt(mean(x^2) + eps) * g).  One warp per row.
__global__ void embed_norm_kernel(const int* __restrict__ tok, int T, const bf16* __restrict__ E,
                                  const bf16* __restrict__ g, float* __restrict__ x,
                                  bf16* __restrict__ n, int d, float eps) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const bf16* e = E + (size_t)tok[t] * d;
  float* xr = x + (size_t)t * d;
  float ss = 0.f;
  for (int c = lane * 8; c < d; c += 256) {
    float f[8];
    load8(e + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += f[i] * f[i];
    *reinterpret_cast<float4*>(xr + c) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(xr + c + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
  ss = warp_sum(ss);
  const float rs = rsqrtf(ss / (float)d + eps);
  for (int c = lane * 8; c < d; c += 256) {
    float f[8], gg[8];
    load8(e + c, f);
    load8(g + c, gg);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * rs * gg[i];
    store8(n + (size_t)t * d + c, f);
  }
}

// n[t] = bf16(rmsnorm(x[t]) * g).  One warp per row.
__global__ void rmsnorm_kernel(const float* __restrict__ x, const bf16* __restrict__ g,
                               bf16* __restrict__ n, int T, int d, float eps) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* xr = x + (size_t)t * d;
  float ss = 0.f;
  for (int c = lane * 8; c < d; c += 256) {
    const float4 a = *reinterpret_cast<const float4*>(xr + c);
    const float4 b = *reinterpret_cast<const float4*>(xr + c + 4);
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z +
          b.w * b.w;
  }
  ss = warp_sum(ss);
  const float rs = rsqrtf(ss / (float)d + eps);
  for (int c = lane * 8; c < d; c += 256) {
    const float4 a = *reinterpret_cast<const float4*>(xr + c);
    const float4 b = *reinterpret_cast<const float4*>(xr + c + 4);
    float gg[8];
    load8(g + c, gg);
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * rs * gg[i];
    store8(n + (size_t)t * d + c, f);
  }
}

// Applies RoPE (rotate-half) to q and k of one token row, rounds q/k/v to bf16, writes q
// to [T][H][dh] and k/v to their Pre-Write destination, and re-zeroes the fp32 q/k/v
// accumulator row for the next layer.  Row t is position i = t % Bq of branch b = t / Bq
// at absolute position P + i.  K/V go to the branch scratch [b][i] or, when
// kv_to_cache, straight to the static cache row P + i (prompt prefill).
__global__ void rope_prewrite_kernel(float* __restrict__ qkv, int T, int H, int Hk, int dh,
                                     bf16* __restrict__ q, bf16* __restrict__ kdst,
                                     bf16* __restrict__ vdst, int kv_to_cache, int Bq,
                                     const float* __restrict__ cos_t,
                                     const float* __restrict__ sin_t, const int* __restrict__ dP) {
  const int t = blockIdx.x;
  if (t >= T) return;
  const int P = dP ? *dP : 0;
  const int b = t / Bq, i = t - b * Bq;
  const int pos = P + i;
  const int half = dh / 2;
  const int nqk = (H + Hk) * half;   // rotation pairs in q and k
  const int nv = Hk * dh;
  const int row_w = (H + 2 * Hk) * dh;
  float* row = qkv + (size_t)t * row_w;
  const size_t kv_row = kv_to_cache ? (size_t)(P + i) : (size_t)t;
  for (int e = threadIdx.x; e < nqk; e += blockDim.x) {
    const int head = e / half, j = e - head * half;
    float* src = row + head * dh;
    const float x1 = src[j], x2 = src[j + half];
    const float c = cos_t[(size_t)pos * half + j], s = sin_t[(size_t)pos * half + j];
    const float y1 = x1 * c - x2 * s, y2 = x2 * c + x1 * s;
    if (head < H) {
      bf16* qd = q + ((size_t)t * H + head) * dh;
      qd[j] = __float2bfloat16_rn(y1);
      qd[j + half] = __float2bfloat16_rn(y2);
    } else {
      bf16* kd = kdst + (kv_row * Hk + (head - H)) * dh;
      kd[j] = __float2bfloat16_rn(y1);
      kd[j + half] = __float2bfloat16_rn(y2);
    }
    src[j] = 0.f;
    src[j + half] = 0.f;
  }
  for (int e = threadIdx.x; e < nv; e += blockDim.x) {
    float* src = row + (H + Hk) * dh + e;
    vdst[kv_row * Hk * dh + e] = __float2bfloat16_rn(*src);
    *src = 0.f;
  }
}

struct Stat {
  float m, s;
  int i;
};

__device__ __forceinline__ Stat merge(Stat a, Stat b) {
  if (b.m == -INFINITY) return a;
  if (a.m == -INFINITY) return b;
  Stat r;
  r.m = fmaxf(a.m, b.m);
  r.s = a.s * __expf(a.m - r.m) + b.s * __expf(b.m - r.m);
  r.i = a.m > b.m ? a.i : (b.m > a.m ? b.i : min(a.i, b.i));
  return r;
}

// Merges the per-vocab-tile (max, sum exp, argmax) partials of each token row into the
// greedy token and its probability maxp = 1 / sum exp(z - max z).  One warp per row,
// fixed reduction order (deterministic).
__global__ void lm_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                                const int* __restrict__ pi, int nvt, int part_ld, int T,
                                int* __restrict__ am, float* __restrict__ mp) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  Stat acc{-INFINITY, 0.f, 0};
  for (int v = lane; v < nvt; v += 32) {
    const size_t o = (size_t)v * part_ld + t;
    acc = merge(acc, Stat{pm[o], ps[o], pi[o]});
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Stat o;
    o.m = __shfl_xor_sync(0xffffffffu, acc.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, acc.s, off);
    o.i = __shfl_xor_sync(0xffffffffu, acc.i, off);
    acc = (lane & off) ? merge(o, acc) : merge(acc, o);
  }
  if (lane == 0) {
    am[t] = acc.i;
    mp[t] = 1.0f / acc.s;
  }
}

// cos/sin of pos * base^(-2j/dh), evaluated in double and rounded to fp32.
__global__ void rope_table_kernel(float* cos_t, float* sin_t, int S, int dh, double base) {
  const int half = dh / 2;
  const long long n = (long long)S * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(e / half), j = (int)(e % half);
    const double ang = (double)pos * pow(base, -2.0 * j / dh);
    cos_t[e] = (float)cos(ang);
    sin_t[e] = (float)sin(ang);
  }
}

}  // namespace

cudaError_t launch_embed_norm(const int* tok, int T, const bf16* E, const bf16* g, float* x,
                              bf16* n, int d, float eps, cudaStream_t s) {
  embed_norm_kernel<<<(T + 7) / 8, 256, 0, s>>>(tok, T, E, g, x, n, d, eps);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, const bf16* g, bf16* n, int T, int d, float eps,
                           cudaStream_t s) {
  rmsnorm_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, g, n, T, d, eps);
  return cudaGetLastError();
}

cudaError_t launch_rope_prewrite(float* qkv, int T, int H, int Hk, int dh, bf16* q,
                                 bf16* kdst, bf16* vdst, int kv_to_cache, int Bq,
                                 const float* cos_t, const float* sin_t, const int* dP,
                                 cudaStream_t s) {
  rope_prewrite_kernel<<<T, 256, 0, s>>>(qkv, T, H, Hk, dh, q, kdst, vdst, kv_to_cache, Bq, cos_t,
                                         sin_t, dP);
  return cudaGetLastError();
}

cudaError_t launch_lm_merge(const float* pm, const float* ps, const int* pi, int nvt,
                            int part_ld, int T, int* am, float* mp, cudaStream_t s) {
  lm_merge_kernel<<<(T + 7) / 8, 256, 0, s>>>(pm, ps, pi, nvt, part_ld, T, am, mp);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int S, int dh, double base,
                              cudaStream_t s) {
  rope_table_kernel<<<256, 256, 0, s>>>(cos_t, sin_t, S, dh, base);
  return cudaGetLastError();
}

}  // namespace lopa
