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
  pdl_wait();
  pdl_trigger();
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

// Sums 4 consecutive floats over the split-K partials, in split order, with the loads
// issued eight at a time.
__device__ __forceinline__ float4 sum_splits4(const float* p, int nsplit, size_t stride) {
  float4 a = *reinterpret_cast<const float4*>(p);
  for (int s0 = 1; s0 < nsplit; s0 += 8) {
    float4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < nsplit) q[u] = *reinterpret_cast<const float4*>(p + (size_t)(s0 + u) * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < nsplit) {
        a.x += q[u].x; a.y += q[u].y; a.z += q[u].z; a.w += q[u].w;
      }
  }
  return a;
}

__device__ __forceinline__ void store4_bf16(bf16* p, float a, float b, float c, float d) {
  uint2 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
  h[0] = __floats2bfloat162_rn(a, b);
  h[1] = __floats2bfloat162_rn(c, d);
  *reinterpret_cast<uint2*>(p) = u;
}

// Sums the q/k/v split-K partials of one token row, applies RoPE (rotate-half) to q and
// k, rounds q/k/v to bf16, writes q to [T][H][dh] and k/v to their Pre-Write destination.
// Row t is position i = t % Bq of branch b = t / Bq at absolute position P + i.  K/V go
// to the branch scratch [b][i] or, when kv_to_cache, straight to the static cache row
// P + i (prompt prefill).  One CTA per row; a work item is 4 consecutive elements of a
// head (j..j+3 with their rotation partners j+dh/2..+3).
__global__ void rope_prewrite_kernel(const float* __restrict__ qkv, int nsplit, size_t split_stride,
                                     int T, int H, int Hk, int dh, bf16* __restrict__ q,
                                     bf16* __restrict__ kdst, bf16* __restrict__ vdst,
                                     int kv_to_cache, int Bq, const float* __restrict__ cos_t,
                                     const float* __restrict__ sin_t, const int* __restrict__ dP) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  if (t >= T) return;
  const int P = dP ? *dP : 0;
  const int b = t / Bq, i = t - b * Bq;
  const int pos = P + i;
  const int half = dh / 2, hq = half / 4;
  const int nqk = (H + Hk) * hq;  // 4-wide rotation items in q and k
  const int nv = Hk * dh / 4;
  const int row_w = (H + 2 * Hk) * dh;
  const float* row = qkv + (size_t)t * row_w;
  const size_t kv_row = kv_to_cache ? (size_t)(P + i) : (size_t)t;
  const float* ct = cos_t + (size_t)pos * half;
  const float* st = sin_t + (size_t)pos * half;
  for (int e = threadIdx.x; e < nqk + nv; e += blockDim.x) {
    if (e < nqk) {
      const int head = e / hq, j = (e - head * hq) * 4;
      const float* src = row + head * dh;
      const float4 x1 = sum_splits4(src + j, nsplit, split_stride);
      const float4 x2 = sum_splits4(src + j + half, nsplit, split_stride);
      const float4 c = *reinterpret_cast<const float4*>(ct + j);
      const float4 sn = *reinterpret_cast<const float4*>(st + j);
      bf16* dst = head < H ? q + ((size_t)t * H + head) * dh
                           : kdst + (kv_row * Hk + (head - H)) * dh;
      store4_bf16(dst + j, x1.x * c.x - x2.x * sn.x, x1.y * c.y - x2.y * sn.y,
                  x1.z * c.z - x2.z * sn.z, x1.w * c.w - x2.w * sn.w);
      store4_bf16(dst + j + half, x2.x * c.x + x1.x * sn.x, x2.y * c.y + x1.y * sn.y,
                  x2.z * c.z + x1.z * sn.z, x2.w * c.w + x1.w * sn.w);
    } else {
      const int e4 = (e - nqk) * 4;
      const float4 v = sum_splits4(row + (H + Hk) * dh + e4, nsplit, split_stride);
      store4_bf16(vdst + kv_row * Hk * dh + e4, v.x, v.y, v.z, v.w);
    }
  }
  __syncthreads();
  if (row_w % 32 == 0) discard_partial_row(row, split_stride, nsplit, row_w);
}

// Block-wide sum; every thread gets the total.  blockDim.x is a multiple of 32, <= 1024.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// Sums nsplit float4 partials at p, p + stride, ... onto acc in split order.  Loads are
// issued eight at a time so that they are in flight together.
__device__ __forceinline__ void add_splits4(float4& acc, const float* p, int nsplit,
                                            size_t stride) {
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < nsplit) q[u] = *reinterpret_cast<const float4*>(p + (size_t)(s0 + u) * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < nsplit) {
        acc.x += q[u].x; acc.y += q[u].y; acc.z += q[u].z; acc.w += q[u].w;
      }
  }
}

// x[t] += sum_s part[s][t] (splits added in order), then n[t] = bf16(rmsnorm(x[t]) * g).
// One CTA per row, four columns per thread.
__global__ void __launch_bounds__(1024)
    residual_norm_kernel(float* __restrict__ x, const float* __restrict__ part, int nsplit,
                         size_t split_stride, const bf16* __restrict__ g, bf16* __restrict__ n,
                         int T, int d, float eps) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int c = threadIdx.x * 4;
  const bool active = c < d;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active) {
    float* xr = x + (size_t)t * d + c;
    acc = *reinterpret_cast<const float4*>(xr);
    add_splits4(acc, part + (size_t)t * d + c, nsplit, split_stride);
    *reinterpret_cast<float4*>(xr) = acc;
  }
  float ss = acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
  ss = block_sum(ss, red);  // also a barrier: every thread has read its partials
  const float rs = rsqrtf(ss / (float)d + eps);
  if (active) {
    const uint2 gu = *reinterpret_cast<const uint2*>(g + c);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gu);
    const float2 g01 = __bfloat1622float2(g2[0]), g23 = __bfloat1622float2(g2[1]);
    store4_bf16(n + (size_t)t * d + c, acc.x * rs * g01.x, acc.y * rs * g01.y, acc.z * rs * g23.x,
                acc.w * rs * g23.y);
  }
  if (d % 32 == 0) discard_partial_row(part + (size_t)t * d, split_stride, nsplit, d);
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
  pdl_wait();
  pdl_trigger();
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

cudaError_t pointwise_set_carveout() {
  const int c = cudaSharedmemCarveoutMaxShared;
  const void* ks[] = {(const void*)embed_norm_kernel, (const void*)rope_prewrite_kernel,
                      (const void*)residual_norm_kernel, (const void*)lm_merge_kernel};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_embed_norm(const int* tok, int T, const bf16* E, const bf16* g, float* x,
                              bf16* n, int d, float eps, cudaStream_t s) {
  return launch_pdl(embed_norm_kernel, dim3((T + 7) / 8), dim3(256), 0, s, tok, T, E, g, x, n, d,
                    eps);
}

cudaError_t launch_rope_prewrite(const float* qkv, int nsplit, size_t split_stride, int T, int H,
                                 int Hk, int dh, bf16* q, bf16* kdst, bf16* vdst,
                                 int kv_to_cache, int Bq, const float* cos_t, const float* sin_t,
                                 const int* dP, cudaStream_t s) {
  return launch_pdl(rope_prewrite_kernel, dim3(T), dim3(256), 0, s, qkv, nsplit, split_stride, T,
                    H, Hk, dh, q, kdst, vdst, kv_to_cache, Bq, cos_t, sin_t, dP);
}

cudaError_t launch_residual_norm(float* x, const float* part, int nsplit, size_t split_stride,
                                 const bf16* g, bf16* n, int T, int d, float eps, cudaStream_t s) {
  const int threads = ((d / 4 + 31) / 32) * 32;
  if (threads > 1024) return cudaErrorInvalidValue;
  return launch_pdl(residual_norm_kernel, dim3(T), dim3(threads), 0, s, x, part, nsplit,
                    split_stride, g, n, T, d, eps);
}

cudaError_t launch_lm_merge(const float* pm, const float* ps, const int* pi, int nvt,
                            int part_ld, int T, int* am, float* mp, cudaStream_t s) {
  return launch_pdl(lm_merge_kernel, dim3((T + 7) / 8), dim3(256), 0, s, pm, ps, pi, nvt, part_ld,
                    T, am, mp);
}

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int S, int dh, double base,
                              cudaStream_t s) {
  rope_table_kernel<<<256, 256, 0, s>>>(cos_t, sin_t, S, dh, base);
  return cudaGetLastError();
}

}  // namespace lopa
