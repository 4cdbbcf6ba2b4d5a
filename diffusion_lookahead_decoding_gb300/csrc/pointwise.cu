// Memory-bound kernels of the verification forward: embedding + RMSNorm, split-K sum +
// residual add + RMSNorm, the LM-head partial merge, and the RoPE table.
#include "common.cuh"
#include "internal.h"
#include "timeline.cuh"

namespace lopa {

LOPA_TL_UNIT(pointwise)

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
                                  bf16* __restrict__ n, int d, float eps, int V, int* err) {
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int id = tok[t];
  if (id < 0 || id >= V) {
    if (lane == 0 && err) atomicExch(err, DEV_BAD_INDEX);
    id = 0;
  }
  const bf16* e = E + (size_t)id * d;
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
  TL_END(tl::EMBED_NORM);
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

// x[t] += sum_s part[s][t] (splits added in order after x), then
// n[t] = bf16(x[t] * rsqrt(mean(x[t]^2) + eps) * g).  One CTA per row, eight columns per
// thread; the partial loads of four splits are in flight together, and two CTAs fit an
// SM, so a 256-row batch is resident in one wave.  Consumed partials are dropped from L2.
__global__ void __launch_bounds__(512, 2)
    residual_norm_kernel(float* __restrict__ x, const float* __restrict__ part, int nsplit,
                         size_t split_stride, const bf16* __restrict__ g, bf16* __restrict__ n,
                         int d, float eps) {
  __shared__ float red[32];
  TL_DECL;
  TL_START();
  const int t = blockIdx.x;
  const int c = threadIdx.x * 8;
  const bool active = c < d;
  // The norm weight is a constant of the model: loaded before the wait on the producer of
  // the partials, so its latency is off the critical path.
  float gg[8];
  if (active) load8(g + c, gg);
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  if (active) {
    float* xr = x + (size_t)t * d + c;
    a0 = *reinterpret_cast<const float4*>(xr);
    a1 = *reinterpret_cast<const float4*>(xr + 4);
    const float* p = part + (size_t)t * d + c;
    for (int s0 = 0; s0 < nsplit; s0 += 4) {
      float4 q0[4], q1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (s0 + u < nsplit) {
          const float* ps = p + (size_t)(s0 + u) * split_stride;
          q0[u] = *reinterpret_cast<const float4*>(ps);
          q1[u] = *reinterpret_cast<const float4*>(ps + 4);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (s0 + u < nsplit) {
          a0.x += q0[u].x; a0.y += q0[u].y; a0.z += q0[u].z; a0.w += q0[u].w;
          a1.x += q1[u].x; a1.y += q1[u].y; a1.z += q1[u].z; a1.w += q1[u].w;
        }
    }
    *reinterpret_cast<float4*>(xr) = a0;
    *reinterpret_cast<float4*>(xr + 4) = a1;
  }
  float ss = a0.x * a0.x + a0.y * a0.y + a0.z * a0.z + a0.w * a0.w;
  ss += a1.x * a1.x + a1.y * a1.y + a1.z * a1.z + a1.w * a1.w;
  ss = block_sum(ss, red);  // also a barrier: every thread has read its partials
  const float rs = rsqrtf(ss / (float)d + eps);
  if (active) {
    float f[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * rs * gg[i];
    store8(n + (size_t)t * d + c, f);
  }
  // Drop the consumed partial rows from L2 without write-back (128-byte lines).
  if (d % 32 == 0) {
    const int lines = d / 32;
    const float* rowp = part + (size_t)t * d;
    for (int e = threadIdx.x; e < lines * nsplit; e += blockDim.x) {
      const int sp = e / lines, l = e - sp * lines;
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(rowp + (size_t)sp * split_stride + (size_t)l * 32)
                   : "memory");
    }
  }
  TL_END(tl::RESIDUAL_NORM);
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
// greedy token and its probability maxp = 1 / sum exp(z - max z).  A CTA serves 32 rows
// (lane = row, so the partial loads [tile][row] are coalesced); its kMergeWarps warps each
// fold a contiguous range of vocabulary tiles, and warp 0 merges the warps' states in warp
// order (a fixed order: deterministic).
constexpr int kMergeWarps = 16;

__global__ void __launch_bounds__(32 * kMergeWarps)
    lm_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                    const int* __restrict__ pi, int nvt, int part_ld, int T,
                    int* __restrict__ am, float* __restrict__ mp) {
  __shared__ Stat part[kMergeWarps][32];
  TL_DECL;
  TL_START();
  pdl_wait();
  TL_WAITED();
  pdl_trigger();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t = blockIdx.x * 32 + lane;
  const int v0 = (int)((long long)w * nvt / kMergeWarps);
  const int v1 = (int)((long long)(w + 1) * nvt / kMergeWarps);
  Stat acc{-INFINITY, 0.f, 0};
  if (t < T) {
    int v = v0;
    for (; v + 4 <= v1; v += 4) {  // four tiles' loads in flight
      Stat s4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const size_t o = (size_t)(v + u) * part_ld + t;
        s4[u] = Stat{pm[o], ps[o], pi[o]};
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) acc = merge(acc, s4[u]);
    }
    for (; v < v1; ++v) {
      const size_t o = (size_t)v * part_ld + t;
      acc = merge(acc, Stat{pm[o], ps[o], pi[o]});
    }
  }
  part[w][lane] = acc;
  __syncthreads();
  if (w == 0 && t < T) {
    Stat r = part[0][lane];
    for (int j = 1; j < kMergeWarps; ++j) r = merge(r, part[j][lane]);
    am[t] = r.i;
    mp[t] = 1.0f / r.s;
  }
  TL_END(tl::LM_MERGE);
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
  const void* ks[] = {(const void*)embed_norm_kernel, (const void*)residual_norm_kernel,
                      (const void*)lm_merge_kernel};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_embed_norm(const int* tok, int T, const bf16* E, const bf16* g, float* x,
                              bf16* n, int d, float eps, int V, int* err, cudaStream_t s) {
  return launch_pdl(embed_norm_kernel, dim3((T + 7) / 8), dim3(256), 0, s, tok, T, E, g, x, n, d,
                    eps, V, err);
}

cudaError_t launch_residual_norm(float* x, const float* part, int nsplit, size_t split_stride,
                                 const bf16* g, bf16* n, int T, int d, float eps, cudaStream_t s) {
  const int threads = ((d / 8 + 31) / 32) * 32;
  if (threads > 512 || d % 8 != 0) return cudaErrorInvalidValue;
  return launch_pdl(residual_norm_kernel, dim3(T), dim3(threads), 0, s, x, part, nsplit,
                    split_stride, g, n, d, eps);
}

cudaError_t launch_lm_merge(const float* pm, const float* ps, const int* pi, int nvt,
                            int part_ld, int T, int* am, float* mp, cudaStream_t s) {
  return launch_pdl(lm_merge_kernel, dim3((T + 31) / 32), dim3(32 * kMergeWarps), 0, s, pm, ps, pi,
                    nvt, part_ld, T, am, mp);
}

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int S, int dh, double base,
                              cudaStream_t s) {
  rope_table_kernel<<<256, 256, 0, s>>>(cos_t, sin_t, S, dh, base);
  return cudaGetLastError();
}

}  // namespace lopa
