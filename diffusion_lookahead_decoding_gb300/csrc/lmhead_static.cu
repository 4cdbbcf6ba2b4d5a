// LM head + online softmax without any allocation by the library.
//
// lopa_lmhead_argmax needs a caller-provided device workspace for its per-vocab-tile
// partial results.  Some callers cannot obtain one: code that runs where allocation is
// not allowed (for example between the steps of an externally managed memory pool, in a
// real-time loop that must never call into the allocator, or in a host that owns all
// device memory and hands out only fixed buffers).  This variant keeps its workspace in
// a fixed-size array in the library's own device memory instead, so the caller passes
// only inputs and outputs.
//
// The array lives as long as the library is loaded on that device.  Every call on a
// device uses the same array, so calls that may overlap on the GPU (different streams,
// no ordering between them) race on it; calls on one stream are ordered and safe.  A
// second file-scope word beside it records a device-side wait that gave up; the caller
// reads it with lopa_kernel_status.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// Partial (max, sum exp, argmax) per (vocabulary tile of 256, row): 12 bytes each.
constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB

static __device__ __align__(256) unsigned char g_lmhead_scratch[kStaticScratchBytes];
static __device__ int g_lmhead_status;  // DeviceError code of a wait that gave up

// Device addresses of the two variables, per device, valid for the context they were
// looked up in (a context created later, e.g. after cudaDeviceReset, looks them up again).
struct Addrs {
  unsigned long long ctx_id = 0;
  void* scratch = nullptr;
  int* status = nullptr;
};
std::mutex g_mu;
Addrs g_addr[lopa::kMaxDevices];

thread_local char g_err[256];

// Failures are reported through lopa_last_error(NULL).
int fail_static(int code, const char* msg) {
  lopa::set_global_error(msg);
  return code;
}

// Set-up, with the device current: looks up the device addresses of the scratch array and
// the status word (host code must never use the variables' names as pointers).  Runs on
// the first call on a device and again only if that device's context changed.
cudaError_t resolve(Addrs* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= lopa::kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long id = lopa::current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  Addrs& a = g_addr[dev];
  if (!a.scratch || id == 0 || a.ctx_id != id) {
    void* p = nullptr;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&q, g_lmhead_status);
    if (e != cudaSuccess) return e;
    if (!p || !q) return cudaErrorInvalidSymbol;
    e = lopa::gemm_set_smem_limits();
    if (e != cudaSuccess) return e;
    a.scratch = p;
    a.status = static_cast<int*>(q);
    a.ctx_id = id;
  }
  *out = a;
  return cudaSuccess;
}

}  // namespace

namespace lopa {

cudaError_t lmhead_static_take_status(cudaStream_t s, int* code) {
  *code = 0;
  Addrs a;
  cudaError_t e = resolve(&a);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(code, a.status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.status, 0, sizeof(int), s);
  return e;
}

}  // namespace lopa

extern "C" int lopa_lmhead_argmax_static(const void* hidden, const void* lm_head, int rows,
                                         int d_model, int vocab, float logit_scale, int mask_id,
                                         int32_t* argmax_out, float* maxp_out, void* stream) {
  using namespace lopa;
  auto aligned16 = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!aligned16(hidden) || !aligned16(lm_head) || !argmax_out || !maxp_out)
    return fail_static(LOPA_ERR_INVALID_ARG, "null or unaligned pointer");
  if (rows < 1 || vocab < 2 || d_model < 64 || d_model % 64 || mask_id < 0 || mask_id >= vocab)
    return fail_static(LOPA_ERR_INVALID_ARG, "bad shape");
  const int nvt = (vocab + 255) / 256;
  const size_t need = (size_t)nvt * rows * 12;
  if (need > kStaticScratchBytes) {
    snprintf(g_err, sizeof(g_err),
             "rows x ceil(vocab/256) x 12 bytes = %zu exceeds the fixed %zu-byte scratch", need,
             kStaticScratchBytes);
    return fail_static(LOPA_ERR_INVALID_ARG, g_err);
  }
  Addrs addr;
  const cudaError_t re = resolve(&addr);
  if (re != cudaSuccess) {
    snprintf(g_err, sizeof(g_err), "looking up the fixed scratch failed: %s", cudaGetErrorString(re));
    return fail_static(LOPA_ERR_CUDA, g_err);
  }
  // Every partial the merge reads is written first by the GEMM, so nothing needs clearing.
  float* pm = static_cast<float*>(addr.scratch);
  float* ps = pm + (size_t)nvt * rows;
  int* pi = reinterpret_cast<int*>(ps + (size_t)nvt * rows);
  GemmLaunch G;
  const char* e = plan_gemm(&G, GEMM_LMSTATS, hidden, rows, rows, lm_head, vocab, d_model,
                            rows > 128 ? 2 : 1, 1, 0, 0);
  if (e[0]) return fail_static(LOPA_ERR_UNSUPPORTED, e);
  GemmArgs& a = G.args;
  a.V = vocab;
  a.mask_id = mask_id;
  a.scale = logit_scale;
  a.part_m = pm;
  a.part_s = ps;
  a.part_i = pi;
  a.part_ld = rows;
  a.err = addr.status;
  a.wait_ns = call_wait_limit_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = launch_gemm(G, s);
  if (ce == cudaSuccess) ce = launch_lm_merge(pm, ps, pi, nvt, rows, rows, argmax_out, maxp_out, s);
  if (ce != cudaSuccess) {
    snprintf(g_err, sizeof(g_err), "launch failed: %s", cudaGetErrorString(ce));
    return fail_static(LOPA_ERR_CUDA, g_err);
  }
  return LOPA_OK;
}
