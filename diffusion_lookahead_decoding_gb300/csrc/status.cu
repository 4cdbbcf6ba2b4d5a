// Device-side status of the kernel-level entry points, and the per-context lookup of the
// library's file-scope device variables.
//
// The kernel-level calls (lopa_linear_accumulate, lopa_lmhead_argmax, lopa_branch_attention)
// run without a context, so the error word their bounded waits write is a file-scope
// __device__ int of the library, one per device.  lopa_kernel_status reads and clears it.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ int g_call_status;  // DeviceError code of a kernel-level call's wait

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::atomic<unsigned long long> g_wait_ns{0};

std::mutex g_mu;
lopa::SymbolCache g_status_cache;

thread_local char g_msg[256];

}  // namespace

namespace lopa {

// Identifier of the calling thread's current CUDA context (unique for the life of the
// process: a context created after a reset gets a new one), or 0 when it is unknown.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the file-scope __device__ variable `sym` (a host-side stand-in that
// must never be passed to a kernel itself) in the current device's context.  The address
// is looked up once per device and again whenever that device's context changes (e.g.
// after cudaDeviceReset); callers hold the lock that guards `cache`.
cudaError_t symbol_address(const void* sym, SymbolCache& cache, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long id = current_context_id();
  if (!cache.addr[dev] || id == 0 || cache.ctx_id[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, sym);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    cache.addr[dev] = p;
    cache.ctx_id[dev] = id;
  }
  *out = cache.addr[dev];
  return cudaSuccess;
}

int* call_status_word(cudaError_t* e) {
  std::lock_guard<std::mutex> lock(g_mu);
  void* p = nullptr;
  *e = symbol_address(&g_call_status, g_status_cache, &p);
  return static_cast<int*>(p);
}

unsigned long long call_wait_limit_ns() { return g_wait_ns.load(); }

}  // namespace lopa

extern "C" {

int lopa_kernel_status(void* stream) {
  using namespace lopa;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  int* word = call_status_word(&e);
  int code = 0, code_static = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&code, word, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(int), s);
  if (e == cudaSuccess) e = lmhead_static_take_status(s, &code_static);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof(g_msg), "kernel status: %s", cudaGetErrorString(e));
    set_global_error(g_msg);
    return LOPA_ERR_CUDA;
  }
  if (code || code_static) {
    snprintf(g_msg, sizeof(g_msg), "a device-side wait of a kernel-level call gave up (code %d)",
             code ? code : code_static);
    set_global_error(g_msg);
    return LOPA_ERR_DEVICE_TIMEOUT;
  }
  return LOPA_OK;
}

int lopa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_ns.store(ns);
  return LOPA_OK;
}

}  // extern "C"
