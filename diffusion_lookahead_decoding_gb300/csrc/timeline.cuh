// Optional per-CTA device timeline (compiled in only with -DLOPA_TIMELINE).
//
// Every instrumented kernel records, per CTA, the %globaltimer value at entry, at the point
// where its dependent work can start (after the programmatic wait, or when a GEMM's
// accumulator is complete) and at exit, into a caller-provided device buffer.  Kernels
// overlap under programmatic dependent launch, and a profiler that serialises them cannot
// show where the critical path of a forward goes; this can.  Without the macro every hook
// is empty and the kernels are unchanged.
#pragma once

#include <stdint.h>

namespace lopa {
namespace tl {

enum Tag : unsigned {
  GEMM = 10,  // + GemmMode
  ATTN_TC = 20,
  ATTN_MMA = 21,
  RESIDUAL_NORM = 30,
  EMBED_NORM = 31,
  LM_MERGE = 32,
  DECIDE = 40,
  SELECT = 41,
  COMMIT = 42,
  FINALIZE = 43,
};

// Buffer layout: a 16-byte header {count, capacity, 0, 0} then `capacity` records.
struct Rec {
  unsigned tag, cta, sm, pad;
  unsigned long long t0, tw, t1;
};

}  // namespace tl
}  // namespace lopa

#ifdef LOPA_TIMELINE
// One pointer per translation unit, set by timeline_set_buffer_<unit>() on the host.
#define LOPA_TL_UNIT(unit)                                                                  \
  static __constant__ unsigned* g_tl_buf;                                                   \
  cudaError_t timeline_set_buffer_##unit(unsigned* p) {                                     \
    return cudaMemcpyToSymbol(g_tl_buf, &p, sizeof(p));                                     \
  }
#define TL_DECL uint64_t tl_t0 = 0, tl_tw = 0
#define TL_START()                                                                          \
  do {                                                                                      \
    if (threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tl_t0));          \
  } while (0)
#define TL_STAMP(var)                                                                       \
  do {                                                                                      \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(var));                                  \
  } while (0)
#define TL_WAITED()                                                                         \
  do {                                                                                      \
    if (threadIdx.x == 0) TL_STAMP(tl_tw);                                                  \
  } while (0)
// Called by thread 0 at the very end of the kernel.
#define TL_END(tag_value)                                                                   \
  do {                                                                                      \
    unsigned* b_ = g_tl_buf;                                                                \
    if (b_ && threadIdx.x == 0) {                                                           \
      const unsigned i_ = atomicAdd(b_, 1u);                                                \
      if (i_ < b_[1]) {                                                                     \
        lopa::tl::Rec* r_ = reinterpret_cast<lopa::tl::Rec*>(b_ + 4) + i_;                   \
        unsigned sm_;                                                                       \
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                     \
        uint64_t t1_;                                                                       \
        TL_STAMP(t1_);                                                                      \
        r_->tag = (tag_value);                                                              \
        r_->cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);           \
        r_->sm = sm_;                                                                       \
        r_->t0 = tl_t0;                                                                     \
        r_->tw = tl_tw;                                                                     \
        r_->t1 = t1_;                                                                       \
      }                                                                                     \
    }                                                                                       \
  } while (0)
#else
#define LOPA_TL_UNIT(unit)
#define TL_DECL
#define TL_START() \
  do {             \
  } while (0)
#define TL_STAMP(var) \
  do {                \
  } while (0)
#define TL_WAITED() \
  do {              \
  } while (0)
#define TL_END(tag_value) \
  do {                    \
  } while (0)
#endif
