// Device-side helpers shared by the kernels of libhogwild.
#pragma once

#include <cuda_bf16.h>

#include "hw_internal.h"

namespace hw {

// Row of q / out / lse of query row v (worker, or (worker, token) with several query tokens per
// worker) of problem p; -1 for a padding row.
__device__ __forceinline__ int query_row(const AttnArgs& a, int p, int v) {
  return a.qrow ? a.qrow[(size_t)p * a.W + v] : p * a.W + v;
}

// Record a failed range check without trapping: OR the bits into the error word and keep the
// details of the first failure.
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t bits, uint32_t kid,
                                             uint32_t a, uint32_t b) {
  atomicOr(err, bits);
  if (atomicCAS(err + 1, 0u, kid) == 0u) {
    err[2] = a;
    err[3] = b;
  }
}

__device__ __forceinline__ unsigned long long plan_seq_now(const PlanGate& g) {
  unsigned long long v = 0;
  if (g.plan_seq)
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(g.plan_seq) : "memory");
  return v;
}

// Wait (one thread) until the plan behind `g` has arrived, given a first reading `v` of its
// sequence word; false, with ERR_TIMEOUT recorded, if it has not after about a second.
__device__ __forceinline__ bool plan_arrived(const PlanGate& g, unsigned long long v, uint32_t* err,
                                             uint32_t kid) {
  if (!g.plan_seq) return true;
  unsigned long long t0 = 0, t = 0;
  for (int it = 0;; ++it) {
    if (it > 0) v = plan_seq_now(g);
    if (v == g.plan_expect) return true;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (it == 0) t0 = t;
    if (t - t0 > 1000000000ull) {
      record_error(err, ERR_TIMEOUT, kid, blockIdx.x, 7);
      return false;
    }
    __nanosleep(128);
  }
}

}  // namespace hw

// Timeline spans, compiled in only with -DHW_TRACE (a separate debug build of the library):
// per translation unit, the earliest CTA start and latest CTA end of its kernels, in
// %globaltimer nanoseconds, read back through hw_span_<name>_read / _clear.
#ifdef HW_TRACE
static __device__ unsigned long long g_span[8];
__device__ __forceinline__ unsigned long long span_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define HW_SPAN_BEGIN(k) \
  do { if (threadIdx.x == 0) atomicMin(&g_span[2 * (k)], span_now()); } while (0)
#define HW_SPAN_END(k) \
  do { if (threadIdx.x == 0) atomicMax(&g_span[2 * (k) + 1], span_now()); } while (0)
#define HW_SPAN_EXPORT(name)                                                      \
  extern "C" int hw_span_##name##_read(unsigned long long* dst) {                 \
    return (int)cudaMemcpyFromSymbol(dst, g_span, sizeof(g_span));                \
  }                                                                               \
  extern "C" int hw_span_##name##_clear(void) {                                   \
    unsigned long long h[8];                                                      \
    for (int i = 0; i < 8; ++i) h[i] = (i & 1) ? 0ull : ~0ull;                    \
    return (int)cudaMemcpyToSymbol(g_span, h, sizeof(h));                         \
  }
#else
#define HW_SPAN_BEGIN(k) do { } while (0)
#define HW_SPAN_END(k) do { } while (0)
#define HW_SPAN_EXPORT(name)
#endif
