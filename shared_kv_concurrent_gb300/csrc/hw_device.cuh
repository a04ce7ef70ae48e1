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

// Fused append (Hogwild! Inference summary, section 9: tokens of a block at block-local
// positions): the appended tokens [f0, f1) of the FreshTok table are written for KV head h --
// key rotated to its position with the fp32 table and stored as bf16, value copied -- into the
// pool, exactly as the append kernel would.  NT threads (tid in [0, NT)); each takes 8 rotation
// pairs (16-byte loads and stores) of one token.  kid names the calling kernel in error records.
template <int D, int NT>
__device__ __forceinline__ void append_fresh(const AttnArgs& a, int h, int f0, int f1, int tid,
                                             uint32_t kid) {
  constexpr int half = D / 2;
  constexpr int CH = half / 8;                 // 8-pair chunks per token
  constexpr int TPP = NT / CH;                 // tokens per pass
  static_assert(NT % CH == 0, "whole tokens per pass");
  const int c = tid % CH;
#pragma unroll 1
  for (int f = f0 + tid / CH; f < f1; f += TPP) {
    const FreshTok ft = a.fresh[f];
    if (ft.page < 0 || ft.page >= a.num_pages || ft.slot < 0 || ft.slot >= a.S) {
      if (c == 0) record_error(a.err, ERR_PAGE_RANGE, kid, blockIdx.x, ft.page);
      continue;
    }
    if (ft.pos < 0 || ft.pos >= a.max_position || ft.src < 0) {
      if (c == 0) record_error(a.err, ERR_POS_RANGE, kid, blockIdx.x, ft.pos);
      continue;
    }
    const size_t src = ((size_t)ft.src * a.H_kv + h) * D + 8 * c;
    const size_t dst = (((size_t)ft.page * a.H_kv + h) * a.S + ft.slot) * D + 8 * c;
    const size_t tab = (size_t)ft.pos * half + 8 * c;
    const uint4 k1 = *reinterpret_cast<const uint4*>(a.k_raw + src);
    const uint4 k2 = *reinterpret_cast<const uint4*>(a.k_raw + src + half);
    const uint4 v1 = *reinterpret_cast<const uint4*>(a.v_raw + src);
    const uint4 v2 = *reinterpret_cast<const uint4*>(a.v_raw + src + half);
    const float4 ca = *reinterpret_cast<const float4*>(a.rope_cos + tab);
    const float4 cb = *reinterpret_cast<const float4*>(a.rope_cos + tab + 4);
    const float4 sa = *reinterpret_cast<const float4*>(a.rope_sin + tab);
    const float4 sb = *reinterpret_cast<const float4*>(a.rope_sin + tab + 4);
    const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
    const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    const __nv_bfloat16* x1 = reinterpret_cast<const __nv_bfloat16*>(&k1);
    const __nv_bfloat16* x2 = reinterpret_cast<const __nv_bfloat16*>(&k2);
    __align__(16) __nv_bfloat16 y1[8], y2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float u1 = __bfloat162float(x1[e]), u2 = __bfloat162float(x2[e]);
      y1[e] = __float2bfloat16_rn(u1 * cv[e] - u2 * sv[e]);
      y2[e] = __float2bfloat16_rn(u2 * cv[e] + u1 * sv[e]);
    }
    *reinterpret_cast<uint4*>(a.k_layer + dst) = *reinterpret_cast<const uint4*>(y1);
    *reinterpret_cast<uint4*>(a.k_layer + dst + half) = *reinterpret_cast<const uint4*>(y2);
    *reinterpret_cast<uint4*>(a.v_layer + dst) = v1;
    *reinterpret_cast<uint4*>(a.v_layer + dst + half) = v2;
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
