// hw_merge_attention -- log-sum-exp merge of normalised partial attention results.
//
// Hogwild! Inference summary (gentlecold.top), section 9: the attention work is split over KV
// entries and the partial results are reduced afterwards; section 5: softmax partials combine
// through their log-sum-exp.  For parts i = 1..n of the same query rows over disjoint sets of
// keys, each given as its normalised output o_i and natural-log lse_i:
//     LSE = log sum_i exp(lse_i),   out = sum_i exp(lse_i - LSE) o_i,
// with empty parts (lse_i = -inf) contributing nothing and out = 0, LSE = -inf when all are.
// The parts may come from hw_concurrent_attention_range calls on this GPU or, gathered, from
// other GPUs that hold other ranges of the entries.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "hw_internal.h"

namespace {

constexpr int kWarps = 4;      // query rows per CTA (a warp per row, a float4 column per lane)

__global__ void __launch_bounds__(kWarps * 32)
    merge_parts_kernel(int n, int64_t rows, int D, const float* __restrict__ parts_out,
                       const float* __restrict__ parts_lse, void* out, int out_f32, float* lse) {
  const int64_t r = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float M = -CUDART_INF_F;
  for (int i = 0; i < n; ++i) M = fmaxf(M, parts_lse[(size_t)i * rows + r]);
  float L = 0.f;
  for (int i = 0; i < n; ++i) {
    const float li = parts_lse[(size_t)i * rows + r];
    L += (M == -CUDART_INF_F || li == -CUDART_INF_F) ? 0.f : expf(li - M);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int c = lane; c < D / 4; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float li = parts_lse[(size_t)i * rows + r];
      if (M == -CUDART_INF_F || li == -CUDART_INF_F) continue;
      const float w = expf(li - M);
      const float4 o = reinterpret_cast<const float4*>(parts_out + ((size_t)i * rows + r) * D)[c];
      acc.x = fmaf(o.x, w, acc.x);
      acc.y = fmaf(o.y, w, acc.y);
      acc.z = fmaf(o.z, w, acc.z);
      acc.w = fmaf(o.w, w, acc.w);
    }
    acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (out_f32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)r * D)[c] = acc;
    } else {
      const __nv_bfloat162 v0 = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 v1 = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&v0);
      pk.y = *reinterpret_cast<const uint32_t*>(&v1);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)r * D)[c] = pk;
    }
  }
  if (lse && lane == 0) lse[r] = L > 0.f ? M + logf(L) : -CUDART_INF_F;
}

}  // namespace

extern "C" hw_status hw_merge_attention(int32_t n_parts, int64_t rows, int32_t head_dim,
                                        const float* parts_out, const float* parts_lse,
                                        void* out, int32_t out_dtype, float* lse, void* stream) {
  if (n_parts < 1 || n_parts > 4096 || rows < 0 || head_dim < 4 || head_dim > 4096 ||
      head_dim % 4)
    return HW_ERR_INVALID_ARG;
  if (out_dtype != HW_OUT_BF16 && out_dtype != HW_OUT_F32) return HW_ERR_INVALID_ARG;
  if (rows == 0) return HW_OK;
  if (!parts_out || !parts_lse || !out) return HW_ERR_INVALID_ARG;
  if (((uintptr_t)parts_out | (uintptr_t)out) % 16 || (uintptr_t)parts_lse % 4 ||
      (uintptr_t)lse % 4)
    return HW_ERR_INVALID_ARG;
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  if (blocks > 0x7fffffff) return HW_ERR_CAPACITY;
  merge_parts_kernel<<<(unsigned)blocks, kWarps * 32, 0, (cudaStream_t)stream>>>(
      n_parts, rows, head_dim, parts_out, parts_lse, out, out_dtype == HW_OUT_F32, lse);
  return hw::cuda_status(cudaGetLastError());
}
