// K3 -- merge of the split-K partials (Hogwild! Inference summary, gentlecold.top, section 9:
// the work is split over KV entries and the partial results reduced; section 5: per-block
// softmax statistics combine by log-sum-exp):
//   out = sum_u o_u 2^(m_u - M) / sum_u l_u 2^(m_u - M),  M = max_u m_u,
//   lse = (M + log2 L) ln 2,
// with (o_u, m_u, l_u) the unit partials in the log2 domain.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "hw_internal.h"

namespace hw {

// Running merge state of one query row in one warp: (M, L) and the lane's float4 of O.
struct MergeAcc {
  float M, L;
  float4 O;
};

// Fold units [k_begin, k_end) of the group (plan entry g) into `acc` for query row r, by one
// warp (lane = float4 column).  The units are taken kChunk at a time with all their loads in
// flight; the running (M, L, O) is rescaled when M grows.
template <int D, int kChunk>
__device__ __forceinline__ void merge_units(const AttnArgs& a, int r, const Group& g, int k_begin,
                                            int k_end, int lane, MergeAcc& acc) {
  constexpr int PS = part_stride(D);
  const bool act = lane < D / 4;
  const size_t stride = (size_t)a.rows * PS;
  const float* base = a.partials + ((size_t)g.unit_begin * a.rows + r) * PS;
  float M = acc.M, L = acc.L;
  float4 O = acc.O;
  for (int k0 = k_begin; k0 < k_end; k0 += kChunk) {
    float2 ml[kChunk];
    float4 o[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int k = k0 + j;
      ml[j] = make_float2(-CUDART_INF_F, 0.f);
      o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < k_end) {
        ml[j] = *reinterpret_cast<const float2*>(base + k * stride + D);
        if (act) o[j] = *reinterpret_cast<const float4*>(base + k * stride + 4 * lane);
      }
    }
    float cm = M;
#pragma unroll
    for (int j = 0; j < kChunk; ++j) cm = fmaxf(cm, ml[j].x);
    if (cm == -CUDART_INF_F) continue;
    const float sc = (M == -CUDART_INF_F) ? 0.f : exp2f(M - cm);
    L *= sc;
    O.x *= sc;
    O.y *= sc;
    O.z *= sc;
    O.w *= sc;
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const float wj = (ml[j].x == -CUDART_INF_F) ? 0.f : exp2f(ml[j].x - cm);
      L = fmaf(ml[j].y, wj, L);
      O.x = fmaf(o[j].x, wj, O.x);
      O.y = fmaf(o[j].y, wj, O.y);
      O.z = fmaf(o[j].z, wj, O.z);
      O.w = fmaf(o[j].w, wj, O.w);
    }
    M = cm;
  }
  acc.M = M;
  acc.L = L;
  acc.O = O;
}

// Combine a second running state into the first (both over disjoint units of the same row).
__device__ __forceinline__ void merge_combine(MergeAcc& x, const MergeAcc& y) {
  const float cm = fmaxf(x.M, y.M);
  if (cm == -CUDART_INF_F) return;
  const float sx = (x.M == -CUDART_INF_F) ? 0.f : exp2f(x.M - cm);
  const float sy = (y.M == -CUDART_INF_F) ? 0.f : exp2f(y.M - cm);
  x.L = x.L * sx + y.L * sy;
  x.O = make_float4(x.O.x * sx + y.O.x * sy, x.O.y * sx + y.O.y * sy, x.O.z * sx + y.O.z * sy,
                    x.O.w * sx + y.O.w * sy);
  x.M = cm;
}

// Is the group entry usable (else the row is skipped and the error recorded)?
__device__ __forceinline__ bool merge_group_ok(const AttnArgs& a, int gi, int r, const Group& g,
                                               int lane) {
  if (g.p < 0 || g.p >= a.P || g.h < 0 || g.h >= a.H_kv || g.unit_begin < 0 ||
      g.unit_begin > g.unit_end || g.unit_end > a.num_units) {
    if (lane == 0) record_error(a.err, ERR_PLAN, KID_MERGE, gi, r);   // skipped, not trusted
    return false;
  }
  return true;
}

// out (and lse) of query row r of group g from its merged state.
template <int D>
__device__ __forceinline__ void merge_store(const AttnArgs& a, int r, const Group& g, int lane,
                                            const MergeAcc& acc) {
  const bool act = lane < D / 4;
  const float inv = (acc.L > 0.f) ? 1.f / acc.L : 0.f;
  const int qr = query_row(a, g.p, r / a.G), hq = g.h * a.G + r % a.G;
  if (qr < 0) return;                           // padding row: no output
  const size_t oi = (size_t)qr * a.H_q + hq;
  const float4 O = acc.O;
  if (act) {
    if (a.out_f32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + oi * D)[lane] =
          make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
    } else {
      const __nv_bfloat162 v0 = __floats2bfloat162_rn(O.x * inv, O.y * inv);
      const __nv_bfloat162 v1 = __floats2bfloat162_rn(O.z * inv, O.w * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&v0);
      pk.y = *reinterpret_cast<const uint32_t*>(&v1);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + oi * D)[lane] = pk;
    }
  }
  if (a.lse && lane == 0)
    a.lse[oi] = (acc.L > 0.f) ? (acc.M + log2f(acc.L)) * 0.6931471805599453f : -CUDART_INF_F;
}

}  // namespace hw
