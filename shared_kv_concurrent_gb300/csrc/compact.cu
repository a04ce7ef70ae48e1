// Compaction of committed segments into one RoPE frame (Hogwild! Inference summary,
// gentlecold.top, section 8: a finished block moves to the end of the common history and its
// representation is "corrected by RoPE offset" -- here reading 1 of that correction: the keys
// are re-rotated to their positions in the merged segment).  Keys are stored rotated at their
// block-local position j; rho(rho(k, j), o) = rho(k, j + o), so a key of a segment that starts
// at offset o of the merge is turned by o and stored at merged position j + o.  Values are
// copied.  Between steps only; a few MB per call, so the kernel is written for clarity.
#include <cuda_bf16.h>

#include "hw_device.cuh"

namespace hw {
namespace {

constexpr int kThreads = 256;

// One CTA per (run, layer); a thread per (token, KV head, 8 rotation pairs).
__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
  const CompactRun r = a.runs[blockIdx.x];
  const int layer = blockIdx.y;
  if (r.src_page < 0 || r.src_page >= a.num_pages || r.dst_page < 0 || r.dst_page >= a.num_pages) {
    if (threadIdx.x == 0) record_error(a.err, ERR_PAGE_RANGE, KID_COMPACT, blockIdx.x, r.src_page);
    return;
  }
  if (r.n < 1 || r.src_slot < 0 || r.src_slot + r.n > a.S || r.dst_slot < 0 ||
      r.dst_slot + r.n > a.S) {
    if (threadIdx.x == 0) record_error(a.err, ERR_SLOT_RANGE, KID_COMPACT, blockIdx.x, r.src_slot);
    return;
  }
  if (r.rot < 0 || r.rot >= a.max_position) {
    if (threadIdx.x == 0) record_error(a.err, ERR_POS_RANGE, KID_COMPACT, blockIdx.x, r.rot);
    return;
  }
  const int half = a.D >> 1, ch = half / 8;              // 8-pair chunks per head row
  const size_t lbase = (size_t)layer * a.layer_elems;
  const float* cs = a.rope_cos + (size_t)r.rot * half;
  const float* sn = a.rope_sin + (size_t)r.rot * half;
  const int work = r.n * a.H_kv * ch;
  for (int idx = threadIdx.x; idx < work; idx += kThreads) {
    const int c = idx % ch;
    const int th = idx / ch;
    const int h = th % a.H_kv;
    const int t = th / a.H_kv;
    const size_t src = lbase + (((size_t)r.src_page * a.H_kv + h) * a.S + r.src_slot + t) * a.D;
    const size_t dst = lbase + (((size_t)r.dst_page * a.H_kv + h) * a.S + r.dst_slot + t) * a.D;
    const uint4 k1 = *reinterpret_cast<const uint4*>(a.k_pool + src + 8 * c);
    const uint4 k2 = *reinterpret_cast<const uint4*>(a.k_pool + src + half + 8 * c);
    const __nv_bfloat162* x1 = reinterpret_cast<const __nv_bfloat162*>(&k1);
    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&k2);
    uint4 y1, y2;
    __nv_bfloat162* o1 = reinterpret_cast<__nv_bfloat162*>(&y1);
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&y2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a1 = __bfloat1622float2(x1[e]);
      const float2 a2 = __bfloat1622float2(x2[e]);
      const float c0 = cs[8 * c + 2 * e], c1 = cs[8 * c + 2 * e + 1];
      const float s0 = sn[8 * c + 2 * e], s1 = sn[8 * c + 2 * e + 1];
      o1[e] = __floats2bfloat162_rn(a1.x * c0 - a2.x * s0, a1.y * c1 - a2.y * s1);
      o2[e] = __floats2bfloat162_rn(a2.x * c0 + a1.x * s0, a2.y * c1 + a1.y * s1);
    }
    *reinterpret_cast<uint4*>(a.k_pool + dst + 8 * c) = y1;
    *reinterpret_cast<uint4*>(a.k_pool + dst + half + 8 * c) = y2;
    *reinterpret_cast<uint4*>(a.v_pool + dst + 8 * c) =
        *reinterpret_cast<const uint4*>(a.v_pool + src + 8 * c);
    *reinterpret_cast<uint4*>(a.v_pool + dst + half + 8 * c) =
        *reinterpret_cast<const uint4*>(a.v_pool + src + half + 8 * c);
  }
}

}  // namespace

void launch_compact(const CompactArgs& a, cudaStream_t s) {
  if (a.num_runs <= 0 || a.num_layers <= 0) return;
  compact_kernel<<<dim3(a.num_runs, a.num_layers), kThreads, 0, s>>>(a);
}

}  // namespace hw
