// K2 (FMA form) and K3 -- concurrent attention with per-(worker, block) query rotation, and
// the log-sum-exp merge of the per-unit partial results.
//
// Method (Hogwild! Inference summary, gentlecold.top): keys are stored rotated at block-local
// positions; for a block at offset o in worker w's view the query is rotated by (i_q - o)
// (section 5), so one KV tile serves every worker and every query head of its GQA group, each
// with its own rotated query.  Work is split over KV entries, not over blocks, and the partial
// results are reduced afterwards (section 9, Flash-Decoding style kernel).
//
// This form uses FP32 FMA and is meant for small row counts (W * G below a 16-row tile); one
// CTA per unit (a run of pieces of one (problem, KV head)), 8 warps, each warp owning rows
// r = warp, warp + 8, ...; lane = token of a 32-token tile staged in shared memory.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "hw_merge.cuh"

namespace hw {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 32;
constexpr int kMaxRowsPerWarp = 16;   // rows <= 128

template <int D>
__global__ void __launch_bounds__(kThreads) attn_fma_kernel(const AttnArgs a) {
  extern __shared__ float sm[];
  constexpr int DJ = D / 32;
  constexpr int KS = D + 1;                     // padded key row: conflict-free lane = token
  const int rows = a.rows;
  float* qs = sm;                               // [rows][D] rotated, pre-scaled queries
  float* ks = qs + rows * D;                    // [kTile][D + 1]
  float* vs = ks + kTile * KS;                  // [kTile][D]
  __shared__ int plan_ok;
  if (threadIdx.x == 0) plan_ok = plan_arrived(a.gate, plan_seq_now(a.gate), a.err, KID_ATTN_FMA);
  __syncthreads();
  if (!plan_ok) {
    // No plan: this unit's partial rows are written empty (m = -inf, l = 0, o = 0), so the
    // merge gives zero for them; the error word says why.
    float* part = a.partials + (size_t)blockIdx.x * rows * part_stride(D);
    for (int e = threadIdx.x; e < rows * part_stride(D); e += blockDim.x)
      part[e] = (e % part_stride(D) == D) ? -CUDART_INF_F : 0.f;
    return;
  }
  const Unit u = a.units[blockIdx.x];
  const Group g = a.groups[u.group];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float m[kMaxRowsPerWarp], l[kMaxRowsPerWarp], o[kMaxRowsPerWarp][DJ];
#pragma unroll
  for (int k = 0; k < kMaxRowsPerWarp; ++k) {
    m[k] = -CUDART_INF_F;
    l[k] = 0.f;
#pragma unroll
    for (int j = 0; j < DJ; ++j) o[k][j] = 0.f;
  }

  int cur_slot = -1;
  for (int pi = u.piece_begin; pi < u.piece_end; ++pi) {
    const Piece pc = a.pieces[pi];
    if (pc.page < 0 || pc.page >= a.num_pages || pc.slot0 < 0 || pc.ntok < 1 ||
        pc.slot0 + pc.ntok > a.S || pc.seg_slot < 0 || pc.seg_slot >= a.num_seg_slots) {
      if (threadIdx.x == 0) record_error(a.err, ERR_PLAN, KID_ATTN_FMA, blockIdx.x, pi);
      continue;
    }
    const int* dl = a.delta + (size_t)pc.seg_slot * a.W;
    if (pc.seg_slot != cur_slot) {
      // New segment: rotate every row's query by (i_q - view offset) of this segment.
      __syncthreads();
      const int half = D / 2;
      for (int idx = threadIdx.x; idx < rows * half; idx += kThreads) {
        const int r = idx / half, i = idx % half;
        const int w = r / a.G, hq = g.h * a.G + r % a.G;
        const int delta = dl[w];
        float y1 = 0.f, y2 = 0.f;
        if (delta >= 0 && delta < a.max_position) {
          const size_t qo = ((size_t)query_row(a, g.p, w) * a.H_q + hq) * D;
          const float q1 = __bfloat162float(a.q[qo + i]);
          const float q2 = __bfloat162float(a.q[qo + i + half]);
          const float c = a.rope_cos[(size_t)delta * half + i];
          const float s = a.rope_sin[(size_t)delta * half + i];
          y1 = (q1 * c - q2 * s) * a.scale_log2;
          y2 = (q2 * c + q1 * s) * a.scale_log2;
        } else if (delta >= a.max_position && i == 0) {
          record_error(a.err, ERR_POS_RANGE, KID_ATTN_FMA, blockIdx.x, delta);
        }
        qs[r * D + i] = y1;
        qs[r * D + i + half] = y2;
      }
      cur_slot = pc.seg_slot;
    }
    const size_t base = (((size_t)pc.page * a.H_kv + g.h) * a.S + pc.slot0) * D;
    for (int t0 = 0; t0 < pc.ntok; t0 += kTile) {
      const int nt = min(kTile, pc.ntok - t0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < kTile * (D / 8); idx += kThreads) {
        const int tok = idx / (D / 8), c8 = (idx % (D / 8)) * 8;
        uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
        if (tok < nt) {
          kr = *reinterpret_cast<const uint4*>(a.k_layer + base + (size_t)(t0 + tok) * D + c8);
          vr = *reinterpret_cast<const uint4*>(a.v_layer + base + (size_t)(t0 + tok) * D + c8);
        }
        const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&kr);
        const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(&vr);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 kf = __bfloat1622float2(kp[j]);
          const float2 vf = __bfloat1622float2(vp[j]);
          ks[tok * KS + c8 + 2 * j] = kf.x;
          ks[tok * KS + c8 + 2 * j + 1] = kf.y;
          vs[tok * D + c8 + 2 * j] = vf.x;
          vs[tok * D + c8 + 2 * j + 1] = vf.y;
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxRowsPerWarp; ++k) {
        const int r = warp + k * kWarps;
        if (r >= rows) continue;
        if (dl[r / a.G] < 0) continue;              // this worker does not see the segment
        // causal cut (several query tokens per worker): tokens of the segment it may see
        const int cap = a.vlen ? a.vlen[(size_t)pc.seg_slot * a.W + r / a.G] : pc.pos0 + pc.ntok;
        const float* qr = qs + r * D;
        const float* kr = ks + lane * KS;
        float s = 0.f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) s = fmaf(qr[d], kr[d], s);
        if (lane >= nt || pc.pos0 + t0 + lane >= cap) s = -CUDART_INF_F;
        float tmax = s;
#pragma unroll
        for (int off = 16; off; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        if (tmax == -CUDART_INF_F) continue;        // nothing of this tile is visible to the row
        const float mn = fmaxf(m[k], tmax);
        const float alpha = exp2f(m[k] - mn);
        const float p = exp2f(s - mn);
        float ps = p;
#pragma unroll
        for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l[k] = l[k] * alpha + ps;
#pragma unroll
        for (int j = 0; j < DJ; ++j) o[k][j] *= alpha;
        for (int t = 0; t < nt; ++t) {
          const float pt = __shfl_sync(0xffffffffu, p, t);
#pragma unroll
          for (int j = 0; j < DJ; ++j) o[k][j] = fmaf(pt, vs[t * D + lane + 32 * j], o[k][j]);
        }
        m[k] = mn;
      }
    }
  }
  // Partial result of this unit: o (unnormalised), m, l in the log2 domain.
#pragma unroll
  for (int k = 0; k < kMaxRowsPerWarp; ++k) {
    const int r = warp + k * kWarps;
    if (r >= rows) continue;
    float* part = a.partials + ((size_t)blockIdx.x * rows + r) * part_stride(D);
#pragma unroll
    for (int j = 0; j < DJ; ++j) part[lane + 32 * j] = o[k][j];
    if (lane == 0) {
      part[D] = m[k];
      part[D + 1] = l[k];
    }
  }
}

// K3: the log-sum-exp merge of the units' partials (merge_row, hw_merge.cuh), one warp per
// (group, query row), as a kernel of its own: used after the CUDA-core attention and after the
// tensor-core attention when that kernel does not merge itself.
//
// Register budget: at most 144 registers, with 20 units' loads in flight per row at once (the
// benchmark workload has 19 units per group).  Measured: 32.85 -> 32.63 us per decode step on
// the 32K-common, 8-worker workload, 1.359 -> 1.326 ms per 64-layer step on the 16K-common one.
// (At 144 registers a merge CTA and a CTA of the next call's attention kernel, 8 warps at
// 184 registers as allocated, fit one SM's 65,536 registers; the shared-memory split still
// keeps them apart, and forcing the large split made the step slower.)
constexpr int kMergeWarps = 4;
constexpr int kMergeChunk = 20;

template <int D>
__global__ void __maxnreg__(144) merge_kernel(const AttnArgs a) {
  // May be launched as a programmatic dependent of the attention kernel: wait for its writes.
  // Whatever follows may start its own prologue now (the library's kernels wait for this grid
  // before they read anything it writes or overwrite the partials it reads).
  HW_SPAN_BEGIN(0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * kMergeWarps + warp;
  const bool valid = item < a.num_groups * a.rows;
  const int gi = valid ? item / a.rows : 0, r = item - gi * a.rows;
  // The group entry belongs to the call's plan, not to what the attention kernel writes: it is
  // read before the wait once the plan's sequence word shows that the plan has arrived (an
  // acquire load; plans without a word were copied before the attention kernel started).
  Group g{};
  bool have_g = false;
  if (valid && plan_seq_now(a.gate) == a.gate.plan_expect) {
    g = a.groups[gi];
    have_g = true;
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  HW_SPAN_BEGIN(1);
  if (valid) {
    if (!have_g) g = a.groups[gi];
    merge_row<D, kMergeChunk>(a, gi, r, g, lane);
  }
  HW_SPAN_END(0);
}

template <int D>
constexpr size_t fma_smem_bytes(int rows) {
  return ((size_t)rows * D + kTile * (D + 1) + kTile * D) * sizeof(float);
}

template <int D>
void launch_fma_d(const AttnArgs& a, cudaStream_t s) {
  attn_fma_kernel<D><<<a.num_units, kThreads, fma_smem_bytes<D>(a.rows), s>>>(a);
}

}  // namespace

HW_SPAN_EXPORT(merge)

cudaError_t prepare_attention_fma(int D) {
  // Shared-memory limit for the largest row count a context may have (128 query rows).
  if (D == 64)
    return cudaFuncSetAttribute(attn_fma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)fma_smem_bytes<64>(128));
  return cudaFuncSetAttribute(attn_fma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)fma_smem_bytes<128>(128));
}

void launch_attention_fma(const AttnArgs& a, cudaStream_t s) {
  if (a.num_units <= 0) return;
  if (a.D == 64)
    launch_fma_d<64>(a, s);
  else
    launch_fma_d<128>(a, s);
}

void launch_merge(const AttnArgs& a, cudaStream_t s, bool pdl) {
  if (a.num_groups <= 0) return;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.num_groups * a.rows + kMergeWarps - 1) / kMergeWarps);
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.D == 64)
    cudaLaunchKernelEx(&cfg, merge_kernel<64>, a);
  else
    cudaLaunchKernelEx(&cfg, merge_kernel<128>, a);
}

}  // namespace hw
