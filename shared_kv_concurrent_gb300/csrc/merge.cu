// K3 -- the log-sum-exp merge of the per-unit partial results of either attention kernel
// (Hogwild! Inference summary, gentlecold.top, section 9: the work is split over KV entries and
// the partial results reduced; section 5: per-block softmax statistics combine by log-sum-exp).
// The arithmetic of one query row is in hw_merge.cuh.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "hw_merge.cuh"

namespace hw {
namespace {

// K3: the log-sum-exp merge of the units' partials (hw_merge.cuh), `split` warps per (group,
// query row) -- one, or two or four when a group has more units than one warp keeps in flight
// (each warp folds its share of the units, the first combines the others' states through shared
// memory) -- as a kernel of its own, after either attention kernel.
//
// Register budget: at most 144 registers, with 20 units' loads in flight per warp at once (the
// benchmark workload has 19 units per group).  Measured: 32.85 -> 32.63 us per decode step on
// the 32K-common, 8-worker workload, 1.359 -> 1.326 ms per 64-layer step on the 16K-common one.
// (At 144 registers a merge CTA and a CTA of the next call's attention kernel, 8 warps at
// 184 registers as allocated, fit one SM's 65,536 registers; the shared-memory split still
// keeps them apart, and forcing the large split made the step slower.)
constexpr int kMergeWarps = 4;
constexpr int kMergeChunk = 20;
constexpr int64_t kMergeSplitWarps = 1024;   // rows are split only while the grid stays this small

template <int D, int split>
__global__ void __maxnreg__(144) merge_kernel(const AttnArgs a) {
  // May be launched as a programmatic dependent of the attention kernel: wait for its writes.
  // Whatever follows may start its own prologue now (the library's kernels wait for this grid
  // before they read anything it writes or overwrite the partials it reads).
  __shared__ MergeAcc others[split > 1 ? kMergeWarps : 1][32];
  HW_SPAN_BEGIN(0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = warp % split;                    // this warp's share of the row's units
  const int item = blockIdx.x * (kMergeWarps / split) + warp / split;
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
  MergeAcc acc{-CUDART_INF_F, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  bool ok = false;
  if (valid) {
    if (!have_g) g = a.groups[gi];
    ok = merge_group_ok(a, gi, r, g, lane);
    if (ok) {
      const int nu = g.unit_end - g.unit_begin;
      const int share = (nu + split - 1) / split;
      const int kb = min(nu, part * share), ke = min(nu, kb + share);
      merge_units<D, kMergeChunk>(a, r, g, kb, ke, lane, acc);
    }
  }
  if constexpr (split > 1) {
    if (part > 0) others[warp][lane] = acc;
    __syncthreads();
    if (part == 0)
      for (int k = 1; k < split; ++k) merge_combine(acc, others[warp + k][lane]);
  }
  if (ok && part == 0) merge_store<D>(a, r, g, lane, acc);
  HW_SPAN_END(0);
}

}  // namespace

HW_SPAN_EXPORT(merge)

void launch_merge(const AttnArgs& a, cudaStream_t s, bool pdl, int max_group_units) {
  if (a.num_groups <= 0) return;
  // Warps per row: enough that each folds at most one batch of units (up to kMergeWarps), for a
  // merge of few rows only.  With many rows the grid is large already, and splitting every row
  // for the sake of a few long groups made the 16-problem workload's step slower
  // (150.5-151.7 -> 154.8 us).
  int split = max_group_units > 2 * kMergeChunk ? 4 : max_group_units > kMergeChunk ? 2 : 1;
  while (split > 1 && (int64_t)a.num_groups * a.rows * split > kMergeSplitWarps) split /= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.num_groups * a.rows * split + kMergeWarps - 1) / kMergeWarps);
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const bool d64 = a.D == 64;
  if (split == 1)
    cudaLaunchKernelEx(&cfg, d64 ? merge_kernel<64, 1> : merge_kernel<128, 1>, a);
  else if (split == 2)
    cudaLaunchKernelEx(&cfg, d64 ? merge_kernel<64, 2> : merge_kernel<128, 2>, a);
  else
    cudaLaunchKernelEx(&cfg, d64 ? merge_kernel<64, 4> : merge_kernel<128, 4>, a);
}

}  // namespace hw
