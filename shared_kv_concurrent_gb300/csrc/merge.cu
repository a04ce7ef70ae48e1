// K3 -- the log-sum-exp merge of the per-unit partial results of either attention kernel
// (Hogwild! Inference summary, gentlecold.top, section 9: the work is split over KV entries and
// the partial results reduced; section 5: per-block softmax statistics combine by log-sum-exp).
// The arithmetic of one query row is merge_row (hw_merge.cuh).
#include <cuda_bf16.h>

#include "hw_device.cuh"
#include "hw_merge.cuh"

namespace hw {
namespace {

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

}  // namespace

HW_SPAN_EXPORT(merge)

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
