// K1 -- KV append: each new token's key is rotated to its block-local position and stored as
// bf16 into its page; the value is copied (Hogwild! Inference summary, gentlecold.top,
// section 9: tokens of a block are stored at local positions 0 .. len-1; section 8: every
// worker appends its K/V to its own block before attention).
//
// Work: one CTA per (run, 16-token chunk); a thread per (token, KV head, rotation pair).  The
// kernel is a few KB per decode step, so it is written for clarity, not for bandwidth.
#include <cuda_bf16.h>

#include "hw_device.cuh"

namespace hw {
namespace {

constexpr int kTokPerCta = 16;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
  // The next kernels of the step (query rotation, attention) may start their own prologue now;
  // they wait for this grid before reading what it writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched as a programmatic dependent of whatever precedes it on the stream (which may
  // produce k_raw / v_raw): wait for that grid before reading anything it could write.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  HW_SPAN_BEGIN(0);
  __shared__ int plan_ok;
  if (threadIdx.x == 0) plan_ok = plan_arrived(a.gate, plan_seq_now(a.gate), a.err, KID_APPEND);
  __syncthreads();
  if (!plan_ok) return;
  const AppendRun run = a.runs[blockIdx.y];
  const int t0 = blockIdx.x * kTokPerCta;
  if (t0 >= run.ntok) return;
  if (run.page < 0 || run.page >= a.num_pages) {
    if (threadIdx.x == 0) record_error(a.err, ERR_PAGE_RANGE, KID_APPEND, blockIdx.y, run.page);
    return;
  }
  if (run.slot0 < 0 || run.slot0 + run.ntok > a.S) {
    if (threadIdx.x == 0) record_error(a.err, ERR_SLOT_RANGE, KID_APPEND, blockIdx.y, run.slot0);
    return;
  }
  if (run.pos0 < 0 || run.pos0 + run.ntok > a.max_position) {
    if (threadIdx.x == 0) record_error(a.err, ERR_POS_RANGE, KID_APPEND, blockIdx.y, run.pos0);
    return;
  }
  const int nt = min(kTokPerCta, run.ntok - t0);
  const int half = a.D >> 1;
  const int work = nt * a.H_kv * half;
  for (int idx = threadIdx.x; idx < work; idx += kThreads) {
    const int i = idx % half;
    const int th = idx / half;
    const int h = th % a.H_kv;
    const int t = t0 + th / a.H_kv;
    const size_t src = ((size_t)(run.src_tok + t) * a.H_kv + h) * a.D;
    const size_t dst = (((size_t)run.page * a.H_kv + h) * a.S + run.slot0 + t) * a.D;
    const size_t tab = (size_t)(run.pos0 + t) * half + i;
    const float c = a.rope_cos[tab];
    const float s = a.rope_sin[tab];
    const float x1 = __bfloat162float(a.k_raw[src + i]);
    const float x2 = __bfloat162float(a.k_raw[src + i + half]);
    a.k_layer[dst + i] = __float2bfloat16_rn(x1 * c - x2 * s);
    a.k_layer[dst + i + half] = __float2bfloat16_rn(x2 * c + x1 * s);
    a.v_layer[dst + i] = a.v_raw[src + i];
    a.v_layer[dst + i + half] = a.v_raw[src + i + half];
  }
  HW_SPAN_END(0);
}

}  // namespace

HW_SPAN_EXPORT(append)

void launch_append(const AppendArgs& a, cudaStream_t s) {
  for (int r0 = 0; r0 < a.num_runs; r0 += 65535) {
    AppendArgs b = a;
    b.runs = a.runs + r0;
    b.num_runs = a.num_runs - r0 < 65535 ? a.num_runs - r0 : 65535;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.max_run + kTokPerCta - 1) / kTokPerCta, b.num_runs);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, append_kernel, b);
  }
}

}  // namespace hw
