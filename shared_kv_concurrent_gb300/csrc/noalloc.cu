// hw_concurrent_attention_noalloc: the concurrent-attention call for callers that cannot
// allocate device memory when they call it.
//
// The regular call keeps its per-call plan and its split-K partial results in the workspace
// the caller sized with hw_workspace_size() and allocated up front.  Some callers cannot do
// that: a host framework that owns all device memory and exposes no allocator to plug-ins, or
// code that must not call cudaMalloc at that point (for example while another component is
// capturing a CUDA graph on the device, where an allocation would break the capture).  This
// entry point needs no caller scratch at all: its scratch is one fixed-size array in device
// global memory, defined below, which every GPU that loads this library holds until the
// process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
#include <mutex>

#include "hw_internal.h"

namespace {

// 16 MiB: room for the plan and the partial results of well over 200 units of 64 rows at
// head_dim 128 (one unit needs rows * (head_dim + 4) * 4 bytes: o, m, l and two pad floats).
constexpr size_t kScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the array's name
// is only a stand-in, not a device address, so it is looked up once per device.
hw_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return HW_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HW_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return HW_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return HW_OK;
}

}  // namespace

extern "C" hw_status hw_concurrent_attention_noalloc(hw_ctx* ctx, int32_t layer, const void* q,
                                                     void* out, int32_t out_dtype, float* lse,
                                                     void* stream) {
  if (!ctx || !q || !out) return HW_ERR_INVALID_ARG;
  // Each call copies its plan from a pinned staging slot that later calls reuse, and may wait
  // on events recorded on `stream`: neither can be replayed from a graph, so a capturing stream
  // is refused before anything is enqueued.  (Another stream's capture does not matter.)
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    return HW_ERR_UNSUPPORTED;
  }
  if (cap != cudaStreamCaptureStatusNone) return HW_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const hw_status st = scratch_address(&scratch);
  if (st != HW_OK) return st;
  return hw::attention_into_scratch(ctx, layer, q, out, out_dtype, lse, stream,
                                    static_cast<char*>(scratch), kScratchBytes);
}
