// Device-side helpers shared by the kernels of libhogwild.
#pragma once

#include <cuda_bf16.h>

#include "hw_internal.h"

namespace hw {

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

}  // namespace hw
