// dsa_host.h - host-side helpers shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "dsa.h"

namespace dsa {

// Records a failed CUDA call for dsa_last_cuda_error() and returns DSA_ERR_CUDA.
dsa_status_t cuda_fail(cudaError_t e);

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};

// Properties of the current device (cached per device). Returns DSA_ERR_NO_DEVICE when the
// current device is not compute capability 10.3.
dsa_status_t current_device(DeviceInfo* out);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace dsa
