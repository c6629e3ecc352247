// Device-side plumbing shared by the CUDA translation units: stream conversion, the
// per-device properties a launch needs, launch-error mapping.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "gtp.h"
#include "status.h"

namespace gtp {

inline cudaStream_t as_stream(gtp_stream s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};

// Properties of the current device (queried once per device and cached).
gtp_status current_device(DeviceInfo *out);

// Returns GTP_E_DEVICE unless the current device is compute capability 10.3.
gtp_status require_sm103(DeviceInfo *out);

// Maps the state after a launch to a status (GTP_E_CUDA with the CUDA message).
gtp_status check_launch(const char *what);

}  // namespace gtp
