// Device-side plumbing shared by the CUDA translation units: stream conversion, the
// per-device properties a launch needs, launch-error mapping.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <utility>

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

// Launches `kernel` with programmatic stream serialization, so that its launch and set-up
// overlap the tail of the previous kernel in the stream; the kernel itself waits for that
// kernel (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
gtp_status launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             const char *what, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = std::getenv("GTP_NO_LAUNCH_OVERLAP") ? 0 : 1;  // plain stream order (A/B timing)
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return fail(GTP_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return check_launch(what);
}

}  // namespace gtp
