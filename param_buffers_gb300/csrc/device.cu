#include <mutex>

#include "device.h"

namespace gtp {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];
}  // namespace

gtp_status current_device(DeviceInfo *out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GTP_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GTP_E_DEVICE, "device ordinal %d unsupported", dev);
  cudaError_t qerr = cudaSuccess;
  std::call_once(g_once[dev], [&] {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if ((qerr = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev))) return;
    if ((qerr = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev))) return;
    if ((qerr = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev))) return;
    if ((qerr = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev))) return;
    d.smem_optin = size_t(v);
    g_info[dev] = d;
  });
  if (qerr != cudaSuccess) return fail(GTP_E_CUDA, "device query: %s", cudaGetErrorString(qerr));
  if (g_info[dev].device != dev) return fail(GTP_E_CUDA, "device %d properties unavailable", dev);
  *out = g_info[dev];
  return GTP_OK;
}

gtp_status require_sm103(DeviceInfo *out) {
  gtp_status s = current_device(out);
  if (s != GTP_OK) return s;
  if (out->cc_major != 10 || out->cc_minor != 3)
    return fail(GTP_E_DEVICE, "compute capability %d.%d: this library is built for sm_103a only",
                out->cc_major, out->cc_minor);
  return GTP_OK;
}

gtp_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(GTP_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return GTP_OK;
}

}  // namespace gtp
