// api_common.cu -- status strings, thread-local error text, device properties.
#include <mutex>

#include "api_common.h"

namespace ra {

static thread_local char g_last_error[512] = "";

ra_status fail(ra_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = '\0'; }

ra_status current_device(DeviceInfo* out) {
  constexpr int kMaxDevices = 64;
  static DeviceInfo cache[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].device != dev) {
    DeviceInfo d;
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
      return fail(RA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    }
    cache[dev] = d;
  }
  *out = cache[dev];
  return RA_OK;
}

ra_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  return RA_OK;
}

}  // namespace ra

extern "C" const char* ra_status_string(ra_status status) {
  switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported shape";
    case RA_ERR_WORKSPACE: return "workspace too small";
    case RA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

extern "C" const char* ra_last_error_message(void) { return ra::g_last_error; }

extern "C" int32_t ra_abi_version(void) { return RA_ABI_VERSION; }
