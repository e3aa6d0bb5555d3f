// api_common.cu -- status strings, thread-local error text, device properties.
#include <mutex>

#include "api_common.h"
#include "ra_ptx.cuh"

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

namespace ra {
namespace {

__device__ int32_t g_never_counted = 0;  // no thread ever writes it

// One CTA: warp 0 waits on an mbarrier no thread arrives at, warp 1 on a counter no thread raises, both
// with the caller's deadline and the same bounded-wait primitives every kernel of the library uses.
// Both waits run out; each warp flags RA_DEVERR_TIMEOUT and the kernel returns.
__global__ void selftest_bounded_wait_kernel(long long deadline, uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = threadIdx.x < 32 ? mbar_wait(smem_u32(&bar), 0, deadline)
                                   : wait_count(&g_never_counted, 1, deadline);
  if (!ok && (threadIdx.x & 31) == 0) flag_error(err, RA_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace ra

extern "C" ra_status ra_selftest_bounded_wait(int64_t deadline_cycles, uint32_t* device_error, ra_stream_t stream) {
  using namespace ra;
  clear_error();
  RA_REQUIRE(deadline_cycles > 0 && deadline_cycles <= (int64_t(1) << 32), "deadline_cycles must be in (0, 2^32]");
  RA_REQUIRE(device_error && aligned4(device_error), "device_error must be a non-null, 4-byte aligned pointer");
  selftest_bounded_wait_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(deadline_cycles, device_error);
  return check_launch("selftest_bounded_wait_kernel");
}
