// api_common.h -- host-side helpers shared by the C-ABI entry points:
// thread-local error text, argument checks, per-device properties.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <utility>

#include "../../include/ra.h"

namespace ra {

// Record a formatted failure message for ra_last_error_message() and return `st`.
ra_status fail(ra_status st, const char* fmt, ...);
// Clear the thread's last message (called at the start of each entry point).
void clear_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int max_smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};

// Properties of the current device (queried once per device, then cached).
ra_status current_device(DeviceInfo* out);

// Map the last launch error (if any) to RA_ERR_CUDA with a message.
ra_status check_launch(const char* what);

// Launch `kern` on `stream` with programmatic stream serialization: it may start while the previous
// kernel on the stream runs, once every CTA of that kernel has called griddepcontrol.launch_dependents.
// Every kernel of this library calls griddepcontrol.wait before it touches memory its predecessor may
// still be writing or reading, so the early start only overlaps launch latency, prologues and tails.
template <typename... KArgs, typename... Args>
ra_status launch_pdl(const char* what, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  return RA_OK;
}

}  // namespace ra

#define RA_REQUIRE(cond, ...)                                              \
  do {                                                                     \
    if (!(cond)) return ::ra::fail(RA_ERR_INVALID_ARGUMENT, __VA_ARGS__);  \
  } while (0)
