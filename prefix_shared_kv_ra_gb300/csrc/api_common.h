// api_common.h -- host-side helpers shared by the C-ABI entry points:
// thread-local error text, argument checks, per-device properties.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>

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

}  // namespace ra

#define RA_REQUIRE(cond, ...)                                              \
  do {                                                                     \
    if (!(cond)) return ::ra::fail(RA_ERR_INVALID_ARGUMENT, __VA_ARGS__);  \
  } while (0)
