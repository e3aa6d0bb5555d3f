// decode_static.cu -- ra_decode_attention_static: decode attention for callers
// that cannot allocate device memory.
//
// ra_decode_attention needs a caller-provided workspace for its split-KV
// partial results.  Some callers have no way to get one: a plugin that runs
// inside a host framework's pre-planned memory budget and may not call
// cudaMalloc after start-up, a runtime without a device allocator of its own,
// or code that must not touch the allocator at all.  This entry point takes the
// same inputs and outputs but keeps its scratch in one file-scope device array
// of RA_DECODE_STATIC_SCRATCH_BYTES (32 MiB), which every GPU that loads this
// library holds until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (the array's name in host
// code is only a host-side stand-in) and caches it per device, together with
// the CUDA context it belongs to.  The address is valid for that context's
// lifetime: after the context is destroyed and another one is created on the
// device (cudaDeviceReset, for instance), the module is loaded again and the
// array may sit elsewhere, so the first call in the new context looks it up
// again (so does the first call of a host thread that has not used CUDA
// before).  Make the first call in each context outside any stream capture.
// The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
// library routine.  It then runs the normal decode
// path with the array as its workspace, so its results are those of
// ra_decode_attention.  All calls share the one array and it keeps the last
// call's contents (the decode path writes every partial before reading it and
// clears the one field that must start at zero itself), so calls that overlap
// on the GPU -- on different streams, or on one stream from several threads
// without ordering -- race on it.
#include <cuda.h>

#include <mutex>

#include "api_common.h"

namespace ra {
namespace {

__device__ __align__(256) uint8_t g_decode_scratch[RA_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The driver's cuCtxGetCurrent, taken through the runtime (the library does not link libcuda).
using CtxGetCurrent = CUresult (*)(CUcontext*);
CtxGetCurrent ctx_get_current() {
  static CtxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrent>(ptr);
  });
  return fn;
}

// Device address of g_decode_scratch on the current device, looked up once per device and context.
ra_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_CUDA, "device ordinal %d out of range", dev);
  CtxGetCurrent get_ctx = ctx_get_current();
  if (!get_ctx) return fail(RA_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
  // null on a host thread that has not used CUDA yet: the lookup below makes the device's context current
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(RA_ERR_CUDA, "cudaGetSymbolAddress(static decode scratch): %s", cudaGetErrorString(e));
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return fail(RA_ERR_CUDA, "no current CUDA context");
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return RA_OK;
}

}  // namespace
}  // namespace ra

extern "C" ra_status ra_decode_attention_static(
    const void* k_pool, const void* v_pool, int64_t num_slots, int32_t num_kv_heads, int32_t head_dim, const void* q,
    void* o, int32_t num_q_heads, float sm_scale, const int32_t* req_to_token, int64_t table_stride,
    int64_t table_rows, const int32_t* req_pool_indices, const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
    int32_t num_groups, const int32_t* group_indptr, const int32_t* group_reqs, const int32_t* group_prefix_start,
    const int32_t* group_prefix_len, const int32_t* group_level, int32_t max_group_prefix_len, int32_t max_group_size,
    int32_t max_group_levels, uint32_t* device_error, ra_stream_t stream) {
  using namespace ra;
  clear_error();
  void* scratch = nullptr;
  if (ra_status st = scratch_for_current_device(&scratch)) return st;
  const size_t need = ra_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                                num_groups, max_group_prefix_len, max_group_size, max_group_levels);
  if (need > static_cast<size_t>(RA_DECODE_STATIC_SCRATCH_BYTES))
    return fail(RA_ERR_WORKSPACE,
                "this decode needs %zu bytes of scratch; the static scratch holds %zu "
                "(use ra_decode_attention with a caller workspace)",
                need, static_cast<size_t>(RA_DECODE_STATIC_SCRATCH_BYTES));
  return ra_decode_attention(k_pool, v_pool, num_slots, num_kv_heads, head_dim, q, o, num_q_heads, sm_scale,
                             req_to_token, table_stride, table_rows, req_pool_indices, seq_lens, batch, max_seq_len,
                             num_groups, group_indptr, group_reqs, group_prefix_start, group_prefix_len, group_level,
                             max_group_prefix_len, max_group_size, max_group_levels, scratch,
                             static_cast<size_t>(RA_DECODE_STATIC_SCRATCH_BYTES), device_error, stream);
}
