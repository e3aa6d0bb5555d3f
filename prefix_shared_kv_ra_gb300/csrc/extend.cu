// extend.cu -- placeholder until the tensor-core extend kernel lands.
#include "api_common.h"
#include "decode_internal.h"

namespace ra {
ra_status launch_cascade_prefix(const DecodeParams&, const CascadeArgs&, int32_t, cudaStream_t) {
  return fail(RA_ERR_UNSUPPORTED, "cascade decode not built yet");
}
}  // namespace ra

extern "C" ra_status ra_extend_attention(const void*, const void*, int64_t, int32_t, int32_t, const void*, void*,
                                         int32_t, float, const int32_t*, int64_t, int64_t, const int32_t*,
                                         const int32_t*, const int32_t*, const int32_t*, int32_t, int64_t, int32_t,
                                         int32_t, uint32_t*, ra_stream_t) {
  ra::clear_error();
  return ra::fail(RA_ERR_UNSUPPORTED, "extend not built yet");
}
