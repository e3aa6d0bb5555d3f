// kv_store.cu -- ra_kv_store: scatter this step's new K/V rows into pool slots.
//
// The pool is token-granular: one slot holds one token's K (and V) for every
// kv head, Hkv * D bf16 = 2 KB contiguous at Hkv = 8, D = 128.  A slot row is
// therefore a contiguous run of 16-byte vectors, and the scatter is a plain
// vectorised copy whose only irregularity is the destination row: each thread
// moves one 16-byte vector of K and the same vector of V, consecutive threads
// take consecutive vectors of a row, so both the reads and the writes of a row
// coalesce into full 128-byte lines.  The work is HBM-bound (read N rows,
// write N rows); the grid is a few waves of the SMs with a grid-stride loop.
// Source: anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一 (new
// tokens are written at out_cache_loc, graph padding writes slot 0).
#include "api_common.h"
#include "ra_ptx.cuh"

namespace ra {

__global__ void __launch_bounds__(256) kv_store_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                       int64_t num_slots, int32_t row_vecs,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int32_t* __restrict__ loc, int64_t total_vecs,
                                                       uint32_t* __restrict__ err) {
  griddep_wait();  // earlier kernels may still read the pool rows this store overwrites
  griddep_launch();
  // kU vectors of K and of V per thread and step, all loads issued before the stores (bytes in flight)
  constexpr int kU = 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total_vecs;
       i0 += kU * stride) {
    uint4 kv[kU], vv[kU];
    int32_t slot[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total_vecs) {
        slot[u] = __ldg(loc + i / row_vecs);
        kv[u] = __ldg(k_new + i);
        vv[u] = __ldg(v_new + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= total_vecs) break;
      const int64_t tok = i / row_vecs;
      const int32_t c = static_cast<int32_t>(i - tok * row_vecs);
      if (slot[u] < 0 || slot[u] >= num_slots) {
        if (c == 0) flag_error(err, RA_DEVERR_SLOT);
        continue;
      }
      const int64_t dst = static_cast<int64_t>(slot[u]) * row_vecs + c;
      k_pool[dst] = kv[u];
      v_pool[dst] = vv[u];
    }
  }
}

}  // namespace ra

extern "C" ra_status ra_kv_store(void* k_pool, void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                                 int32_t head_dim, const void* k_new, const void* v_new,
                                 const int32_t* out_cache_loc, int64_t num_tokens, uint32_t* device_error,
                                 ra_stream_t stream) {
  using namespace ra;
  clear_error();
  RA_REQUIRE(num_tokens >= 0, "num_tokens must be >= 0 (got %lld)", (long long)num_tokens);
  RA_REQUIRE(num_slots > 0, "num_slots must be > 0");
  RA_REQUIRE(num_kv_heads > 0 && head_dim > 0, "num_kv_heads and head_dim must be > 0");
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
  RA_REQUIRE(row_bytes % 16 == 0, "a slot row (num_kv_heads*head_dim*2 = %lld bytes) must be a multiple of 16",
             (long long)row_bytes);
  if (num_tokens == 0) return RA_OK;
  RA_REQUIRE(k_pool && v_pool && k_new && v_new && out_cache_loc, "null pointer argument");
  RA_REQUIRE(aligned16(k_pool) && aligned16(v_pool) && aligned16(k_new) && aligned16(v_new),
             "pools and new rows must be 16-byte aligned");
  RA_REQUIRE(aligned4(out_cache_loc), "out_cache_loc must be 4-byte aligned");
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  const int32_t row_vecs = static_cast<int32_t>(row_bytes / 16);
  const int64_t total = num_tokens * row_vecs;
  const int threads = 256;
  const int64_t want = (total + threads * 4 - 1) / (threads * 4);  // 4 vectors per thread
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  return launch_pdl("kv_store_kernel", kv_store_kernel, dim3(blocks), dim3(threads), 0,
                    reinterpret_cast<cudaStream_t>(stream), static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                    num_slots, row_vecs, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    out_cache_loc, total, device_error);
}
