// extend.cu -- ra_extend_attention and the cascade prefix pass of
// ra_decode_attention, both on the tcgen05 attention tile kernel.
//
// Extend is the dense contraction of this path: 128 query rows (128 / G
// suffix tokens x the G q heads of one kv head) against 128-key tiles of the
// request's context, QK^T and PV on the 5th-generation tensor cores with the
// accumulators in TMEM.  Grid: (query tile, kv head, request); CTAs of one
// (request, kv head) are adjacent so their shared prefix K/V tiles are served
// from L2.
// Sources: SGLang paper summary, §3 (reuse the cached prefix KV, compute
// only the suffix); yaopepe.com explainer, §04 (the matched prefix is
// referenced, the unmatched suffix is prefilled against it).
#include <cudaTypedefs.h>

#include <mutex>

#include "api_common.h"
#include "attn_tc.cuh"
#include "decode_internal.h"

namespace ra {

namespace {

// ------------------------------------------------------------------ work list
// The extend CTAs of a batch differ in length by two orders of magnitude (a query tile of a request
// with a 32K-token prefix sweeps 256 key tiles, one of a fresh request a single tile).  Launched in
// (tile, head, request) order, the longest can start last and leave most SMs idle at the end.  A
// one-CTA pass lists the (request, query tile) pairs by key-tile count, longest first (a counting
// sort); extend CTA x then takes entry x / Hkv, so the block scheduler hands out work longest first
// (greedy LPT list scheduling) and the Hkv CTAs of an entry, which gather rows of the same slots,
// run side by side.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBins = 4096;  // key-tile counts above kPlanBins - 1 share the first bin

struct ExtendWorkspace {
  int32_t* count;    // entries listed
  int32_t* counter;  // item claim counter of the persistent kernel
  int32_t* items;    // [2 * cap]
  int64_t cap;
  size_t total;
};

// Entries are at most sum_b ceil(E_b / tokens_per_cta) <= total_q / tokens_per_cta + batch.
ExtendWorkspace layout_extend_workspace(int32_t batch, int64_t total_q, int32_t tokens_per_cta, void* base) {
  ExtendWorkspace w{};
  w.cap = (total_q + tokens_per_cta - 1) / tokens_per_cta + batch;
  w.total = 16 + static_cast<size_t>(w.cap) * 8;
  uint8_t* b = static_cast<uint8_t*>(base);
  w.count = reinterpret_cast<int32_t*>(b);
  w.counter = reinterpret_cast<int32_t*>(b ? b + 4 : nullptr);
  w.items = reinterpret_cast<int32_t*>(b ? b + 16 : nullptr);
  return w;
}

__device__ __forceinline__ int32_t plan_bin(int32_t P, int32_t E, int32_t t, int32_t tokens_per_cta) {
  const int32_t kend = P + min(E, (t + 1) * tokens_per_cta);
  const int32_t cost = (kend + tc::kKeys - 1) / tc::kKeys;
  return kPlanBins - 1 - min(cost, kPlanBins - 1);  // bin 0 = longest
}

__global__ void __launch_bounds__(kPlanThreads) extend_plan_kernel(const int32_t* extend_lens,
                                                                  const int32_t* prefix_lens, int32_t batch,
                                                                  int32_t max_extend_len, int32_t max_prefix_len,
                                                                  int64_t table_stride, int32_t tokens_per_cta,
                                                                  int32_t* count, int32_t* counter, int32_t* items,
                                                                  int64_t cap, uint32_t* err) {
  __shared__ int32_t s_bin[kPlanBins];
  __shared__ int32_t s_warp[kPlanThreads / 32];
  griddep_launch();  // the extend kernel may start its launch; it waits for this grid before reading the list
  // (this grid waits for the previous one before its first write, so its completion implies that one's)
  for (int i = threadIdx.x; i < kPlanBins; i += kPlanThreads) s_bin[i] = 0;
  __syncthreads();
  // a request's tiles, or 0 if its lengths are invalid (flagged here, once)
  auto tiles_of = [&](int b, int32_t& P, int32_t& E, bool report) -> int32_t {
    E = __ldg(extend_lens + b);
    P = __ldg(prefix_lens + b);
    if (E < 0 || E > max_extend_len || P < 0 || P > max_prefix_len) {
      if (report) flag_error(err, RA_DEVERR_LENGTH);
      E = min(max(E, 0), max_extend_len);  // the rows within the bound are still computed
      if (P < 0 || P > max_prefix_len) return 0;
    }
    if (static_cast<int64_t>(P) + E > table_stride) {
      if (report) flag_error(err, RA_DEVERR_LENGTH);
      return 0;
    }
    return (E + tokens_per_cta - 1) / tokens_per_cta;
  };
  for (int b = threadIdx.x; b < batch; b += kPlanThreads) {
    int32_t P, E;
    const int32_t n = tiles_of(b, P, E, true);
    for (int32_t t = 0; t < n; ++t) atomicAdd(&s_bin[plan_bin(P, E, t, tokens_per_cta)], 1);
  }
  __syncthreads();
  // exclusive scan of the bins: thread i owns bins [4i, 4i + 4)
  constexpr int kPer = kPlanBins / kPlanThreads;
  int32_t v[kPer], run = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    v[e] = run;
    run += s_bin[threadIdx.x * kPer + e];
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int32_t base = (warp > 0 ? s_warp[warp - 1] : 0) + incl - run;
  const int32_t total = s_warp[kPlanThreads / 32 - 1];
#pragma unroll
  for (int e = 0; e < kPer; ++e) s_bin[threadIdx.x * kPer + e] = base + v[e];
  __syncthreads();
  // Everything above read only the call's inputs.  The writes below wait for the previous kernel: it may
  // be the previous call's extend kernel on this workspace, still claiming from its list and counter.
  griddep_wait();
  for (int b = threadIdx.x; b < batch; b += kPlanThreads) {
    int32_t P, E;
    const int32_t n = tiles_of(b, P, E, false);
    for (int32_t t = 0; t < n; ++t) {
      const int32_t pos = atomicAdd(&s_bin[plan_bin(P, E, t, tokens_per_cta)], 1);
      if (pos < cap) {
        items[2 * pos] = b;
        items[2 * pos + 1] = t;
      } else {
        flag_error(err, RA_DEVERR_LENGTH);  // extend_lens sum above total_q
      }
    }
  }
  if (threadIdx.x == 0) {
    *count = static_cast<int32_t>(static_cast<int64_t>(total) < cap ? total : cap);
    *counter = 0;
  }
}

// K ring / V ring depths: the tensor core waits on K first, so K gets the deeper ring.
template <int D>
constexpr int k_stages() { return D == 128 ? 3 : 4; }
template <int D>
constexpr int v_stages() { return D == 128 ? 2 : 4; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view [rows, head_dim] of a bf16 array whose rows are head_dim contiguous elements, read as
// one 64-element (128-byte, 128B-swizzled) column block of 1 row: the box a TMA gather4 takes.
ra_status row_gather_map(CUtensorMap* map, const void* base, int64_t rows, int32_t head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (rows <= 0 || rows > INT32_MAX) return fail(RA_ERR_UNSUPPORTED, "%lld rows exceed a TMA row coordinate", (long long)rows);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t elem[2] = {1, 1};
  CUresult cr = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled(rows) failed (%d)", static_cast<int>(cr));
  return RA_OK;
}

// Opt the kernel into its dynamic shared memory and check that it was compiled to the per-thread
// register count its setmaxnreg split is balanced against (a split above the block's launch
// allocation would leave the softmax warps waiting for registers that never come).
template <typename Kern>
ra_status set_smem(Kern kern, int bytes, bool* configured, int device) {
  if (configured[device]) return RA_OK;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaFuncGetAttributes(attn_tc): %s", cudaGetErrorString(e));
  if (fa.numRegs != tc::kLaunchRegs)
    return fail(RA_ERR_UNSUPPORTED, "attn_tc kernel compiled to %d registers per thread, its register split needs %d",
                fa.numRegs, tc::kLaunchRegs);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaFuncSetAttribute(attn_tc): %s", cudaGetErrorString(e));
  configured[device] = true;
  return RA_OK;
}

template <int D>
ra_status launch_extend(const TcParams& p, const CUtensorMap& qmap, int64_t entries, cudaStream_t s) {
  CUtensorMap kmap, vmap;
  if (ra_status st = row_gather_map(&kmap, p.k_pool, p.num_slots * p.hkv, D)) return st;
  if (ra_status st = row_gather_map(&vmap, p.v_pool, p.num_slots * p.hkv, D)) return st;
  using L = tc::Layout<D, k_stages<D>(), v_stages<D>()>;
  auto kern = attn_tc_kernel<D, k_stages<D>(), v_stages<D>(), true>;
  static bool configured[64] = {};
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  if (L::kDynSmem > dev.max_smem_optin)
    return fail(RA_ERR_UNSUPPORTED, "extend kernel needs %d bytes of shared memory", L::kDynSmem);
  if (ra_status st = set_smem(kern, L::kDynSmem, configured, dev.device)) return st;
  // persistent: one CTA per SM (at most one per item)
  const int64_t items = entries * p.hkv;
  dim3 grid(static_cast<unsigned>(items < dev.num_sms ? items : dev.num_sms));
  return launch_pdl("attn_tc_kernel<extend>", kern, grid, dim3(tc::kThreads), L::kDynSmem, s, p, qmap, kmap, vmap);
}

template <int D>
ra_status launch_prefix(const TcParams& p, int grid_x, int num_groups, int32_t wave, cudaStream_t s, int32_t* ctas) {
  using L = tc::Layout<D, k_stages<D>(), v_stages<D>()>;
  auto kern = attn_tc_kernel<D, k_stages<D>(), v_stages<D>(), false>;
  static bool configured[64] = {};
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  if (L::kDynSmem > dev.max_smem_optin)
    return fail(RA_ERR_UNSUPPORTED, "prefix kernel needs %d bytes of shared memory", L::kDynSmem);
  if (ra_status st = set_smem(kern, L::kDynSmem, configured, dev.device)) return st;
  CUtensorMap qmap, kmap, vmap;
  if (ra_status st = row_gather_map(&qmap, p.q, static_cast<int64_t>(p.batch) * p.hq, D)) return st;
  if (ra_status st = row_gather_map(&kmap, p.k_pool, p.num_slots * p.hkv, D)) return st;
  if (ra_status st = row_gather_map(&vmap, p.v_pool, p.num_slots * p.hkv, D)) return st;
  // persistent: one CTA per SM (at most one per item)
  const int64_t items = static_cast<int64_t>(grid_x) * p.hkv * num_groups;
  // at most the wave the splits were planned for: the SMs beyond it run the private decode beside the pass
  // (multi-turn mix: 230 -> 223 us for the decode call, the other workloads unchanged)
  int64_t cap = dev.num_sms;
  if (wave > 0 && wave < cap) cap = wave;
  dim3 grid(static_cast<unsigned>(items < cap ? items : cap));
  *ctas = static_cast<int32_t>(grid.x);
  return launch_pdl("attn_tc_kernel<cascade prefix>", kern, grid, dim3(tc::kThreads), L::kDynSmem, s, p, qmap, kmap,
                    vmap);
}

}  // namespace

ra_status launch_cascade_prefix(const DecodeParams& d, const CascadeArgs& ca, int32_t head_dim,
                                cudaStream_t stream, int32_t* ctas) {
  if (128 % d.group != 0)
    return fail(RA_ERR_UNSUPPORTED, "GQA group %d does not divide the 128-row tile", d.group);
  TcParams p{};
  p.k_pool = d.k_pool;
  p.v_pool = d.v_pool;
  p.num_slots = d.num_slots;
  p.hkv = d.hkv;
  p.q = d.q;
  p.hq = d.hq;
  p.group = d.group;
  p.scale_log2 = d.scale_log2;
  p.table = d.table;
  p.table_stride = d.table_stride;
  p.table_rows = d.table_rows;
  p.err = d.err;
  p.rpi = d.rpi;
  p.group_indptr = ca.group_indptr;
  p.group_reqs = ca.group_reqs;
  p.group_prefix_start = ca.group_prefix_start;
  p.group_prefix_len = ca.group_prefix_len;
  p.group_level = ca.group_level;
  p.casc_levels = ca.max_group_levels;
  p.casc_slots = d.casc_slots;
  p.batch = d.batch;
  p.max_seq_len = d.max_seq_len;
  p.cchunk = d.cchunk;
  p.max_csplits = d.max_csplits;
  p.casc_o = d.casc_o;
  p.casc_lse = d.casc_lse;
  p.work_counter = d.prefix_counter;
  p.done_counter = d.prefix_done;
  p.num_groups = ca.num_groups;
  const int members_per_cta = tc::kTiles * (128 / d.group);
  const int mtiles = (ca.max_group_size + members_per_cta - 1) / members_per_cta;
  const int grid_x = mtiles * d.max_csplits;
  p.grid_x = grid_x;
  return head_dim == 128 ? launch_prefix<128>(p, grid_x, ca.num_groups, d.prefix_wave, stream, ctas)
                         : launch_prefix<64>(p, grid_x, ca.num_groups, d.prefix_wave, stream, ctas);
}

}  // namespace ra

extern "C" ra_status ra_extend_attention(const void* k_pool, const void* v_pool, int64_t num_slots,
                                         int32_t num_kv_heads, int32_t head_dim, const void* q, void* o,
                                         int32_t num_q_heads, float sm_scale, const int32_t* req_to_token,
                                         int64_t table_stride, int64_t table_rows, const int32_t* req_pool_indices,
                                         const int32_t* prefix_lens, const int32_t* extend_lens,
                                         const int32_t* qo_indptr, int32_t batch, int64_t total_q,
                                         int32_t max_extend_len, int32_t max_prefix_len, void* workspace,
                                         size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream) {
  using namespace ra;
  clear_error();
  RA_REQUIRE(batch >= 0 && batch <= 65535, "batch must be in [0, 65535] (got %d)", batch);
  RA_REQUIRE(total_q >= 0 && total_q < (int64_t(1) << 31), "total_q out of range");
  RA_REQUIRE(num_kv_heads > 0 && num_q_heads > 0, "head counts must be > 0");
  RA_REQUIRE(num_q_heads % num_kv_heads == 0, "num_q_heads (%d) must be a multiple of num_kv_heads (%d)",
             num_q_heads, num_kv_heads);
  RA_REQUIRE(num_slots > 0, "num_slots must be > 0");
  RA_REQUIRE(std::isfinite(sm_scale) && sm_scale > 0.f, "sm_scale must be finite and > 0");
  if (head_dim != 64 && head_dim != 128) return fail(RA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  const int32_t group = num_q_heads / num_kv_heads;
  if (128 % group != 0) return fail(RA_ERR_UNSUPPORTED, "GQA group %d must divide 128", group);
  if (batch == 0 || total_q == 0) return RA_OK;
  RA_REQUIRE(max_extend_len >= 1 && max_prefix_len >= 0, "max_extend_len must be >= 1, max_prefix_len >= 0");
  // each request needs prefix_lens[b] + extend_lens[b] <= table_stride (checked per request on the device)
  RA_REQUIRE(table_stride >= max_extend_len && table_stride > max_prefix_len,
             "table_stride (%lld) narrower than max_extend_len or max_prefix_len + 1", (long long)table_stride);
  RA_REQUIRE(table_rows > 0, "table_rows must be > 0");
  RA_REQUIRE(k_pool && v_pool && q && o && req_to_token && req_pool_indices && prefix_lens && extend_lens &&
                 qo_indptr,
             "null pointer argument");
  RA_REQUIRE(aligned16(k_pool) && aligned16(v_pool) && aligned16(q) && aligned16(o),
             "pools, q and o must be 16-byte aligned");
  RA_REQUIRE(aligned4(req_to_token) && aligned4(req_pool_indices) && aligned4(prefix_lens) &&
                 aligned4(extend_lens) && aligned4(qo_indptr),
             "index arrays must be 4-byte aligned");
  const int tokens_per_cta = tc::kTiles * (128 / group);
  const ExtendWorkspace ws = layout_extend_workspace(batch, total_q, tokens_per_cta, workspace);
  if (!workspace || workspace_bytes < ws.total)
    return fail(RA_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace ? workspace_bytes : 0, ws.total);
  RA_REQUIRE(aligned16(workspace), "workspace must be 16-byte aligned");
  RA_REQUIRE(ws.cap * num_kv_heads < (int64_t(1) << 31), "too many extend tiles for one grid");

  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  // q viewed as [total_q][Hq][D]; one box = 128/G tokens x the G heads of a kv head x 64 dims
  const int rows_per_tile = 128 / group;
  CUtensorMap qmap;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                        static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(rows_per_tile)};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult cr = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, elem,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (%d)", static_cast<int>(cr));

  TcParams p{};
  p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  p.num_slots = num_slots;
  p.hkv = num_kv_heads;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.hq = num_q_heads;
  p.group = group;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.table = req_to_token;
  p.table_stride = table_stride;
  p.table_rows = table_rows;
  p.err = device_error;
  p.rpi = req_pool_indices;
  p.prefix_lens = prefix_lens;
  p.extend_lens = extend_lens;
  p.qo_indptr = qo_indptr;
  p.max_extend_len = max_extend_len;
  p.max_prefix_len = max_prefix_len;
  p.total_q = total_q;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.work_count = ws.count;
  p.work_counter = ws.counter;
  p.work_items = ws.items;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (ra_status st = launch_pdl("extend_plan_kernel", extend_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s,
                                extend_lens, prefix_lens, batch, max_extend_len, max_prefix_len, table_stride,
                                tokens_per_cta, ws.count, ws.counter, ws.items, ws.cap, device_error))
    return st;
  // at most sum_b ceil(E_b / tokens_per_cta) entries; CTAs past the listed count return at once
  const int64_t entries = std::min<int64_t>(ws.cap, static_cast<int64_t>(batch) *
                                                        ((max_extend_len + tokens_per_cta - 1) / tokens_per_cta));
  return head_dim == 128 ? launch_extend<128>(p, qmap, entries, s) : launch_extend<64>(p, qmap, entries, s);
}

extern "C" size_t ra_extend_workspace_bytes(int32_t batch, int64_t total_q, int32_t num_q_heads,
                                            int32_t num_kv_heads) {
  if (batch < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int32_t group = num_q_heads / num_kv_heads;
  if (128 % group != 0) return 0;
  return ra::layout_extend_workspace(batch, total_q, ra::tc::kTiles * (128 / group), nullptr).total;
}
