// decode.cu -- ra_decode_attention: split-KV GQA decode over the slot pool.
//
// Decode streams every context key of every request once per kv head: it is
// HBM-bound (4 flop/byte at GQA group 4, 8 at group 8).  The design is built
// around keeping enough bytes in flight and touching each byte once:
//
//  * grid (split, kv head, request): each CTA owns a range of `chunk` keys of
//    one (request, kv head) and all G query heads of that kv head, so a K/V
//    row is fetched once for the whole GQA group;
//  * each warp owns 16-key slabs of the range and runs its own NSTAGE-deep
//    pipeline: one lane per row issues a 1-D bulk copy (cp.async.bulk, the TMA
//    engine) of that key's 256-byte K or V row, gathered through
//    req_to_token, into a padded shared-memory tile, completion tracked by a
//    per-stage mbarrier -- no register staging, no cross-warp barrier;
//  * QK^T and PV run on the tensor cores with the keys on the M side and the
//    GQA group on N (m16n8k16): S^T = K Q^T puts 16 keys x 8 q heads in one
//    fragment, the probabilities are re-laid out for P^T with movmatrix, and
//    O^T = V^T P^T accumulates in registers.  At decode shapes a tcgen05 tile
//    (M >= 64) would be mostly padding; this warp-level form uses the whole
//    fragment and leaves the HBM stream as the only bound;
//  * online softmax in the log2 domain per q head, reduced across the 8
//    lanes that share a column with shuffles; the CTA's warps merge through
//    shared memory; a single-split request writes its bf16 output directly,
//    otherwise (output, log-sum-exp) partials go to the workspace and a
//    combine pass merges them.
//
// Sources: anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一 (decode
// reads each request's slots through req_pool_indices / seq_lens); SGLang
// paper summary, §3 (shared prefixes live once in the pool).
#include <math.h>

#include "api_common.h"
#include "decode_internal.h"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr int kSlab = 16;

template <int D>
struct DecodeShape {
  static constexpr int kRowStride = D * 2 + 16;  // padded: 8 rows of a ldmatrix hit 8 distinct bank groups
  static constexpr int kStageBytes = 2 * kSlab * kRowStride;
  static constexpr int kKT = D / 16;
};

template <int D, int NWARPS, int NSTAGE>
constexpr int decode_smem_bytes() {
  return 128 + NWARPS * NSTAGE * DecodeShape<D>::kStageBytes;
}

__device__ __forceinline__ int32_t load_slot(const int32_t* __restrict__ row_ptr, int32_t key,
                                             int64_t num_slots, uint32_t* err) {
  int32_t s = __ldg(row_ptr + key);
  if (s < 0 || s >= num_slots) {
    flag_error(err, RA_DEVERR_SLOT);
    s = 0;
  }
  return s;
}

template <int D, int NWARPS, int NSTAGE>
__global__ void __launch_bounds__(NWARPS * 32, 2) decode_split_kernel(const DecodeParams p) {
  using Sh = DecodeShape<D>;
  constexpr int RS = Sh::kRowStride;
  constexpr int KT = Sh::kKT;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kh = blockIdx.y;
  const int b = blockIdx.z;

  // ---- per-request range (uniform over the CTA)
  int32_t L = __ldg(p.seq_lens + b);
  const int32_t row = __ldg(p.rpi + b);
  if (row < 0 || row >= p.table_rows || L < 1) {
    if (split == 0 && kh == 0 && threadIdx.x == 0)
      flag_error(p.err, (row < 0 || row >= p.table_rows) ? RA_DEVERR_TABLE : RA_DEVERR_LENGTH);
    return;
  }
  if (L > p.max_seq_len) {
    if (split == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_LENGTH);
    L = p.max_seq_len;
  }
  int32_t start = p.key_start ? __ldg(p.key_start + b) : 0;
  start = start < 0 ? 0 : (start > L ? L : start);
  const int32_t n_keys_total = L - start;
  const int32_t n_splits = (n_keys_total + p.chunk - 1) / p.chunk;
  if (split >= n_splits) return;
  const int32_t k0 = start + split * p.chunk;
  const int32_t k1 = min(L, k0 + p.chunk);
  const int32_t n_slabs = (k1 - k0 + kSlab - 1) / kSlab;
  const int32_t my_slabs = warp < n_slabs ? (n_slabs - warp + NWARPS - 1) / NWARPS : 0;
  const int32_t* __restrict__ row_ptr = p.table + static_cast<int64_t>(row) * p.table_stride;

  // ---- shared memory: [barriers (128 B)] [warp 0 stages] [warp 1 stages] ...
  const uint32_t bar0 = smem_u32(smem) + warp * NSTAGE * 8;
  const uint32_t data0 = smem_u32(smem) + 128 + warp * NSTAGE * Sh::kStageBytes;
  if (threadIdx.x == 0) s_abort = 0;
  if (lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(bar0 + s * 8, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- Q^T fragments (B operand): column g = lane/4 is q head kh*G + g
  const int g = lane >> 2;
  const int tq = lane & 3;
  uint32_t qf[KT][2];
  {
    const bool live = g < p.group;
    const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(b) * p.hq + kh * p.group + (live ? g : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      qf[kk][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq)) : 0u;
      qf[kk][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq)) : 0u;
    }
  }

  const __nv_bfloat16* kv_base = (lane < 16 ? p.k_pool : p.v_pool) + static_cast<int64_t>(kh) * D;
  const int64_t slot_stride = static_cast<int64_t>(p.hkv) * D;
  // key handled by this lane's copy in slab i (rows past the range repeat the last key: finite data, weight 0)
  auto slab_key = [&](int32_t i) {
    const int32_t key = k0 + (warp + i * NWARPS) * kSlab + (lane & 15);
    return key < k1 ? key : k1 - 1;
  };
  auto issue = [&](int32_t i, int32_t slot) {
    const int st = i % NSTAGE;
    if (lane == 0) mbar_arrive_expect_tx(bar0 + st * 8, 2 * kSlab * D * 2);
    __syncwarp();
    const uint32_t dst = data0 + st * Sh::kStageBytes + (lane < 16 ? 0 : kSlab * RS) + (lane & 15) * RS;
    bulk_g2s(dst, kv_base + static_cast<int64_t>(slot) * slot_stride, D * 2, bar0 + st * 8);
  };

  const int32_t n_pro = my_slabs < NSTAGE ? my_slabs : NSTAGE;
  for (int32_t i = 0; i < n_pro; ++i) issue(i, load_slot(row_ptr, slab_key(i), p.num_slots, p.err));

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[KT][4];
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // lane's ldmatrix row addresses inside a stage
  const uint32_t a_off = (lane & 15) * RS + (lane >> 4) * 16;                                  // K, non-transposed
  const uint32_t v_off = kSlab * RS + ((lane & 7) + ((lane >> 4) << 3)) * RS + ((lane >> 3) & 1) * 16;  // V, transposed

  int32_t i = 0;
  bool timed_out = false;
  for (; i < my_slabs; ++i) {
    const int st = i % NSTAGE;
    const bool refill = i + NSTAGE < my_slabs;
    const int32_t next_slot = refill ? load_slot(row_ptr, slab_key(i + NSTAGE), p.num_slots, p.err) : 0;
    if (!mbar_wait(bar0 + st * 8, (i / NSTAGE) & 1)) {
      timed_out = true;
      break;
    }
    const uint32_t stage = data0 + st * Sh::kStageBytes;

    // S^T[16 keys x 8 heads] = K Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(stage + a_off + kk * 32, a0, a1, a2, a3);
      mma_bf16_16816(s, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
    }
    // mask keys past the range, log2-domain scores
    const int32_t kbase = k0 + (warp + i * NWARPS) * kSlab;
    const bool v_lo = kbase + g < k1;
    const bool v_hi = kbase + g + 8 < k1;
    const float x0 = v_lo ? s[0] * p.scale_log2 : -INFINITY;
    const float x1 = v_lo ? s[1] * p.scale_log2 : -INFINITY;
    const float x2 = v_hi ? s[2] * p.scale_log2 : -INFINITY;
    const float x3 = v_hi ? s[3] * p.scale_log2 : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // key 0 of a slab is always in range, so the new maxima are finite
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const float p0 = ex2(x0 - mn0), p1 = ex2(x1 - mn1), p2 = ex2(x2 - mn0), p3 = ex2(x3 - mn1);
    l0 = l0 * al0 + p0 + p2;
    l1 = l1 * al1 + p1 + p3;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
    // P^T as the B operand: transpose the two 8x8 key blocks
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
    // O^T[D x 8] += V^T P^T
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(stage + v_off + mt * 32, a0, a1, a2, a3);
      mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (refill) {
      fence_proxy_async_smem();
      issue(i + NSTAGE, next_slot);
    }
  }
  if (timed_out) {
    // drain this warp's copies still in flight (bounded), then give up on the CTA
    const int32_t issued = my_slabs < i + NSTAGE ? my_slabs : i + NSTAGE;
    for (int32_t j = i; j < issued; ++j) mbar_wait(bar0 + (j % NSTAGE) * 8, (j / NSTAGE) & 1);
    if (lane == 0) {
      flag_error(p.err, RA_DEVERR_TIMEOUT);
      s_abort = 1;
    }
  }

  // full row sums: the 8 lanes of a column share m
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every warp's copies are consumed: the stage buffers can be reused
  if (s_abort) return;

  // ---- merge the warps: smem floats [NWARPS][8] m, [NWARPS][8] l, [NWARPS][D][8] O^T
  float* fm = reinterpret_cast<float*>(smem + 128);
  float* fl = fm + NWARPS * 8;
  float* fo = fl + NWARPS * 8;
  if (g == 0) {
    fm[warp * 8 + 2 * tq] = m0;
    fm[warp * 8 + 2 * tq + 1] = m1;
    fl[warp * 8 + 2 * tq] = l0;
    fl[warp * 8 + 2 * tq + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) {
    const int d = mt * 16 + g;
    float* o = fo + (warp * D + d) * 8 + 2 * tq;
    o[0] = acc[mt][0];
    o[1] = acc[mt][1];
    o[8 * 8] = acc[mt][2];
    o[8 * 8 + 1] = acc[mt][3];
  }
  __syncthreads();

  const bool direct = (n_splits == 1) && (start == 0);
  for (int idx = threadIdx.x; idx < p.group * D; idx += NWARPS * 32) {
    const int gg = idx / D;
    const int d = idx - gg * D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) mm = fmaxf(mm, fm[w * 8 + gg]);
    float ll = 0.f, oo = 0.f;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
      const float mw = fm[w * 8 + gg];
      if (mw == -INFINITY) continue;
      const float sc = ex2(mw - mm);
      ll += fl[w * 8 + gg] * sc;
      oo += fo[(w * D + d) * 8 + gg] * sc;
    }
    const int h = kh * p.group + gg;
    const int64_t bh = static_cast<int64_t>(b) * p.hq + h;
    if (direct) {
      p.o[bh * D + d] = __float2bfloat16_rn(oo / ll);
    } else {
      const int64_t ps = bh * p.max_splits + split;
      p.part_o[ps * D + d] = oo / ll;
      if (d == 0) p.part_lse[ps] = mm + __log2f(ll);
    }
  }
}

// Merge per-split partials (and the shared-prefix partial of a cascade member).
// One warp per (request, q head); each lane owns D/32 output dims.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  constexpr int V = D / 32;
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.batch * p.hq) return;
  const int b = warp_global / p.hq;
  int32_t L = __ldg(p.seq_lens + b);
  const int32_t row = __ldg(p.rpi + b);
  if (row < 0 || row >= p.table_rows || L < 1) return;
  if (L > p.max_seq_len) L = p.max_seq_len;
  int32_t start = p.key_start ? __ldg(p.key_start + b) : 0;
  start = start < 0 ? 0 : (start > L ? L : start);
  const int32_t n_splits = (L - start + p.chunk - 1) / p.chunk;
  const bool has_prefix = start > 0;
  if (n_splits == 1 && !has_prefix) return;  // written directly by the split kernel
  const int64_t bh = warp_global;
  const int32_t n_pre = has_prefix ? (start + p.cchunk - 1) / p.cchunk : 0;  // prefix-pass splits
  float mm = -INFINITY;
  for (int s = 0; s < n_pre; ++s) mm = fmaxf(mm, p.casc_lse[bh * p.max_csplits + s]);
  for (int s = 0; s < n_splits; ++s) mm = fmaxf(mm, p.part_lse[bh * p.max_splits + s]);
  float acc[V];
  float wsum = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int s = 0; s < n_pre; ++s) {
    const int64_t ps = bh * p.max_csplits + s;
    const float w = ex2(p.casc_lse[ps] - mm);
    wsum += w;
    const float* src = p.casc_o + ps * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] += w * src[v];
  }
  for (int s = 0; s < n_splits; ++s) {
    const int64_t ps = bh * p.max_splits + s;
    const float w = ex2(p.part_lse[ps] - mm);
    wsum += w;
    const float* src = p.part_o + ps * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] += w * src[v];
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int v = 0; v < V; v += 2) {
    __nv_bfloat162 pr = __floats2bfloat162_rn(acc[v] * inv, acc[v + 1] * inv);
    *reinterpret_cast<__nv_bfloat162*>(p.o + bh * D + lane * V + v) = pr;
  }
}

// key_start[b] = prefix length of b's cascade group (0 for requests in no group).
__global__ void cascade_key_start_kernel(int32_t* key_start, int32_t batch, const int32_t* group_indptr,
                                         const int32_t* group_reqs, const int32_t* group_prefix_len,
                                         int32_t num_groups, uint32_t* err) {
  const int32_t total = __ldg(group_indptr + num_groups);
  for (int32_t m = blockIdx.x * blockDim.x + threadIdx.x; m < total; m += gridDim.x * blockDim.x) {
    int32_t lo = 0, hi = num_groups;  // group g with indptr[g] <= m < indptr[g+1]
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (__ldg(group_indptr + mid) <= m) lo = mid; else hi = mid;
    }
    const int32_t b = __ldg(group_reqs + m);
    if (b < 0 || b >= batch) {
      flag_error(err, RA_DEVERR_TABLE);
      continue;
    }
    key_start[b] = __ldg(group_prefix_len + lo);
  }
}

constexpr int kNWarps = 4;
constexpr int kNStage = 3;

template <int D>
ra_status launch_decode(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = decode_smem_bytes<D, kNWarps, kNStage>();
  auto kern = decode_split_kernel<D, kNWarps, kNStage>;
  static bool configured[64] = {};
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  if (!configured[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaFuncSetAttribute(decode): %s", cudaGetErrorString(e));
    configured[dev.device] = true;
  }
  dim3 grid(p.max_splits, p.hkv, p.batch);
  kern<<<grid, kNWarps * 32, smem, stream>>>(p);
  if (ra_status st = check_launch("decode_split_kernel")) return st;
  const int nwarps = p.batch * p.hq;
  decode_combine_kernel<D><<<(nwarps + 3) / 4, 128, 0, stream>>>(p);
  return check_launch("decode_combine_kernel");
}

}  // namespace

// Private keys per split: at least 128, at most 1024, aiming at ~2K (request, kv head, split) work items.
// Shared-prefix pass (cascade): 128-row tiles of (member, q head) per group and kv head; the prefix is
// split in multiples of 128 keys until there are about two CTAs per SM of work.
DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t max_seq_len,
                       int32_t num_groups, int32_t max_group_prefix_len, int32_t max_group_size) {
  DecodePlan pl;
  const int64_t work = static_cast<int64_t>(batch) * num_kv_heads * (max_seq_len > 0 ? max_seq_len : 1);
  int64_t chunk = (work + 2047) / 2048;
  chunk = (chunk + 63) / 64 * 64;
  if (chunk < 128) chunk = 128;
  if (chunk > 1024) chunk = 1024;
  pl.chunk = static_cast<int32_t>(chunk);
  pl.max_splits = static_cast<int32_t>((static_cast<int64_t>(max_seq_len) + chunk - 1) / chunk);
  if (pl.max_splits < 1) pl.max_splits = 1;
  if (num_groups > 0 && max_group_prefix_len > 0) {
    const int32_t group = num_q_heads / num_kv_heads;
    const int32_t rows_per_tile = 128 / (group > 0 ? group : 1);
    const int64_t mtiles = (max_group_size + rows_per_tile - 1) / rows_per_tile;
    const int64_t base = static_cast<int64_t>(num_groups) * num_kv_heads * mtiles;
    const int64_t key_tiles = (max_group_prefix_len + 127) / 128;
    int64_t want = (304 + base - 1) / base;
    if (want < 1) want = 1;
    if (want > key_tiles) want = key_tiles;
    const int64_t tiles_per_split = (key_tiles + want - 1) / want;
    pl.cchunk = static_cast<int32_t>(tiles_per_split * 128);
    pl.max_csplits = static_cast<int32_t>((max_group_prefix_len + pl.cchunk - 1) / pl.cchunk);
  }
  return pl;
}

DecodeWorkspace layout_decode_workspace(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                        const DecodePlan& pl, bool cascade) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  DecodeWorkspace w;
  const size_t bh = static_cast<size_t>(batch) * num_q_heads;
  size_t off = 0;
  w.part_o = off;
  off += up(bh * pl.max_splits * head_dim * sizeof(float));
  w.part_lse = off;
  off += up(bh * pl.max_splits * sizeof(float));
  if (cascade) {
    w.casc_o = off;
    off += up(bh * pl.max_csplits * head_dim * sizeof(float));
    w.casc_lse = off;
    off += up(bh * pl.max_csplits * sizeof(float));
    w.key_start = off;
    off += up(static_cast<size_t>(batch) * sizeof(int32_t));
  }
  w.total = off;
  return w;
}

}  // namespace ra

extern "C" size_t ra_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t max_seq_len, int32_t num_groups,
                                            int32_t max_group_prefix_len, int32_t max_group_size) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (num_groups > 0 && (max_group_prefix_len <= 0 || max_group_size <= 0)) return 0;
  const ra::DecodePlan pl = ra::plan_decode(batch, num_q_heads, num_kv_heads, max_seq_len, num_groups,
                                            max_group_prefix_len, max_group_size);
  return ra::layout_decode_workspace(batch, num_q_heads, head_dim, pl, num_groups > 0).total;
}

extern "C" ra_status ra_decode_attention(const void* k_pool, const void* v_pool, int64_t num_slots,
                                         int32_t num_kv_heads, int32_t head_dim, const void* q, void* o,
                                         int32_t num_q_heads, float sm_scale, const int32_t* req_to_token,
                                         int64_t table_stride, int64_t table_rows, const int32_t* req_pool_indices,
                                         const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                         int32_t num_groups, const int32_t* group_indptr,
                                         const int32_t* group_reqs, const int32_t* group_prefix_len,
                                         int32_t max_group_prefix_len, int32_t max_group_size, void* workspace,
                                         size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream) {
  using namespace ra;
  clear_error();
  RA_REQUIRE(batch >= 0 && batch <= 65535, "batch must be in [0, 65535] (got %d)", batch);
  RA_REQUIRE(num_kv_heads > 0 && num_q_heads > 0, "head counts must be > 0");
  RA_REQUIRE(num_q_heads % num_kv_heads == 0, "num_q_heads (%d) must be a multiple of num_kv_heads (%d)",
             num_q_heads, num_kv_heads);
  RA_REQUIRE(num_slots > 0, "num_slots must be > 0");
  RA_REQUIRE(std::isfinite(sm_scale) && sm_scale > 0.f, "sm_scale must be finite and > 0");
  RA_REQUIRE(num_groups >= 0, "num_groups must be >= 0");
  if (head_dim != 64 && head_dim != 128) return fail(RA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  const int32_t group = num_q_heads / num_kv_heads;
  if (group > 8) return fail(RA_ERR_UNSUPPORTED, "GQA group %d (decode supports up to 8)", group);
  if (batch == 0) return RA_OK;
  RA_REQUIRE(max_seq_len >= 1, "max_seq_len must be >= 1");
  RA_REQUIRE(table_stride >= max_seq_len, "table_stride (%lld) < max_seq_len (%d)", (long long)table_stride,
             max_seq_len);
  RA_REQUIRE(table_rows > 0, "table_rows must be > 0");
  RA_REQUIRE(k_pool && v_pool && q && o && req_to_token && req_pool_indices && seq_lens, "null pointer argument");
  RA_REQUIRE(aligned16(k_pool) && aligned16(v_pool) && aligned16(q) && aligned16(o),
             "pools, q and o must be 16-byte aligned");
  RA_REQUIRE(aligned4(req_to_token) && aligned4(req_pool_indices) && aligned4(seq_lens),
             "index arrays must be 4-byte aligned");
  if (num_groups > 0) {
    RA_REQUIRE(group_indptr && group_reqs && group_prefix_len, "cascade arrays must be non-null");
    RA_REQUIRE(max_group_prefix_len >= 1 && max_group_prefix_len <= max_seq_len,
               "max_group_prefix_len must be in [1, max_seq_len]");
    RA_REQUIRE(max_group_size >= 1 && max_group_size <= batch, "max_group_size must be in [1, batch]");
  }
  const DecodePlan pl = plan_decode(batch, num_q_heads, num_kv_heads, max_seq_len, num_groups,
                                    max_group_prefix_len, max_group_size);
  const DecodeWorkspace wl = layout_decode_workspace(batch, num_q_heads, head_dim, pl, num_groups > 0);
  if (workspace_bytes < wl.total)
    return fail(RA_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", workspace_bytes, wl.total);
  RA_REQUIRE(workspace && aligned16(workspace), "workspace must be non-null and 16-byte aligned");

  DecodeParams p{};
  p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
  p.num_slots = num_slots;
  p.hkv = num_kv_heads;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.hq = num_q_heads;
  p.group = group;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.table = req_to_token;
  p.table_stride = table_stride;
  p.table_rows = table_rows;
  p.rpi = req_pool_indices;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.max_seq_len = max_seq_len;
  p.chunk = pl.chunk;
  p.max_splits = pl.max_splits;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws + wl.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + wl.part_lse);
  p.err = device_error;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (num_groups > 0) {
    p.cchunk = pl.cchunk;
    p.max_csplits = pl.max_csplits;
    p.casc_o = reinterpret_cast<float*>(ws + wl.casc_o);
    p.casc_lse = reinterpret_cast<float*>(ws + wl.casc_lse);
    int32_t* key_start = reinterpret_cast<int32_t*>(ws + wl.key_start);
    p.key_start = key_start;
    cudaError_t e = cudaMemsetAsync(key_start, 0, sizeof(int32_t) * batch, s);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    cascade_key_start_kernel<<<(batch + 127) / 128, 128, 0, s>>>(key_start, batch, group_indptr, group_reqs,
                                                                  group_prefix_len, num_groups, device_error);
    if (ra_status st = check_launch("cascade_key_start_kernel")) return st;
    CascadeArgs ca{group_indptr, group_reqs, group_prefix_len, num_groups, max_group_prefix_len, max_group_size};
    if (ra_status st = launch_cascade_prefix(p, ca, head_dim, s)) return st;
  }
  return head_dim == 128 ? launch_decode<128>(p, s) : launch_decode<64>(p, s);
}
