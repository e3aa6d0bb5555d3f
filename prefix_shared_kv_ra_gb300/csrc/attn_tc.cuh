// attn_tc.cuh -- tcgen05 / TMEM attention tile kernel over the slot pool.
//
// One CTA computes 128 query rows of one kv head against a range of keys
// gathered from the pool through a req_to_token row.  The rows are a GQA
// block: 128 / G tokens (or decode requests) x the G q heads of the kv head,
// so every gathered K/V tile feeds 128 rows of tensor-core work.  Two users:
//
//  * extend (EXTEND = true): rows are suffix tokens of one request; row
//    (token i, head g) sees keys 0 .. P + i (cached prefix + causal suffix);
//    the bf16 output is written directly.
//  * cascade prefix pass (EXTEND = false): rows are the decode queries of the
//    members of one prefix group; all rows see the same range of the shared
//    prefix, read once for the whole group; (output, log2-sum-exp) partials
//    are written for the decode combine pass.
//
// Warp roles (288 threads):
//  warps 0-3  softmax + epilogue, one thread per row = TMEM lane;
//  warps 4-7  producers: gather K (warps 4,5) and V (warps 6,7) rows of a
//             128-key tile with 16-byte cp.async into the 128-byte-swizzled
//             K-major (K) / MN-major (V) layouts tcgen05 reads, completion
//             signalled on per-stage mbarriers; the query tile of an extend
//             CTA is one 3-D TMA tile load (cp.async.bulk.tensor) instead;
//  warp 8     allocates TMEM and issues tcgen05.mma from one thread:
//             S = Q K^T (SS form, M=128 N=128) into one of two TMEM S buffers,
//             O += P V (TS form: P read from TMEM where softmax stored it over
//             its own S buffer) into the TMEM O accumulator.
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D); 512 allocated.
//
// Online softmax in the log2 domain with a lazy rescale: a row's reference
// maximum moves only when the running maximum exceeds it by more than 8
// (a factor 256), and only then is the row's O accumulator rescaled in TMEM.
// Probabilities are therefore <= 256 and the final O / l is exact softmax.
//
// Every mbarrier wait is bounded; on a timeout the CTA flags
// RA_DEVERR_TIMEOUT, every role drains and leaves, and TMEM is freed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "ra_ptx.cuh"

namespace ra {

struct TcParams {
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int64_t num_slots;
  int32_t hkv;
  const __nv_bfloat16* q;
  int32_t hq;
  int32_t group;
  float scale_log2;
  const int32_t* table;
  int64_t table_stride;
  int64_t table_rows;
  uint32_t* err;
  // extend
  const int32_t* rpi;
  const int32_t* prefix_lens;
  const int32_t* extend_lens;
  const int32_t* qo_indptr;
  int32_t max_extend_len;
  int32_t max_prefix_len;
  __nv_bfloat16* o;
  // cascade prefix pass
  const int32_t* group_indptr;
  const int32_t* group_reqs;
  const int32_t* group_prefix_len;
  int32_t batch;  // decode batch (bound for group_reqs entries)
  int32_t max_seq_len;
  int32_t cchunk;
  int32_t max_csplits;
  float* casc_o;
  float* casc_lse;
};

namespace tc {

constexpr int kRows = 128;     // query rows per CTA (MMA M)
constexpr int kKeys = 128;     // keys per tile (MMA N of S, K of PV)
constexpr int kThreads = 288;  // 9 warps
constexpr int kProducerBase = 128;
constexpr int kMmaWarp = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS1 = 128;
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int NS>
struct Layout {
  static constexpr int kTileBytes = kKeys * D * 2;  // one K or V tile (also the Q tile: 128 rows)
  static constexpr int kQ = 0;
  static constexpr int kK = kTileBytes;
  static constexpr int kV = kK + NS * kTileBytes;
  static constexpr int kBytes = kV + NS * kTileBytes;
  static constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk c (0 .. D/8-1) of row r in a [128 rows x D] bf16 tile
// stored as D/64 blocks of 128-byte swizzled rows (the layout of a SWIZZLE_128B
// TMA box and of tcgen05's K-major / MN-major 128B-swizzled operands).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (c >> 3) * (kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

}  // namespace tc

template <int D, int NS, bool EXTEND>
__global__ void __launch_bounds__(tc::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap qmap) {
  using namespace tc;
  using L = Layout<D, NS>;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_kf[NS], bar_ke[NS], bar_vf[NS], bar_ve[NS], bar_s[2], bar_p[2],
      bar_o, bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int T = kRows / G;  // tokens (or members) per CTA
  const int kh = blockIdx.y;

  // ------------------------------------------------------------------ job (CTA-uniform)
  int32_t kbeg = 0, kend = 0, table_row = 0;
  int32_t n_valid = 0;   // valid tokens / members in this CTA
  int32_t causal0 = 0;   // extend: key limit of token 0 is causal0 + 1
  int64_t q_tok0 = 0;    // extend: first q token
  int32_t mem0 = 0;      // cascade: first member index into group_reqs
  int32_t csplit = 0;
  if constexpr (EXTEND) {
    const int b = blockIdx.z;
    const int tile = blockIdx.x;
    int32_t E = __ldg(p.extend_lens + b);
    const int32_t P = __ldg(p.prefix_lens + b);
    table_row = __ldg(p.rpi + b);
    if (E > p.max_extend_len || P > p.max_prefix_len || E < 0 || P < 0) {
      if (tile == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      E = min(max(E, 0), p.max_extend_len);
      if (P < 0 || P > p.max_prefix_len) return;
    }
    if (tile * T >= E) return;
    if (table_row < 0 || table_row >= p.table_rows) {
      if (tile == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return;
    }
    n_valid = min(T, E - tile * T);
    causal0 = P + tile * T;
    kbeg = 0;
    kend = causal0 + n_valid;
    if (kend > p.table_stride) {
      if (tile == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      return;
    }
    q_tok0 = static_cast<int64_t>(__ldg(p.qo_indptr + b)) + tile * T;
  } else {
    const int g = blockIdx.z;
    const int32_t m_begin = __ldg(p.group_indptr + g);
    const int32_t n_mem = __ldg(p.group_indptr + g + 1) - m_begin;
    const int mt = blockIdx.x / p.max_csplits;
    csplit = blockIdx.x - mt * p.max_csplits;
    if (mt * T >= n_mem) return;
    const int32_t Pg = __ldg(p.group_prefix_len + g);
    if (Pg < 1 || Pg > p.max_seq_len) {
      if (blockIdx.x == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      return;
    }
    if (csplit * p.cchunk >= Pg) return;
    kbeg = csplit * p.cchunk;
    kend = min(Pg, kbeg + p.cchunk);
    mem0 = m_begin + mt * T;
    n_valid = min(T, n_mem - mt * T);
    const int32_t leader = __ldg(p.group_reqs + m_begin);
    if (leader < 0 || leader >= p.batch) {
      if (blockIdx.x == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return;
    }
    table_row = __ldg(p.rpi + leader);
    if (table_row < 0 || table_row >= p.table_rows) {
      if (blockIdx.x == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return;
    }
  }
  const int32_t nt = (kend - kbeg + kKeys - 1) / kKeys;  // >= 1
  const int32_t* __restrict__ row_ptr = p.table + static_cast<int64_t>(table_row) * p.table_stride;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + L::kQ;
  auto sK = [&](int st) { return sbase + L::kK + st * L::kTileBytes; };
  auto sV = [&](int st) { return sbase + L::kV + st * L::kTileBytes; };

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&bar_q), EXTEND ? 1 : 128);
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&bar_kf[s]), 64);
      mbar_init(smem_u32(&bar_vf[s]), 64);
      mbar_init(smem_u32(&bar_ke[s]), 1);
      mbar_init(smem_u32(&bar_ve[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_s[s]), 1);
      mbar_init(smem_u32(&bar_p[s]), 128);
    }
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_done), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(p.err, RA_DEVERR_TIMEOUT);
  };

  if (warp >= 4 && warp < 8) {
    // ================================================================ producers
    const int ptid = threadIdx.x - kProducerBase;
    const int pw = ptid >> 5;
    const bool is_v = pw >= 2;
    const int half = pw & 1;
    // ---- query tile
    if constexpr (EXTEND) {
      if (ptid == 0) {
        prefetch_tensormap(&qmap);
        const uint32_t bq = smem_u32(&bar_q);
        mbar_arrive_expect_tx(bq, kRows * D * 2);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sQ + h * (kRows * 128)),
              "l"(&qmap), "r"(h * 64), "r"(kh * G), "r"(static_cast<int32_t>(q_tok0)), "r"(bq)
              : "memory");
        }
      }
    } else {
      // gather the members' decode query rows: row r = (member r / G, q head kh*G + r % G)
      constexpr int RPI = 32 / CH;  // rows per warp instruction
      for (int it = 0; it < kRows * CH / 128; ++it) {
        const int r = (it * 4 + pw) * RPI + lane / CH;
        const int c = lane % CH;
        const int k = r / G;
        const int32_t m = mem0 + (k < n_valid ? k : 0);
        int32_t b = __ldg(p.group_reqs + m);
        b = (b < 0 || b >= p.batch) ? 0 : b;
        const __nv_bfloat16* src = p.q + (static_cast<int64_t>(b) * p.hq + kh * G + (r % G)) * D + c * 8;
        cp_async16(sQ + swz(r, c), src);
      }
      cp_async_arrive_noinc(smem_u32(&bar_q));
    }
    // ---- K / V tiles
    const __nv_bfloat16* pool = (is_v ? p.v_pool : p.k_pool) + static_cast<int64_t>(kh) * D;
    const int64_t slot_stride = static_cast<int64_t>(p.hkv) * D;
    uint64_t* full = is_v ? bar_vf : bar_kf;
    uint64_t* empty = is_v ? bar_ve : bar_ke;
    constexpr int RPI = 32 / CH;
    for (int j = 0; j < nt; ++j) {
      if (aborted(abort_flag)) break;
      const int st = j % NS;
      // slots of this warp's 64 keys (keys past the range repeat the last key: finite, masked)
      const int32_t key_a = kbeg + j * kKeys + half * 64 + lane;
      int32_t slot_a = __ldg(row_ptr + min(key_a, kend - 1));
      int32_t slot_b = __ldg(row_ptr + min(key_a + 32, kend - 1));
      if (slot_a < 0 || slot_a >= p.num_slots) { flag_error(p.err, RA_DEVERR_SLOT); slot_a = 0; }
      if (slot_b < 0 || slot_b >= p.num_slots) { flag_error(p.err, RA_DEVERR_SLOT); slot_b = 0; }
      if (j >= NS && !mbar_wait(smem_u32(&empty[st]), ((j / NS) + 1) & 1)) {
        give_up();
        break;
      }
      const uint32_t tile = is_v ? sV(st) : sK(st);
#pragma unroll 4
      for (int it = 0; it < 64 / RPI; ++it) {
        const int rl = it * RPI + lane / CH;  // 0..63
        const int c = lane % CH;
        const int32_t sa = __shfl_sync(0xffffffffu, slot_a, rl & 31);
        const int32_t sb = __shfl_sync(0xffffffffu, slot_b, rl & 31);
        const int32_t slot = rl < 32 ? sa : sb;
        cp_async16(tile + swz(half * 64 + rl, c), pool + static_cast<int64_t>(slot) * slot_stride + c * 8);
      }
      cp_async_arrive_noinc(smem_u32(&full[st]));
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, 0, 1);
      bool ok = mbar_wait(smem_u32(&bar_q), 0);
      fence_proxy_async_smem();
      tc_fence_after();
      bool issued = false;
      auto issue_qk = [&](int j) -> bool {
        const int st = j % NS;
        if (!mbar_wait(smem_u32(&bar_kf[st]), (j / NS) & 1)) return false;
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t d_tmem = tmem + (j & 1) * kColS1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kRows * 128) + (kk & 3) * 32;
          tc_mma_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK(st) + off, 16, 1024), idesc_qk,
                    kk > 0);
        }
        tc_commit(smem_u32(&bar_s[j & 1]));
        tc_commit(smem_u32(&bar_ke[st]));
        issued = true;
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < nt; ++j) {
        if (aborted(abort_flag)) { ok = false; break; }
        if (j + 1 < nt && !issue_qk(j + 1)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&bar_p[j & 1]), (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const int st = j % NS;
        if (!mbar_wait(smem_u32(&bar_vf[st]), (j / NS) & 1)) { ok = false; break; }
        fence_proxy_async_smem();
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          tc_mma_ts(tmem + kColO, tmem + (j & 1) * kColS1 + kk * 8,
                    sdesc_sw128(sV(st) + kk * 2048, kRows * 128, 1024), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&bar_ve[st]));
        tc_commit(smem_u32(&bar_o));
      }
      if (!ok) give_up();
      if (issued) {
        tc_commit(smem_u32(&bar_done));  // all MMAs of this CTA retired before TMEM is freed
        mbar_wait(smem_u32(&bar_done), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax (warps 0-3)
    const int r = threadIdx.x;  // row = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const int tok = r / G;
    const bool row_valid = tok < n_valid;
    int32_t lim;  // exclusive key limit of this row
    if constexpr (EXTEND) lim = row_valid ? causal0 + tok + 1 : kend;
    else lim = kend;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      const bool fail_here = aborted(abort_flag) || !mbar_wait(smem_u32(&bar_s[sb]), (j >> 1) & 1);
      if (__any_sync(0xffffffffu, fail_here)) { ok = false; break; }  // warp-uniform: tcgen05.ld/st are collective
      tc_fence_after();
      uint32_t sr[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) {
        uint32_t (&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]);
        tmem_ld32(tmem + lane_addr + sb * kColS1 + c * 32, chunk);
      }
      tc_wait_ld();
      const int32_t key0 = kbeg + j * kKeys;
      // row max of the raw scores (scale > 0 commutes with max), 8 independent chains
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      if (key0 + kKeys > lim) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          if (key0 + c >= lim) sr[c] = __float_as_uint(-INFINITY);
          mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(sr[c]));
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(sr[c]));
      }
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
      const float m_new = fmaxf(m_used, mx);
      const bool resc = m_new > m_used + kRescaleThreshold;
      const float m_ref = resc ? m_new : m_used;
      const float m_sub = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float alpha = resc ? ex2(m_used - m_sub) : 1.f;
      // p = 2^(s * scale_log2 - m_ref): one FMA + one MUFU per score; 8 independent partial sums
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c * 32 + 2 * e]), p.scale_log2, -m_sub));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c * 32 + 2 * e + 1]), p.scale_log2, -m_sub));
          sum8[(2 * e) & 7] += p0;
          sum8[(2 * e + 1) & 7] += p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + lane_addr + sb * kColS1 + c * 16, pk);
      }
      const float rowsum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l = l * alpha + rowsum;
      if (j > 0) {
        // Observe PV_{j-1} before releasing P_j: bar_o then never runs two phases ahead of
        // this warp's parity waits, and O is complete for tile j-1 if it must be rescaled.
        const bool late = !mbar_wait(smem_u32(&bar_o), (j - 1) & 1);
        if (__any_sync(0xffffffffu, late)) { ok = false; break; }
        if (__any_sync(0xffffffffu, resc)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_addr + kColO + c * 32, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tmem + lane_addr + kColO + c * 32, ov);
          }
        }
      }
      m_used = m_ref;
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p[sb]));
    }
    if (!ok) give_up();
    // ---- epilogue: O / l
    ok = ok && mbar_wait(smem_u32(&bar_o), (nt - 1) & 1);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      if constexpr (EXTEND) {
        __nv_bfloat16* dst = p.o + ((q_tok0 + tok) * p.hq + kh * G + (r % G)) * static_cast<int64_t>(D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_addr + kColO + c * 32, ov);
          tc_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      } else {
        int32_t b = __ldg(p.group_reqs + mem0 + (row_valid ? tok : 0));
        const bool write = row_valid && b >= 0 && b < p.batch;
        const int64_t ps = ((static_cast<int64_t>(write ? b : 0) * p.hq + kh * G + (r % G)) * p.max_csplits + csplit);
        float* dst = p.casc_o + ps * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_addr + kColO + c * 32, ov);
          tc_wait_ld();
          if (write) {
            float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(__uint_as_float(ov[4 * e]) * inv_l, __uint_as_float(ov[4 * e + 1]) * inv_l,
                                  __uint_as_float(ov[4 * e + 2]) * inv_l, __uint_as_float(ov[4 * e + 3]) * inv_l);
          }
        }
        if (write) p.casc_lse[ps] = m_used + __log2f(l);
      }
    } else {
      give_up();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace ra
