// attn_tc.cuh -- tcgen05 / TMEM attention tile kernel over the slot pool.
//
// One CTA computes 256 query rows of one kv head -- two 128-row tiles, each a
// GQA block of 128 / G tokens (or decode requests) x the G q heads of the kv
// head -- against a range of keys gathered from the pool through a
// req_to_token row.  Every gathered 128-key K/V tile feeds both query tiles,
// i.e. 256 rows of tensor-core work.  Two users:
//
//  * extend (EXTEND = true): rows are suffix tokens of one request; row
//    (token i, head g) sees keys 0 .. P + i (cached prefix + causal suffix);
//    the bf16 output is written directly.
//  * cascade prefix pass (EXTEND = false): rows are the decode queries of the
//    members of one prefix group; all rows see the same range of the shared
//    prefix, read once for the whole group; (output, log2-sum-exp) partials
//    are written for the decode combine pass.
//
// Warp roles (352 threads):
//  warps 0-3  softmax + epilogue of query tile 0, one thread per row = TMEM lane;
//  warps 4-7  the same for query tile 1;
//  warp 8     gathers K rows, warp 9 gathers V rows of each 128-key tile with
//             16-byte cp.async into the 128-byte-swizzled K-major (K) and
//             MN-major (V) layouts tcgen05 reads (completion on per-stage
//             mbarriers); an extend CTA's query tiles arrive by 3-D TMA tile
//             loads (cp.async.bulk.tensor), a prefix-pass CTA's are gathered
//             by the same two warps;
//  warp 10    allocates TMEM and issues tcgen05.mma from one thread, in the
//             order S0 = Q0 K^T, S1 = Q1 K^T, then per key tile
//             O0 += P0 V, S0' = Q0 K'^T, O1 += P1 V, S1' = Q1 K'^T, so the
//             tensor core works on one query tile while the other tile's
//             softmax warps run (ping-pong).
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); P_i is
// stored by the softmax warps over the first 64 columns of S_i (bf16 pairs)
// and read from there by the TS-form MMA.
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
  const int32_t* work_count;  // number of (request, query tile) entries in work_items
  const int32_t* work_items;  // [2 * entries]: request, query tile; longest key range first
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

constexpr int kRows = 128;     // query rows per tile (MMA M)
constexpr int kTiles = 2;      // query tiles per CTA
constexpr int kKeys = 128;     // keys per tile (MMA N of S, K of PV)
constexpr int kKWarps = 4;                 // TMA gather throughput grows with the number of issuing warps;
constexpr int kVWarps = 3;                 // the tensor core waits on K first, so K gets one warp more
constexpr int kKWarp0 = 8;                 // K gather warps 8..11
constexpr int kVWarp0 = kKWarp0 + kKWarps;  // V gather warps 12..14
constexpr int kMmaWarp = kVWarp0 + kVWarps;  // warp 15
constexpr int kThreads = 32 * (kMmaWarp + 1);  // 512
constexpr int kGroups = kKeys / 4;          // 4-key gather groups per tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kFastSumLimit = 32768.0f;  // single-pass acceptance: every p of the row <= 2^15
// Register split: the softmax warpgroups (0, 1) hold a 128-key P row and two 32-column S chunks; the
// gather and MMA warpgroups (2, 3) need few.  setmaxnreg moves registers between them within the
// block's launch allocation (kThreads x kLaunchRegs), which the split must add up to exactly.
constexpr int kLaunchRegs = 65536 / kThreads;  // what __launch_bounds__(kThreads, 1) compiles to
constexpr int kSoftmaxRegs = 184;
constexpr int kOtherRegs = 72;
static_assert(2 * 128 * kSoftmaxRegs + 2 * 128 * kOtherRegs == kThreads * kLaunchRegs, "register split");

template <int D, int KS, int VS>
struct Layout {
  static constexpr int kTileBytes = kKeys * D * 2;  // one K or V tile (also one query tile: 128 rows)
  static constexpr int kQ = 0;
  static constexpr int kK = kTiles * kTileBytes;
  static constexpr int kV = kK + KS * kTileBytes;
  static constexpr int kBytes = kV + VS * kTileBytes;
  static constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk c (0 .. D/8-1) of row r in a [128 rows x D] bf16 tile
// stored as D/64 blocks of 128-byte swizzled rows (the layout of a SWIZZLE_128B
// TMA box and of tcgen05's K-major / MN-major 128B-swizzled operands).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (c >> 3) * (kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

}  // namespace tc

template <int D, int KS, int VS, bool EXTEND>
__global__ void __launch_bounds__(tc::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using namespace tc;
  using L = Layout<D, KS, VS>;
  constexpr int HALVES = D / 64;  // 128-byte (64-element) column blocks of a row
  extern __shared__ uint8_t smem_raw[];
  // K/V stage release: one barrier per key tile t (ring of KVF), committed after the last MMA reading
  // K_t and V_t (PV of query tile 1).  KVF > max(KS, VS): a producer waiting for tile t's release
  // cannot see the ring slot complete tile t + KVF first (that tile needs its own next copy).
  constexpr int KVF = (KS > VS ? KS : VS) + 1;
  __shared__ __align__(8) uint64_t bar_q, bar_kf[KS], bar_vf[VS], bar_kvfree[KVF], bar_s[kTiles], bar_p[kTiles],
      bar_o[kTiles], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  griddep_wait();  // the previous kernel (e.g. the KV store of this step) has completed
  griddep_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int T = kRows / G;  // tokens (or members) per query tile
  const int kh = EXTEND ? static_cast<int>(blockIdx.x % p.hkv) : static_cast<int>(blockIdx.y);

  // ------------------------------------------------------------------ job (CTA-uniform)
  int32_t kbeg = 0, kend = 0, table_row = 0;
  int32_t n_valid = 0;   // valid tokens / members in this CTA (of 2T)
  int32_t causal0 = 0;   // extend: token t of the CTA sees keys < causal0 + t + 1
  int64_t q_tok0 = 0;    // extend: first q token
  int32_t mem0 = 0;      // cascade: first member index into group_reqs
  int32_t csplit = 0;
  if constexpr (EXTEND) {
    // entry blockIdx.x / Hkv of the work list (the kv heads of an entry are adjacent CTAs: they read
    // the same slots' rows at the same time); the list holds only valid, non-empty query tiles
    // (lengths were checked and flagged when it was built)
    const int32_t entry = static_cast<int32_t>(blockIdx.x / p.hkv);
    if (entry >= __ldg(p.work_count)) return;
    const int b = __ldg(p.work_items + 2 * entry);
    const int tile = __ldg(p.work_items + 2 * entry + 1);
    const int32_t E = min(max(__ldg(p.extend_lens + b), 0), p.max_extend_len);
    const int32_t P = __ldg(p.prefix_lens + b);
    table_row = __ldg(p.rpi + b);
    if (table_row < 0 || table_row >= p.table_rows) {
      if (tile == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return;
    }
    n_valid = min(kTiles * T, E - tile * kTiles * T);
    causal0 = P + tile * kTiles * T;
    kbeg = 0;
    kend = causal0 + n_valid;
    q_tok0 = static_cast<int64_t>(__ldg(p.qo_indptr + b)) + tile * kTiles * T;
  } else {
    const int g = blockIdx.z;
    const int32_t m_begin = __ldg(p.group_indptr + g);
    const int32_t n_mem = __ldg(p.group_indptr + g + 1) - m_begin;
    const int mt = blockIdx.x / p.max_csplits;
    csplit = blockIdx.x - mt * p.max_csplits;
    if (mt * kTiles * T >= n_mem) return;
    const int32_t Pg = __ldg(p.group_prefix_len + g);
    if (Pg < 1 || Pg > p.max_seq_len) {
      if (blockIdx.x == 0 && kh == 0 && threadIdx.x == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      return;
    }
    if (csplit * p.cchunk >= Pg) return;
    kbeg = csplit * p.cchunk;
    kend = min(Pg, kbeg + p.cchunk);
    mem0 = m_begin + mt * kTiles * T;
    n_valid = min(kTiles * T, n_mem - mt * kTiles * T);
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
  auto sQ = [&](int i) { return sbase + L::kQ + i * L::kTileBytes; };
  auto sK = [&](int st) { return sbase + L::kK + st * L::kTileBytes; };
  auto sV = [&](int st) { return sbase + L::kV + st * L::kTileBytes; };

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&bar_q), EXTEND ? 1 : kKWarps);
    for (int s = 0; s < KS; ++s) mbar_init(smem_u32(&bar_kf[s]), kKWarps);
    for (int s = 0; s < VS; ++s) mbar_init(smem_u32(&bar_vf[s]), kVWarps);
    for (int s = 0; s < KVF; ++s) mbar_init(smem_u32(&bar_kvfree[s]), 1);
    for (int i = 0; i < kTiles; ++i) {
      mbar_init(smem_u32(&bar_s[i]), 1);
      mbar_init(smem_u32(&bar_p[i]), 128);
      mbar_init(smem_u32(&bar_o[i]), 1);
    }
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

  if (warp >= kKWarp0 && warp < kMmaWarp) {
    // ================================================================ producers (TMA)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    const bool is_v = warp >= kVWarp0;
    const int nw = is_v ? kVWarps : kKWarps;
    const int pw = warp - (is_v ? kVWarp0 : kKWarp0);  // 0 .. nw-1
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    if (lane == 0) prefetch_tensormap(map);
    // ---- query tiles (K warps)
    if (!is_v) {
      const uint32_t bq = smem_u32(&bar_q);
      if constexpr (EXTEND) {
        if (pw == 0 && lane == 0) {
          prefetch_tensormap(&qmap);
          mbar_arrive_expect_tx(bq, kTiles * kRows * D * 2);
#pragma unroll
          for (int i = 0; i < kTiles; ++i) {
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
              asm volatile(
                  "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                  " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sQ(i) + h * (kRows * 128)),
                  "l"(&qmap), "r"(h * 64), "r"(kh * G), "r"(static_cast<int32_t>(q_tok0 + i * T)), "r"(bq)
                  : "memory");
            }
          }
        }
      } else {
        // the members' decode query rows, 4 rows per TMA gather: CTA row R = (member R / G, q head kh*G + R % G);
        // each K warp gathers a quarter of the 256 rows (16 groups of 4)
        constexpr int kQGroups = kTiles * kRows / 4 / kKWarps;
        if (lane == 0) mbar_arrive_expect_tx(bq, kQGroups * 4 * D * 2);
        __syncwarp();
        if (lane < kQGroups) {
          const int grp = pw * kQGroups + lane;
          int32_t qrow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int R = grp * 4 + e;
            const int k = R / G;
            int32_t b = __ldg(p.group_reqs + mem0 + (k < n_valid ? k : 0));
            b = (b < 0 || b >= p.batch) ? 0 : b;
            qrow[e] = b * p.hq + kh * G + (R % G);
          }
          const int R0 = grp * 4;
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            tma_gather4(sQ(R0 >> 7) + h * (kRows * 128) + (R0 & 127) * 128, &qmap, h * 64, qrow[0], qrow[1], qrow[2],
                        qrow[3], bq);
        }
      }
    }
    // ---- K or V tiles: warp pw of nw gathers 4-key groups g0 .. g1-1 of each 128-key tile (keys 4*g0 ..),
    // lane i < g1-g0 issuing the gather4 of group g0+i.  Slot ids: lane l holds keys 4*g0 + l and 4*g0 + 32 + l.
    // The slot ids of tile j+1 are loaded while tile j is issued.
    const int g0 = pw * kGroups / nw, g1 = (pw + 1) * kGroups / nw;
    const int nkeys = 4 * (g1 - g0);  // <= 44
    uint64_t* full = is_v ? bar_vf : bar_kf;

    const int ns = is_v ? VS : KS;
    auto load_row = [&](int j, int k) -> int32_t {  // tensor-map row (slot * Hkv + kh) of key 4*g0 + k
      if (k >= nkeys) return 0;
      const int32_t key = kbeg + j * kKeys + 4 * g0 + k;  // keys past the range repeat the last key
      int32_t s = __ldg(row_ptr + min(key, kend - 1));
      if (s < 0 || s >= p.num_slots) {
        flag_error(p.err, RA_DEVERR_SLOT);
        s = 0;
      }
      return s * p.hkv + kh;
    };
    int issued = 0;
    int32_t ca = load_row(0, lane), cb = load_row(0, lane + 32);
    for (int j = 0; j < nt; ++j) {
      if (aborted(abort_flag)) break;
      const int st = j % ns;
      const int32_t na = j + 1 < nt ? load_row(j + 1, lane) : 0;
      const int32_t nb = j + 1 < nt ? load_row(j + 1, lane + 32) : 0;
      // stage st held tile j - ns: wait for that tile's release
      if (j >= ns && !mbar_wait(smem_u32(&bar_kvfree[(j - ns) % KVF]), ((j - ns) / KVF) & 1)) {
        give_up();
        break;
      }
      const uint32_t tile = is_v ? sV(st) : sK(st);
      int32_t r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = lane * 4 + e;  // key of this lane's group (meaningful for lane < g1-g0)
        const int32_t va = __shfl_sync(0xffffffffu, ca, k & 31);
        const int32_t vb = __shfl_sync(0xffffffffu, cb, k & 31);
        r[e] = k < 32 ? va : vb;
      }
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&full[st]), nkeys * D * 2);
      __syncwarp();
      if (lane < g1 - g0) {
        const int row = 4 * (g0 + lane);  // first tile row of this gather
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
          tma_gather4(tile + h * (kRows * 128) + row * 128, map, h * 64, r[0], r[1], r[2], r[3], smem_u32(&full[st]));
      }
      issued = j + 1;
      ca = na;
      cb = nb;
    }
    // copies this warp issued land before the CTA can leave (normally consumed already)
    for (int j = (issued > ns ? issued - ns : 0); j < issued; ++j)
      mbar_wait(smem_u32(&full[j % ns]), (j / ns) & 1);
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, 0, 1);
      bool ok = mbar_wait(smem_u32(&bar_q), 0);
      fence_proxy_async_smem();
      tc_fence_after();
      bool issued = false;
      auto qk = [&](int i, int j) -> bool {  // S_i = Q_i K_j^T
        const int st = j % KS;
        if (i == 0) {
          if (!mbar_wait(smem_u32(&bar_kf[st]), (j / KS) & 1)) return false;
          fence_proxy_async_smem();
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kRows * 128) + (kk & 3) * 32;
          tc_mma_ss(tmem + i * kKeys, sdesc_sw128(sQ(i) + off, 16, 1024), sdesc_sw128(sK(st) + off, 16, 1024),
                    idesc_qk, kk > 0);
        }
        tc_commit(smem_u32(&bar_s[i]));
        issued = true;
        return true;
      };
      auto pv = [&](int i, int j) -> bool {  // O_i += P_i V_j
        const int st = j % VS;
        if (!mbar_wait(smem_u32(&bar_p[i]), j & 1)) return false;
        tc_fence_after();
        if (i == 0) {
          if (!mbar_wait(smem_u32(&bar_vf[st]), (j / VS) & 1)) return false;
          fence_proxy_async_smem();
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          tc_mma_ts(tmem + kColO + i * 128, tmem + i * kKeys + kk * 8,
                    sdesc_sw128(sV(st) + kk * 2048, kRows * 128, 1024), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        // Each commit stalls the tensor pipe briefly, so there are three per key tile: S_0, S_1 and the
        // K/V release here.  O_i needs none until the last tile: S_i(j+1)'s commit also covers PV_i(j).
        if (i == kTiles - 1) tc_commit(smem_u32(&bar_kvfree[j % KVF]));
        if (j == nt - 1) tc_commit(smem_u32(&bar_o[i]));
        return true;
      };
      ok = ok && qk(0, 0) && qk(1, 0);
      for (int j = 0; ok && j < nt; ++j) {
        if (aborted(abort_flag)) { ok = false; break; }
        ok = pv(0, j) && (j + 1 >= nt || qk(0, j + 1)) && pv(1, j) && (j + 1 >= nt || qk(1, j + 1));
      }
      if (!ok) give_up();
      if (issued) {
        tc_commit(smem_u32(&bar_done));  // all MMAs of this CTA retired before TMEM is freed
        mbar_wait(smem_u32(&bar_done), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax (warps 0-7)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    const int ti = warp >> 2;              // query tile
    const int r = threadIdx.x & 127;        // row of the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t col_s = ti * kKeys;
    const uint32_t col_o = kColO + ti * 128;
    const int tok = ti * T + r / G;         // token / member of the CTA
    const bool row_valid = tok < n_valid;
    int32_t lim;  // exclusive key limit of this row
    if constexpr (EXTEND) lim = row_valid ? causal0 + tok + 1 : kend;
    else lim = kend;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const bool fail_here = aborted(abort_flag) || !mbar_wait(smem_u32(&bar_s[ti]), j & 1);
      if (__any_sync(0xffffffffu, fail_here)) { ok = false; break; }  // warp-uniform: tcgen05.ld/st are collective
      tc_fence_after();
      const int32_t key0 = kbeg + j * kKeys;
      const bool masked = key0 + kKeys > lim;
      // Tiles after the first are exponentiated against the current reference in a single pass.  The
      // row sum bounds every probability of the row (p <= sum), so a sum above kFastSumLimit, or one
      // that is not finite, marks the reference as stale: the warp then redoes the tile on the exact
      // path -- row maximum first, lazy reference update, then the exponentials -- which the first
      // tile always takes.  P is held in registers until the pass is accepted, since it overwrites S.
      uint32_t pk[2][32];
      float rowsum = 0.f, alpha = 1.f, m_ref = m_used;
      bool resc = false;
      bool exact = j == 0;
#pragma unroll 1
      for (int attempt = 0; attempt < 2; ++attempt) {
        if (exact) {
          // row max of the raw scores (scale > 0 commutes with max), 8 independent chains; the next
          // 32-column TMEM load is in flight while the current chunk is reduced
          float mx8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
          auto max_chunk = [&](const uint32_t (&sr)[32], int c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float x = (masked && key0 + c * 32 + e >= lim) ? -INFINITY : __uint_as_float(sr[e]);
              mx8[e & 7] = fmaxf(mx8[e & 7], x);
            }
          };
          uint32_t ba[32], bb[32];
          tmem_ld32(tmem + lane_addr + col_s, ba);
          tc_wait_ld_regs(ba);
          tmem_ld32(tmem + lane_addr + col_s + 32, bb);
          max_chunk(ba, 0);
          tc_wait_ld_regs(bb);
          tmem_ld32(tmem + lane_addr + col_s + 64, ba);
          max_chunk(bb, 1);
          tc_wait_ld_regs(ba);
          tmem_ld32(tmem + lane_addr + col_s + 96, bb);
          max_chunk(ba, 2);
          tc_wait_ld_regs(bb);
          max_chunk(bb, 3);
          const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
          const float m_new = fmaxf(m_used, mx);
          resc = m_new > m_used + kRescaleThreshold;
          m_ref = resc ? m_new : m_used;
        }
        const float m_sub = (m_ref == -INFINITY) ? 0.f : m_ref;
        alpha = resc ? ex2(m_used - m_sub) : 1.f;
        // p = 2^(s * scale_log2 - m_ref): packed FMA pairs + one MUFU per score, packed to bf16 pairs
        const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
        const uint64_t neg_m2 = f2_pack(-m_sub, -m_sub);
        uint64_t sum2[4] = {0, 0, 0, 0};  // 4 independent chains of (even, odd) partial sums
        auto exp_chunk = [&](const uint32_t (&sr)[32], int c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float s0 = __uint_as_float(sr[2 * e]), s1 = __uint_as_float(sr[2 * e + 1]);
            if (masked) {
              if (key0 + c * 32 + 2 * e >= lim) s0 = -INFINITY;
              if (key0 + c * 32 + 2 * e + 1 >= lim) s1 = -INFINITY;
            }
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(s0, s1), scale2, neg_m2), t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            sum2[e & 3] = f2_add(sum2[e & 3], f2_pack(p0, p1));
            pk[c >> 1][(c & 1) * 16 + e] = pack_bf16x2(p0, p1);
          }
        };
        {
          uint32_t ba[32], bb[32];
          tmem_ld32(tmem + lane_addr + col_s, ba);
          tc_wait_ld_regs(ba);
          tmem_ld32(tmem + lane_addr + col_s + 32, bb);
          exp_chunk(ba, 0);
          tc_wait_ld_regs(bb);
          tmem_ld32(tmem + lane_addr + col_s + 64, ba);
          exp_chunk(bb, 1);
          tc_wait_ld_regs(ba);
          tmem_ld32(tmem + lane_addr + col_s + 96, bb);
          exp_chunk(ba, 2);
          tc_wait_ld_regs(bb);
          exp_chunk(bb, 3);
        }
        float sum8[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(sum2[e], sum8[2 * e], sum8[2 * e + 1]);
        rowsum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        if (exact) break;
        const bool stale = !(rowsum <= kFastSumLimit);
        if (!__any_sync(0xffffffffu, stale)) break;
        exact = true;
      }
      // P (bf16 pairs) over the first 64 columns of S, read by the PV MMA
      tmem_st32(tmem + lane_addr + col_s, pk[0]);
      tmem_st32(tmem + lane_addr + col_s + 32, pk[1]);
      l = l * alpha + rowsum;
      if (j > 0) {
        // O_i holds PV_i(j-1): the commit that signalled S_i(j) covers every earlier MMA
        if (__any_sync(0xffffffffu, resc)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_addr + col_o + c * 32, ov);
            tc_wait_ld_regs(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tmem + lane_addr + col_o + c * 32, ov);
          }
        }
      }
      m_used = m_ref;
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p[ti]));
    }
    if (!ok) give_up();
    // ---- epilogue: O / l
    ok = ok && mbar_wait(smem_u32(&bar_o[ti]), 0);  // committed once, after the last PV
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      if constexpr (EXTEND) {
        __nv_bfloat16* dst = p.o + ((q_tok0 + tok) * p.hq + kh * G + (r % G)) * static_cast<int64_t>(D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_addr + col_o + c * 32, ov);
          tc_wait_ld_regs(ov);
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
          tmem_ld32(tmem + lane_addr + col_o + c * 32, ov);
          tc_wait_ld_regs(ov);
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
