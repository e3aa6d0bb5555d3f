// attn_tc.cuh -- persistent tcgen05 / TMEM attention kernel over the slot pool.
//
// One CTA per SM runs a stream of work items.  An item is 256 query rows of one kv head -- two
// 128-row tiles, each a GQA block of 128 / G tokens (or decode requests) x the G q heads of the kv
// head -- against a range of keys gathered from the pool through a req_to_token row.  Every
// gathered 128-key K/V tile feeds both query tiles, i.e. 256 rows of tensor-core work.  Two users:
//
//  * extend (EXTEND = true): rows are suffix tokens of one request; row (token i, head g) sees
//    keys 0 .. P + i (cached prefix + causal suffix); the bf16 output is written directly.  Items
//    come from a (request, query tile) list sorted longest first, times the kv heads.
//  * cascade prefix pass (EXTEND = false): rows are the decode queries of the members of one
//    prefix group; all rows see the same range of the shared prefix, read once for the group;
//    (output, log2-sum-exp) partials are written for the decode combine pass.
//
// Warp roles (512 threads):
//  warps 0-3  softmax + epilogue of query tile 0, one thread per row = TMEM lane;
//  warps 4-7  the same for query tile 1;
//  warps 8-11 gather the K rows of each 128-key tile with TMA tile::gather4 (4 rows per
//             instruction) into the 128B-swizzled K-major layout tcgen05 reads; warp 8 also
//             claims the items and publishes them through a shared ring (one mbarrier each);
//  warps 12-14 gather the V rows into the MN-major layout;
//  warp 15    one thread issues tcgen05.mma in the order S0 = Q0 K^T, S1 = Q1 K^T, then per key
//             tile O0 += P0 V, S0' = Q0 K'^T, O1 += P1 V, S1' = Q1 K'^T, so the tensor core
//             works on one query tile while the other tile's softmax runs (ping-pong); the warp
//             also loads the next item's query tiles (a 3-D TMA tile load, or a gather4 of the
//             members' rows) as soon as the current item's last QK on that tile has completed.
// The K and V gathers, and so the tensor core, run on from one item into the next; the epilogue
// of an item (O / l from TMEM) overlaps the next item's first QKs, and its first PV waits on an
// "O free" barrier the epilogue releases.  TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384),
// O1 [384,512); P_i is stored by the softmax warps over the first 64 columns of S_i (bf16 pairs)
// and read from there by the TS-form MMA.
//
// Online softmax in the log2 domain with a lazy rescale: a row's reference maximum moves only
// when the running maximum exceeds it by more than 8 (a factor 256), and only then is the row's
// O accumulator rescaled in TMEM.  Tiles after an item's first are exponentiated in one pass
// against the current reference and accepted when the row sum stays <= 2^15; otherwise the
// warp redoes the tile on the exact path (row maximum first).  O / l is exact softmax.
//
// Every mbarrier wait is bounded; on a timeout the CTA flags RA_DEVERR_TIMEOUT, every role
// drains and leaves (the producers at once through the CTA's abort flag, the MMA and softmax warps at
// the deadline of their next wait), and TMEM is freed.
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
  int32_t* work_counter;  // item claim counter, zero before the launch
  int32_t* done_counter;  // cascade prefix pass: each CTA adds one once all its partials are written
  // extend
  const int32_t* rpi;
  const int32_t* prefix_lens;
  const int32_t* extend_lens;
  const int32_t* qo_indptr;
  int32_t max_extend_len;
  int32_t max_prefix_len;
  int64_t total_q;  // rows of q and o: every written row index is checked against it
  __nv_bfloat16* o;
  const int32_t* work_count;  // number of (request, query tile) entries in work_items
  const int32_t* work_items;  // [2 * entries]: request, query tile; longest key range first
  // cascade prefix pass
  const int32_t* group_indptr;
  const int32_t* group_reqs;
  const int32_t* group_prefix_start;  // nullable: 0
  const int32_t* group_prefix_len;    // end of the group's range
  const int32_t* group_level;         // nullable: 0
  int32_t casc_levels;                // levels of prefix partials per member
  int32_t casc_slots;                 // casc_levels x max_csplits
  int32_t num_groups;
  int32_t grid_x;  // member tiles x prefix splits per group
  int32_t batch;   // decode batch (bound for group_reqs entries)
  int32_t max_seq_len;
  int32_t cchunk;
  int32_t max_csplits;
  float* casc_o;    // [casc_slots, batch, hq, D]
  float* casc_lse;  // [casc_slots, batch, hq]
};

namespace tc {

constexpr int kRows = 128;     // query rows per tile (MMA M)
constexpr int kTiles = 2;      // query tiles per item
constexpr int kKeys = 128;     // keys per tile (MMA N of S, K of PV)
constexpr int kKWarps = 4;                 // TMA gather throughput grows with the number of issuing warps;
constexpr int kVWarps = 3;                 // the tensor core waits on K first, so K gets one warp more
constexpr int kKWarp0 = 8;                 // K gather warps 8..11
constexpr int kVWarp0 = kKWarp0 + kKWarps;  // V gather warps 12..14
constexpr int kMmaWarp = kVWarp0 + kVWarps;  // warp 15
constexpr int kThreads = 32 * (kMmaWarp + 1);  // 512
constexpr int kGroups = kKeys / 4;          // 4-key gather groups per tile
constexpr int kItemRing = 8;                // published items (the claimer runs <= KS + 2 items ahead)
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

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// One work item: key range, table row and query rows.
struct Job {
  int32_t kh;
  int32_t kbeg, kend, nt;  // keys [kbeg, kend) in nt 128-key tiles
  int32_t table_row;
  int32_t n_valid;   // valid tokens / members (of 2T)
  int32_t causal0;   // extend: token t of the item sees keys < causal0 + t + 1
  int64_t q_tok0;    // extend: first q token
  int32_t mem0;      // cascade: first member index into group_reqs
  int32_t csplit;    // cascade: prefix split
  int32_t slot;      // cascade: partial slot of the members (level x max_csplits + split)
  int32_t tiles;     // query tiles holding valid rows (1: tile 1 is empty; its MMAs and softmax are skipped,
                     // while every barrier still completes its phases as for two tiles)
};

// Item -> job; false for an empty or invalid item (reported once, when `report`).
template <bool EXTEND>
__device__ __forceinline__ bool tc_job(const TcParams& p, int32_t item, Job& j, bool report) {
  const int T = kRows / p.group;
  j.kh = item % p.hkv;
  const int32_t rest = item / p.hkv;
  j.causal0 = 0;
  j.q_tok0 = 0;
  j.mem0 = 0;
  j.csplit = 0;
  j.slot = 0;
  if constexpr (EXTEND) {
    // entry `rest` of the work list: it holds only non-empty query tiles of requests whose lengths
    // were checked (and flagged) when it was built
    const int b = __ldg(p.work_items + 2 * rest);
    const int tile = __ldg(p.work_items + 2 * rest + 1);
    const int32_t E = min(max(__ldg(p.extend_lens + b), 0), p.max_extend_len);
    const int32_t P = __ldg(p.prefix_lens + b);
    j.table_row = __ldg(p.rpi + b);
    if (j.table_row < 0 || j.table_row >= p.table_rows) {
      if (report && tile == 0 && j.kh == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return false;
    }
    // the request's rows qo_indptr[b] .. qo_indptr[b] + E - 1 must lie inside o: a request whose
    // lengths disagree with total_q writes nothing (flagged once)
    const int64_t q_first = __ldg(p.qo_indptr + b);
    if (q_first < 0 || q_first + E > p.total_q) {
      if (report && tile == 0 && j.kh == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      return false;
    }
    j.n_valid = min(kTiles * T, E - tile * kTiles * T);
    j.causal0 = P + tile * kTiles * T;
    j.kbeg = 0;
    j.kend = j.causal0 + j.n_valid;
    j.q_tok0 = q_first + tile * kTiles * T;
  } else {
    const int x = rest % p.grid_x;
    const int g = rest / p.grid_x;
    const int32_t m_begin = __ldg(p.group_indptr + g);
    const int32_t n_mem = __ldg(p.group_indptr + g + 1) - m_begin;
    const int mt = x / p.max_csplits;
    j.csplit = x - mt * p.max_csplits;
    if (mt * kTiles * T >= n_mem) return false;
    // the group's range [g0, Pg) of its members' positions, split into cchunk-key pieces
    const int32_t Pg = __ldg(p.group_prefix_len + g);
    const int32_t g0 = p.group_prefix_start ? __ldg(p.group_prefix_start + g) : 0;
    const int32_t lvl = p.group_level ? __ldg(p.group_level + g) : 0;
    if (Pg < 1 || Pg > p.max_seq_len || g0 < 0 || g0 >= Pg || lvl < 0 || lvl >= p.casc_levels) {
      if (report && x == 0 && j.kh == 0) flag_error(p.err, RA_DEVERR_LENGTH);
      return false;
    }
    if (j.csplit * p.cchunk >= Pg - g0) return false;
    j.kbeg = g0 + j.csplit * p.cchunk;
    j.kend = min(Pg, j.kbeg + p.cchunk);
    j.slot = lvl * p.max_csplits + j.csplit;
    j.mem0 = m_begin + mt * kTiles * T;
    j.n_valid = min(kTiles * T, n_mem - mt * kTiles * T);
    const int32_t leader = __ldg(p.group_reqs + m_begin);
    if (leader < 0 || leader >= p.batch) {
      if (report && x == 0 && j.kh == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return false;
    }
    j.table_row = __ldg(p.rpi + leader);
    if (j.table_row < 0 || j.table_row >= p.table_rows) {
      if (report && x == 0 && j.kh == 0) flag_error(p.err, RA_DEVERR_TABLE);
      return false;
    }
  }
  j.nt = (j.kend - j.kbeg + kKeys - 1) / kKeys;
  j.tiles = j.n_valid > T ? 2 : 1;
  return j.nt > 0;
}

}  // namespace tc

template <int D, int KS, int VS, bool EXTEND>
__global__ void __launch_bounds__(tc::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using namespace tc;
  using L = Layout<D, KS, VS>;
  constexpr int HALVES = D / 64;  // 128-byte (64-element) column blocks of a row
  // K/V stage release: one barrier per key tile t (ring of KVF), committed after the last MMA reading
  // K_t and V_t (PV of query tile 1).  KVF > max(KS, VS): a producer waiting for tile t's release
  // cannot see the ring slot complete tile t + KVF first (that tile needs its own next copy).
  constexpr int KVF = (KS > VS ? KS : VS) + 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q[kTiles], bar_kf[KS], bar_vf[VS], bar_kvfree[KVF], bar_s[kTiles],
      bar_p[kTiles], bar_o[kTiles], bar_ofree[kTiles], bar_item[kItemRing], bar_done;
  __shared__ int32_t s_item[kItemRing];
  __shared__ Job s_job[kItemRing];  // decoded by the claimer: no role reads the work list itself
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  griddep_wait();  // the previous kernel (the work-list pass / the key-start scatter) has completed
  griddep_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int T = kRows / G;  // tokens (or members) per query tile

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto sQ = [&](int i) { return sbase + L::kQ + i * L::kTileBytes; };
  auto sK = [&](int st) { return sbase + L::kK + st * L::kTileBytes; };
  auto sV = [&](int st) { return sbase + L::kV + st * L::kTileBytes; };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < KS; ++s) mbar_init(smem_u32(&bar_kf[s]), kKWarps);
    for (int s = 0; s < VS; ++s) mbar_init(smem_u32(&bar_vf[s]), kVWarps);
    for (int s = 0; s < KVF; ++s) mbar_init(smem_u32(&bar_kvfree[s]), 1);
    for (int i = 0; i < kTiles; ++i) {
      mbar_init(smem_u32(&bar_q[i]), EXTEND ? 1 : kKWarps / kTiles);
      mbar_init(smem_u32(&bar_s[i]), 1);
      mbar_init(smem_u32(&bar_p[i]), 128);
      mbar_init(smem_u32(&bar_o[i]), 1);
      mbar_init(smem_u32(&bar_ofree[i]), 128);
    }
    for (int s = 0; s < kItemRing; ++s) mbar_init(smem_u32(&bar_item[s]), 1);
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
  // item n of this CTA: 1 = `jb` holds its job, 0 = no more work, -1 = a bounded wait ran out
  auto wait_item = [&](int32_t n, Job& jb) -> int {
    if (!mbar_wait(smem_u32(&bar_item[n % kItemRing]), (n / kItemRing) & 1)) return -1;
    if (s_item[n % kItemRing] < 0) return 0;
    jb = s_job[n % kItemRing];
    return 1;
  };

  if (warp >= kKWarp0 && warp < kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    // ================================================================ producers (TMA)
    const bool is_v = warp >= kVWarp0;
    const int nw = is_v ? kVWarps : kKWarps;
    const int pw = warp - (is_v ? kVWarp0 : kKWarp0);  // 0 .. nw-1
    const bool claimer = !is_v && pw == 0;
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    if (lane == 0) prefetch_tensormap(map);
    // the claimer hands out items in order (the extend list is longest first), skipping empty ones
    int32_t n_items = 0;
    if (claimer) {
      n_items = EXTEND ? __ldg(p.work_count) * p.hkv : p.num_groups * p.grid_x * p.hkv;
    }
    // claim the next non-empty item and publish it, decoded, as entry n of the ring (warp-collective).
    // Item blockIdx.x is this CTA's first without a claim; the counter hands out the items after the grid.
    bool own_first = true;
    auto claim_publish = [&](int32_t n) {
      int32_t idx;
      Job cj;
      for (;;) {
        idx = static_cast<int32_t>(blockIdx.x);
        if (!own_first) {
          if (lane == 0) idx = static_cast<int32_t>(gridDim.x) + atomicAdd(p.work_counter, 1);
          idx = __shfl_sync(0xffffffffu, idx, 0);
        }
        own_first = false;
        if (idx >= n_items) {
          idx = -1;
          break;
        }
        if (tc_job<EXTEND>(p, idx, cj, lane == 0)) break;
      }
      if (lane == 0) {
        s_item[n % kItemRing] = idx;
        if (idx >= 0) s_job[n % kItemRing] = cj;
        mbar_arrive(smem_u32(&bar_item[n % kItemRing]));
      }
    };
    if (claimer) claim_publish(0);
    // warp pw of nw gathers 4-key groups g0 .. g1-1 of each 128-key tile (keys 4*g0 ..), lane i < g1-g0
    // issuing the gather4 of group g0+i.  Slot ids: lane l holds keys 4*g0 + l and 4*g0 + 32 + l of a
    // tile; the next tile's (possibly the next item's first) are loaded while this one is issued.
    const int g0 = pw * kGroups / nw, g1 = (pw + 1) * kGroups / nw;
    const int nkeys = 4 * (g1 - g0);  // <= 44
    uint64_t* full = is_v ? bar_vf : bar_kf;
    const int ns = is_v ? VS : KS;
    auto load_row = [&](const Job& jb, int j, int k) -> int32_t {  // tensor-map row (slot * Hkv + kh)
      if (k >= nkeys) return 0;
      const int32_t key = jb.kbeg + j * kKeys + 4 * g0 + k;  // keys past the range repeat the last key
      int32_t s = __ldg(p.table + static_cast<int64_t>(jb.table_row) * p.table_stride + min(key, jb.kend - 1));
      if (s < 0 || s >= p.num_slots) {
        flag_error(p.err, RA_DEVERR_SLOT);
        s = 0;
      }
      return s * p.hkv + jb.kh;
    };
    int32_t gt = 0;  // key tiles issued by this warp (all items)
    bool ok = true;
    int32_t n = 0;
    Job jb{};
    int r = wait_item(0, jb);
    if (!__all_sync(0xffffffffu, r >= 0)) ok = false;
    int32_t ca = ok && r > 0 ? load_row(jb, 0, lane) : 0, cb = ok && r > 0 ? load_row(jb, 0, lane + 32) : 0;
    while (ok && r > 0) {
      for (int j = 0; j < jb.nt; ++j) {
        if (aborted(abort_flag)) { ok = false; break; }
        // the next tile's slot ids: this item's, or the next item's first
        int32_t na = 0, nb = 0;
        if (j + 1 < jb.nt) {
          na = load_row(jb, j + 1, lane);
          nb = load_row(jb, j + 1, lane + 32);
        }
        const int st = gt % ns;
        // stage st held tile gt - ns: wait for that tile's release
        if (gt >= ns &&
            !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_kvfree[(gt - ns) % KVF]), ((gt - ns) / KVF) & 1))) {
          ok = false;
          break;
        }
        const uint32_t tile = is_v ? sV(st) : sK(st);
        int32_t rr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = lane * 4 + e;  // key of this lane's group (meaningful for lane < g1-g0)
          const int32_t va = __shfl_sync(0xffffffffu, ca, k & 31);
          const int32_t vb = __shfl_sync(0xffffffffu, cb, k & 31);
          rr[e] = k < 32 ? va : vb;
        }
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&full[st]), nkeys * D * 2);
        __syncwarp();
        if (lane < g1 - g0) {
          const int row = 4 * (g0 + lane);  // first tile row of this gather
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            tma_gather4(tile + h * (kRows * 128) + row * 128, map, h * 64, rr[0], rr[1], rr[2], rr[3],
                        smem_u32(&full[st]));
        }
        ++gt;
        if constexpr (!EXTEND) {
          // The members' query rows of this item: K warps 0-1 gather query tile 0, warps 2-3 tile 1, 16
          // groups of 4 rows each (one gather4 per 64-column half).  The tile is free once the previous
          // item's last QK on it has completed, which the commit of that S signals.
          if (!is_v && j == 0) {
            const int qt = pw / 2;
            if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[qt]), (gt - 2) & 1))) {
              ok = false;
              break;
            }
            const uint32_t bq = smem_u32(&bar_q[qt]);
            if (lane == 0) mbar_arrive_expect_tx(bq, 16 * 4 * D * 2);
            __syncwarp();
            if (lane < 16) {
              const int grp = (pw & 1) * 16 + lane;  // group of the tile
              int32_t qrow[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int R = grp * 4 + e;
                const int k = qt * T + R / G;
                int32_t b = __ldg(p.group_reqs + jb.mem0 + (k < jb.n_valid ? k : 0));
                b = (b < 0 || b >= p.batch) ? 0 : b;
                qrow[e] = b * p.hq + jb.kh * G + (R % G);
              }
#pragma unroll
              for (int h = 0; h < HALVES; ++h)
                tma_gather4(sQ(qt) + h * (kRows * 128) + grp * 4 * 128, &qmap, h * 64, qrow[0], qrow[1], qrow[2],
                            qrow[3], bq);
            }
          }
        }
        // the next item is claimed once this one's first tile is on its way
        if (claimer && j == 0) claim_publish(n + 1);
        ca = na;
        cb = nb;
      }
      if (!ok) break;
      ++n;
      r = wait_item(n, jb);
      if (!__all_sync(0xffffffffu, r >= 0)) { ok = false; break; }
      if (r > 0) {
        ca = load_row(jb, 0, lane);
        cb = load_row(jb, 0, lane + 32);
      }
    }
    if (!ok) {
      give_up();
      // copies this warp issued land before the CTA can leave
      for (int32_t t = (gt > ns ? gt - ns : 0); t < gt; ++t) mbar_wait(smem_u32(&full[t % ns]), (t / ns) & 1);
    }
  } else if (warp == kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    // ================================================================ MMA issuer + query loads
    if (lane == 0) prefetch_tensormap(&qmap);
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, kKeys, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, 0, 1);
    // Every Q, K and V tile sits at a fixed shared-memory offset: one descriptor per operand kind, a
    // tile's and a K step's offsets added to its start-address field (addresses / 16 stay below 2^14).
    const uint64_t desc_q0 = sdesc_sw128(sQ(0), 16, 1024), desc_k0 = sdesc_sw128(sK(0), 16, 1024);
    const uint64_t desc_v0 = sdesc_sw128(sV(0), kRows * 128, 1024);
    constexpr uint32_t kTile16 = L::kTileBytes >> 4;
    // query tile i of an extend job into sQ(i): one 3-D TMA tile load per 64-column half (the K warps
    // gather the prefix pass's member rows)
    auto load_q = [&](const Job& jb, int i) {
      const uint32_t bq = smem_u32(&bar_q[i]);
      if constexpr (EXTEND) {
        if (lane == 0) mbar_arrive_expect_tx(bq, kRows * D * 2);
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < HALVES; ++h) {
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sQ(i) + h * (kRows * 128)),
                "l"(&qmap), "r"(h * 64), "r"(jb.kh * G), "r"(static_cast<int32_t>(jb.q_tok0 + i * T)), "r"(bq)
                : "memory");
          }
        }
      }
    };
    // every lane waits (the warp is otherwise idle but for lane 0); the outcome is made warp-uniform.
    // (Parking lanes 1-31 in a shuffle while lane 0 waits measured ~20% slower on GB300.)
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity));
    };
    bool ok = true;
    int32_t n = 0, g = 0;  // items done, key tiles done (all items)
    Job jb{}, jn{};
    int r = wait_item(0, jb);
    if (!__all_sync(0xffffffffu, r >= 0)) ok = false;
    int next = -2;  // the item after jb: -2 not looked up yet, 0 none, 1 in jn
    auto lookup_next = [&]() -> bool {  // published when jb's first K tile was issued
      if (next != -2) return true;
      const int rn = wait_item(n + 1, jn);
      if (!__all_sync(0xffffffffu, rn >= 0)) return false;
      next = rn;
      return true;
    };
    if (ok && r > 0 && EXTEND) {
      load_q(jb, 0);
      load_q(jb, 1);
    }
    // S_i = Q_i K_gg^T; for an empty query tile (live false) only the commit, which keeps bar_s's phases
    auto qk = [&](int i, int gg, bool live) -> bool {
      const int st = gg % KS;
      if (i == 0) {
        if (!wait_all(bar_kf[st], (gg / KS) & 1)) return false;
        tc_fence_after();
      }
      if (lane == 0) {
        const uint64_t qd = desc_q0 + i * kTile16, kd = desc_k0 + st * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16 && live; ++kk) {
          const uint32_t off16 = ((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4;
          tc_mma_ss(tmem + i * kKeys, qd + off16, kd + off16, idesc_qk, kk > 0);
        }
        tc_commit(smem_u32(&bar_s[i]));
      }
      __syncwarp();
      return true;
    };
    // O_i += P_i V_gg; j = key tile within the item.  After the last P of the item, query tile i is
    // free (the softmax saw S_i, so its QK has completed): the next item's tile is loaded then.
    auto pv = [&](int i, int gg, int j) -> bool {
      const int st = gg % VS;
      if (!wait_all(bar_p[i], gg & 1)) return false;
      tc_fence_after();
      if (j == 0 && n > 0) {
        // the previous item's epilogue has read O_i
        if (!wait_all(bar_ofree[i], (n - 1) & 1)) return false;
        tc_fence_after();
      }
      if (i == 0) {
        if (!wait_all(bar_vf[st], (gg / VS) & 1)) return false;
        tc_fence_after();
      }
      if (lane == 0) {
        const bool live = i < jb.tiles;  // an empty query tile issues no PV (its O is never read)
        const uint64_t vd = desc_v0 + st * kTile16;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16 && live; ++kk) {
          tc_mma_ts(tmem + kColO + i * 128, tmem + i * kKeys + kk * 8, vd + kk * (2048 >> 4), idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        // Each commit stalls the tensor pipe briefly, so there are three per key tile: S_0, S_1 and the
        // K/V release here.  O_i needs none until the item's last tile: S_i's commit also covers PV_i.
        if (i == kTiles - 1) tc_commit(smem_u32(&bar_kvfree[gg % KVF]));
        if (j == jb.nt - 1) tc_commit(smem_u32(&bar_o[i]));
      }
      __syncwarp();
      return true;
    };
    // Query tile i of this item is free once its last QK (key tile gl) has completed: the commit of
    // S_i signals that (the softmax warps wait on the same phase).  The next item's tile is loaded then,
    // a whole softmax ahead of the QK that needs it.
    auto reload_q = [&](int i, int gl) -> bool {
      if (!lookup_next()) return false;
      if constexpr (EXTEND) {
        if (!wait_all(bar_s[i], gl & 1)) return false;
        if (next > 0) load_q(jn, i);
      }
      return true;
    };
    // The key tiles of consecutive items form one stream: per tile PV_0, QK_0', PV_1, QK_1', where the
    // QKs after an item's last tile are the next item's first.
    if (ok && r > 0) {
      ok = wait_all(bar_q[0], 0) && wait_all(bar_q[1], 0);
      if (ok) {
        tc_fence_after();
        ok = qk(0, 0, true) && qk(1, 0, jb.tiles > 1);
      }
    }
    while (ok && r > 0) {
      // (no per-tile look at the abort flag: after a failure elsewhere this warp leaves through the
      // deadline of its next wait; the check on the loop's back edge measured ~1% of the kernel)
      for (int j = 0; ok && j < jb.nt; ++j) {
        const int gg = g + j;
        const bool last = j + 1 == jb.nt;
        // The QK on tile i after this key tile's PV: this item's next key tile, or after its last the next
        // item's first, once that item's query tile has landed.  One call site per query tile: the loop
        // body exists once (a copy for an item's last tile measured 6-8% slower: the MMA warp's code
        // shares an instruction cache with the softmax warps of its sub-partition).
        auto qk_after = [&](int i) -> bool {
          bool live = i == 0 || jb.tiles > 1;
          if (last) {
            if (next == 0) return true;
            if (!wait_all(bar_q[i], (n + 1) & 1)) return false;
            tc_fence_after();
            live = i < jn.tiles;
          }
          return qk(i, gg + 1, live);
        };
        ok = (!last || reload_q(0, gg)) && pv(0, gg, j) && (!last || reload_q(1, gg)) && qk_after(0) &&
             pv(1, gg, j) && qk_after(1);
      }
      if (!ok) break;
      g += jb.nt;
      ++n;
      r = next;
      jb = jn;
      next = -2;
    }
    if (!ok) give_up();
    if (lane == 0) tc_commit(smem_u32(&bar_done));  // all MMAs of this CTA retired before TMEM is freed
    __syncwarp();
    mbar_wait(smem_u32(&bar_done), 0);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ================================================================ softmax (warps 0-7)
    const int ti = warp >> 2;              // query tile
    const int r = threadIdx.x & 127;        // row of the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t col_s = ti * kKeys;
    const uint32_t col_o = kColO + ti * 128;
    const int tok = ti * T + r / G;         // token / member of the item
    bool ok = true;
    int32_t n = 0, g = 0;
    for (;; ++n) {
      Job jb;
      const int ri = wait_item(n, jb);
      if (__any_sync(0xffffffffu, ri < 0)) { ok = false; break; }
      if (ri == 0) break;
      const bool row_valid = tok < jb.n_valid;
      int32_t lim;  // exclusive key limit of this row
      if constexpr (EXTEND) lim = row_valid ? jb.causal0 + tok + 1 : jb.kend;
      else lim = jb.kend;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < jb.nt; ++j) {
        const int gg = g + j;
        // (as in the MMA warp, no per-tile look at the abort flag: the wait's deadline ends a failed CTA)
        const bool fail_here = !mbar_wait(smem_u32(&bar_s[ti]), gg & 1);
        if (__any_sync(0xffffffffu, fail_here)) { ok = false; break; }  // warp-uniform: tcgen05.ld/st are collective
        if (ti >= jb.tiles) {  // an empty query tile: no S was computed; keep bar_p's phase
          mbar_arrive(smem_u32(&bar_p[ti]));
          continue;
        }
        tc_fence_after();
        const int32_t key0 = jb.kbeg + j * kKeys;
        const bool masked = key0 + kKeys > lim;
        const bool warp_masked = __any_sync(0xffffffffu, masked);
        // Every tile is exponentiated against a reference in a single pass: the current one, or on the
        // item's first tile the maximum of its first 32 columns.  The row sum bounds every probability
        // of the row (p <= sum), so a sum above kFastSumLimit, or one that is not finite, marks the
        // reference as stale: the warp then redoes the tile on the exact path -- row maximum first, lazy
        // reference update, then the exponentials.  P is held in registers until the pass is accepted,
        // since it overwrites S.
        uint32_t pk[2][32];
        float rowsum = 0.f, alpha = 1.f, m_ref = m_used;
        bool resc = false;
        bool exact = false;
#pragma unroll 1
        for (int attempt = 0; attempt < 2; ++attempt) {
          // row max of the raw scores (scale > 0 commutes with max), 8 independent chains
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
          auto max_of = [&]() {
            return fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
          };
          if (exact) {
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
            const float m_new = fmaxf(m_used, max_of());
            resc = m_new > m_used + kRescaleThreshold;
            m_ref = resc ? m_new : m_used;
          } else if (j == 0) {
            // the item's first tile: the reference is the maximum of chunk 0 (it holds a key of every
            // row: the row's first key is the tile's first).  O and l are empty, nothing to rescale.
            uint32_t ba[32];
            tmem_ld32(tmem + lane_addr + col_s, ba);
            tc_wait_ld_regs(ba);
            max_chunk(ba, 0);
            m_ref = max_of();
          }
          const float m_sub = (m_ref == -INFINITY) ? 0.f : m_ref;
          alpha = resc ? ex2(m_used - m_sub) : 1.f;
          // p = 2^(s * scale_log2 - m_ref): packed FMA pairs + one MUFU per score, packed to bf16 pairs
          const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
          const uint64_t neg_m2 = f2_pack(-m_sub, -m_sub);
          uint64_t sum2[4] = {0, 0, 0, 0};  // 4 independent chains of (even, odd) partial sums
          // The causal / range mask is compiled only into the variant a warp takes when one of its rows
          // ends inside this tile: the other tiles issue no compare or select per score.
          auto exp_chunk = [&](const uint32_t (&sr)[32], int c, auto mask_tag) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float s0 = __uint_as_float(sr[2 * e]), s1 = __uint_as_float(sr[2 * e + 1]);
              if constexpr (decltype(mask_tag)::value) {
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
          auto exp_tile = [&](auto mask_tag) {
            uint32_t ba[32], bb[32];
            tmem_ld32(tmem + lane_addr + col_s, ba);
            tc_wait_ld_regs(ba);
            tmem_ld32(tmem + lane_addr + col_s + 32, bb);
            exp_chunk(ba, 0, mask_tag);
            tc_wait_ld_regs(bb);
            tmem_ld32(tmem + lane_addr + col_s + 64, ba);
            exp_chunk(bb, 1, mask_tag);
            tc_wait_ld_regs(ba);
            tmem_ld32(tmem + lane_addr + col_s + 96, bb);
            exp_chunk(ba, 2, mask_tag);
            tc_wait_ld_regs(bb);
            exp_chunk(bb, 3, mask_tag);
          };
          if (warp_masked) exp_tile(BoolTag<true>{});
          else exp_tile(BoolTag<false>{});
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
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O_i holds PV_i(j-1): the commit that signalled S_i(j) covers every earlier MMA
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
        m_used = m_ref;
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p[ti]));
      }
      if (!ok) break;
      g += jb.nt;
      // ---- epilogue: O / l, then O_i is released to the next item's first PV
      const bool late = !mbar_wait(smem_u32(&bar_o[ti]), n & 1);
      if (__any_sync(0xffffffffu, late)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.f / l;
      if constexpr (EXTEND) {
        __nv_bfloat16* dst = p.o + ((jb.q_tok0 + tok) * p.hq + jb.kh * G + (r % G)) * static_cast<int64_t>(D);
        uint32_t oa[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_addr + col_o + c * 32, oa[c]);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc_wait_ld_regs(oa[c]);  // ties each array to the wait (one real wait)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t (&ov)[32] = oa[c];
          uint32_t pko[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pko[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pko[4 * e], pko[4 * e + 1], pko[4 * e + 2], pko[4 * e + 3]);
          }
        }
      } else {
        // fp32 partial rows, one per thread, at [slot][member][q head] (the G heads of a member contiguous),
        // written in whole 32-byte sectors
        const int32_t member = __ldg(p.group_reqs + jb.mem0 + (row_valid ? tok : 0));
        const bool write = row_valid && member >= 0 && member < p.batch;
        const int64_t ps = (static_cast<int64_t>(jb.slot) * p.batch + (write ? member : 0)) * p.hq + jb.kh * G + (r % G);
        float* dst = p.casc_o + ps * D;
        uint32_t oa[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_addr + col_o + c * 32, oa[c]);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc_wait_ld_regs(oa[c]);  // ties each array to the wait (one real wait)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t (&ov)[32] = oa[c];
          if (write) {
#pragma unroll
            for (int e = 0; e < 4; ++e)  // whole 32-byte sectors
              st_global_v8(dst + c * 32 + 8 * e, __uint_as_float(ov[8 * e]) * inv_l,
                           __uint_as_float(ov[8 * e + 1]) * inv_l, __uint_as_float(ov[8 * e + 2]) * inv_l,
                           __uint_as_float(ov[8 * e + 3]) * inv_l, __uint_as_float(ov[8 * e + 4]) * inv_l,
                           __uint_as_float(ov[8 * e + 5]) * inv_l, __uint_as_float(ov[8 * e + 6]) * inv_l,
                           __uint_as_float(ov[8 * e + 7]) * inv_l);
          }
        }
        if (write) p.casc_lse[ps] = m_used + __log2f(l);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_ofree[ti]));
    }
    if (!ok) give_up();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (!EXTEND) {
    // the prefix partials of this CTA are written (the barrier orders every warp's stores before this
    // thread's fence): the decode combine merges a request's partials once every CTA has counted itself
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(p.done_counter, 1);
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace ra
