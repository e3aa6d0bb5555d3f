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

constexpr int kSlab = 16;          // keys per ring stage (the MMA M side)
constexpr int kMaxStages = 8;
constexpr int kItemRing = 16;      // published items; the leader runs at most nstage + 1 items ahead
constexpr int kProducers = 4;      // warps issuing the bulk copies of a slab (TMA issue rate grows with them)
constexpr int kRowsPerProducer = 2 * kSlab / kProducers;  // K rows then V rows of a slab, split evenly
constexpr int kHdrBytes = 640;     // full/empty barriers, item ring, abort flag, item / done / free barriers
constexpr int kSmemLimit = 227 * 1024;
constexpr int kPlanThreads = 1024;  // one CTA plans the call
constexpr int kRemBuckets = 64;     // size classes of the requests' last (short) items
constexpr int kCombineWarps = 4;    // (request, q head) merges per combine CTA
constexpr float kDecodeRescale = 8.0f;  // log2 units: the decode softmax's reference moves past this

// One work item: keys [k0, k1) of request b for the kv heads of head group hg; d is its dense index
// (request-major: the item's partial results live at d).
struct Item {
  int32_t b, split, hg, k0, k1, start, n_splits, row, d;
};

// Claim `idx` = (position in the plan's longest-first order) * n_hgroups + hg.  The plan (written by
// decode_plan_kernel) lists only non-empty items of valid requests.  Plan arrays are read with plain
// loads: they are written on the device by the kernel before this one.
__device__ __forceinline__ void decode_item(const DecodeParams& p, int32_t idx, Item& it) {
  it.hg = idx % p.n_hgroups;
  it.d = p.order[idx / p.n_hgroups];
  it.b = p.item_req[it.d];
  const int32_t i0 = p.req_item0[it.b];
  it.split = it.d - i0;
  it.n_splits = p.req_item0[it.b + 1] - i0;
  it.row = __ldg(p.rpi + it.b);
  const int32_t L = min(__ldg(p.seq_lens + it.b), p.max_seq_len);
  const int32_t start = p.key_start ? __ldg(p.key_start + it.b) : 0;
  it.start = start < 0 ? 0 : (start > L ? L : start);
  const int32_t chunk = p.plan[1];
  it.k0 = it.start + it.split * chunk;
  it.k1 = min(L, it.k0 + chunk);
}

// Persistent split-KV decode.  One CTA per SM pulls (request, split, head group) items from a
// counter.  Warps hpc .. hpc+3 are producers: per 16-key slab, producer w copies a quarter of the
// slab's 32 rows -- each key's K row and V row of the whole head group, hpc * D * 2 contiguous bytes
// -- with one cp.async.bulk each into a ring stage.  The first producer also claims the items and
// publishes them through a shared ring (with one mbarrier per entry) as soon as it claims them, a
// few slabs ahead, so every producer looks one slab ahead across items for its slot ids.  Consumer
// warp w owns kv head hg * hpc + w of every item.  Warp hpc+4 signals finished partials: once every
// consumer warp is done with an item whose request goes through the combine, it makes the partials
// visible device-wide (a gpu-scope fence) and adds one to the request's count, so the combine can merge
// the request as soon as its count is complete -- the fence stays off the consumer warps' path.
template <int D>
__global__ void __launch_bounds__(32 * (kMaxHeadsPerCta + kProducers + 1), 1) decode_kernel(const DecodeParams p) {
  constexpr int KT = D / 16;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nc = p.hpc;
  const int ns = p.nstage;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase;        // ns mbarriers (kProducers arrivals + bytes)
  const uint32_t empty0 = sbase + 64;  // ns mbarriers (nc consumer arrivals)
  volatile int32_t* s_items = reinterpret_cast<volatile int32_t*>(smem + 128);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(smem + 192);
  const uint32_t item0 = sbase + 256;  // kItemRing mbarriers: entry published
  const uint32_t done0 = sbase + 384;  // kItemRing mbarriers: every consumer warp is done with the entry
  const uint32_t free0 = sbase + 512;  // kItemRing mbarriers: the signal warp has read the entry (slot free)
  const uint32_t stage0 = sbase + kHdrBytes;
  const int RS = p.row_stride;
  // Without groups the plan kernel is the call's first kernel: wait for it (its plan, the reset counters and
  // a fused store) before anything else.  With groups the plan kernel made its writes visible before it let
  // this kernel launch, and it completes only after the prefix pass: this kernel reads nothing the pass
  // writes, so it does not wait here (it runs beside the pass).  It waits before leaving, so that its
  // completion implies the plan's and the prefix pass's.  Then the combine may launch: the plan it reads is
  // visible, and it waits per request for the partials it merges.
  if (p.key_start == nullptr) griddep_wait();
  griddep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full0 + 8 * s, kProducers);
      mbar_init(empty0 + 8 * s, nc);
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(item0 + 8 * s, 1);
      mbar_init(done0 + 8 * s, nc);
      mbar_init(free0 + 8 * s, 1);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int row_bytes = p.hpc * D * 2;

  if (warp >= nc && warp < nc + kProducers) {
    // ================================================================ producers
    const int pw = warp - nc;
    const bool leader = pw == 0;
    const int row_id = pw * kRowsPerProducer + lane;  // this lane's row of a slab (lane < kRowsPerProducer)
    const bool is_v = row_id >= kSlab;
    const int key_in_slab = row_id & (kSlab - 1);
    const __nv_bfloat16* pool = is_v ? p.v_pool : p.k_pool;
    const uint32_t row_off = (is_v ? kSlab * RS : 0) + key_in_slab * RS;
    int32_t n_claims = 0;  // plan items x head groups (read once the plan is visible)
    auto claim = [&]() -> int32_t {  // warp-collective
      int32_t idx = 0;
      if (lane == 0) idx = atomicAdd(p.counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      return idx < n_claims ? idx : -1;
    };
    // entry n reuses the ring slot of entry n - kItemRing: the signal warp, the last reader, must have read it
    auto publish = [&](int32_t n, int32_t idx) -> bool {
      if (n >= kItemRing && !mbar_wait(free0 + 8 * (n % kItemRing), ((n / kItemRing) - 1) & 1)) return false;
      if (lane == 0) {
        s_items[n % kItemRing] = idx;
        mbar_arrive(item0 + 8 * (n % kItemRing));
      }
      return true;
    };
    // 1: item n in `it`; 0: end of work; -1: a bounded wait ran out
    auto next_item = [&](int32_t n, Item& it) -> int {
      if (!mbar_wait(item0 + 8 * (n % kItemRing), (n / kItemRing) & 1)) return -1;
      const int32_t idx = s_items[n % kItemRing];
      if (idx < 0) return 0;
      decode_item(p, idx, it);
      return 1;
    };
    auto load_slot = [&](const Item& it, int32_t s) -> int32_t {  // rows past the range repeat the last key
      if (lane >= kRowsPerProducer) return 0;
      const int32_t nk = it.k1 - it.k0;
      int32_t key = s * kSlab + key_in_slab;
      key = key < nk ? key : nk - 1;
      return __ldg(p.table + static_cast<int64_t>(it.row) * p.table_stride + it.k0 + key);
    };
    n_claims = p.plan[0] * p.n_hgroups;
    bool ok = true;
    if (leader) ok = __all_sync(0xffffffffu, publish(0, claim()));
    int32_t n = 0, c = 0, s = 0;
    Item it;
    int r = ok ? next_item(0, it) : -1;
    ok = r >= 0;
    int32_t slot = r > 0 ? load_slot(it, 0) : 0;
    while (ok && r > 0) {
      const int32_t n_slabs = (it.k1 - it.k0 + kSlab - 1) / kSlab;
      // the leader claims the next item when this one has ns slabs left to issue: the claim overlaps
      // them, and items stay unclaimed for CTAs that start late (behind a cascade prefix pass that
      // holds their SMs) instead of queueing behind this one
      if (leader && s == (n_slabs > ns ? n_slabs - ns : 0) && !__all_sync(0xffffffffu, publish(n + 1, claim()))) {
        ok = false;
        break;
      }
      // one slab ahead: the next (item, slab) and its slot id
      Item it2 = it;
      int32_t s2 = s + 1, n2 = n;
      int r2 = 1;
      if (s2 == n_slabs) {
        n2 = n + 1;
        s2 = 0;
        r2 = next_item(n2, it2);
        if (r2 < 0) { ok = false; break; }
      }
      const int32_t slot2 = r2 > 0 ? load_slot(it2, s2) : 0;
      // slab s of item n into stage c % ns
      const int st = c % ns;
      if (c >= ns && !mbar_wait(empty0 + 8 * st, ((c / ns) + 1) & 1)) { ok = false; break; }
      if (*s_abort) { ok = false; break; }
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, kRowsPerProducer * row_bytes);
      __syncwarp();
      if (lane < kRowsPerProducer) {
        int32_t sl = slot;
        if (sl < 0 || sl >= p.num_slots) {
          flag_error(p.err, RA_DEVERR_SLOT);
          sl = 0;
        }
        bulk_g2s(stage0 + st * p.stage_bytes + row_off,
                 pool + static_cast<int64_t>(sl) * p.hkv * D + static_cast<int64_t>(it.hg) * p.hpc * D, row_bytes,
                 full0 + 8 * st);
      }
      ++c;
      it = it2;
      s = s2;
      n = n2;
      r = r2;
      slot = slot2;
    }
    if (ok) {
      // end of work (entry n holds -1): every producer arrives on the next stage, the consumers read
      // the marker from it
      const int st = c % ns;
      if (c >= ns && !mbar_wait(empty0 + 8 * st, ((c / ns) + 1) & 1)) ok = false;
      if (ok && lane == 0) mbar_arrive(full0 + 8 * st);
    }
    if (!ok) {
      if (lane == 0) {
        *s_abort = 1;
        flag_error(p.err, RA_DEVERR_TIMEOUT);
      }
      // copies this warp issued must land before the CTA leaves
      for (int32_t j = (c > ns ? c - ns : 0); j < c; ++j) mbar_wait(full0 + 8 * (j % ns), (j / ns) & 1);
    }
    griddep_wait();
    return;
  }
  if (warp == nc + kProducers) {
    // ================================================================ signaller
    for (int32_t n = 0;; ++n) {
      const int e = n % kItemRing;
      if (!mbar_wait(done0 + 8 * e, (n / kItemRing) & 1)) {
        if (lane == 0) {
          *s_abort = 1;
          flag_error(p.err, RA_DEVERR_TIMEOUT);
        }
        break;
      }
      const int32_t idx = s_items[e];
      __syncwarp();
      if (lane == 0) mbar_arrive(free0 + 8 * e);
      if (idx < 0) break;
      if (lane == 0) {
        Item it;
        decode_item(p, idx, it);
        if (!(it.n_splits == 1 && it.start == 0)) {  // partials, merged by the combine
          __threadfence();  // the consumers' partials (ordered before this by the done barrier) first
          atomicAdd(p.req_done + it.b, 1);
        }
      }
      __syncwarp();
    }
    griddep_wait();
    return;
  }
  if (warp > nc + kProducers) {
    griddep_wait();
    return;
  }

  // ================================================================ consumers
  const int g = lane >> 2;  // q head within the GQA group (MMA N index)
  const int tq = lane & 3;
  const uint32_t a_off = (lane & 15) * RS + (lane >> 4) * 16 + warp * D * 2;
  const uint32_t v_off = kSlab * RS + ((lane & 7) + ((lane >> 4) << 3)) * RS + ((lane >> 3) & 1) * 16 + warp * D * 2;
  int32_t n = 0, c = 0;
  bool clean = false;  // left through the end marker
  for (;; ++n) {
    int st = c % ns;
    if (!mbar_wait(full0 + 8 * st, (c / ns) & 1) || *s_abort) break;
    const int32_t idx = s_items[n % kItemRing];
    if (idx < 0) {
      clean = true;
      __syncwarp();
      if (lane == 0) mbar_arrive(done0 + 8 * (n % kItemRing));  // the signal warp reads the end marker
      break;
    }
    Item it;
    decode_item(p, idx, it);
    const int kh = it.hg * p.hpc + warp;
    // Q^T fragments (B operand): column g is q head kh*G + g
    uint32_t qf[KT][2];
    {
      const bool live = g < p.group;
      const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(it.b) * p.hq + kh * p.group + (live ? g : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qf[kk][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq)) : 0u;
        qf[kk][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq)) : 0u;
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[KT][4];
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    const int32_t n_slabs = (it.k1 - it.k0 + kSlab - 1) / kSlab;
    bool ok = true;
    for (int32_t s = 0; s < n_slabs; ++s, ++c) {
      st = c % ns;
      if (s > 0 && !mbar_wait(full0 + 8 * st, (c / ns) & 1)) { ok = false; break; }
      const uint32_t stage = stage0 + st * p.stage_bytes;
      // S^T[16 keys x 8 heads] = K Q^T, two independent MMA chains
      float s1[4] = {0.f, 0.f, 0.f, 0.f};
      float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KT; kk += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(stage + a_off + kk * 32, a0, a1, a2, a3);
        ldsm_x4(stage + a_off + (kk + 1) * 32, b0, b1, b2, b3);
        mma_bf16_16816(s1, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        mma_bf16_16816(s2, b0, b1, b2, b3, qf[kk + 1][0], qf[kk + 1][1]);
      }
      const int32_t kbase = it.k0 + s * kSlab;
      const bool v_lo = kbase + g < it.k1;
      const bool v_hi = kbase + g + 8 < it.k1;
      const float x0 = v_lo ? (s1[0] + s2[0]) * p.scale_log2 : -INFINITY;
      const float x1 = v_lo ? (s1[1] + s2[1]) * p.scale_log2 : -INFINITY;
      const float x2 = v_hi ? (s1[2] + s2[2]) * p.scale_log2 : -INFINITY;
      const float x3 = v_hi ? (s1[3] + s2[3]) * p.scale_log2 : -INFINITY;
      // Lazy reference: the running maximum moves (and O and l are rescaled) only when a score of the slab
      // exceeds it by more than kDecodeRescale, which a warp vote finds; otherwise the slab is exponentiated
      // against the reference as it stands (every p <= 2^kDecodeRescale).  The first slab of an item always
      // moves it (the reference starts at -inf).
      if (__any_sync(0xffffffffu, x0 > m0 + kDecodeRescale || x2 > m0 + kDecodeRescale ||
                                      x1 > m1 + kDecodeRescale || x3 > m1 + kDecodeRescale)) {
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
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          acc[mt][0] *= al0;
          acc[mt][1] *= al1;
          acc[mt][2] *= al0;
          acc[mt][3] *= al1;
        }
      }
      const float p0 = ex2(x0 - m0), p1 = ex2(x1 - m1), p2 = ex2(x2 - m0), p3 = ex2(x3 - m1);
      l0 += p0 + p2;
      l1 += p1 + p3;
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
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }
    if (!ok) break;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // outputs: thread holds (d = mt*16 + g [+8], q head 2*tq [+1]) of this kv head
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const bool h0 = 2 * tq < p.group, h1 = 2 * tq + 1 < p.group;
    const int64_t bh0 = static_cast<int64_t>(it.b) * p.hq + kh * p.group + 2 * tq;
    if (it.n_splits == 1 && it.start == 0) {
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int d = mt * 16 + g;
        if (h0) {
          p.o[bh0 * D + d] = __float2bfloat16_rn(acc[mt][0] * inv0);
          p.o[bh0 * D + d + 8] = __float2bfloat16_rn(acc[mt][2] * inv0);
        }
        if (h1) {
          p.o[(bh0 + 1) * D + d] = __float2bfloat16_rn(acc[mt][1] * inv1);
          p.o[(bh0 + 1) * D + d + 8] = __float2bfloat16_rn(acc[mt][3] * inv1);
        }
      }
    } else {
      const int64_t ps0 = static_cast<int64_t>(it.d) * p.hq + kh * p.group + 2 * tq;  // partial row of (item, head)
      const int64_t ps1 = ps0 + 1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int d = mt * 16 + g;
        if (h0) {
          p.part_o[ps0 * D + d] = acc[mt][0] * inv0;
          p.part_o[ps0 * D + d + 8] = acc[mt][2] * inv0;
        }
        if (h1) {
          p.part_o[ps1 * D + d] = acc[mt][1] * inv1;
          p.part_o[ps1 * D + d + 8] = acc[mt][3] * inv1;
        }
      }
      if (g == 0) {
        if (h0) p.part_lse[ps0] = m0 + __log2f(l0);
        if (h1) p.part_lse[ps1] = m1 + __log2f(l1);
      }
    }
    // this warp's part of the entry is written (__syncwarp orders the lanes' stores before lane 0's release)
    __syncwarp();
    if (lane == 0) mbar_arrive(done0 + 8 * (n % kItemRing));
  }
  if (!clean && lane == 0) {
    // a bounded wait ran out: stop the producer as well
    *s_abort = 1;
    flag_error(p.err, RA_DEVERR_TIMEOUT);
  }
  griddep_wait();
}

// Merge the partials of every request that has more than one (its private splits' and the shared-prefix
// pass's): o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).  One warp per (request, q head), each lane
// owning D/32 dims.  The kernel launches while the decode kernel still runs (every decode CTA has started)
// and a warp waits only for its own request: until the request's count of (item, head group) partials is
// complete (the decode kernel's signal warp adds to it) and, when the request has prefix partials, until
// every CTA of the prefix pass is done.  Requests whose last items finish early are merged while the rest
// of the decode kernel runs.  Partials are read through L2 (they were written by other SMs during this
// call).  The merge is latency-bound, so a warp keeps its loads in flight together: the request's
// description with both counts, then the log-sum-exps of 32 partials (one per lane) with the first kRows
// rows known to be written (private partials always are; with one-level groups so are the first
// ceil(key_start / cchunk) prefix slots), the weights from warp shuffles, and the other rows kRows at a
// time -- with multi-level groups, prefix rows only where a group wrote them (a finite log-sum-exp).
// Partials are taken private first, then prefix, in chunks of 32 folded with a running maximum.
template <int D>
__device__ __forceinline__ void merge_request_head(const DecodeParams& p) {
  constexpr int V = D / 32;
  constexpr int kRows = 8;
  const int warp_global = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.batch * p.hq) return;
  const int b = warp_global / p.hq;
  // the request's description and, on lane 0, both counts, loaded together (one round trip)
  int32_t L = __ldg(p.seq_lens + b);
  const int32_t row = __ldg(p.rpi + b);
  int32_t start = p.key_start ? __ldcg(p.key_start + b) : 0;
  const int32_t i0 = __ldcg(p.req_item0 + b);  // the request's private items are i0 .. i0 + n_splits - 1
  const int32_t i1 = __ldcg(p.req_item0 + b + 1);
  int32_t done_seen = 0, pre_seen = 0;
  if (lane == 0) {
    done_seen = ld_relaxed_gpu(p.req_done + b);
    if (p.key_start) pre_seen = ld_relaxed_gpu(p.prefix_done);
  }
  const int32_t n_splits = i1 - i0;
  if (row < 0 || row >= p.table_rows || L < 1) return;
  if (L > p.max_seq_len) L = p.max_seq_len;
  start = start < 0 ? 0 : (start > L ? L : start);
  // prefix partials: with one-level groups the slots the pass wrote, else every slot of every level (those
  // no group wrote hold -inf: weight 0, skipped)
  const int32_t n_pre = start > 0 ? (p.casc_one_level ? (start + p.cchunk - 1) / p.cchunk : p.casc_slots) : 0;
  if (n_splits == 1 && n_pre == 0) return;  // written directly by the decode kernel
  // wait for this request's partials: lane 0 polls; then every lane reads both counts itself and fences,
  // so that each lane's own loads of the partials follow an acquire of the counts it saw complete
  const int32_t expect = n_splits * p.n_hgroups;
  bool ready = true;
  if (lane == 0) {
    if (expect > 0 && done_seen < expect) ready = wait_count(p.req_done + b, expect);
    if (ready && n_pre > 0 && pre_seen < p.prefix_ctas) ready = wait_count(p.prefix_done, p.prefix_ctas);
    if (!ready) flag_error(p.err, RA_DEVERR_TIMEOUT);
  }
  if (!__shfl_sync(0xffffffffu, ready, 0)) return;
  if (expect > 0) (void)ld_relaxed_gpu(p.req_done + b);
  if (n_pre > 0) (void)ld_relaxed_gpu(p.prefix_done);
  fence_acq_rel_gpu();
  const int32_t n = n_splits + n_pre;
  // partials known to be written: their rows are loaded with the log-sum-exps, the others once weighed
  const int32_t n_written = p.casc_one_level ? n : n_splits;
  const int64_t bh = warp_global;
  const int64_t h = bh - static_cast<int64_t>(b) * p.hq;
  const int64_t slot_stride = static_cast<int64_t>(p.batch) * p.hq;  // prefix partials: [slot][request][q head]
  auto lse_of = [&](int s) {
    return s < n_splits ? __ldcg(p.part_lse + (i0 + s) * p.hq + h)
                        : __ldcg(p.casc_lse + (s - n_splits) * slot_stride + bh);
  };
  auto load_row = [&](int s, float (&x)[V]) {
    const float* src = (s < n_splits ? p.part_o + ((i0 + s) * p.hq + h) * D
                                     : p.casc_o + ((s - n_splits) * slot_stride + bh) * D) + lane * V;
    if constexpr (V == 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
      x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
    } else {
      const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
      x[0] = t.x, x[1] = t.y;
    }
  };
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float mrun = -INFINITY, wsum = 0.f;  // wsum: this lane's partials' weights (relative to mrun)
  for (int base = 0; base < n; base += 32) {
    const int cnt = n - base < 32 ? n - base : 32;
    const float ls = lane < cnt ? lse_of(base + lane) : -INFINITY;
    float x[kRows][V];
#pragma unroll
    for (int k = 0; k < kRows; ++k)
      if (k < cnt && base + k < n_written) load_row(base + k, x[k]);  // written: load at once
    float mc = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
    const float mnew = fmaxf(mrun, mc);
    if (mnew == -INFINITY) continue;  // no partial written so far
    const float sc = ex2(mrun - mnew);  // 0 while mrun is -inf (acc and wsum are 0 then)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= sc;
    wsum *= sc;
    mrun = mnew;
    const float wl = ex2(ls - mnew);  // weight of partial base + lane (0 for an empty prefix slot)
    wsum += wl;
    for (int k0 = 0; k0 < cnt; k0 += kRows) {
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int s = base + k0 + k;
        const bool loaded = k0 == 0 && s < n_written;
        const float w = __shfl_sync(0xffffffffu, wl, (k0 + k) & 31);
        if (k0 + k < cnt && w > 0.f && !loaded) load_row(s, x[k]);
      }
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, (k0 + k) & 31);
        if (k0 + k < cnt && w > 0.f) {
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = fmaf(w, x[k][v], acc[v]);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = 1.f / wsum;
#pragma unroll
  for (int v = 0; v < V; v += 2)
    *reinterpret_cast<__nv_bfloat162*>(p.o + bh * D + lane * V + v) =
        __floats2bfloat162_rn(acc[v] * inv, acc[v + 1] * inv);
}

template <int D>
__global__ void __launch_bounds__(32 * kCombineWarps) decode_combine_kernel(const DecodeParams p) {
  griddep_launch();
  merge_request_head<D>(p);
  // every CTA waits before it leaves, so that this grid's completion implies the decode kernel's (and,
  // through it, the plan kernel's and the prefix pass's): the next kernel on the stream may rely on it
  griddep_wait();
}

// Block-wide exclusive scan of (a, b) pairs over kPlanThreads threads; totals returned in ta, tb.
__device__ __forceinline__ void plan_scan2(int32_t& a, int32_t& b, int32_t& ta, int32_t& tb, int32_t* s_wa,
                                           int32_t* s_wb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t ia = a, ib = b;  // inclusive within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t xa = __shfl_up_sync(0xffffffffu, ia, off), xb = __shfl_up_sync(0xffffffffu, ib, off);
    if (lane >= off) ia += xa, ib += xb;
  }
  if (lane == 31) s_wa[warp] = ia, s_wb[warp] = ib;
  __syncthreads();
  if (warp == 0) {
    int32_t wa = s_wa[lane], wb = s_wb[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t xa = __shfl_up_sync(0xffffffffu, wa, off), xb = __shfl_up_sync(0xffffffffu, wb, off);
      if (lane >= off) wa += xa, wb += xb;
    }
    s_wa[lane] = wa, s_wb[lane] = wb;  // inclusive warp totals
  }
  __syncthreads();
  const int32_t pa = warp > 0 ? s_wa[warp - 1] : 0, pb = warp > 0 ? s_wb[warp - 1] : 0;
  ta = s_wa[31], tb = s_wb[31];
  a = pa + ia - a;
  b = pb + ib - b;
  __syncthreads();  // the scratch may be reused
}

// Fused store (ra_decode_attention_store): pool[st_loc[b]] = new row b for K and V, one 16-byte vector
// per thread and step, consecutive threads on consecutive vectors of a row (as ra_kv_store).  Run by
// the call's first kernel after it waited for the kernels before it (they may still read the slots).
__device__ __forceinline__ void scatter_new_rows(const DecodeParams& p, int64_t first, int64_t stride) {
  uint4* kp = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.k_pool));
  uint4* vp = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.v_pool));
  for (int64_t i = first; i < p.st_total; i += stride) {
    const int64_t b = i / p.st_row_vecs;
    const int32_t c = static_cast<int32_t>(i - b * p.st_row_vecs);
    const int32_t slot = __ldg(p.st_loc + b);
    if (slot < 0 || slot >= p.num_slots) {
      if (c == 0) flag_error(p.err, RA_DEVERR_SLOT);
      continue;
    }
    const uint4 kv = __ldg(p.st_k + i), vv = __ldg(p.st_v + i);
    const int64_t dst = static_cast<int64_t>(slot) * p.st_row_vecs + c;
    kp[dst] = kv;
    vp[dst] = vv;
  }
}

// The private-key work plan of one decode call, made on the device from the real lengths (the host only
// knows bounds).  T = the batch's private keys (seq_len minus the cascade start, over valid requests);
// chunk = max(kDecodeMinChunk, T / kDecodePlanItems rounded up to 16), so a call has at most
// kDecodePlanItems + batch items however long its contexts are.  Request b's items get the dense indices
// req_item0[b] .. req_item0[b+1]-1 (where their partials live); the claim order lists every full-chunk
// item first, then each request's shorter last item by decreasing size (longest processing time first),
// so the CTAs that finish last finish on short items.  One CTA of kPlanThreads threads; each thread owns
// a contiguous run of requests.  It also resets the work counter.  With a fused store (and no groups)
// CTAs 1.. of the grid scatter the step's new rows instead.
__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const DecodeParams p) {
  if (blockIdx.x > 0) {  // the fused store's CTAs (only without groups; CTA 0 plans)
    griddep_launch();
    griddep_wait();
    scatter_new_rows(p, static_cast<int64_t>(blockIdx.x - 1) * blockDim.x + threadIdx.x,
                     static_cast<int64_t>(gridDim.x - 1) * blockDim.x);
    return;
  }
  __shared__ int32_t s_wa[32], s_wb[32];
  __shared__ int32_t s_hist[kRemBuckets];
  __shared__ unsigned long long s_total;
  // Without groups this is the call's first kernel: it lets the decode kernel launch at once (the decode
  // kernel waits for this grid before its first claim) and plans from the call's inputs, which no kernel
  // of this library writes, while the kernel before it finishes; it waits for that kernel only before its
  // first write to the workspace (the kernel may be the previous call's combine, still reading it).
  // With groups it runs behind the prefix pass, which let it launch only after the key starts were
  // complete; it does not wait for the pass, so that the decode kernel can run beside it.
  const bool behind_pass = p.key_start != nullptr;
  if (!behind_pass) griddep_launch();
  const int t = threadIdx.x;
  const int32_t per = (p.batch + kPlanThreads - 1) / kPlanThreads;
  const int32_t r0 = min(p.batch, t * per), r1 = min(p.batch, r0 + per);
  auto len_of = [&](int32_t b, bool report) -> int32_t {
    const int32_t row = __ldg(p.rpi + b);
    int32_t L = __ldg(p.seq_lens + b);
    if (row < 0 || row >= p.table_rows || L < 1) {
      if (report) flag_error(p.err, (row < 0 || row >= p.table_rows) ? RA_DEVERR_TABLE : RA_DEVERR_LENGTH);
      return 0;
    }
    if (L > p.max_seq_len) {
      if (report) flag_error(p.err, RA_DEVERR_LENGTH);
      L = p.max_seq_len;
    }
    int32_t start = p.key_start ? p.key_start[b] : 0;
    start = start < 0 ? 0 : (start > L ? L : start);
    return L - start;
  };
  if (t == 0) s_total = 0ull;
  if (t < kRemBuckets) s_hist[t] = 0;
  __syncthreads();
  unsigned long long tot = 0;
  for (int32_t b = r0; b < r1; ++b) tot += static_cast<unsigned long long>(len_of(b, true));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  if ((t & 31) == 0) atomicAdd(&s_total, tot);
  __syncthreads();
  const unsigned long long per_item = (s_total + kDecodePlanItems - 1) / kDecodePlanItems;
  // (the host bounds batch x max_seq_len by kDecodePlanItems x 2^30, so the chunk fits in 31 bits)
  const int32_t chunk = static_cast<int32_t>(
      per_item <= kDecodeMinChunk ? kDecodeMinChunk : ((per_item + 15) / 16) * 16);
  // item counts (all, full-chunk) of this thread's requests, scanned over the block
  int32_t cnt = 0, full = 0;
  for (int32_t b = r0; b < r1; ++b) {
    const int32_t len = len_of(b, false);
    cnt += (len + chunk - 1) / chunk;
    full += len / chunk;
    const int32_t rem = len % chunk;
    if (rem > 0) atomicAdd(&s_hist[static_cast<int64_t>(chunk - rem) * kRemBuckets / chunk], 1);
  }
  int32_t n_items, n_full;
  plan_scan2(cnt, full, n_items, n_full, s_wa, s_wb);
  if (t < 32) {  // bucket starts, largest remainders first, after the full items: a warp scan, 2 buckets a lane
    const int32_t c0 = s_hist[2 * t], c1 = s_hist[2 * t + 1];
    int32_t incl = c0 + c1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (t >= off) incl += y;
    }
    const int32_t excl = n_full + incl - (c0 + c1);
    s_hist[2 * t] = excl;
    s_hist[2 * t + 1] = excl + c0;
  }
  __syncthreads();
  if (!behind_pass) griddep_wait();  // the workspace is free
  for (int32_t b = r0; b < r1; ++b) {
    const int32_t len = len_of(b, false);
    const int32_t c = (len + chunk - 1) / chunk, f = len / chunk, rem = len % chunk;
    p.req_item0[b] = cnt;
    p.req_done[b] = 0;
    for (int32_t s = 0; s < c; ++s) p.item_req[cnt + s] = b;
    for (int32_t s = 0; s < f; ++s) p.order[full + s] = cnt + s;
    if (rem > 0) p.order[atomicAdd(&s_hist[static_cast<int64_t>(chunk - rem) * kRemBuckets / chunk], 1)] = cnt + f;
    cnt += c;
    full += f;
  }
  if (t == 0) {
    p.req_item0[p.batch] = n_items;
    p.plan[0] = n_items;
    p.plan[1] = chunk;
    *p.counter = 0;
  }
  if (behind_pass) {
    // The decode kernel launches once every thread's plan writes are visible device-wide (it reads the
    // plan without waiting for this grid); this grid completes only after the prefix pass, so that the
    // decode kernel's completion, and through it the combine, implies the pass's.
    __threadfence();
    __syncthreads();
    griddep_launch();
    griddep_wait();
  }
}

// First kernel of a call with cascade groups.  CTA 0 clears the workspace's leading integer block (key
// starts, the work counters, the prefix pass's completion count), then sets key_start[b] to the largest range
// end of b's groups (0 for requests in no group); CTAs 1 .. lse_ctas set every prefix-partial log-sum-exp to
// -inf (slots no group writes stay so); the CTAs after them run the fused store.
__global__ void cascade_setup_kernel(const DecodeParams p, int32_t* ints, int32_t n_zero, const int32_t* group_indptr,
                                     const int32_t* group_reqs, const int32_t* group_prefix_len, int32_t num_groups,
                                     int64_t n_lse, int32_t lse_ctas) {
  griddep_wait();  // earlier kernels on the stream may still use the workspace and the pool
  griddep_launch();
  if (blockIdx.x == 0) {
    for (int32_t i = threadIdx.x; i < n_zero; i += blockDim.x) ints[i] = 0;
    __syncthreads();
    const int32_t total = __ldg(group_indptr + num_groups);
    for (int32_t m = threadIdx.x; m < total; m += blockDim.x) {
      int32_t lo = 0, hi = num_groups;  // group g with indptr[g] <= m < indptr[g+1]
      while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(group_indptr + mid) <= m) lo = mid; else hi = mid;
      }
      const int32_t b = __ldg(group_reqs + m);
      if (b < 0 || b >= p.batch) {
        flag_error(p.err, RA_DEVERR_TABLE);
        continue;
      }
      atomicMax(ints + b, __ldg(group_prefix_len + lo));
    }
  } else if (static_cast<int32_t>(blockIdx.x) <= lse_ctas) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n_lse;
         i += static_cast<int64_t>(lse_ctas) * blockDim.x)
      p.casc_lse[i] = -INFINITY;
  } else {
    const int64_t cta = blockIdx.x - 1 - lse_ctas;
    scatter_new_rows(p, cta * blockDim.x + threadIdx.x, static_cast<int64_t>(gridDim.x - 1 - lse_ctas) * blockDim.x);
  }
}

template <int D>
ra_status launch_decode(const DecodeParams& p, int grid, int smem, cudaStream_t stream) {
  auto kern = decode_kernel<D>;
  static int configured[64] = {};
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  if (smem > dev.max_smem_optin) return fail(RA_ERR_UNSUPPORTED, "decode needs %d bytes of shared memory", smem);
  if (configured[dev.device] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, "cudaFuncSetAttribute(decode): %s", cudaGetErrorString(e));
    configured[dev.device] = kSmemLimit;
  }
  if (ra_status st = launch_pdl("decode_kernel", kern, dim3(grid), dim3(32 * (p.hpc + kProducers + 1)), smem, stream, p))
    return st;
  const int nwarps = p.batch * p.hq;
  return launch_pdl("decode_combine_kernel", decode_combine_kernel<D>, dim3((nwarps + kCombineWarps - 1) / kCombineWarps),
                    dim3(32 * kCombineWarps), 0, stream, p);
}

}  // namespace

// kv heads per work item: the largest divisor of Hkv that is <= 8 (one consumer warp each).
static int32_t heads_per_cta(int32_t num_kv_heads) {
  for (int32_t h = kMaxHeadsPerCta; h > 1; --h)
    if (num_kv_heads % h == 0) return h;
  return 1;
}

// Private keys are cut into items on the device (decode_plan_kernel); the host only bounds their number.
// Shared-prefix pass (cascade): 256-row items of (member, q head) per group and kv head, each covering
// at most `cchunk` prefix keys.  The persistent private decode is launched programmatically after it
// and runs on the SMs the prefix pass leaves free.
DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len,
                       int32_t num_groups, int32_t max_group_prefix_len, int32_t max_group_size) {
  DecodePlan pl;
  pl.max_items = kDecodePlanItems + batch;
  if (num_groups > 0 && max_group_prefix_len > 0) {
    // Prefix keys per prefix-pass CTA (a multiple of the 128-key tile, at most 2048): the split count
    // that minimises the pass's makespan, waves x (tiles per CTA + the ~3 tiles' worth of fill and
    // drain a CTA costs), one CTA per SM; on a tie the fewer CTAs.
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t members_per_cta = 2 * (128 / (group > 0 ? group : 1));  // two 128-row query tiles
    const int64_t mtiles = (max_group_size + members_per_cta - 1) / members_per_cta;
    const int64_t base = static_cast<int64_t>(num_groups) * num_kv_heads * mtiles;
    const int64_t tiles = (max_group_prefix_len + 127) / 128;
    // CTAs per wave: GB300's 152 SMs in the share the shared prefix takes of the longest context (the
    // host-side bounds), at least two thirds of them; the pass's grid is capped at the wave, and the rest
    // run the private decode beside the pass.  Measured: a forked batch (8192 shared + <= 257 private
    // keys) 64 -> 58 us with all SMs for the pass, while the 8B-shape batch (1024 shared of <= 4096) loses
    // 10% unless a third is left to its private keys; the multi-turn mix (prefixes up to 13.7K of 32K)
    // takes 223 us with the grid capped at 104 CTAs, 230 us with all 152, 225-244 us with a wave of
    // 88 / 76 / 64.  Computed from the call's bounds, not the device: the workspace size (sized on the
    // host, possibly with no device current) must not depend on which device runs the call.
    const int64_t share = 152 * static_cast<int64_t>(max_group_prefix_len) / (max_seq_len > 0 ? max_seq_len : 1);
    const int64_t sms = share < 104 ? 104 : (share > 152 ? 152 : share);
    // Batches whose contexts are the shared prefix plus a short private tail (its bound at most 1/8 of the
    // prefix): the SMs beyond the pass decode the tails -- on average half the bound, ~105 KB per SM per
    // key tile of the pass (~50 GB/s per SM while HBM is not saturated, measured), starting ~4 tiles
    // after the pass -- and the split balances the two.  Measured on a forked batch (8192 shared keys,
    // tails of 0..256): 1024 / 1280 / 1408 / 1536 / 1664 / 1792 keys per CTA took 54.2 / 49.0 / 50.6 /
    // 52.1 / 53.1 / 56.3 us; this picks 1280.
    const int64_t tail = static_cast<int64_t>(max_seq_len) - max_group_prefix_len;
    const bool short_tails = tail >= 0 && 8 * tail <= max_group_prefix_len;
    const double tail_bytes = 0.5 * static_cast<double>(batch) * static_cast<double>(tail) * num_kv_heads *
                              static_cast<double>(head_dim) * 2 * 2;
    int64_t best_tiles = 16;
    double best_cost = -1.0;
    for (int64_t per = 16; per >= 1; --per) {  // tiles per CTA
      const int64_t splits = (tiles + per - 1) / per;
      const int64_t waves = (base * splits + sms - 1) / sms;
      double cost = static_cast<double>(waves * (per + 3));
      if (short_tails) {
        const int64_t ctas = base * splits < sms ? base * splits : sms;
        const double tail_cost = tail_bytes / (static_cast<double>(152 - ctas) * 105e3) + 4.0;
        if (tail_cost > cost) cost = tail_cost;
      }
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_tiles = per;
      }
    }
    if (best_tiles > tiles) best_tiles = tiles;
    pl.cchunk = static_cast<int32_t>(best_tiles * 128);
    pl.prefix_wave = static_cast<int32_t>(sms);
    pl.max_csplits = static_cast<int32_t>((max_group_prefix_len + pl.cchunk - 1) / pl.cchunk);
  }
  return pl;
}

DecodeWorkspace layout_decode_workspace(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, const DecodePlan& pl, int32_t cascade_levels) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  DecodeWorkspace w;
  const size_t bh = static_cast<size_t>(batch) * num_q_heads;
  size_t off = 0;
  const size_t ih = static_cast<size_t>(pl.max_items) * num_q_heads;
  w.part_o = off;
  off += up(ih * head_dim * sizeof(float));
  w.part_lse = off;
  off += up(ih * sizeof(float));
  if (cascade_levels > 0) {
    const size_t slots = static_cast<size_t>(cascade_levels) * pl.max_csplits;
    w.casc_o = off;
    off += up(bh * slots * head_dim * sizeof(float));
    w.casc_lse = off;
    off += up(bh * slots * sizeof(float));
  }
  w.ints = off;
  (void)num_kv_heads;
  w.zero_bytes = (static_cast<size_t>(batch) + 3) * sizeof(int32_t);
  w.ints_bytes = w.zero_bytes + (2 + static_cast<size_t>(batch) + 1 + 2 * static_cast<size_t>(pl.max_items) +
                                 static_cast<size_t>(batch)) * sizeof(int32_t);
  off += up(w.ints_bytes);
  w.total = off;
  return w;
}

}  // namespace ra

extern "C" size_t ra_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t max_seq_len, int32_t num_groups,
                                            int32_t max_group_prefix_len, int32_t max_group_size,
                                            int32_t max_group_levels) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (num_groups > 0 && (max_group_prefix_len <= 0 || max_group_size <= 0 || max_group_levels <= 0)) return 0;
  const ra::DecodePlan pl = ra::plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_groups,
                                            max_group_prefix_len, max_group_size);
  return ra::layout_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, pl,
                                     num_groups > 0 ? max_group_levels : 0)
      .total;
}

// ra_decode_attention, and with k_new / v_new / out_cache_loc non-null ra_decode_attention_store.
static ra_status decode_call(const void* k_pool, const void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                             int32_t head_dim, const void* k_new, const void* v_new, const int32_t* out_cache_loc,
                             const void* q, void* o, int32_t num_q_heads, float sm_scale,
                             const int32_t* req_to_token, int64_t table_stride, int64_t table_rows,
                             const int32_t* req_pool_indices, const int32_t* seq_lens, int32_t batch,
                             int32_t max_seq_len, int32_t num_groups, const int32_t* group_indptr,
                             const int32_t* group_reqs, const int32_t* group_prefix_start,
                             const int32_t* group_prefix_len, const int32_t* group_level,
                             int32_t max_group_prefix_len, int32_t max_group_size, int32_t max_group_levels,
                             void* workspace, size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream) {
  using namespace ra;
  const bool fused = k_new != nullptr || v_new != nullptr || out_cache_loc != nullptr;
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
  if (fused) {
    RA_REQUIRE(k_new && v_new && out_cache_loc, "k_new, v_new and out_cache_loc must all be non-null");
    RA_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned4(out_cache_loc),
               "k_new and v_new must be 16-byte aligned, out_cache_loc 4-byte aligned");
  }
  if (num_groups > 0) {
    RA_REQUIRE(group_indptr && group_reqs && group_prefix_len, "cascade arrays must be non-null");
    RA_REQUIRE(max_group_prefix_len >= 1 && max_group_prefix_len <= max_seq_len,
               "max_group_prefix_len must be in [1, max_seq_len]");
    RA_REQUIRE(max_group_size >= 1 && max_group_size <= batch, "max_group_size must be in [1, batch]");
    RA_REQUIRE(max_group_levels >= 1 && max_group_levels <= 64, "max_group_levels must be in [1, 64]");
    RA_REQUIRE(group_level || max_group_levels == 1, "max_group_levels > 1 needs group_level");
    RA_REQUIRE(aligned4(group_indptr) && aligned4(group_reqs) && aligned4(group_prefix_len) &&
                   (!group_prefix_start || aligned4(group_prefix_start)) && (!group_level || aligned4(group_level)),
               "group arrays must be 4-byte aligned");
  }
  // the device plan's item length must fit in 31 bits (it is at most batch x max_seq_len / kDecodePlanItems)
  RA_REQUIRE(static_cast<int64_t>(batch) * max_seq_len <= static_cast<int64_t>(kDecodePlanItems) << 30,
             "batch x max_seq_len too large");
  const DecodePlan pl = plan_decode(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, num_groups,
                                    max_group_prefix_len, max_group_size);
  const int32_t levels = num_groups > 0 ? max_group_levels : 0;
  const DecodeWorkspace wl = layout_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, pl, levels);
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
  p.max_items = pl.max_items;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws + wl.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + wl.part_lse);
  p.err = device_error;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // fused store: extra CTAs of the call's first kernel scatter the new rows (a few waves of 4 vectors
  // per thread, at most one CTA per SM)
  int store_ctas = 0;
  if (fused) {
    DeviceInfo d0;
    if (ra_status st = current_device(&d0)) return st;
    p.st_k = static_cast<const uint4*>(k_new);
    p.st_v = static_cast<const uint4*>(v_new);
    p.st_loc = out_cache_loc;
    p.st_row_vecs = num_kv_heads * head_dim * 2 / 16;
    p.st_total = static_cast<int64_t>(batch) * p.st_row_vecs;
    const int64_t per_cta = (num_groups > 0 ? 256 : kPlanThreads) * 4;
    const int64_t want = (p.st_total + per_cta - 1) / per_cta;
    store_ctas = static_cast<int>(want < d0.num_sms ? want : d0.num_sms);
    if (store_ctas < 1) store_ctas = 1;
  }

  int32_t* ints = reinterpret_cast<int32_t*>(ws + wl.ints);
  p.counter = ints + batch;
  p.prefix_counter = ints + batch + 1;
  p.prefix_done = ints + batch + 2;
  p.plan = ints + batch + 3;
  p.req_item0 = p.plan + 2;
  p.item_req = p.req_item0 + batch + 1;
  p.order = p.item_req + pl.max_items;
  p.req_done = p.order + pl.max_items;
  // Kernels rather than memsets, so that the launches of the call stay chained programmatically:
  // with groups, [set-up: counters, key starts, empty prefix partials] -> [prefix pass] -> [plan] ->
  // [decode] -> [combine]; without, [plan] -> [decode] -> [combine].
  if (num_groups > 0) {
    p.cchunk = pl.cchunk;
    p.max_csplits = pl.max_csplits;
    p.prefix_wave = pl.prefix_wave;
    p.casc_slots = levels * pl.max_csplits;
    p.casc_one_level = (max_group_levels == 1 && group_prefix_start == nullptr) ? 1 : 0;
    p.casc_o = reinterpret_cast<float*>(ws + wl.casc_o);
    p.casc_lse = reinterpret_cast<float*>(ws + wl.casc_lse);
    p.key_start = ints;
    const int64_t n_lse = static_cast<int64_t>(batch) * num_q_heads * p.casc_slots;
    const int64_t lse_want = (n_lse + 256 * 8 - 1) / (256 * 8);  // ~8 values per thread
    const int32_t lse_ctas = static_cast<int32_t>(lse_want < 128 ? (lse_want > 0 ? lse_want : 1) : 128);
    if (ra_status st = launch_pdl("cascade_setup_kernel", cascade_setup_kernel, dim3(1 + lse_ctas + store_ctas),
                                  dim3(256), 0, s, p, ints, static_cast<int32_t>(wl.zero_bytes / sizeof(int32_t)),
                                  group_indptr, group_reqs, group_prefix_len, num_groups, n_lse, lse_ctas))
      return st;
    CascadeArgs ca{group_indptr,         group_reqs,           group_prefix_start, group_prefix_len, group_level,
                   num_groups,           max_group_prefix_len, max_group_size,     max_group_levels};
    if (ra_status st = launch_cascade_prefix(p, ca, head_dim, s, &p.prefix_ctas)) return st;
  }
  // (with groups the set-up kernel did the fused store: the plan kernel runs behind the prefix pass)
  if (ra_status st = launch_pdl("decode_plan_kernel", decode_plan_kernel, dim3(1 + (num_groups > 0 ? 0 : store_ctas)),
                                dim3(kPlanThreads), 0, s, p))
    return st;
  // persistent decode geometry
  p.hpc = heads_per_cta(num_kv_heads);
  p.n_hgroups = num_kv_heads / p.hpc;
  p.row_stride = p.hpc * head_dim * 2 + 16;
  p.stage_bytes = 2 * 16 * p.row_stride;
  p.nstage = (kSmemLimit - kHdrBytes) / p.stage_bytes;
  if (p.nstage > kMaxStages) p.nstage = kMaxStages;
  if (p.nstage < 2) return fail(RA_ERR_UNSUPPORTED, "decode ring does not fit in shared memory");
  const int smem = kHdrBytes + p.nstage * p.stage_bytes;
  const int64_t n_items = static_cast<int64_t>(pl.max_items) * p.n_hgroups;  // bound of the claims
  DeviceInfo dev;
  if (ra_status st = current_device(&dev)) return st;
  const int grid = static_cast<int>(n_items < dev.num_sms ? n_items : dev.num_sms);
  return head_dim == 128 ? launch_decode<128>(p, grid, smem, s) : launch_decode<64>(p, grid, smem, s);
}

extern "C" ra_status ra_decode_attention(const void* k_pool, const void* v_pool, int64_t num_slots,
                                         int32_t num_kv_heads, int32_t head_dim, const void* q, void* o,
                                         int32_t num_q_heads, float sm_scale, const int32_t* req_to_token,
                                         int64_t table_stride, int64_t table_rows, const int32_t* req_pool_indices,
                                         const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                         int32_t num_groups, const int32_t* group_indptr,
                                         const int32_t* group_reqs, const int32_t* group_prefix_start,
                                         const int32_t* group_prefix_len, const int32_t* group_level,
                                         int32_t max_group_prefix_len, int32_t max_group_size,
                                         int32_t max_group_levels, void* workspace, size_t workspace_bytes,
                                         uint32_t* device_error, ra_stream_t stream) {
  ra::clear_error();
  return decode_call(k_pool, v_pool, num_slots, num_kv_heads, head_dim, nullptr, nullptr, nullptr, q, o,
                     num_q_heads, sm_scale, req_to_token, table_stride, table_rows, req_pool_indices, seq_lens, batch,
                     max_seq_len, num_groups, group_indptr, group_reqs, group_prefix_start, group_prefix_len,
                     group_level, max_group_prefix_len, max_group_size, max_group_levels, workspace, workspace_bytes,
                     device_error, stream);
}

extern "C" ra_status ra_decode_attention_store(void* k_pool, void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                                               int32_t head_dim, const void* k_new, const void* v_new,
                                               const int32_t* out_cache_loc, const void* q, void* o,
                                               int32_t num_q_heads, float sm_scale, const int32_t* req_to_token,
                                               int64_t table_stride, int64_t table_rows,
                                               const int32_t* req_pool_indices, const int32_t* seq_lens,
                                               int32_t batch, int32_t max_seq_len, int32_t num_groups,
                                               const int32_t* group_indptr, const int32_t* group_reqs,
                                               const int32_t* group_prefix_start, const int32_t* group_prefix_len,
                                               const int32_t* group_level, int32_t max_group_prefix_len,
                                               int32_t max_group_size, int32_t max_group_levels, void* workspace,
                                               size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream) {
  ra::clear_error();
  if (!k_new || !v_new || !out_cache_loc)
    return ra::fail(RA_ERR_INVALID_ARGUMENT, "k_new, v_new and out_cache_loc must all be non-null");
  return decode_call(k_pool, v_pool, num_slots, num_kv_heads, head_dim, k_new, v_new, out_cache_loc, q, o,
                     num_q_heads, sm_scale, req_to_token, table_stride, table_rows, req_pool_indices, seq_lens, batch,
                     max_seq_len, num_groups, group_indptr, group_reqs, group_prefix_start, group_prefix_len,
                     group_level, max_group_prefix_len, max_group_size, max_group_levels, workspace, workspace_bytes,
                     device_error, stream);
}
