// decode_internal.h -- parameter blocks shared by the decode kernels and the
// tensor-core prefix pass of the cascade (grouped) decode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cmath>

#include "../../include/ra.h"

namespace ra {

struct DecodeParams {
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int64_t num_slots;
  int32_t hkv;
  const __nv_bfloat16* q;  // [batch, hq, D]
  __nv_bfloat16* o;        // [batch, hq, D]
  int32_t hq;
  int32_t group;     // hq / hkv
  float scale_log2;  // sm_scale * log2(e)
  const int32_t* table;
  int64_t table_stride;
  int64_t table_rows;
  const int32_t* rpi;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_seq_len;
  const int32_t* key_start;  // [batch] first private position (cascade), or nullptr
  int32_t hpc;               // kv heads per CTA item (consumer warps)
  int32_t n_hgroups;         // hkv / hpc
  int32_t nstage;            // ring stages
  int32_t row_stride;        // bytes between keys in a ring stage (hpc * D * 2 + 16)
  int32_t stage_bytes;       // 2 * 16 * row_stride
  int32_t max_items;         // kDecodePlanItems + batch: bound of the plan's items
  int32_t* counter;          // work-item counter (reset by the plan kernel)
  int32_t* prefix_counter;   // cascade prefix pass's work-item counter (zeroed with the key starts)
  int32_t* prefix_done;      // cascade prefix pass: CTAs that have written all their partials (zeroed likewise)
  int32_t prefix_ctas;       // cascade prefix pass: CTAs launched
  int32_t prefix_wave;       // cascade prefix pass: the wave size its splits were planned for
  int32_t* req_done;         // [batch]: (item, head group) partials written per request (reset by the plan kernel)
  int32_t* plan;             // [2]: items, keys per item (chunk), written by the plan kernel
  int32_t* req_item0;        // [batch + 1]: request b's items are req_item0[b] .. req_item0[b+1]-1
  int32_t* item_req;         // [max_items]: request of each item
  int32_t* order;            // [max_items]: items in claim order (longest first)
  float* part_o;    // [max_items, hq, D] per item and q head
  float* part_lse;  // [max_items, hq] (log2 domain)
  int32_t cchunk;      // shared-prefix keys per prefix-pass split (cascade)
  int32_t max_csplits;  // prefix-pass splits per group range
  int32_t casc_slots;   // prefix partials per (request, q head): levels x max_csplits
  int32_t casc_one_level;  // every group starts at position 0 at level 0: a member's written prefix partials
                           // are exactly slots 0 .. ceil(key_start / cchunk) - 1
  float* casc_o;        // [casc_slots, batch, hq, D] shared-prefix partials (cascade)
  float* casc_lse;      // [casc_slots, batch, hq]; -inf marks a slot no group wrote
  uint32_t* err;
  // fused store (ra_decode_attention_store): the step's new rows, scattered by the call's first kernel
  const uint4* st_k;       // [batch, hkv, D] bf16 as 16-byte vectors, or nullptr (no store)
  const uint4* st_v;
  const int32_t* st_loc;   // [batch] destination slots
  int32_t st_row_vecs;     // 16-byte vectors per slot row (hkv * D * 2 / 16)
  int64_t st_total;        // batch * st_row_vecs
};

// The private keys of a decode call are cut into items on the device (decode_plan_kernel): at most
// kDecodePlanItems items of equal length (>= kDecodeMinChunk keys) plus one shorter item per request.
// Three full-length items per SM of GB300 (152 SMs): measured against 320 and 640, the best or tied on
// the decode workloads (forked 70B 185 / 244 / 210 us, multi-turn mix 266 / 265 / 278 us).  A constant,
// not the device's SM count: the workspace size must not depend on the device that runs the call.
constexpr int32_t kDecodePlanItems = 456;
constexpr int32_t kDecodeMinChunk = 128;

struct DecodePlan {
  int32_t max_items = 0;    // kDecodePlanItems + batch
  int32_t cchunk = 0;       // shared-prefix keys per prefix-pass split (cascade)
  int32_t max_csplits = 0;
  int32_t prefix_wave = 0;  // prefix-pass CTAs (of GB300's 152 SMs) the cost model planned the splits for
};

struct DecodeWorkspace {
  size_t part_o = 0, part_lse = 0, casc_o = 0, casc_lse = 0;
  size_t ints = 0, ints_bytes = 0;  // key_start [batch], counter, prefix counter, prefix done (zeroed with
                                    // groups); plan [2], req_item0 [batch+1], item_req, order [max_items],
                                    // req_done [batch]
  size_t zero_bytes = 0;            // leading part of the block cleared before the key-start scatter
  size_t total = 0;
};

constexpr int kMaxHeadsPerCta = 8;  // consumer warps of the decode kernel

struct CascadeArgs {
  const int32_t* group_indptr;
  const int32_t* group_reqs;
  const int32_t* group_prefix_start;  // nullable: 0
  const int32_t* group_prefix_len;    // end position of the group's range
  const int32_t* group_level;         // nullable: 0
  int32_t num_groups;
  int32_t max_group_prefix_len;
  int32_t max_group_size;
  int32_t max_group_levels;
};

DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len,
                       int32_t num_groups, int32_t max_group_prefix_len, int32_t max_group_size);
DecodeWorkspace layout_decode_workspace(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, const DecodePlan& pl, int32_t cascade_levels);

// Tensor-core pass over each group's shared prefix: writes p.casc_o / p.casc_lse
// for every member (defined with the tcgen05 attention kernel).
// Returns the pass's grid size in *ctas (each of its CTAs adds one to p.prefix_done when it is done).
ra_status launch_cascade_prefix(const DecodeParams& p, const CascadeArgs& ca, int32_t head_dim,
                                cudaStream_t stream, int32_t* ctas);

}  // namespace ra
