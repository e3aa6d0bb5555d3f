/*
 * CPU oracle for the RadixAttention hot path -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct fp64 restatement of what the GPU path must
 * compute.  Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
 * leg may load it; the product library never does, and this file shares no
 * code, header or constant with it.
 *
 * What it follows:
 *  - KV store: a token's K/V row is written into the pool slot the allocator
 *    gave it (anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍",
 *    来源一: each step's new tokens go to `out_cache_loc`).  The oracle is the
 *    definition: pool' = pool with row loc[i] replaced by new[i].
 *  - Attention over a shared prefix: KV depends only on the prefix tokens, so
 *    a request reuses the cached prefix KV and only computes its suffix (SGLang
 *    paper summary, §3 "Efficient KV Cache Reuse with RadixAttention"; the
 *    yaopepe.com explainer, §04: the prefix KV is referenced, the unmatched
 *    suffix is prefilled).  The result is plain softmax attention of each new
 *    query over every key of its context up to and including its own
 *    position, with the context's slots read from req_to_token (the per-request
 *    slot rows of the v0.2 runtime, `req_pool_indices`, same handbook page).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - GQA: q head h reads kv head h / (Hq / Hkv).
 *  - scores are sm_scale * <q, k>, softmax over the visible keys, output
 *    sum_j w_j v_j; computed here in double from exactly decoded bf16 inputs.
 *  - an extend row i of request b sits at position P_b + i and sees keys
 *    0 .. P_b + i (itself included); a decode row sees keys 0 .. L_b - 1.
 *  - all keys, prefix and suffix, are read from the pool through the table
 *    (the caller stores the suffix and fills the table first).
 *
 * Pool addressing: the pools hold only the rows in use, [U, Hkv, D]; slot_row
 * maps a slot id to its row (-1 = not in use).  This is bookkeeping for large
 * pools, not part of the arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* pool' = pool with the row of slot loc[i] replaced by new[i] (K and V). */
int ora_kv_store(uint16_t* pool_k, uint16_t* pool_v, int64_t num_slots, int64_t row_elems,
                 const uint16_t* k_new, const uint16_t* v_new, const int32_t* loc, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    if (loc[i] < 0 || loc[i] >= num_slots) return -1;
  }
  for (int64_t i = 0; i < n; ++i) {
    memcpy(pool_k + (int64_t)loc[i] * row_elems, k_new + i * row_elems, (size_t)row_elems * 2);
    memcpy(pool_v + (int64_t)loc[i] * row_elems, v_new + i * row_elems, (size_t)row_elems * 2);
  }
  return 0;
}

/*
 * One query row against n_keys keys whose slots are key_slots[0..n_keys).
 *   s_j = scale * sum_d q[d] k_j[d];  w_j = exp(s_j - max s) / sum exp(s - max s);
 *   out[d] = sum_j w_j v_j[d].
 * Returns 0, or -1 if a slot is out of range or not in use.
 */
static int attend_row(const uint16_t* q, const uint16_t* pool_k, const uint16_t* pool_v,
                      const int64_t* slot_row, int64_t num_slots, int32_t hkv, int32_t d, int32_t kv_head,
                      const int32_t* key_slots, int64_t n_keys, double scale, double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  double* qd = (double*)malloc(sizeof(double) * (size_t)d);
  if (!s || !qd) { free(s); free(qd); return -2; }
  for (int32_t e = 0; e < d; ++e) qd[e] = bf16_to_double(q[e]);
  for (int32_t e = 0; e < d; ++e) out[e] = 0.0;
  double m = -INFINITY;
  for (int64_t j = 0; j < n_keys; ++j) {
    int32_t slot = key_slots[j];
    if (slot < 0 || slot >= num_slots || slot_row[slot] < 0) { free(s); free(qd); return -1; }
    const uint16_t* k = pool_k + (slot_row[slot] * hkv + kv_head) * (int64_t)d;
    double dot = 0.0;
    for (int32_t e = 0; e < d; ++e) dot += qd[e] * bf16_to_double(k[e]);
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    s[j] = exp(s[j] - m);
    z += s[j];
  }
  for (int64_t j = 0; j < n_keys; ++j) {
    const uint16_t* v = pool_v + (slot_row[key_slots[j]] * hkv + kv_head) * (int64_t)d;
    double w = s[j] / z;
    for (int32_t e = 0; e < d; ++e) out[e] += w * bf16_to_double(v[e]);
  }
  free(s);
  free(qd);
  return 0;
}

/*
 * Extend attention.  q: [total_q, hq, d] (rows of request b are
 * qo_indptr[b] .. qo_indptr[b+1]); row i of request b is at position
 * prefix_lens[b] + i and sees keys at positions 0 .. prefix_lens[b] + i,
 * slot = req_to_token[rpi[b] * stride + position].
 * sel: flat indices t * hq + h to evaluate (NULL: all, in that order).
 * out: [n_sel (or total_q * hq), d] doubles.
 */
int ora_extend(const uint16_t* pool_k, const uint16_t* pool_v, const int64_t* slot_row, int64_t num_slots,
               int32_t hkv, int32_t d, const uint16_t* q, int32_t hq,
               const int32_t* req_to_token, int64_t stride, int64_t table_rows,
               const int32_t* rpi, const int32_t* prefix_lens, const int32_t* extend_lens,
               const int32_t* qo_indptr, int32_t batch, double scale,
               const int64_t* sel, int64_t n_sel, double* out) {
  if (hkv <= 0 || hq % hkv != 0) return -3;
  const int32_t group = hq / hkv;
  const int64_t total_q = batch > 0 ? qo_indptr[batch] : 0;
  const int64_t n = sel ? n_sel : total_q * hq;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(min : err)
  for (int64_t r = 0; r < n; ++r) {
    int64_t flat = sel ? sel[r] : r;
    int64_t t = flat / hq;
    int32_t h = (int32_t)(flat % hq);
    int32_t b = 0;
    while (b + 1 <= batch && qo_indptr[b + 1] <= t) ++b; /* request owning token t */
    if (b >= batch || rpi[b] < 0 || rpi[b] >= table_rows) { err = -1; continue; }
    int64_t i = t - qo_indptr[b];
    if (i >= extend_lens[b]) { err = -1; continue; }
    int64_t n_keys = (int64_t)prefix_lens[b] + i + 1;
    int rc = attend_row(q + flat * d, pool_k, pool_v, slot_row, num_slots, hkv, d, h / group,
                        req_to_token + (int64_t)rpi[b] * stride, n_keys, scale, out + r * d);
    if (rc != 0) err = rc;
  }
  return err;
}

/*
 * Decode attention.  q: [batch, hq, d]; request b's single query sits at
 * position seq_lens[b] - 1 and sees keys at positions 0 .. seq_lens[b] - 1.
 * sel: flat indices b * hq + h (NULL: all).  out: [n, d] doubles.
 */
int ora_decode(const uint16_t* pool_k, const uint16_t* pool_v, const int64_t* slot_row, int64_t num_slots,
               int32_t hkv, int32_t d, const uint16_t* q, int32_t hq,
               const int32_t* req_to_token, int64_t stride, int64_t table_rows,
               const int32_t* rpi, const int32_t* seq_lens, int32_t batch, double scale,
               const int64_t* sel, int64_t n_sel, double* out) {
  if (hkv <= 0 || hq % hkv != 0) return -3;
  const int32_t group = hq / hkv;
  const int64_t n = sel ? n_sel : (int64_t)batch * hq;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(min : err)
  for (int64_t r = 0; r < n; ++r) {
    int64_t flat = sel ? sel[r] : r;
    int32_t b = (int32_t)(flat / hq);
    int32_t h = (int32_t)(flat % hq);
    if (b >= batch || rpi[b] < 0 || rpi[b] >= table_rows || seq_lens[b] < 1) { err = -1; continue; }
    int rc = attend_row(q + flat * d, pool_k, pool_v, slot_row, num_slots, hkv, d, h / group,
                        req_to_token + (int64_t)rpi[b] * stride, seq_lens[b], scale, out + r * d);
    if (rc != 0) err = rc;
  }
  return err;
}

/* Threads the oracle's parallel loops use (1 without OpenMP). */
int ora_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
