"""Pins for the CPU oracle (no GPU): brute force, closed forms, invariants.

Each test is chosen so that a plausible mistake in the oracle (a dropped key,
an off-by-one causal bound, a wrong kv-head index, a transposed operand, a
missing max-subtraction or normalisation) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("seed,hq,hkv,d", [(0, 4, 2, 8), (1, 6, 3, 4), (2, 8, 2, 16), (3, 2, 2, 8), (4, 8, 1, 8)])
def test_oracle_matches_brute_force(seed, hq, hkv, d):
    b = W.random_mixed(seed, n_extend=3, n_decode=4, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, max_len=24)
    o_e = oracle.extend_batch(b)
    o_d = oracle.decode_batch(b)
    np.testing.assert_allclose(o_e, np.array(brute.extend(b)).reshape(o_e.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_d, np.array(brute.decode(b)).reshape(o_d.shape), rtol=0, atol=1e-12)


def test_oracle_matches_brute_force_tiny_config():
    e, d = W.tiny_extend_decode()
    np.testing.assert_allclose(oracle.extend_batch(e), np.array(brute.extend(e)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.decode_batch(d), np.array(brute.decode(d)), rtol=0, atol=1e-12)


def _golden_rows():
    rows = []
    for line in open(os.path.join(GOLDEN, "two_key_softmax.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(float(x) for x in line.split()))
    return rows


@pytest.mark.parametrize("scale,o0,o1", _golden_rows())
def test_two_key_closed_form(scale, o0, o1):
    # one request: cached prefix = 1 key, suffix = 1 token (itself)
    pool = oracle.CompactPool(4, np.array([1, 2]), _bits([[[1, 0]], [[0, 0]]]), _bits([[[1, 0]], [[0, 1]]]))
    table = np.array([[1, 2]], np.int32)
    out = oracle.extend(pool, _bits([[[1, 0]]]), table, np.array([0]), np.array([1]), np.array([1]),
                        np.array([0, 1]), scale)
    np.testing.assert_allclose(out[0], [o0, o1], rtol=0, atol=1e-15)
    # the same row as a decode step (L = 2)
    out_d = oracle.decode(pool, _bits([[[1, 0]]]), table, np.array([0]), np.array([2]), scale)
    np.testing.assert_allclose(out_d[0], [o0, o1], rtol=0, atol=1e-15)


def test_single_key_returns_its_value():
    b = W.random_mixed(11, n_extend=2, n_decode=2, num_q_heads=4, num_kv_heads=2, head_dim=16, max_len=1,
                       min_len=1, share_prob=0.0)
    pool = oracle.pool_after_store(b)
    for which, out, rows in (("e", oracle.extend_batch(b), None), ("d", oracle.decode_batch(b), None)):
        hq = b.num_q_heads
        for r in range(out.shape[0]):
            t, h = divmod(r, hq)
            rpi = b.ext_rpi[t] if which == "e" else b.dec_rpi[t]
            slot = b.req_to_token[rpi, 0]
            v = W.bf16_bits_to_f32(pool.v[pool.slot_row[slot], h // 2]).astype(np.float64)
            np.testing.assert_array_equal(out[r], v)


def test_constant_v_returns_v_and_zero_q_returns_mean():
    b = W.random_mixed(12, n_extend=3, n_decode=3, num_q_heads=4, num_kv_heads=2, head_dim=8, max_len=30)
    # constant V per kv head
    cval = _bits(np.arange(16, dtype=np.float32).reshape(2, 8) / 4 - 1)
    b.pool_v[:] = cval
    b.v_new[:] = cval
    ref = W.bf16_bits_to_f32(cval).astype(np.float64)
    oe, od = oracle.extend_batch(b), oracle.decode_batch(b)
    for out in (oe, od):
        for r in range(out.shape[0]):
            np.testing.assert_allclose(out[r], ref[(r % 4) // 2], rtol=0, atol=1e-13)
    # q = 0 -> uniform weights -> mean of the visible V rows
    b = W.random_mixed(13, n_extend=3, n_decode=3, num_q_heads=4, num_kv_heads=2, head_dim=8, max_len=30)
    b.ext_q[:] = 0
    b.dec_q[:] = 0
    pool = oracle.pool_after_store(b)
    od = oracle.decode_batch(b)
    for bi in range(b.n_decode):
        ctx = b.req_to_token[b.dec_rpi[bi], :b.dec_seq_lens[bi]]
        for h in range(4):
            vs = W.bf16_bits_to_f32(pool.v[pool.slot_row[ctx], h // 2]).astype(np.float64)
            np.testing.assert_allclose(od[bi * 4 + h], vs.mean(axis=0), rtol=0, atol=1e-13)
    oe = oracle.extend_batch(b)
    for bi in range(b.n_extend):
        for i in range(b.ext_extend_lens[bi]):
            t = b.ext_qo_indptr[bi] + i
            ctx = b.req_to_token[b.ext_rpi[bi], :b.ext_prefix_lens[bi] + i + 1]
            vs = W.bf16_bits_to_f32(pool.v[pool.slot_row[ctx], 1]).astype(np.float64)
            np.testing.assert_allclose(oe[t * 4 + 3], vs.mean(axis=0), rtol=0, atol=1e-13)


def test_weights_sum_to_one_via_linearity():
    """out(V + c) - out(V) = c * sum_j w_j: shifting every V row by the same amount
    shifts the output by exactly that amount iff the weights sum to one."""
    b = W.random_mixed(14, n_extend=2, n_decode=3, num_q_heads=4, num_kv_heads=1, head_dim=8, max_len=40)
    # V values that are multiples of 1/4 in [-4, 4): v + 8 is exact in bf16
    rng = np.random.default_rng(3)
    b.pool_v[:] = _bits(rng.integers(-16, 16, size=b.pool_v.shape) / 4.0)
    b.v_new[:] = _bits(rng.integers(-16, 16, size=b.v_new.shape) / 4.0)
    o1d, o1e = oracle.decode_batch(b), oracle.extend_batch(b)
    b.pool_v[:] = _bits(W.bf16_bits_to_f32(b.pool_v) + 8.0)
    b.v_new[:] = _bits(W.bf16_bits_to_f32(b.v_new) + 8.0)
    o2d, o2e = oracle.decode_batch(b), oracle.extend_batch(b)
    np.testing.assert_allclose(o2d - o1d, 8.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2e - o1e, 8.0, rtol=0, atol=1e-12)


def test_prefix_reuse_equals_full_attention_on_fresh_pool():
    """Attention of a suffix over a reused cached prefix = the last rows of full causal
    attention over the concatenated sequence, computed with no cache in other slots."""
    b = W.random_mixed(21, n_extend=4, n_decode=0, num_q_heads=4, num_kv_heads=2, head_dim=16, max_len=48,
                       share_prob=0.9)
    out = oracle.extend_batch(b)
    pool = oracle.pool_after_store(b)
    rng = np.random.default_rng(5)
    S2 = 4096
    for bi in range(b.n_extend):
        P, E = int(b.ext_prefix_lens[bi]), int(b.ext_extend_lens[bi])
        L = P + E
        ctx = b.req_to_token[b.ext_rpi[bi], :L]
        # a fresh pool: the whole sequence re-prefilled into new slots
        new_slots = rng.permutation(np.arange(1, S2))[:L]
        fresh = oracle.CompactPool(S2, new_slots, pool.k[pool.slot_row[ctx]], pool.v[pool.slot_row[ctx]])
        q_full = np.zeros((L, 4, 16), np.uint16)
        q_full[P:] = b.ext_q[b.ext_qo_indptr[bi]:b.ext_qo_indptr[bi + 1]]
        q_full[:P] = b.ext_q[0]  # arbitrary queries for the prefix rows (not compared)
        full = oracle.extend(fresh, q_full, new_slots[None, :].astype(np.int32), np.array([0]), np.array([0]),
                             np.array([L]), np.array([0, L]), b.sm_scale)
        mine = out[b.ext_qo_indptr[bi] * 4:b.ext_qo_indptr[bi + 1] * 4]
        np.testing.assert_allclose(mine, full[P * 4:], rtol=0, atol=1e-13)


def test_chunked_prefill_equals_one_extend():
    """Prefilling a suffix in chunks, each chunk attending to the cached prefix plus the earlier
    chunks, gives the rows of one extend over the whole suffix (the KV of a position depends only
    on the tokens before it, SGLang paper summary §3)."""
    from helpers import prefill_chunks
    b = W.random_mixed(23, n_extend=5, n_decode=0, num_q_heads=8, num_kv_heads=2, head_dim=16, max_len=90,
                       share_prob=0.7)
    full = oracle.extend_batch(b).reshape(-1, b.num_q_heads, b.head_dim)
    pool = oracle.pool_after_store(b)
    seen = np.zeros(b.total_q_extend, bool)
    for q, plen, elen, qo, toks in prefill_chunks(b, 13):
        part = oracle.extend(pool, q, b.req_to_token, b.ext_rpi, plen, elen, qo, b.sm_scale)
        np.testing.assert_allclose(part.reshape(-1, b.num_q_heads, b.head_dim), full[toks], rtol=0, atol=1e-13)
        seen[toks] = True
    assert seen.all()


def test_slot_permutation_invariance():
    b = W.random_mixed(31, n_extend=3, n_decode=5, num_q_heads=8, num_kv_heads=2, head_dim=8, max_len=40)
    oe, od = oracle.extend_batch(b), oracle.decode_batch(b)
    perm = np.random.default_rng(9).permutation(b.num_slots)
    b.pool_slots = perm[b.pool_slots]
    b.out_cache_loc = perm[b.out_cache_loc].astype(np.int32)
    t = b.req_to_token
    b.req_to_token = np.where(t >= 0, perm[np.maximum(t, 0)], t).astype(np.int32)
    np.testing.assert_array_equal(oracle.extend_batch(b), oe)
    np.testing.assert_array_equal(oracle.decode_batch(b), od)


def test_decode_equals_extend_row_at_same_position():
    b = W.random_mixed(41, n_extend=3, n_decode=0, num_q_heads=4, num_kv_heads=2, head_dim=16, max_len=30)
    oe = oracle.extend_batch(b)
    pool = oracle.pool_after_store(b)
    for bi in range(b.n_extend):
        for i in range(int(b.ext_extend_lens[bi])):
            t = int(b.ext_qo_indptr[bi]) + i
            L = int(b.ext_prefix_lens[bi]) + i + 1
            od = oracle.decode(pool, b.ext_q[t:t + 1], b.req_to_token, b.ext_rpi[bi:bi + 1], np.array([L]),
                               b.sm_scale)
            np.testing.assert_array_equal(od, oe[t * 4:(t + 1) * 4])


def test_causal_bound_includes_self_and_excludes_future():
    """Changing the K/V of the token right after row i leaves row i unchanged; changing
    its own K/V changes it."""
    b = W.random_mixed(51, n_extend=1, n_decode=0, num_q_heads=2, num_kv_heads=1, head_dim=8, max_len=12,
                       min_len=8, ext_lens=[6])
    base = oracle.extend_batch(b)
    P = int(b.ext_prefix_lens[0])
    i = 2
    slot_next = b.req_to_token[b.ext_rpi[0], P + i + 1]
    slot_self = b.req_to_token[b.ext_rpi[0], P + i]
    for slot, same in ((slot_next, True), (slot_self, False)):
        c = W.random_mixed(51, n_extend=1, n_decode=0, num_q_heads=2, num_kv_heads=1, head_dim=8, max_len=12,
                           min_len=8, ext_lens=[6])
        k = list(c.out_cache_loc).index(slot)
        c.k_new[k] = _bits(np.full((1, 8), 3.0))
        c.v_new[k] = _bits(np.full((1, 8), -5.0))
        o = oracle.extend_batch(c)
        row = slice(i * 2, i * 2 + 2)
        if same:
            np.testing.assert_array_equal(o[row], base[row])
        else:
            assert np.abs(o[row] - base[row]).max() > 1e-3


def test_gqa_head_mapping_is_consecutive():
    """q head h reads kv head h // G: zero every kv head but one and check which q heads see it."""
    b = W.random_mixed(61, n_extend=0, n_decode=2, num_q_heads=6, num_kv_heads=3, head_dim=8, max_len=10)
    b.pool_v[:, [0, 2]] = 0
    b.v_new[:, [0, 2]] = 0
    od = oracle.decode_batch(b).reshape(2, 6, 8)
    assert np.all(od[:, [0, 1, 4, 5]] == 0)
    assert np.all(np.abs(od[:, [2, 3]]).max(axis=-1) > 0)


def test_kv_store_definition():
    rng = np.random.default_rng(0)
    pk = rng.integers(0, 65535, size=(16, 2, 8), dtype=np.uint16)
    pv = rng.integers(0, 65535, size=(16, 2, 8), dtype=np.uint16)
    kn = rng.integers(0, 65535, size=(3, 2, 8), dtype=np.uint16)
    vn = rng.integers(0, 65535, size=(3, 2, 8), dtype=np.uint16)
    loc = np.array([5, 0, 15], np.int32)
    k2, v2 = oracle.kv_store(pk, pv, kn, vn, loc)
    mask = np.ones(16, bool)
    mask[loc] = False
    np.testing.assert_array_equal(k2[mask], pk[mask])
    np.testing.assert_array_equal(v2[mask], pv[mask])
    np.testing.assert_array_equal(k2[loc], kn)
    np.testing.assert_array_equal(v2[loc], vn)
    with pytest.raises(ValueError):
        oracle.kv_store(pk, pv, kn, vn, np.array([1, 16, 2], np.int32))


def test_oracle_rejects_unused_slot():
    b = W.random_mixed(71, n_extend=0, n_decode=2, num_q_heads=2, num_kv_heads=1, head_dim=8, max_len=10)
    b.req_to_token[b.dec_rpi[0], 0] = 0   # slot 0 is never in use
    with pytest.raises(ValueError):
        oracle.decode_batch(b)
