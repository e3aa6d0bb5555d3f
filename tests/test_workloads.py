"""Invariants of the seeded inputs (no GPU): slots, sharing, table layout, sizes."""
import numpy as np
import pytest

import workloads as W


def _check_batch(b):
    S = b.num_slots
    all_new = b.out_cache_loc
    assert np.all((all_new >= 1) & (all_new < S)), "slot 0 is the reserved dummy slot"
    assert np.unique(all_new).size == all_new.size, "new slots must be distinct"
    assert np.intersect1d(all_new, b.pool_slots).size == 0, "new slots must not hold cached tokens"
    assert np.unique(b.pool_slots).size == b.pool_slots.size
    assert np.all((b.pool_slots >= 1) & (b.pool_slots < S))
    cached = set(b.pool_slots.tolist()) | set(all_new.tolist())
    for rpi, L in list(zip(b.dec_rpi, b.dec_seq_lens)) + \
            list(zip(b.ext_rpi, b.ext_prefix_lens + b.ext_extend_lens)):
        row = b.req_to_token[rpi]
        assert np.all(row[L:] == W.NO_SLOT)
        assert set(row[:L].tolist()) <= cached
        assert np.unique(row[:L]).size == L, "a request never holds a slot twice"
    # table rows are distinct per request
    rows = np.concatenate([b.ext_rpi, b.dec_rpi])
    assert np.unique(rows).size == rows.size
    if b.has_cascade():
        for g in range(b.casc_group_indptr.size - 1):
            mem = b.casc_group_reqs[b.casc_group_indptr[g]:b.casc_group_indptr[g + 1]]
            P = b.casc_group_prefix_len[g]
            lead = b.req_to_token[b.dec_rpi[mem[0]], :P]
            for m in mem:
                assert b.dec_seq_lens[m] >= P
                np.testing.assert_array_equal(b.req_to_token[b.dec_rpi[m], :P], lead)


def test_tiny_config_shapes():
    e, d = W.tiny_extend_decode()
    assert list(e.ext_extend_lens) == [8, 12, 16, 24] and list(e.ext_prefix_lens) == [32] * 4
    assert (e.num_q_heads, e.num_kv_heads, e.head_dim, e.num_slots) == (8, 2, 64, 512)
    assert list(d.dec_seq_lens) == [41, 45, 49, 57]
    assert d.pool_slots.size + d.out_cache_loc.size == 96
    # shared prefix slots identical across requests
    pref = {tuple(e.req_to_token[r, :32]) for r in e.ext_rpi}
    assert len(pref) == 1
    _check_batch(e)
    _check_batch(d)


@pytest.mark.parametrize("name", ["decode_8b_system_prompts", "fewshot_extend", "forked_decode_70b"])
def test_config_invariants(name):
    b = W.WORKLOADS[name]()
    _check_batch(b)
    if name == "decode_8b_system_prompts":
        assert b.n_decode == 64 and (b.num_q_heads, b.num_kv_heads, b.head_dim) == (32, 8, 128)
        assert b.dec_seq_lens.min() >= 512 and b.dec_seq_lens.max() <= 4096
        assert b.casc_group_indptr.size == 9
    if name == "fewshot_extend":
        assert b.n_extend == 16 and np.all(b.ext_prefix_lens == 3000)
        assert b.ext_extend_lens.min() >= 200 and b.ext_extend_lens.max() <= 400
    if name == "forked_decode_70b":
        assert b.n_decode == 64 and (b.num_q_heads, b.num_kv_heads) == (64, 8)
        assert np.all((b.dec_seq_lens >= 8193) & (b.dec_seq_lens <= 8192 + 257))
        assert list(b.casc_group_prefix_len) == [8192]


@pytest.mark.parametrize("seed", range(4))
def test_random_mixed_invariants(seed):
    _check_batch(W.random_mixed(seed, n_extend=5, n_decode=7, num_q_heads=8, num_kv_heads=2, head_dim=64,
                                max_len=300, with_cascade=True))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0], np.float32)
    b = W.f32_to_bf16_bits(x)
    np.testing.assert_array_equal(W.bf16_bits_to_f32(b), [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 65536.0])


def _check_new_tokens_and_sharing(b):
    """The step's new tokens sit where the calls read them, and the rows are radix-consistent."""
    loc = b.out_cache_loc
    n_ext = int(b.ext_extend_lens.sum())
    assert loc.size == n_ext + b.n_decode
    for i, (r, P, E) in enumerate(zip(b.ext_rpi, b.ext_prefix_lens, b.ext_extend_lens)):
        q0, q1 = b.ext_qo_indptr[i], b.ext_qo_indptr[i + 1]
        assert q1 - q0 == E
        np.testing.assert_array_equal(b.req_to_token[r, P:P + E], loc[q0:q1])   # suffix after the prefix
        assert not set(b.req_to_token[r, :P].tolist()) & set(loc.tolist())      # the prefix is cached
    for j, (r, L) in enumerate(zip(b.dec_rpi, b.dec_seq_lens)):
        assert b.req_to_token[r, L - 1] == loc[n_ext + j]                        # the new token is last
        assert not set(b.req_to_token[r, :L - 1].tolist()) & set(loc.tolist())
    rows = [b.req_to_token[r, :L] for r, L in
            list(zip(b.ext_rpi, b.ext_prefix_lens + b.ext_extend_lens)) + list(zip(b.dec_rpi, b.dec_seq_lens))]
    # a slot is one position of one prefix: every slot has one (position, preceding slot) pair, so by
    # induction over the positions every row that holds it agrees on everything before it
    slot = np.concatenate(rows).astype(np.int64)
    pos = np.concatenate([np.arange(r.size) for r in rows])
    pred = np.concatenate([np.r_[-1, r[:-1]] for r in rows]).astype(np.int64)
    pairs = np.unique(np.stack([slot, pos, pred], axis=1), axis=0)
    assert np.unique(pairs[:, 0]).size == pairs.shape[0]
    if b.has_cascade():
        starts = b.casc_group_start if b.casc_group_start is not None else \
            np.zeros(b.casc_group_indptr.size - 1, np.int32)
        for g in range(b.casc_group_indptr.size - 1):
            mem = b.casc_group_reqs[b.casc_group_indptr[g]:b.casc_group_indptr[g + 1]]
            s, e = int(starts[g]), int(b.casc_group_prefix_len[g])
            assert len(mem) >= 2 and 0 <= s < e
            for m in mem:
                assert e <= b.dec_seq_lens[m] - 1                                 # the new token stays private


@pytest.mark.parametrize("seed", range(24))
def test_random_mixed_new_tokens_and_sharing(seed):
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    b = W.random_mixed(100 + seed, n_extend=int(rng.integers(0, 6)), n_decode=int(rng.integers(1, 9)),
                       num_q_heads=hkv * int(rng.choice([1, 2, 4])), num_kv_heads=hkv, head_dim=64,
                       max_len=int(rng.choice([20, 130, 400])), share_prob=float(rng.uniform(0, 0.95)),
                       with_cascade=bool(seed % 2), page_size=int(rng.choice([1, 1, 4])))
    _check_batch(b)
    _check_new_tokens_and_sharing(b)


@pytest.mark.parametrize("name", ["decode_8b_system_prompts", "fewshot_extend", "forked_decode_70b"])
def test_workload_new_tokens_and_sharing(name):
    _check_new_tokens_and_sharing(W.WORKLOADS[name]())
