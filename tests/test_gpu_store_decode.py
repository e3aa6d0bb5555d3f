"""GPU parity: KV store (bit-exact) and decode attention (1e-2 abs + 1e-2 rel) against
the CPU oracle, through the C ABI, on small ragged cases and the full workloads."""
import numpy as np
import pytest
import torch

import oracle
import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import DeviceBatch, assert_close, bf16, grow_key_scale, i32, to_f64

pytestmark = pytest.mark.gpu


def _pool_rows(t: torch.Tensor, slots: np.ndarray) -> np.ndarray:
    idx = torch.from_numpy(slots.astype(np.int64)).to(t.device)
    return t.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)


def check_decode(db: DeviceBatch, sel=None, cascade=False):
    b = db.b
    db.decode(cascade=cascade)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    got = to_f64(db.dec_o).reshape(-1, b.head_dim)
    ref = oracle.decode_batch(b, sel=sel)
    if sel is not None:
        got = got[sel]
    assert_close(got, ref, f"{b.name} decode")


# ---------------------------------------------------------------- store
def test_store_tiny_bit_exact():
    e, d = W.tiny_extend_decode()
    for b in (e, d):
        db = DeviceBatch(b)
        db.store()
        torch.cuda.synchronize()
        k_ref, v_ref = oracle.kv_store(*b.dense_pool(), b.k_new, b.v_new, b.out_cache_loc)
        got_k = db.k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
        got_v = db.v_pool.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got_k, k_ref)   # the whole pool, bit for bit
        np.testing.assert_array_equal(got_v, v_ref)


def test_store_empty_and_bad_slot_flag():
    b = W.random_mixed(3, n_extend=1, n_decode=3, num_q_heads=4, num_kv_heads=2, head_dim=64, max_len=20)
    db = DeviceBatch(b)
    ra.ra_kv_store(db.k_pool, db.v_pool, db.k_new[:0], db.v_new[:0], db.loc[:0], device_error=db.err)
    bad = db.loc.clone()
    bad[0] = b.num_slots + 5
    before = db.k_pool.clone()
    ra.ra_kv_store(db.k_pool, db.v_pool, db.k_new, db.v_new, bad, device_error=db.err)
    torch.cuda.synchronize()
    assert int(db.err.item()) & ra.DEVERR_SLOT
    # the bad row is skipped, the others written
    assert torch.equal(db.k_pool[b.out_cache_loc[1]], db.k_new[1])
    changed = (db.k_pool != before).any(dim=(1, 2)).nonzero().flatten().cpu().numpy()
    assert set(changed.tolist()) <= set(b.out_cache_loc[1:].tolist())


# ---------------------------------------------------------------- decode
def test_decode_tiny_config():
    _, d = W.tiny_extend_decode()
    db = DeviceBatch(d)
    db.store()
    check_decode(db)


@pytest.mark.parametrize("seed,hq,hkv,d,max_len", [
    (0, 8, 2, 64, 40), (1, 32, 8, 128, 700), (2, 16, 2, 128, 1500), (3, 8, 8, 128, 300),
    (4, 4, 2, 64, 2600), (5, 64, 8, 128, 1200), (6, 6, 3, 128, 260)])
def test_decode_ragged(seed, hq, hkv, d, max_len):
    b = W.random_mixed(seed, n_extend=0, n_decode=9, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       max_len=max_len)
    db = DeviceBatch(b)
    db.store()
    check_decode(db)


@pytest.mark.parametrize("seed,hq,hkv,d,per_tile", [(7, 32, 8, 128, 6.0), (8, 8, 2, 64, 0.5)])
def test_decode_growing_scores_per_slab(seed, hq, hkv, d, per_tile):
    """Keys scaled by 1 + per_tile * (position // 16): every 16-key slab's scores grow past the decode
    softmax's running reference (by far, or -- with the small factor -- by amounts around its 2^8
    rescale threshold), so its rescale of O and l runs on most slabs."""
    b = grow_key_scale(W.random_mixed(seed, n_extend=0, n_decode=12, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      min_len=200, max_len=1500), per_tile=per_tile, tile=16)
    db = DeviceBatch(b)
    db.store()
    check_decode(db)


@pytest.mark.parametrize("seed,n,hq,hkv,d,min_len,max_len", [
    (30, 60, 32, 16, 64, 1, 3000),     # chunk above the minimum, remainders of every size, 2 head groups
    (31, 5, 8, 2, 128, 256, 256),      # every context an exact multiple of the item length: no short items
    (32, 3, 8, 2, 64, 127, 129)])      # lengths around one item
def test_decode_device_plan(seed, n, hq, hkv, d, min_len, max_len):
    """The call's private keys are cut into items on the device from the real lengths (equal items
    first, each request's short last item after them): outputs still match the oracle."""
    b = W.random_mixed(seed, n_extend=0, n_decode=n, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       min_len=min_len, max_len=max_len)
    db = DeviceBatch(b)
    db.store()
    check_decode(db)


def test_decode_device_plan_large_batch():
    """More requests than the plan kernel has threads (each thread plans a run of consecutive requests),
    short contexts; without and with cascade groups."""
    b = W.random_mixed(33, n_extend=0, n_decode=2500, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=40,
                       with_cascade=True)
    db = DeviceBatch(b)
    db.store()
    check_decode(db)
    check_decode(db, cascade=True)


def test_decode_single_token_contexts():
    b = W.random_mixed(8, n_extend=0, n_decode=5, num_q_heads=8, num_kv_heads=2, head_dim=128, max_len=1,
                       min_len=1, share_prob=0.0)
    db = DeviceBatch(b)
    db.store()
    check_decode(db)
    # one key: the output is that key's V row rounded to bf16
    v = to_f64(db.v_new).reshape(5, 2, 128)
    got = to_f64(db.dec_o).reshape(5, 8, 128)
    np.testing.assert_array_equal(got, np.repeat(v, 4, axis=1))


def test_decode_bad_table_row_is_flagged_not_faulted():
    b = W.random_mixed(9, n_extend=0, n_decode=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=50)
    db = DeviceBatch(b)
    db.store()
    db.table[b.dec_rpi[1], 0] = -7           # a corrupt slot id
    db.decode()
    torch.cuda.synchronize()
    assert int(db.err.item()) & ra.DEVERR_SLOT


def test_decode_empty_batch_is_noop():
    b = W.random_mixed(10, n_extend=0, n_decode=2, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=20)
    db = DeviceBatch(b)
    ws = torch.empty(1024, dtype=torch.uint8, device=db.dev)
    ra.ra_decode_attention(db.k_pool, db.v_pool, db.dec_q[:0], db.dec_o[:0], db.table, db.dec_rpi[:0],
                           db.dec_lens[:0], max_seq_len=b.max_seq_len, sm_scale=b.sm_scale, workspace=ws)
    torch.cuda.synchronize()


# ---------------------------------------------------------------- fused store + decode
def _store_decode(db: DeviceBatch, cascade: bool):
    b = db.b
    kw = {}
    if cascade:
        kw = dict(group_indptr=db.g_indptr, group_reqs=db.g_reqs, group_prefix_len=db.g_plen,
                  max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                  max_group_size=int(np.diff(b.casc_group_indptr).max()), group_prefix_start=db.g_start,
                  group_level=db.g_level, max_group_levels=b.casc_levels)
    ra.ra_decode_attention_store(db.k_pool, db.v_pool, db.k_new, db.v_new, db.loc, db.dec_q, db.dec_o, db.table,
                                 db.dec_rpi, db.dec_lens, max_seq_len=b.max_seq_len, sm_scale=b.sm_scale,
                                 workspace=db.decode_ws(cascade), device_error=db.err, **kw)


@pytest.mark.parametrize("case,cascade", [("decode_8b_system_prompts", False), ("decode_8b_system_prompts", True),
                                          ("forked_decode_70b", True), ("random_large", False),
                                          ("random_large", True)])
def test_store_decode_fused_matches_store_then_decode(case, cascade):
    """ra_decode_attention_store writes the same pool rows as ra_kv_store (bit-exact) and returns the same
    outputs as ra_kv_store followed by ra_decode_attention (bit-exact: the same kernels read the same
    pool), within the tolerance of the oracle."""
    if case == "random_large":
        b = W.random_mixed(34, n_extend=0, n_decode=2000, num_q_heads=8, num_kv_heads=2, head_dim=128, max_len=60,
                           with_cascade=True)
    else:
        b = W.WORKLOADS[case]()
    assert b.n_extend == 0 and b.num_new_tokens == b.n_decode
    ref = DeviceBatch(b)
    ref.store()
    ref.decode(cascade=cascade)
    fused = DeviceBatch(b)
    _store_decode(fused, cascade)
    torch.cuda.synchronize()
    assert int(ref.err.item()) == 0 and int(fused.err.item()) == 0
    slots = b.out_cache_loc.astype(np.int64)
    np.testing.assert_array_equal(_pool_rows(fused.k_pool, slots), b.k_new)
    np.testing.assert_array_equal(_pool_rows(fused.v_pool, slots), b.v_new)
    np.testing.assert_array_equal(fused.dec_o.view(torch.int16).cpu().numpy(), ref.dec_o.view(torch.int16).cpu().numpy())
    if case == "random_large":
        assert_close(to_f64(fused.dec_o).reshape(-1, b.head_dim), oracle.decode_batch(b), f"{b.name} fused decode")


def test_store_decode_fused_bad_slot_is_flagged():
    b = W.random_mixed(35, n_extend=0, n_decode=4, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=30)
    db = DeviceBatch(b)
    db.loc = torch.full_like(db.loc, b.num_slots + 5)  # every new row outside the pool: skipped, flagged
    _store_decode(db, False)
    torch.cuda.synchronize()
    assert int(db.err.item()) & ra.DEVERR_SLOT

