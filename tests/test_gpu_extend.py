"""GPU parity: extend attention (tcgen05) and the cascade (prefix-grouped) decode
against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import (DeviceBatch, assert_close, attach_tree_groups, attach_tree_groups_multilevel, grow_key_scale,
                     late_half_key_scale,
                     prefill_chunks, to_f64)

pytestmark = pytest.mark.gpu


def check_extend(db: DeviceBatch, sel=None):
    b = db.b
    db.extend()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0, int(db.err.item())
    got = to_f64(db.ext_o).reshape(-1, b.head_dim)
    ref = oracle.extend_batch(b, sel=sel)
    if sel is not None:
        got = got[sel]
    assert_close(got, ref, f"{b.name} extend")


def test_extend_tiny_config():
    e, _ = W.tiny_extend_decode()
    db = DeviceBatch(e)
    db.store()
    check_extend(db)


@pytest.mark.parametrize("seed,hq,hkv,d,max_len", [
    (0, 8, 2, 64, 40), (1, 32, 8, 128, 300), (2, 16, 2, 128, 700), (3, 8, 8, 128, 200),
    (4, 64, 8, 128, 500), (5, 4, 2, 64, 900), (6, 16, 1, 128, 150), (7, 32, 2, 64, 260)])
def test_extend_ragged(seed, hq, hkv, d, max_len):
    b = W.random_mixed(seed, n_extend=6, n_decode=0, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       max_len=max_len)
    db = DeviceBatch(b)
    db.store()
    check_extend(db)


@pytest.mark.parametrize("d", [128, 64])
def test_extend_output_only_16_byte_aligned(d):
    """An output only as aligned as the interface requires (16 bytes: a view 16 bytes into a buffer)."""
    b = W.random_mixed(40 + d, n_extend=5, n_decode=0, num_q_heads=16, num_kv_heads=4, head_dim=d, max_len=400)
    db = DeviceBatch(b)
    db.store()
    n = db.ext_o.numel()
    big = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device=db.dev)
    db.ext_o = big[8:].view(db.ext_o.shape)
    assert db.ext_o.data_ptr() % 32 == 16
    check_extend(db)


def test_extend_prefix_zero_and_single_token_suffix():
    b = W.random_mixed(11, n_extend=5, n_decode=0, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=300,
                       share_prob=0.0, ext_lens=[1, 300, 1, 129, 128])
    assert (b.ext_prefix_lens == 0).any() and (b.ext_extend_lens == 1).any()
    db = DeviceBatch(b)
    db.store()
    check_extend(db)


@pytest.mark.parametrize("seed,hq,hkv,d", [(21, 32, 8, 128), (22, 16, 2, 64)])
def test_extend_growing_scores(seed, hq, hkv, d):
    """Scores that grow by orders of magnitude from tile to tile: every tile after the first fails the
    single-pass acceptance bound and is redone with the exact maximum and an O rescale."""
    b = grow_key_scale(W.random_mixed(seed, n_extend=5, n_decode=0, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      max_len=700, min_len=300))
    db = DeviceBatch(b)
    db.store()
    check_extend(db)


@pytest.mark.parametrize("seed,hq,hkv,d", [(23, 32, 8, 128), (24, 16, 2, 64)])
def test_extend_late_half_scores(seed, hq, hkv, d):
    """Every key tile's last 64 scores far above its first 64 (which stay within the reference of the
    tile before): the second half of each tile's probabilities needs a reference move after the first
    half has gone to the PV."""
    b = late_half_key_scale(W.random_mixed(seed, n_extend=5, n_decode=0, num_q_heads=hq, num_kv_heads=hkv,
                                           head_dim=d, max_len=700, min_len=300))
    db = DeviceBatch(b)
    db.store()
    check_extend(db)


@pytest.mark.parametrize("chunk", [64, 100])
def test_chunked_prefill(chunk):
    """Chunked prefill through the C ABI: each call extends every request by one chunk over its
    cached prefix plus the chunks before it; the rows equal the oracle's single extend."""
    b = W.random_mixed(24, n_extend=6, n_decode=0, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=600,
                       min_len=200)
    db = DeviceBatch(b)
    db.store()
    db.extend()
    full_gpu = to_f64(db.ext_o).reshape(b.total_q_extend, b.num_q_heads, b.head_dim)
    ref = oracle.extend_batch(b).reshape(b.total_q_extend, b.num_q_heads, b.head_dim)
    dev = db.dev
    got = np.zeros_like(ref)
    for q, plen, elen, qo, toks in prefill_chunks(b, chunk):
        qd = torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16)
        od = torch.empty_like(qd)
        ws = torch.empty(ra.ra_extend_workspace_bytes(b.n_extend, qd.shape[0], b.num_q_heads, b.num_kv_heads),
                         dtype=torch.uint8, device=dev)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
        ra.ra_extend_attention(db.k_pool, db.v_pool, qd, od, db.table, db.ext_rpi, i32(plen), i32(elen), i32(qo),
                               max_extend_len=chunk, max_prefix_len=int(plen.max()), sm_scale=b.sm_scale,
                               workspace=ws, device_error=db.err)
        torch.cuda.synchronize()
        got[toks] = to_f64(od).reshape(-1, b.num_q_heads, b.head_dim)
    assert int(db.err.item()) == 0
    assert_close(got.reshape(-1, b.head_dim), ref.reshape(-1, b.head_dim), "chunked prefill vs oracle")
    assert_close(got.reshape(-1, b.head_dim), full_gpu.reshape(-1, b.head_dim), "chunked vs one extend")


def test_extend_matches_decode_for_the_last_token():
    """The last suffix row of an extend equals a decode of that token (same context)."""
    b = W.random_mixed(12, n_extend=4, n_decode=0, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=600)
    db = DeviceBatch(b)
    db.store()
    db.extend()
    last = b.ext_qo_indptr[1:] - 1
    q = db.ext_q[torch.from_numpy(last.astype(np.int64)).to(db.dev)].contiguous()
    o = torch.empty_like(q)
    lens = torch.from_numpy((b.ext_prefix_lens + b.ext_extend_lens).astype(np.int32)).to(db.dev)
    ws = torch.empty(ra.ra_decode_workspace_bytes(4, 32, 8, 128, int(lens.max())), dtype=torch.uint8,
                     device=db.dev)
    ra.ra_decode_attention(db.k_pool, db.v_pool, q, o, db.table, db.ext_rpi, lens, max_seq_len=int(lens.max()),
                           sm_scale=b.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    a = to_f64(db.ext_o[torch.from_numpy(last.astype(np.int64)).to(db.dev)])
    assert_close(to_f64(o), a, "decode vs last extend row")


def test_extend_rows_outside_o_are_flagged_not_written():
    """A request whose qo_indptr puts its rows past total_q is skipped and flagged RA_DEVERR_LENGTH: nothing
    is written outside o (a guard region after it keeps its fill), the other requests are still exact."""
    b = W.random_mixed(41, n_extend=4, n_decode=0, num_q_heads=16, num_kv_heads=4, head_dim=128, max_len=300,
                       min_len=40)
    db = DeviceBatch(b)
    db.store()
    n, guard = b.total_q_extend, 96
    buf = torch.full((n + guard, b.num_q_heads, b.head_dim), float("nan"), dtype=torch.bfloat16, device=db.dev)
    o = buf[:n]
    qo = b.ext_qo_indptr.copy()
    last = b.n_extend - 1
    qo[last] += 5  # rows qo[last] .. qo[last] + E - 1 now run 5 rows past total_q
    assert qo[last] + b.ext_extend_lens[last] > n
    ws = torch.empty(ra.ra_extend_workspace_bytes(b.n_extend, n, b.num_q_heads, b.num_kv_heads), dtype=torch.uint8,
                     device=db.dev)
    ra.ra_extend_attention(db.k_pool, db.v_pool, db.ext_q, o, db.table, db.ext_rpi, db.ext_prefix, db.ext_len,
                           torch.from_numpy(qo).to(db.dev), max_extend_len=b.max_extend_len,
                           max_prefix_len=b.max_prefix_len, sm_scale=b.sm_scale, workspace=ws, device_error=db.err)
    torch.cuda.synchronize()
    assert int(db.err.item()) & ra.DEVERR_LENGTH
    assert torch.isnan(buf[n:].float()).all(), "a row past total_q was written"
    assert torch.isnan(o[b.ext_qo_indptr[last]:].float()).all(), "the skipped request wrote rows"
    keep = int(b.ext_qo_indptr[last]) * b.num_q_heads
    got = to_f64(o).reshape(-1, b.head_dim)[:keep]
    assert_close(got, oracle.extend_batch(b)[:keep], "requests before the skipped one")


def test_extend_bad_slot_flagged():
    b = W.random_mixed(13, n_extend=2, n_decode=0, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=100)
    db = DeviceBatch(b)
    db.store()
    db.table[b.ext_rpi[0], 0] = b.num_slots  # out of range
    db.extend()
    torch.cuda.synchronize()
    assert int(db.err.item()) & ra.DEVERR_SLOT


# ---------------------------------------------------------------- cascade decode
def check_cascade(db: DeviceBatch, sel=None):
    b = db.b
    assert b.has_cascade()
    db.decode(cascade=False)
    torch.cuda.synchronize()
    plain = to_f64(db.dec_o)
    db.dec_o.zero_()
    db.decode(cascade=True)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0, int(db.err.item())
    casc = to_f64(db.dec_o)
    got = casc.reshape(-1, b.head_dim)
    ref = oracle.decode_batch(b, sel=sel)
    if sel is not None:
        got = got[sel]
    assert_close(got, ref, f"{b.name} cascade decode")
    assert_close(casc, plain, f"{b.name} cascade vs plain")


def test_cascade_tiny_config():
    _, d = W.tiny_extend_decode()
    db = DeviceBatch(d)
    db.store()
    check_cascade(db)


@pytest.mark.parametrize("seed,hq,hkv,d,max_len", [
    (20, 32, 8, 128, 900), (21, 64, 8, 128, 400), (22, 8, 2, 64, 300), (23, 16, 8, 128, 1300)])
def test_cascade_ragged(seed, hq, hkv, d, max_len):
    b = W.random_mixed(seed, n_extend=0, n_decode=24, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       max_len=max_len, share_prob=0.9, with_cascade=True)
    if not b.has_cascade():
        pytest.skip("seed produced no group")
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)


def test_cascade_member_without_private_keys():
    """A member whose whole context is the group prefix (P_g == L) only has prefix partials."""
    b = W.random_mixed(24, n_extend=0, n_decode=6, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=500,
                       share_prob=0.9, with_cascade=True)
    if not b.has_cascade():
        pytest.skip("seed produced no group")
    g0 = b.casc_group_reqs[b.casc_group_indptr[0]:b.casc_group_indptr[1]]
    # shrink the prefix to the shortest member's full length
    b.casc_group_prefix_len[0] = min(b.casc_group_prefix_len[0], int(b.dec_seq_lens[g0].min()))
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)


def test_cascade_growing_scores():
    """The prefix pass's tiles (several per split) under scores that grow tile by tile."""
    b = grow_key_scale(W.decode_8b_system_prompts())  # 8 groups sharing 1024 prompt tokens: 512-key splits of 4 tiles
    assert b.has_cascade()
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)


def test_cascade_late_half_scores():
    """The prefix pass under scores whose last 64 of every key tile exceed the first 64's reference."""
    b = late_half_key_scale(W.decode_8b_system_prompts())
    assert b.has_cascade()
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)


@pytest.mark.parametrize("seed,hq,hkv,d", [(51, 32, 8, 128), (52, 16, 2, 64)])
def test_cascade_multilevel_random(seed, hq, hkv, d):
    """One group per shared node of the decode rows' tree: nested ranges at several levels."""
    b = attach_tree_groups_multilevel(W.random_mixed(seed, n_extend=0, n_decode=24, num_q_heads=hq, num_kv_heads=hkv,
                                                     head_dim=d, max_len=1200, min_len=200, share_prob=0.95))
    assert b.has_cascade() and b.casc_levels >= 2
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)


def test_cascade_multilevel_multiturn_mix():
    """The multi-turn mix's decode with one group per shared node of its tree (every row compared)."""
    b = attach_tree_groups_multilevel(W.multiturn_mix_70b())
    assert b.casc_levels >= 2
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)
