"""GPU parity sweep: randomly drawn mixed batches (shapes, lengths, forks, extend/decode mix, cascade
groups) through the C ABI -- store, extend, decode plain and grouped, and the fused store + decode --
each against the fp64 CPU oracle.  Seeded: every case is reproducible from its seed."""
import numpy as np
import pytest
import torch

import oracle
import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import DeviceBatch, assert_close, to_f64

pytestmark = pytest.mark.gpu

SHAPES = [(8, 2, 64), (16, 4, 128), (32, 8, 128), (64, 8, 128), (8, 8, 64), (12, 3, 128), (16, 2, 64)]  # GQA <= 8 (decode)


def _draw(seed: int) -> W.Batch:
    rng = np.random.default_rng(1000 + seed)
    hq, hkv, d = SHAPES[seed % len(SHAPES)]
    n_ext = int(rng.integers(0, 6))
    n_dec = int(rng.integers(1, 10))
    max_len = int(rng.choice([40, 130, 700, 1500]))
    return W.random_mixed(2000 + seed, n_extend=n_ext, n_decode=n_dec, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim=d, max_len=max_len, min_len=int(rng.integers(1, 4)),
                          share_prob=float(rng.uniform(0.0, 0.9)), with_cascade=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("seed", range(16))
def test_random_batch_matches_oracle(seed):
    b = _draw(seed)
    db = DeviceBatch(b)
    db.store()
    pool = oracle.pool_after_store(b)
    if b.n_extend:
        db.extend()
        torch.cuda.synchronize()
        assert int(db.err.item()) == 0
        assert_close(to_f64(db.ext_o).reshape(-1, b.head_dim), oracle.extend_batch(b, pool=pool),
                     f"sweep {seed} extend")
    ref = oracle.decode_batch(b, pool=pool)
    db.decode(cascade=False)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    assert_close(to_f64(db.dec_o).reshape(-1, b.head_dim), ref, f"sweep {seed} decode")
    if b.has_cascade():
        db.dec_o.fill_(float("nan"))
        db.decode(cascade=True)
        torch.cuda.synchronize()
        assert int(db.err.item()) == 0
        assert_close(to_f64(db.dec_o).reshape(-1, b.head_dim), ref, f"sweep {seed} cascade decode")


@pytest.mark.parametrize("seed", range(16, 24))
def test_random_decode_batch_fused_store(seed):
    """Decode-only draws: the fused store + decode call against the oracle (the pool starts without
    the step's tokens)."""
    b = _draw(seed)
    b = W.random_mixed(3000 + seed, n_extend=0, n_decode=b.n_decode + 2, num_q_heads=b.num_q_heads,
                       num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, max_len=int(b.max_seq_len) + 1,
                       with_cascade=seed % 2 == 0)
    db = DeviceBatch(b)
    kw = {}
    if b.has_cascade():
        kw = dict(group_indptr=db.g_indptr, group_reqs=db.g_reqs, group_prefix_len=db.g_plen,
                  max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                  max_group_size=int(np.diff(b.casc_group_indptr).max()), group_prefix_start=db.g_start,
                  group_level=db.g_level, max_group_levels=b.casc_levels)
    ra.ra_decode_attention_store(db.k_pool, db.v_pool, db.k_new, db.v_new, db.loc, db.dec_q, db.dec_o, db.table,
                                 db.dec_rpi, db.dec_lens, max_seq_len=b.max_seq_len, sm_scale=b.sm_scale,
                                 workspace=db.decode_ws(b.has_cascade()), device_error=db.err, **kw)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    assert_close(to_f64(db.dec_o).reshape(-1, b.head_dim), oracle.decode_batch(b), f"sweep {seed} fused decode")
