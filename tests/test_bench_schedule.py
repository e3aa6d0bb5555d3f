"""The benchmark's decode order (the radix tree's depth-first order, a cache-aware scheduler's order):
rescheduling a batch permutes its decode requests together with their store rows, so the oracle's
outputs of the rescheduled batch are the original batch's outputs in the new order."""
import numpy as np

import bench
import oracle
import workloads as W
from prefix_shared_kv_ra_gb300.radix import dfs_order


def test_rescheduled_batch_is_the_same_batch_in_dfs_order():
    b = W.random_mixed(61, n_extend=3, n_decode=9, num_q_heads=8, num_kv_heads=2, head_dim=64, max_len=90,
                       share_prob=0.8)
    c = bench.schedule_decode_dfs(b)
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    order = dfs_order(rows)
    np.testing.assert_array_equal(c.dec_rpi, b.dec_rpi[order])
    # the store writes the same rows to the same slots
    got = {int(s): (k.tobytes(), v.tobytes()) for s, k, v in zip(c.out_cache_loc, c.k_new, c.v_new)}
    ref = {int(s): (k.tobytes(), v.tobytes()) for s, k, v in zip(b.out_cache_loc, b.k_new, b.v_new)}
    assert got == ref
    # attention: the decode outputs permuted, the extend outputs unchanged
    hq, d = b.num_q_heads, b.head_dim
    dec_b = oracle.decode_batch(b).reshape(b.n_decode, hq, d)
    dec_c = oracle.decode_batch(c).reshape(c.n_decode, hq, d)
    np.testing.assert_array_equal(dec_c, dec_b[order])
    np.testing.assert_array_equal(oracle.extend_batch(c), oracle.extend_batch(b))
    # the rows in the new order are lexicographically sorted
    new_rows = [tuple(c.req_to_token[r, :L].tolist()) for r, L in zip(c.dec_rpi, c.dec_seq_lens)]
    assert new_rows == sorted(new_rows)
