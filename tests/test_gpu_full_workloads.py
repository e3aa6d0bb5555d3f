"""GPU parity on the five workloads at full size, every output compared.

Each workload runs in the launch configuration the benchmark times (store,
then extend, then decode; the multi-turn mix's decode with the radix tree's
one-level cascade groups) and every output row is compared with the fp64
oracle at 1e-2 + 1e-2 |ref| (a request's result is ordinary softmax attention
over its whole context: SGLang paper summary, §3).  After the store the whole
pool is compared bit for bit: the slots of `out_cache_loc` hold the oracle's
stored rows, every other slot its contents from before the store (the store's
definition, anrans handbook "v0.2", 来源一).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import DeviceBatch, assert_close, check_store, to_f64

pytestmark = pytest.mark.gpu


def _extend_all(db: DeviceBatch, pool):
    b = db.b
    db.extend()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    got = to_f64(db.ext_o).reshape(-1, b.head_dim)
    assert_close(got, oracle.extend_batch(b, pool=pool), f"{b.name} extend, all {got.shape[0]} rows")


def _decode_all(db: DeviceBatch, pool, cascade: bool):
    b = db.b
    db.decode(cascade=cascade)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    got = to_f64(db.dec_o).reshape(-1, b.head_dim)
    what = f"{b.name} decode{' (cascade)' if cascade else ''}, all {got.shape[0]} rows"
    assert_close(got, oracle.decode_batch(b, pool=pool), what)


def test_tiny_extend_then_decode_whole():
    e, d = W.tiny_extend_decode()
    for b in (e, d):
        db = DeviceBatch(b)
        check_store(db)
        pool = oracle.pool_after_store(b)
        if b.n_extend:
            _extend_all(db, pool)
        if b.n_decode:
            _decode_all(db, pool, cascade=False)


@pytest.mark.parametrize("name", ["decode_8b_system_prompts", "forked_decode_70b"])
def test_decode_workload_whole(name):
    b = W.WORKLOADS[name]()
    db = DeviceBatch(b)
    check_store(db)
    pool = oracle.pool_after_store(b)
    _decode_all(db, pool, cascade=False)
    _decode_all(db, pool, cascade=True)


def test_fewshot_extend_whole():
    b = W.fewshot_extend()
    db = DeviceBatch(b)
    check_store(db)
    _extend_all(db, oracle.pool_after_store(b))


def test_multiturn_mix_step_whole():
    """The benchmark's step on its own batch (decode requests in the tree's depth-first order): store (9.4K
    new tokens into a 2M-slot pool), extend of the 32 extend requests (all 588,480 rows), cascade decode of
    the 224 decode requests with the tree's groups (all 14,336 rows), and the same decode without groups."""
    import bench
    b = bench.mix_step_batch()
    assert b.has_cascade()
    db = DeviceBatch(b)
    check_store(db)
    pool = oracle.pool_after_store(b)
    _extend_all(db, pool)
    _decode_all(db, pool, cascade=True)
    _decode_all(db, pool, cascade=False)
