"""The boundary's calls are graph-capturable: a whole step (store, extend, cascade decode)
captured once in a CUDA graph and replayed on new inputs written into the same buffers gives
the eager results bit for bit (the CUDA-graph decode of the pages' runtime replays fixed-address
buffers the same way)."""
import numpy as np
import pytest
import torch

import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import DeviceBatch

pytestmark = pytest.mark.gpu


def _step(db):
    db.store()
    db.extend()
    db.decode(cascade=db.b.has_cascade())


def test_step_replays_from_a_cuda_graph():
    b = W.random_mixed(40, n_extend=4, n_decode=12, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=900,
                       share_prob=0.9, with_cascade=True)
    assert b.has_cascade()
    db = DeviceBatch(b)
    _step(db)  # warm-up outside capture: first-call set-up (attributes, workspace)
    torch.cuda.synchronize()
    ref_e, ref_d = db.ext_o.clone(), db.dec_o.clone()

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        _step(db)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            _step(db)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()

    db.ext_o.zero_()
    db.dec_o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(db.ext_o, ref_e) and torch.equal(db.dec_o, ref_d)

    # new queries in the captured buffers: replay equals a fresh eager step
    gen = torch.Generator(device=db.dev).manual_seed(7)
    db.ext_q.copy_(torch.randn(db.ext_q.shape, generator=gen, device=db.dev).to(torch.bfloat16))
    db.dec_q.copy_(torch.randn(db.dec_q.shape, generator=gen, device=db.dev).to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    got_e, got_d = db.ext_o.clone(), db.dec_o.clone()
    _step(db)
    torch.cuda.synchronize()
    assert torch.equal(got_e, db.ext_o) and torch.equal(got_d, db.dec_o)
    assert int(db.err.item()) == 0


def _fused_step(db):
    b = db.b
    ra.ra_decode_attention_store(db.k_pool, db.v_pool, db.k_new, db.v_new, db.loc, db.dec_q, db.dec_o, db.table,
                                 db.dec_rpi, db.dec_lens, max_seq_len=b.max_seq_len, sm_scale=b.sm_scale,
                                 workspace=db.decode_ws(True), device_error=db.err, group_indptr=db.g_indptr,
                                 group_reqs=db.g_reqs, group_prefix_len=db.g_plen,
                                 max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                                 max_group_size=int(np.diff(b.casc_group_indptr).max()),
                                 group_prefix_start=db.g_start, group_level=db.g_level, max_group_levels=b.casc_levels)


def test_fused_store_decode_replays_from_a_cuda_graph():
    """The decode step as one call (store fused into the grouped decode) replays from a graph: new
    queries and new K/V rows written into the captured buffers give the eager result bit for bit."""
    b = W.random_mixed(41, n_extend=0, n_decode=16, num_q_heads=32, num_kv_heads=8, head_dim=128, max_len=700,
                       share_prob=0.9, with_cascade=True)
    assert b.has_cascade()
    db = DeviceBatch(b)
    _fused_step(db)  # warm-up outside capture (workspace, kernel attributes)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            _fused_step(db)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    gen = torch.Generator(device=db.dev).manual_seed(8)
    for buf in (db.dec_q, db.k_new, db.v_new):
        buf.copy_(torch.randn(buf.shape, generator=gen, device=db.dev).to(torch.bfloat16))
    db.dec_o.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = db.dec_o.clone()
    _fused_step(db)
    torch.cuda.synchronize()
    assert torch.equal(got, db.dec_o)
    assert int(db.err.item()) == 0
