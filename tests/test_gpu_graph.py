"""The boundary's calls are graph-capturable: a whole step (store, extend, cascade decode)
captured once in a CUDA graph and replayed on new inputs written into the same buffers gives
the eager results bit for bit (the CUDA-graph decode of the pages' runtime replays fixed-address
buffers the same way)."""
import numpy as np
import pytest
import torch

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
