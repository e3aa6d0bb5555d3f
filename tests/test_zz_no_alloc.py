"""ra_decode_attention_static: the decode entry point for callers that cannot
allocate device memory (for example a plugin running under a host framework's
fixed memory plan, or a runtime with no device allocator of its own).  It keeps
its split-KV scratch in the library's static device array instead of a caller
workspace.

Called here through the C ABI (ctypes) and compared with the workspace entry
point, ra_decode_attention, on two calls in a row.  Both run the same kernels on
the same inputs, so the outputs must agree bit for bit (which also puts them
within the 1e-2 + 1e-2 |ref| tolerance the other parity tests use).  This file
is collected last so that a stop-at-first-failure run has already run every
other test; it also passes on its own in a fresh process (its first call
performs the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import DeviceBatch, assert_close, to_f64

pytestmark = pytest.mark.gpu


def _static_call(db: DeviceBatch, cascade: bool, out: torch.Tensor) -> int:
    """One call of the C entry point with raw pointers; returns its status."""
    lib = ra.load()
    b = db.b
    P = ctypes.c_void_p

    def ptr(t):
        return P(t.data_ptr()) if t is not None else None

    ng, gi, gr, gp, mgp, mgs = 0, None, None, None, 0, 0
    if cascade:
        ng = b.casc_group_indptr.size - 1
        gi, gr, gp = db.g_indptr, db.g_reqs, db.g_plen
        mgp = int(b.casc_group_prefix_len.max())
        mgs = int(np.diff(b.casc_group_indptr).max())
    stream = P(torch.cuda.current_stream(db.dev).cuda_stream)
    return lib.ra_decode_attention_static(
        ptr(db.k_pool), ptr(db.v_pool), b.num_slots, b.num_kv_heads, b.head_dim, ptr(db.dec_q), ptr(out),
        b.num_q_heads, b.sm_scale, ptr(db.table), db.table.shape[1], db.table.shape[0], ptr(db.dec_rpi),
        ptr(db.dec_lens), b.n_decode, b.max_seq_len, ng, ptr(gi), ptr(gr), None, ptr(gp), None, mgp, mgs, 1,
        ptr(db.err), stream)


def _reference(db: DeviceBatch, cascade: bool) -> torch.Tensor:
    db.decode(cascade=cascade)  # the workspace entry point
    torch.cuda.synchronize()
    return db.dec_o.clone()


def _same_bits(got: torch.Tensor, ref: torch.Tensor, what: str):
    assert_close(to_f64(got), to_f64(ref), what)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"{what}: not bit-identical"


def test_static_scratch_decode_matches_workspace_decode_on_two_calls():
    cases = [
        (DeviceBatch(W.decode_8b_system_prompts()), True),   # system-prompt groups, cascade prefix pass + splits
        (DeviceBatch(W.random_mixed(31, n_extend=0, n_decode=12, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                    max_len=2500)), False),
    ]
    for db, _ in cases:
        db.store()
    refs = [_reference(db, casc) for db, casc in cases]
    # two calls in a row, each checked; the second reuses the array the first left behind
    for (db, casc), ref in zip(cases, refs):
        out = torch.full_like(db.dec_o, float("nan"))
        assert _static_call(db, casc, out) == 0, ra.load().ra_last_error_message()
        torch.cuda.synchronize()
        assert int(db.err.item()) == 0
        _same_bits(out, ref, f"{db.b.name} static-scratch decode")
    # and once more on the first case, after the second case overwrote the scratch
    db, casc = cases[0]
    out = torch.full_like(db.dec_o, float("nan"))
    assert _static_call(db, casc, out) == 0
    torch.cuda.synchronize()
    _same_bits(out, refs[0], "static-scratch decode, repeated")


def test_static_scratch_decode_python_binding():
    """The binding's ra_decode_attention_static (it makes the tensors' device current for the call)."""
    b = W.decode_8b_system_prompts()
    db = DeviceBatch(b)
    db.store()
    ref = _reference(db, True)
    out = torch.full_like(db.dec_o, float("nan"))
    ra.ra_decode_attention_static(db.k_pool, db.v_pool, db.dec_q, out, db.table, db.dec_rpi, db.dec_lens,
                                  max_seq_len=b.max_seq_len, sm_scale=b.sm_scale, group_indptr=db.g_indptr,
                                  group_reqs=db.g_reqs, group_prefix_len=db.g_plen,
                                  max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                                  max_group_size=int(np.diff(b.casc_group_indptr).max()), device_error=db.err)
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    _same_bits(out, ref, "static-scratch decode through the binding")


def test_static_scratch_decode_rejects_sizes_beyond_the_array():
    # 4096 requests x 64 q heads need more than 32 MiB of partials
    need = ra.ra_decode_workspace_bytes(4096, 64, 8, 128, 32768)
    assert need > ra.RA_DECODE_STATIC_SCRATCH_BYTES
    b = W.random_mixed(32, n_extend=0, n_decode=2, num_q_heads=64, num_kv_heads=8, head_dim=128, max_len=50)
    db = DeviceBatch(b)
    lib = ra.load()
    P = ctypes.c_void_p
    out = torch.empty_like(db.dec_q)
    st = lib.ra_decode_attention_static(
        P(db.k_pool.data_ptr()), P(db.v_pool.data_ptr()), b.num_slots, 8, 128, P(db.dec_q.data_ptr()),
        P(out.data_ptr()), 64, b.sm_scale, P(db.table.data_ptr()), 32768, db.table.shape[0],
        P(db.dec_rpi.data_ptr()), P(db.dec_lens.data_ptr()), 4096, 32768, 0, None, None, None, None, None, 0, 0, 1,
        None, P(torch.cuda.current_stream(db.dev).cuda_stream))
    assert st == 3  # RA_ERR_WORKSPACE, nothing launched
    assert b"static scratch" in lib.ra_last_error_message()
