"""The C-ABI library: it loads, exports every symbol include/ra.h declares, and its
host-side validation rejects bad arguments before touching a GPU (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import prefix_shared_kv_ra_gb300 as ra
from prefix_shared_kv_ra_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ra.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ra.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("ra_kv_store", "ra_extend_attention", "ra_extend_workspace_bytes", "ra_decode_attention",
              "ra_decode_workspace_bytes", "ra_decode_attention_store", "ra_status_string",
              "ra_last_error_message", "ra_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (ra_[a-z0-9_]+)\b", out))
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    for n in _declared_functions():
        assert hasattr(lib, n)


def test_abi_version_and_status_strings(lib):
    assert ra.ra_abi_version() == 5
    assert lib.ra_status_string(0) == b"ok"
    assert lib.ra_status_string(3) == b"workspace too small"


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first


def _decode_call(lib, **over):
    args = dict(k=FAKE, v=FAKE, S=1024, hkv=8, d=128, q=FAKE, o=FAKE, hq=32, scale=0.088, table=FAKE,
                stride=4096, rows=64, rpi=FAKE, lens=FAKE, batch=4, max_len=4096, ng=0, gi=None, gr=None, gs=None,
                gp=None, gl=None, mgp=0, mgs=0, mgl=1, ws=FAKE, wsb=1 << 30, err=None, stream=None)
    args.update(over)
    return lib.ra_decode_attention(*args.values())


def _store_decode_call(lib, kn=FAKE, vn=FAKE, loc=FAKE, **over):
    args = dict(k=FAKE, v=FAKE, S=1024, hkv=8, d=128, kn=kn, vn=vn, loc=loc, q=FAKE, o=FAKE, hq=32, scale=0.088,
                table=FAKE, stride=4096, rows=64, rpi=FAKE, lens=FAKE, batch=4, max_len=4096, ng=0, gi=None, gr=None,
                gs=None, gp=None, gl=None, mgp=0, mgs=0, mgl=1, ws=FAKE, wsb=1 << 30, err=None, stream=None)
    args.update(over)
    return lib.ra_decode_attention_store(*args.values())


def test_store_decode_validation(lib):
    """The fused store + decode checks the store's arguments as well as the decode's; nothing launches."""
    assert _store_decode_call(lib, kn=None) == 1                                   # missing new rows
    assert _store_decode_call(lib, loc=None) == 1
    assert _store_decode_call(lib, vn=ctypes.c_void_p((1 << 20) + 8)) == 1         # misaligned v_new
    assert _store_decode_call(lib, loc=ctypes.c_void_p((1 << 20) + 2)) == 1        # misaligned slots
    assert _store_decode_call(lib, hq=30) == 1                                     # decode checks still apply
    assert _store_decode_call(lib, wsb=16) == 3
    assert _store_decode_call(lib, batch=0) == 0                                   # empty batch: no-op


def test_decode_validation(lib):
    assert _decode_call(lib, hq=30) == 1                       # Hq % Hkv != 0
    assert _decode_call(lib, d=96) == 2                        # unsupported head_dim
    assert _decode_call(lib, hq=128) == 2                      # group 16 > 8
    assert _decode_call(lib, wsb=16) == 3                      # workspace too small
    assert b"workspace" in lib.ra_last_error_message()
    assert _decode_call(lib, q=ctypes.c_void_p((1 << 20) + 8)) == 1   # misaligned q
    assert _decode_call(lib, stride=100) == 1                  # table narrower than max_seq_len
    assert _decode_call(lib, scale=float("nan")) == 1
    assert _decode_call(lib, batch=-1) == 1
    assert _decode_call(lib, ng=2, gi=None) == 1               # cascade arrays missing
    assert _decode_call(lib, ng=2, gi=FAKE, gr=FAKE, gp=FAKE, mgp=100, mgs=2, mgl=2) == 1  # levels need group_level
    assert _decode_call(lib, ng=2, gi=FAKE, gr=FAKE, gp=FAKE, mgp=100, mgs=2, mgl=0) == 1  # no level
    assert _decode_call(lib, batch=0) == 0                     # empty batch: no-op


def test_decode_workspace_grows_with_bounds(lib):
    a = ra.ra_decode_workspace_bytes(64, 32, 8, 128, 4096)
    b = ra.ra_decode_workspace_bytes(64, 32, 8, 128, 512)
    c = ra.ra_decode_workspace_bytes(64, 32, 8, 128, 4096, 8, 1024, 8)
    c3 = ra.ra_decode_workspace_bytes(64, 32, 8, 128, 4096, 8, 1024, 8, 3)
    assert c3 > c  # three levels of prefix partials
    d = ra.ra_decode_workspace_bytes(64, 32, 8, 128, 32768)
    # private partials are bounded by the device plan's item count (a constant plus one per request),
    # not by the context length
    assert 0 < b == a == d < c
    assert ra.ra_decode_workspace_bytes(128, 32, 8, 128, 4096) > a
    assert ra.ra_decode_workspace_bytes(0, 32, 8, 128, 4096) == 0


def _extend_call(lib, **over):
    args = dict(k=FAKE, v=FAKE, S=1024, hkv=8, d=128, q=FAKE, o=FAKE, hq=32, scale=0.088, table=FAKE,
                stride=4096, rows=64, rpi=FAKE, plen=FAKE, elen=FAKE, qo=FAKE, batch=4, total_q=1000,
                max_e=500, max_p=3000, ws=FAKE, wsb=16, err=None, stream=None)
    args.update(over)
    return lib.ra_extend_attention(*args.values())


def test_extend_validation(lib):
    need = ra.ra_extend_workspace_bytes(4, 1000, 32, 8)
    assert _extend_call(lib, hq=30) == 1                       # Hq % Hkv != 0
    assert _extend_call(lib, d=96) == 2                        # unsupported head_dim
    assert _extend_call(lib, wsb=need - 1) == 3                # workspace too small
    assert b"workspace" in lib.ra_last_error_message()
    assert _extend_call(lib, ws=None, wsb=need) == 3           # no workspace
    assert _extend_call(lib, ws=ctypes.c_void_p((1 << 20) + 4), wsb=need) == 1  # misaligned workspace
    assert _extend_call(lib, stride=400) == 1                  # table narrower than max_extend_len
    assert _extend_call(lib, batch=0, ws=None, wsb=0) == 0     # empty batch: no-op, no workspace needed
    assert _extend_call(lib, total_q=0, ws=None, wsb=0) == 0


def test_extend_workspace_bounds_the_work_list(lib):
    # one (request, query tile) entry per 2 * 128 / G suffix tokens, plus one per request, 8 bytes each
    assert ra.ra_extend_workspace_bytes(4, 1000, 32, 8) == 16 + 8 * ((1000 + 63) // 64 + 4)
    assert ra.ra_extend_workspace_bytes(4, 1000, 64, 8) == 16 + 8 * ((1000 + 31) // 32 + 4)
    assert ra.ra_extend_workspace_bytes(4, 1000, 30, 8) == 0
    assert ra.ra_extend_workspace_bytes(0, 0, 32, 8) == 16


def test_kv_store_validation(lib):
    f = lib.ra_kv_store
    assert f(FAKE, FAKE, 16, 8, 128, FAKE, FAKE, FAKE, 0, None, None) == 0        # zero tokens: no-op
    assert f(FAKE, FAKE, 16, 8, 128, FAKE, FAKE, FAKE, -1, None, None) == 1
    assert f(FAKE, FAKE, 16, 1, 4, FAKE, FAKE, FAKE, 3, None, None) == 1         # 8-byte rows
    assert f(None, FAKE, 16, 8, 128, FAKE, FAKE, FAKE, 3, None, None) == 1
    assert f(ctypes.c_void_p((1 << 20) + 4), FAKE, 16, 8, 128, FAKE, FAKE, FAKE, 3, None, None) == 1


def test_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(ra, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        ra.load()


def test_store_decode_binding_checks_shapes_before_the_call():
    """The Python binding of the fused store + decode rejects new rows or slots of the wrong shape, and
    tensors of the wrong dtype, before anything reaches the library (CPU tensors: no launch)."""
    import torch
    pool = torch.zeros((64, 2, 64), dtype=torch.bfloat16)
    q = torch.zeros((3, 8, 64), dtype=torch.bfloat16)
    table = torch.zeros((3, 16), dtype=torch.int32)
    idx = torch.zeros(3, dtype=torch.int32)
    ws = torch.zeros(256, dtype=torch.uint8)
    args = dict(max_seq_len=16, sm_scale=0.125, workspace=ws)
    kn = torch.zeros((3, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # one new row per request
        ra.ra_decode_attention_store(pool, pool, kn[:2], kn[:2], idx[:2], q, q.clone(), table, idx, idx, **args)
    with pytest.raises(ValueError):  # out_cache_loc has one entry per request
        ra.ra_decode_attention_store(pool, pool, kn, kn, idx[:1], q, q.clone(), table, idx, idx, **args)
    with pytest.raises(TypeError):  # slots are int32
        ra.ra_decode_attention_store(pool, pool, kn, kn, idx.long(), q, q.clone(), table, idx, idx, **args)


def test_selftest_bounded_wait_validates_before_launch(lib):
    """Bad arguments are rejected on the host (nothing is launched, no GPU needed)."""
    assert lib.ra_selftest_bounded_wait(0, FAKE, None) == 1
    assert lib.ra_selftest_bounded_wait((1 << 32) + 1, FAKE, None) == 1
    assert lib.ra_selftest_bounded_wait(1000, None, None) == 1
    assert lib.ra_selftest_bounded_wait(1000, ctypes.c_void_p((1 << 20) + 2), None) == 1


def _decode_workspace_layout(batch, hq, d, csplits, levels=1):
    """The decode workspace's size from its layout: per-item partials, prefix partials, the integer block."""
    up = lambda x: (x + 255) & ~255
    max_items = 456 + batch
    total = up(max_items * hq * d * 4) + up(max_items * hq * 4)
    if csplits:
        slots = levels * csplits
        total += up(batch * hq * slots * d * 4) + up(batch * hq * slots * 4)
    return total + up((batch + 3) * 4 + (2 + batch + 1 + 2 * max_items + batch) * 4)


def test_decode_prefix_split_balances_short_private_tails(lib):
    """The prefix pass's split, seen through the workspace size (one partial slot per split): a batch whose
    contexts are one 8192-key prefix plus tails of at most 257 keys gets 1,280-key splits (7), balanced
    against the tails' decode on the SMs the pass leaves free; a batch with long private parts keeps the
    split that fills the pass's wave (one 1,024-key split of its 1,024-key prefix)."""
    assert ra.ra_decode_workspace_bytes(64, 64, 8, 128, 8449, 1, 8192, 64, 1) == \
        _decode_workspace_layout(64, 64, 128, csplits=7)
    assert ra.ra_decode_workspace_bytes(64, 32, 8, 128, 4096, 8, 1024, 8, 1) == \
        _decode_workspace_layout(64, 32, 128, csplits=1)
    assert ra.ra_decode_workspace_bytes(64, 32, 8, 128, 4096) == _decode_workspace_layout(64, 32, 128, csplits=0)
