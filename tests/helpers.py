"""Shared helpers for the GPU parity tests: move a generator batch to the
device, run the hot path through the Python binding, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import prefix_shared_kv_ra_gb300 as ra
import workloads as W

ATOL = 1e-2
RTOL = 1e-2


def bf16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def i32(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DeviceBatch:
    """A generator batch resident on the GPU (pool before the store)."""

    def __init__(self, b: W.Batch, dev="cuda:0"):
        self.b = b
        self.dev = torch.device(dev)
        S, hkv, d = b.num_slots, b.num_kv_heads, b.head_dim
        self.k_pool = torch.zeros((S, hkv, d), dtype=torch.bfloat16, device=self.dev)
        self.v_pool = torch.zeros((S, hkv, d), dtype=torch.bfloat16, device=self.dev)
        if b.pool_slots.size:
            idx = torch.from_numpy(b.pool_slots.astype(np.int64)).to(self.dev)
            self.k_pool.index_copy_(0, idx, bf16(b.pool_k, self.dev))
            self.v_pool.index_copy_(0, idx, bf16(b.pool_v, self.dev))
        self.k_new = bf16(b.k_new, self.dev)
        self.v_new = bf16(b.v_new, self.dev)
        self.loc = i32(b.out_cache_loc, self.dev)
        self.table = i32(b.req_to_token, self.dev)
        self.ext_q = bf16(b.ext_q, self.dev)
        self.ext_rpi = i32(b.ext_rpi, self.dev)
        self.ext_prefix = i32(b.ext_prefix_lens, self.dev)
        self.ext_len = i32(b.ext_extend_lens, self.dev)
        self.ext_qo = i32(b.ext_qo_indptr, self.dev)
        self.dec_q = bf16(b.dec_q, self.dev)
        self.dec_rpi = i32(b.dec_rpi, self.dev)
        self.dec_lens = i32(b.dec_seq_lens, self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        if b.has_cascade():
            self.g_indptr = i32(b.casc_group_indptr, self.dev)
            self.g_reqs = i32(b.casc_group_reqs, self.dev)
            self.g_plen = i32(b.casc_group_prefix_len, self.dev)
            self.g_start = None if b.casc_group_start is None else i32(b.casc_group_start, self.dev)
            self.g_level = None if b.casc_group_level is None else i32(b.casc_group_level, self.dev)
        self.ext_o = torch.empty_like(self.ext_q)
        self.dec_o = torch.empty_like(self.dec_q)
        self.ws = torch.empty(0, dtype=torch.uint8, device=self.dev)

    # -- the three calls
    def store(self):
        ra.ra_kv_store(self.k_pool, self.v_pool, self.k_new, self.v_new, self.loc, device_error=self.err)

    def extend(self):
        b = self.b
        if b.n_extend == 0:
            return
        ws = torch.empty(ra.ra_extend_workspace_bytes(b.n_extend, b.total_q_extend, b.num_q_heads, b.num_kv_heads),
                         dtype=torch.uint8, device=self.dev)
        ra.ra_extend_attention(self.k_pool, self.v_pool, self.ext_q, self.ext_o, self.table, self.ext_rpi,
                               self.ext_prefix, self.ext_len, self.ext_qo, max_extend_len=b.max_extend_len,
                               max_prefix_len=b.max_prefix_len, sm_scale=b.sm_scale, workspace=ws,
                               device_error=self.err)

    def decode_ws(self, cascade: bool) -> torch.Tensor:
        b = self.b
        ng, mp, ms = 0, 0, 0
        if cascade:
            ng = b.casc_group_indptr.size - 1
            mp = int(b.casc_group_prefix_len.max())
            ms = int(np.diff(b.casc_group_indptr).max())
        n = ra.ra_decode_workspace_bytes(b.n_decode, b.num_q_heads, b.num_kv_heads, b.head_dim, b.max_seq_len,
                                         ng, mp, ms, b.casc_levels if cascade else 1)
        if self.ws.numel() < n:
            self.ws = torch.empty(n, dtype=torch.uint8, device=self.dev)
        return self.ws

    def decode(self, cascade: bool = False):
        b = self.b
        if b.n_decode == 0:
            return
        ws = self.decode_ws(cascade)
        kw = {}
        if cascade:
            kw = dict(group_indptr=self.g_indptr, group_reqs=self.g_reqs, group_prefix_len=self.g_plen,
                      max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                      max_group_size=int(np.diff(b.casc_group_indptr).max()), group_prefix_start=self.g_start,
                      group_level=self.g_level, max_group_levels=b.casc_levels)
        ra.ra_decode_attention(self.k_pool, self.v_pool, self.dec_q, self.dec_o, self.table, self.dec_rpi,
                               self.dec_lens, max_seq_len=b.max_seq_len, sm_scale=b.sm_scale, workspace=ws,
                               device_error=self.err, **kw)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside 1e-2 + 1e-2|ref| "
                             f"(max err {err.max():.3e}; first at {tuple(i)}: got {got[tuple(i)]}, "
                             f"ref {ref[tuple(i)]})")


def check_store(db: DeviceBatch):
    """Run the store and check the whole pool (K and V) bit for bit against the pool before the store with
    the oracle's rows at out_cache_loc."""
    b = db.b
    before_k, before_v = db.k_pool.clone(), db.v_pool.clone()
    db.store()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    # the oracle's store over the slots it writes (rows relabelled 0..N-1: the store commutes with that)
    loc = b.out_cache_loc.astype(np.int64)
    idx = torch.from_numpy(loc).to(db.dev)
    rows_k = before_k.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    rows_v = before_v.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    exp_k, exp_v = oracle.kv_store(rows_k, rows_v, b.k_new, b.v_new, np.arange(loc.size, dtype=np.int32))
    for before, exp, got in ((before_k, exp_k, db.k_pool), (before_v, exp_v, db.v_pool)):
        before.index_copy_(0, idx, torch.from_numpy(exp.view(np.int16)).to(db.dev).view(torch.bfloat16))
        assert torch.equal(before.view(torch.int16), got.view(torch.int16))


def attach_tree_groups(b: W.Batch, min_prefix: int = 256) -> W.Batch:
    """Give a decode batch the one-level cascade groups the radix tree derives from its table rows."""
    from prefix_shared_kv_ra_gb300.radix import cascade_groups
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    b.casc_group_indptr, b.casc_group_reqs, b.casc_group_prefix_len = cascade_groups(rows, min_prefix=min_prefix)
    return b


def grow_key_scale(b: W.Batch, per_tile: float = 6.0, tile: int = 128) -> W.Batch:
    """Scale every key by 1 + per_tile * (its context position // tile), in place: scores then grow from
    one 128-key tile to the next by far more than any lazy softmax reference allows, so kernels that
    exponentiate against a running reference must move it (and rescale O) on every tile."""
    return scale_keys(b, lambda p: 1.0 + per_tile * (p // tile))


def late_half_key_scale(b: W.Batch, per_tile: float = 20.0) -> W.Batch:
    """Scale the keys at positions 64..127 of every 128-position tile by 1 + per_tile * (tile + 1) and
    leave the others, in place.  A key tile's first 64 scores then stay within the reference of the
    tile before while its last 64 exceed it by far: a kernel that hands out the first half's
    probabilities before it has seen the second half must move the reference (and rescale O) between
    the two halves of every tile."""
    return scale_keys(b, lambda p: 1.0 + per_tile * (p // 128 + 1) if p % 128 >= 64 else 1.0)


def scale_keys(b: W.Batch, factor) -> W.Batch:
    """Multiply every key of the pool and of the new rows by factor(its context position), in place."""
    pos = {}
    rows = [(r, int(n)) for r, n in zip(b.ext_rpi, b.ext_prefix_lens + b.ext_extend_lens)] + \
           [(r, int(n)) for r, n in zip(b.dec_rpi, b.dec_seq_lens)]
    for r, n in rows:
        for p, s in enumerate(b.req_to_token[r, :n].tolist()):
            pos[s] = p

    def scaled(bits: np.ndarray, slots: np.ndarray) -> np.ndarray:
        f = np.array([factor(pos.get(int(s), 0)) for s in slots], dtype=np.float32)
        x = W.bf16_bits_to_f32(bits) * f[:, None, None]
        return W.f32_to_bf16_bits(x)

    b.pool_k = scaled(b.pool_k, b.pool_slots)
    b.k_new = scaled(b.k_new, b.out_cache_loc)
    return b


def prefill_chunks(b: W.Batch, chunk: int):
    """Chunked prefill of an extend batch: call k extends every request by its k-th chunk of at most
    `chunk` suffix tokens, with all earlier chunks as cached prefix.  Yields, per call, (q rows,
    prefix_lens, extend_lens, qo_indptr, token index of each row in the unchunked batch)."""
    P, E, qo = b.ext_prefix_lens, b.ext_extend_lens, b.ext_qo_indptr
    n_calls = int(-(-E.max() // chunk))
    for k in range(n_calls):
        done = np.minimum(k * chunk, E)
        ext = np.minimum(chunk, E - done).astype(np.int32)
        toks = np.concatenate([qo[i] + done[i] + np.arange(ext[i]) for i in range(E.size)]).astype(np.int64)
        yield (b.ext_q[toks], (P + done).astype(np.int32), ext,
               np.concatenate([[0], np.cumsum(ext)]).astype(np.int32), toks)


def attach_tree_groups_multilevel(b: W.Batch) -> W.Batch:
    """Give a decode batch the multi-level cascade groups of its table rows' tree (one per shared node)."""
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    (b.casc_group_indptr, b.casc_group_reqs, b.casc_group_start, b.casc_group_prefix_len, b.casc_group_level,
     b.casc_levels) = cascade_groups_multilevel(rows)
    return b
