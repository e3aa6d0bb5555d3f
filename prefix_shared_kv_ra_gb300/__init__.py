"""GB300 (sm_103a) RadixAttention hot path: KV store, extend and decode
attention over a token-granular KV pool shared through a radix-tree prefix
cache.

This module is the thin Python binding of ``libra.so`` (C ABI in
``include/ra.h``).  It only marshals arguments: it checks torch dtypes,
devices, shapes and contiguity, and passes raw device pointers and the
current CUDA stream to the library, where every step of the path runs in
hand-written CUDA kernels.  There is no fallback: if the library is missing
or fails to load, importing the binding raises.

Functions keep the C names: ``ra_kv_store``, ``ra_extend_attention``,
``ra_decode_attention``, ``ra_decode_workspace_bytes``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = ["RAError", "ra_kv_store", "ra_extend_attention", "ra_extend_workspace_bytes", "ra_decode_attention",
           "ra_decode_workspace_bytes", "ra_decode_attention_store",
           "ra_decode_attention_static", "RA_DECODE_STATIC_SCRATCH_BYTES",
           "ra_abi_version", "ra_selftest_bounded_wait", "library_path", "load", "DEVERR_SLOT", "DEVERR_TABLE", "DEVERR_LENGTH",
           "DEVERR_TIMEOUT"]

RA_OK = 0
RA_DECODE_STATIC_SCRATCH_BYTES = 32 << 20  # size of the library's static decode scratch (include/ra.h)
DEVERR_SLOT, DEVERR_TABLE, DEVERR_LENGTH, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
_lib = None


class RAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libra.so (building it first only if asked and it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise ImportError(f"{_build.LIB} is not built; run prefix_shared_kv_ra_gb300._build.build()")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.ra_kv_store.argtypes = [P, P, i64, i32, i32, P, P, P, i64, P, P]
    lib.ra_extend_attention.argtypes = [P, P, i64, i32, i32, P, P, i32, f32, P, i64, i64, P, P, P, P, i32, i64,
                                        i32, i32, P, sz, P, P]
    lib.ra_extend_workspace_bytes.argtypes = [i32, i64, i32, i32]
    lib.ra_extend_workspace_bytes.restype = sz
    lib.ra_decode_attention.argtypes = [P, P, i64, i32, i32, P, P, i32, f32, P, i64, i64, P, P, i32, i32, i32,
                                        P, P, P, P, P, i32, i32, i32, P, sz, P, P]
    lib.ra_decode_attention_store.argtypes = [P, P, i64, i32, i32, P, P, P, P, P, i32, f32, P, i64, i64, P, P, i32,
                                              i32, i32, P, P, P, P, P, i32, i32, i32, P, sz, P, P]
    lib.ra_decode_attention_store.restype = ctypes.c_int
    lib.ra_decode_attention_static.argtypes = [P, P, i64, i32, i32, P, P, i32, f32, P, i64, i64, P, P, i32, i32,
                                               i32, P, P, P, P, P, i32, i32, i32, P, P]
    lib.ra_decode_attention_static.restype = ctypes.c_int
    lib.ra_selftest_bounded_wait.argtypes = [i64, P, P]
    lib.ra_selftest_bounded_wait.restype = ctypes.c_int
    lib.ra_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.ra_decode_workspace_bytes.restype = sz
    for f in (lib.ra_kv_store, lib.ra_extend_attention, lib.ra_decode_attention, lib.ra_abi_version):
        f.restype = ctypes.c_int
    lib.ra_status_string.argtypes = [ctypes.c_int]
    lib.ra_status_string.restype = ctypes.c_char_p
    lib.ra_last_error_message.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != RA_OK:
        lib = load()
        msg = lib.ra_last_error_message().decode() or lib.ra_status_string(status).decode()
        raise RAError(status, msg)


def _ptr(t: Optional[torch.Tensor], dtype: torch.dtype, name: str, device: torch.device):
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device, stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def ra_selftest_bounded_wait(deadline_cycles: int, device_error: torch.Tensor, stream=None) -> None:
    """One kernel whose waits (an mbarrier nobody arrives at, a counter nobody raises) run out after
    deadline_cycles SM cycles: it must flag DEVERR_TIMEOUT in device_error (int32 [1] on the GPU) and
    return."""
    dev = device_error.device
    _check(load().ra_selftest_bounded_wait(int(deadline_cycles), _ptr(device_error, torch.int32, "device_error", dev),
                                           _stream(dev, stream)))


def ra_abi_version() -> int:
    return int(load().ra_abi_version())


def ra_kv_store(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                out_cache_loc: torch.Tensor, device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """pool[out_cache_loc[i]] = new[i] for K and V (bit copy).  Pools [S, Hkv, D] bf16."""
    dev = k_pool.device
    S, hkv, d = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape or tuple(k_new.shape[1:]) != (hkv, d):
        raise ValueError("shape mismatch between pools and new rows")
    if out_cache_loc.shape != (k_new.shape[0],):
        raise ValueError("out_cache_loc must be [num_tokens]")
    bf = torch.bfloat16
    _check(load().ra_kv_store(_ptr(k_pool, bf, "k_pool", dev), _ptr(v_pool, bf, "v_pool", dev), S, hkv, d,
                              _ptr(k_new, bf, "k_new", dev), _ptr(v_new, bf, "v_new", dev),
                              _ptr(out_cache_loc, torch.int32, "out_cache_loc", dev), k_new.shape[0],
                              _ptr(device_error, torch.int32, "device_error", dev), _stream(dev, stream)))


def ra_extend_attention(k_pool: torch.Tensor, v_pool: torch.Tensor, q: torch.Tensor, o: torch.Tensor,
                        req_to_token: torch.Tensor, req_pool_indices: torch.Tensor, prefix_lens: torch.Tensor,
                        extend_lens: torch.Tensor, qo_indptr: torch.Tensor, *, max_extend_len: int,
                        max_prefix_len: int, sm_scale: float, workspace: torch.Tensor,
                        device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Suffix queries over cached prefix + causal suffix; q, o [total_q, Hq, D] bf16; workspace: uint8,
    at least ra_extend_workspace_bytes(batch, total_q, Hq, Hkv) bytes."""
    dev = k_pool.device
    S, hkv, d = k_pool.shape
    total_q, hq, dq = q.shape
    if dq != d or o.shape != q.shape:
        raise ValueError("q/o shape mismatch")
    batch = req_pool_indices.shape[0]
    bf, i32 = torch.bfloat16, torch.int32
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.device != dev:
        raise ValueError("workspace must be a contiguous uint8 tensor on the pool's device")
    _check(load().ra_extend_attention(
        _ptr(k_pool, bf, "k_pool", dev), _ptr(v_pool, bf, "v_pool", dev), S, hkv, d, _ptr(q, bf, "q", dev),
        _ptr(o, bf, "o", dev), hq, float(sm_scale), _ptr(req_to_token, i32, "req_to_token", dev),
        req_to_token.shape[1], req_to_token.shape[0], _ptr(req_pool_indices, i32, "req_pool_indices", dev),
        _ptr(prefix_lens, i32, "prefix_lens", dev), _ptr(extend_lens, i32, "extend_lens", dev),
        _ptr(qo_indptr, i32, "qo_indptr", dev), batch, total_q, int(max_extend_len), int(max_prefix_len),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _ptr(device_error, i32, "device_error", dev),
        _stream(dev, stream)))


def ra_extend_workspace_bytes(batch: int, total_q: int, num_q_heads: int, num_kv_heads: int) -> int:
    return int(load().ra_extend_workspace_bytes(batch, total_q, num_q_heads, num_kv_heads))


def ra_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_seq_len: int,
                              num_groups: int = 0, max_group_prefix_len: int = 0, max_group_size: int = 0,
                              max_group_levels: int = 1) -> int:
    return int(load().ra_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                                num_groups, max_group_prefix_len, max_group_size, max_group_levels))


def ra_decode_attention(k_pool: torch.Tensor, v_pool: torch.Tensor, q: torch.Tensor, o: torch.Tensor,
                        req_to_token: torch.Tensor, req_pool_indices: torch.Tensor, seq_lens: torch.Tensor, *,
                        max_seq_len: int, sm_scale: float, workspace: torch.Tensor,
                        group_indptr: Optional[torch.Tensor] = None, group_reqs: Optional[torch.Tensor] = None,
                        group_prefix_len: Optional[torch.Tensor] = None, max_group_prefix_len: int = 0,
                        max_group_size: int = 0, group_prefix_start: Optional[torch.Tensor] = None,
                        group_level: Optional[torch.Tensor] = None, max_group_levels: int = 1,
                        device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """One query per request over its context; q, o [batch, Hq, D] bf16; optional cascade groups (group g
    covers positions group_prefix_start[g] .. group_prefix_len[g]-1 of its members, at group_level[g])."""
    dev = k_pool.device
    S, hkv, d = k_pool.shape
    batch, hq, dq = q.shape
    if dq != d or o.shape != q.shape:
        raise ValueError("q/o shape mismatch")
    bf, i32 = torch.bfloat16, torch.int32
    ng = 0 if group_indptr is None else group_indptr.shape[0] - 1
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.device != dev:
        raise ValueError("workspace must be a contiguous uint8 tensor on the pool's device")
    _check(load().ra_decode_attention(
        _ptr(k_pool, bf, "k_pool", dev), _ptr(v_pool, bf, "v_pool", dev), S, hkv, d, _ptr(q, bf, "q", dev),
        _ptr(o, bf, "o", dev), hq, float(sm_scale), _ptr(req_to_token, i32, "req_to_token", dev),
        req_to_token.shape[1], req_to_token.shape[0], _ptr(req_pool_indices, i32, "req_pool_indices", dev),
        _ptr(seq_lens, i32, "seq_lens", dev), batch, int(max_seq_len), ng,
        _ptr(group_indptr, i32, "group_indptr", dev), _ptr(group_reqs, i32, "group_reqs", dev),
        _ptr(group_prefix_start, i32, "group_prefix_start", dev), _ptr(group_prefix_len, i32, "group_prefix_len", dev),
        _ptr(group_level, i32, "group_level", dev), int(max_group_prefix_len), int(max_group_size),
        int(max_group_levels), ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
        _ptr(device_error, i32, "device_error", dev), _stream(dev, stream)))


def ra_decode_attention_store(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                              out_cache_loc: torch.Tensor, q: torch.Tensor, o: torch.Tensor,
                              req_to_token: torch.Tensor, req_pool_indices: torch.Tensor, seq_lens: torch.Tensor, *,
                              max_seq_len: int, sm_scale: float, workspace: torch.Tensor,
                              group_indptr: Optional[torch.Tensor] = None, group_reqs: Optional[torch.Tensor] = None,
                              group_prefix_len: Optional[torch.Tensor] = None, max_group_prefix_len: int = 0,
                              max_group_size: int = 0, group_prefix_start: Optional[torch.Tensor] = None,
                              group_level: Optional[torch.Tensor] = None, max_group_levels: int = 1,
                              device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """The decode step's store and attention in one call: pool[out_cache_loc[b]] = k_new[b] / v_new[b]
    ([batch, Hkv, D] bf16), then ra_decode_attention (same arguments and result)."""
    dev = k_pool.device
    S, hkv, d = k_pool.shape
    batch, hq, dq = q.shape
    if dq != d or o.shape != q.shape:
        raise ValueError("q/o shape mismatch")
    if k_new.shape != (batch, hkv, d) or v_new.shape != k_new.shape or out_cache_loc.shape != (batch,):
        raise ValueError("k_new / v_new must be [batch, Hkv, D] and out_cache_loc [batch]")
    bf, i32 = torch.bfloat16, torch.int32
    ng = 0 if group_indptr is None else group_indptr.shape[0] - 1
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.device != dev:
        raise ValueError("workspace must be a contiguous uint8 tensor on the pool's device")
    _check(load().ra_decode_attention_store(
        _ptr(k_pool, bf, "k_pool", dev), _ptr(v_pool, bf, "v_pool", dev), S, hkv, d, _ptr(k_new, bf, "k_new", dev),
        _ptr(v_new, bf, "v_new", dev), _ptr(out_cache_loc, i32, "out_cache_loc", dev), _ptr(q, bf, "q", dev),
        _ptr(o, bf, "o", dev), hq, float(sm_scale), _ptr(req_to_token, i32, "req_to_token", dev),
        req_to_token.shape[1], req_to_token.shape[0], _ptr(req_pool_indices, i32, "req_pool_indices", dev),
        _ptr(seq_lens, i32, "seq_lens", dev), batch, int(max_seq_len), ng,
        _ptr(group_indptr, i32, "group_indptr", dev), _ptr(group_reqs, i32, "group_reqs", dev),
        _ptr(group_prefix_start, i32, "group_prefix_start", dev), _ptr(group_prefix_len, i32, "group_prefix_len", dev),
        _ptr(group_level, i32, "group_level", dev), int(max_group_prefix_len), int(max_group_size),
        int(max_group_levels), ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
        _ptr(device_error, i32, "device_error", dev), _stream(dev, stream)))


def ra_decode_attention_static(k_pool: torch.Tensor, v_pool: torch.Tensor, q: torch.Tensor, o: torch.Tensor,
                               req_to_token: torch.Tensor, req_pool_indices: torch.Tensor, seq_lens: torch.Tensor, *,
                               max_seq_len: int, sm_scale: float, group_indptr: Optional[torch.Tensor] = None,
                               group_reqs: Optional[torch.Tensor] = None,
                               group_prefix_len: Optional[torch.Tensor] = None, max_group_prefix_len: int = 0,
                               max_group_size: int = 0, group_prefix_start: Optional[torch.Tensor] = None,
                               group_level: Optional[torch.Tensor] = None, max_group_levels: int = 1,
                               device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """ra_decode_attention without a workspace argument, for callers that cannot allocate:
    the library's static device scratch (RA_DECODE_STATIC_SCRATCH_BYTES) is used instead."""
    dev = k_pool.device
    S, hkv, d = k_pool.shape
    batch, hq, dq = q.shape
    if dq != d or o.shape != q.shape:
        raise ValueError("q/o shape mismatch")
    bf, i32 = torch.bfloat16, torch.int32
    ng = 0 if group_indptr is None else group_indptr.shape[0] - 1
    # the library resolves its static scratch on the CURRENT device: make it the tensors' device
    with torch.cuda.device(dev):
        _check(load().ra_decode_attention_static(
            _ptr(k_pool, bf, "k_pool", dev), _ptr(v_pool, bf, "v_pool", dev), S, hkv, d, _ptr(q, bf, "q", dev),
            _ptr(o, bf, "o", dev), hq, float(sm_scale), _ptr(req_to_token, i32, "req_to_token", dev),
            req_to_token.shape[1], req_to_token.shape[0], _ptr(req_pool_indices, i32, "req_pool_indices", dev),
            _ptr(seq_lens, i32, "seq_lens", dev), batch, int(max_seq_len), ng,
            _ptr(group_indptr, i32, "group_indptr", dev), _ptr(group_reqs, i32, "group_reqs", dev),
            _ptr(group_prefix_start, i32, "group_prefix_start", dev),
            _ptr(group_prefix_len, i32, "group_prefix_len", dev), _ptr(group_level, i32, "group_level", dev),
            int(max_group_prefix_len), int(max_group_size), int(max_group_levels),
            _ptr(device_error, i32, "device_error", dev), _stream(dev, stream)))
