"""CPU oracle for the RadixAttention hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
library never does; the two share no code.  The arithmetic lives in
``ra_oracle.c`` (plain C, fp64, OpenMP over query rows), the hit-ratio
definitions in ``hit_ratio.py`` and an independent pure-Python restatement
for tiny inputs in ``brute.py``.

This module builds ``ra_oracle.c`` with gcc and wraps it with ctypes.
Inputs are numpy arrays; bf16 values are passed as raw uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ra_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ra_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.ora_kv_store.argtypes = [P, P, i64, i64, P, P, P, i64]
        lib.ora_extend.argtypes = [P, P, P, i64, i32, i32, P, i32, P, i64, i64, P, P, P, P, i32, f64, P, i64, P]
        lib.ora_decode.argtypes = [P, P, P, i64, i32, i32, P, i32, P, i64, i64, P, P, i32, f64, P, i64, P]
        for f in (lib.ora_kv_store, lib.ora_extend, lib.ora_decode, lib.ora_num_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().ora_num_threads())


def _p(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------
# KV store (definition: pool' = pool with rows at loc replaced)
# ----------------------------------------------------------------------------
def kv_store(pool_k: np.ndarray, pool_v: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
             loc: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Return copies of the dense [S, Hkv, D] uint16 pools after the store."""
    pk = np.array(pool_k, dtype=np.uint16, copy=True, order="C")
    pv = np.array(pool_v, dtype=np.uint16, copy=True, order="C")
    kn, vn, lc = _c(k_new, np.uint16), _c(v_new, np.uint16), _c(loc, np.int32)
    row = int(np.prod(pk.shape[1:]))
    rc = _load().ora_kv_store(_p(pk), _p(pv), pk.shape[0], row, _p(kn), _p(vn), _p(lc), lc.size)
    if rc != 0:
        raise ValueError("oracle kv_store: slot out of range")
    return pk, pv


# ----------------------------------------------------------------------------
# attention over a compact pool
# ----------------------------------------------------------------------------
class CompactPool:
    """Rows in use of a [S, Hkv, D] pool plus the slot -> row map."""

    def __init__(self, num_slots: int, slots: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray):
        self.num_slots = int(num_slots)
        self.k = _c(k_rows, np.uint16)
        self.v = _c(v_rows, np.uint16)
        self.slot_row = np.full(self.num_slots, -1, np.int64)
        self.slot_row[np.asarray(slots, np.int64)] = np.arange(len(slots), dtype=np.int64)
        self.hkv, self.d = int(self.k.shape[1]), int(self.k.shape[2])


def pool_after_store(batch) -> CompactPool:
    """Pool of a generator batch once its new tokens are stored (later rows win)."""
    slots = np.concatenate([batch.pool_slots.astype(np.int64), batch.out_cache_loc.astype(np.int64)])
    k = np.concatenate([batch.pool_k, batch.k_new])
    v = np.concatenate([batch.pool_v, batch.v_new])
    return CompactPool(batch.num_slots, slots, k, v)


def extend(pool: CompactPool, q: np.ndarray, req_to_token: np.ndarray, rpi: np.ndarray,
           prefix_lens: np.ndarray, extend_lens: np.ndarray, qo_indptr: np.ndarray, scale: float,
           sel: Optional[np.ndarray] = None) -> np.ndarray:
    """fp64 extend attention; returns [n, D] (rows sel = t * Hq + h, default all)."""
    q = _c(q, np.uint16)
    hq = int(q.shape[1])
    tab = _c(req_to_token, np.int32)
    rpi, pl, el, qo = (_c(x, np.int32) for x in (rpi, prefix_lens, extend_lens, qo_indptr))
    sel_a = None if sel is None else _c(sel, np.int64)
    n = int(qo[-1]) * hq if sel_a is None else sel_a.size
    out = np.zeros((n, pool.d), np.float64)
    rc = _load().ora_extend(_p(pool.k), _p(pool.v), _p(pool.slot_row), pool.num_slots, pool.hkv, pool.d,
                            _p(q), hq, _p(tab), tab.shape[1], tab.shape[0], _p(rpi), _p(pl), _p(el), _p(qo),
                            rpi.size, float(scale), _p(sel_a), 0 if sel_a is None else sel_a.size, _p(out))
    if rc != 0:
        raise ValueError(f"oracle extend failed ({rc})")
    return out


def decode(pool: CompactPool, q: np.ndarray, req_to_token: np.ndarray, rpi: np.ndarray,
           seq_lens: np.ndarray, scale: float, sel: Optional[np.ndarray] = None) -> np.ndarray:
    """fp64 decode attention; returns [n, D] (rows sel = b * Hq + h, default all)."""
    q = _c(q, np.uint16)
    hq = int(q.shape[1])
    tab = _c(req_to_token, np.int32)
    rpi, sl = _c(rpi, np.int32), _c(seq_lens, np.int32)
    sel_a = None if sel is None else _c(sel, np.int64)
    n = rpi.size * hq if sel_a is None else sel_a.size
    out = np.zeros((n, pool.d), np.float64)
    rc = _load().ora_decode(_p(pool.k), _p(pool.v), _p(pool.slot_row), pool.num_slots, pool.hkv, pool.d,
                            _p(q), hq, _p(tab), tab.shape[1], tab.shape[0], _p(rpi), _p(sl), rpi.size,
                            float(scale), _p(sel_a), 0 if sel_a is None else sel_a.size, _p(out))
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out


def extend_batch(batch, sel: Optional[np.ndarray] = None, pool: Optional[CompactPool] = None) -> np.ndarray:
    pool = pool or pool_after_store(batch)
    return extend(pool, batch.ext_q, batch.req_to_token, batch.ext_rpi, batch.ext_prefix_lens,
                  batch.ext_extend_lens, batch.ext_qo_indptr, batch.sm_scale, sel)


def decode_batch(batch, sel: Optional[np.ndarray] = None, pool: Optional[CompactPool] = None) -> np.ndarray:
    pool = pool or pool_after_store(batch)
    return decode(pool, batch.dec_q, batch.req_to_token, batch.dec_rpi, batch.dec_seq_lens, batch.sm_scale, sel)
