"""Second, independent restatement of attention over a slot pool -- TEST
INFRASTRUCTURE ONLY, for tiny inputs (pure-Python loops, Python floats).

It shares nothing with ``ra_oracle.c``: it keeps the pool as a dict from slot
id to its K/V rows, walks each request's context position by position through
the request's table row, and evaluates softmax attention with ``math.exp``.
Its only job is to pin the C oracle (agreement to ~1e-12 on tiny cases).
Definition followed: SGLang paper summary, §3 "Efficient KV Cache Reuse with
RadixAttention" (a request reuses the KV of its cached prefix; the result is
ordinary attention over its whole context).
"""
from __future__ import annotations

import math
import struct
from typing import Dict, List, Tuple


def _bf16(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def _pool_dict(batch) -> Dict[int, Tuple[list, list]]:
    pool: Dict[int, Tuple[list, list]] = {}
    for i, s in enumerate(batch.pool_slots.tolist()):
        pool[s] = (batch.pool_k[i].tolist(), batch.pool_v[i].tolist())
    for i, s in enumerate(batch.out_cache_loc.tolist()):   # this step's store
        pool[s] = (batch.k_new[i].tolist(), batch.v_new[i].tolist())
    return pool


def _attend(qrow: List[int], ctx_slots: List[int], pool, kv_head: int, scale: float) -> List[float]:
    q = [_bf16(x) for x in qrow]
    scores = []
    for s in ctx_slots:
        k = [_bf16(x) for x in pool[s][0][kv_head]]
        scores.append(scale * sum(a * b for a, b in zip(q, k)))
    top = max(scores)
    e = [math.exp(x - top) for x in scores]
    z = sum(e)
    out = [0.0] * len(q)
    for w, s in zip(e, ctx_slots):
        v = [_bf16(x) for x in pool[s][1][kv_head]]
        for c in range(len(q)):
            out[c] += (w / z) * v[c]
    return out


def extend(batch) -> List[List[float]]:
    """Rows in (token, head) order, like the C oracle's default."""
    pool = _pool_dict(batch)
    hq, hkv = batch.num_q_heads, batch.num_kv_heads
    out = []
    for b in range(batch.n_extend):
        row = batch.req_to_token[batch.ext_rpi[b]].tolist()
        p = int(batch.ext_prefix_lens[b])
        for i in range(int(batch.ext_extend_lens[b])):
            t = int(batch.ext_qo_indptr[b]) + i
            ctx = row[:p + i + 1]
            for h in range(hq):
                out.append(_attend(batch.ext_q[t, h].tolist(), ctx, pool, h // (hq // hkv), batch.sm_scale))
    return out


def decode(batch) -> List[List[float]]:
    pool = _pool_dict(batch)
    hq, hkv = batch.num_q_heads, batch.num_kv_heads
    out = []
    for b in range(batch.n_decode):
        ctx = batch.req_to_token[batch.dec_rpi[b]].tolist()[:int(batch.dec_seq_lens[b])]
        for h in range(hq):
            out.append(_attend(batch.dec_q[b, h].tolist(), ctx, pool, h // (hq // hkv), batch.sm_scale))
    return out
