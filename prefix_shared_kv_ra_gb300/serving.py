"""Host driver of the hot path over many steps: the radix-tree prefix cache over the slot pool
feeding the three calls, with a CUDA-graph decode.

Per step (SGLang paper summary, §3 "Efficient KV Cache Reuse with RadixAttention"; yaopepe.com
explainer, §04; anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一):

* admission: each arriving request matches its prompt against the tree and locks the matched
  path; it is admitted if the free slots plus the tokens the tree could evict, less the decode
  tokens the running requests still need, cover its suffix and output (else it waits); it then
  takes a table row and fresh slots for the unmatched suffix (evicting unreferenced leaves, least
  recently used first, when the pool runs short);
* ra_kv_store + ra_extend_attention for the admitted suffixes;
* one decode token for every request past its prefill: a fresh slot each, then ra_kv_store +
  ra_decode_attention replayed from a CUDA graph captured per padded batch size (padding rows
  read and write the dummy slot 0, as the pages' CUDA-graph decode does);
* completion: a finished turn is inserted into the tree (slots of positions another request
  inserted meanwhile are freed), unlocked, and its row released.

The driver times the host work spent in the tree (match, lock, insert, evict) against the step's
wall time; the attention values are synthetic (this drives the data path, not a model).
"""
from __future__ import annotations

import time
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import (ra_decode_attention, ra_decode_workspace_bytes, ra_extend_attention, ra_extend_workspace_bytes,
               ra_kv_store)
from .radix import RadixCache, SlotPool

__all__ = ["ServingReplay", "Request", "multiturn_chat", "run_chat"]


@dataclass
class Request:
    rid: int
    prompt: np.ndarray        # int32 token ids
    out_len: int              # tokens to generate
    slots: np.ndarray         # slots of the positions so far
    row: int                  # req_to_token row
    node: object              # locked tree node (end of the matched prefix)
    cached: int               # prompt tokens served from the cache
    generated: List[int] = field(default_factory=list)


class ServingReplay:
    def __init__(self, *, num_slots: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_len: int,
                 max_running: int, device, seed: int = 0, graph_sizes: Sequence[int] = (8, 16, 32, 64, 128, 256),
                 use_graphs: bool = True):
        self.dev = torch.device(device)
        self.hq, self.hkv, self.d = num_q_heads, num_kv_heads, head_dim
        self.max_len, self.max_running = max_len, max_running
        self.pool = SlotPool(num_slots)
        self.cache = RadixCache(self.pool)
        bf = torch.bfloat16
        self.k_pool = torch.zeros((num_slots, num_kv_heads, head_dim), dtype=bf, device=self.dev)
        self.v_pool = torch.zeros_like(self.k_pool)
        # rows 0 .. max_running-1 for requests; the last row is the padding row (slot 0 everywhere)
        self.table = torch.zeros((max_running + 1, max_len), dtype=torch.int32, device=self.dev)
        self.pad_row = max_running
        self.free_rows = list(range(max_running - 1, -1, -1))
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.gen = torch.Generator(device=self.dev).manual_seed(seed)
        self.rng = np.random.default_rng(seed)
        self.scale = float(head_dim) ** -0.5
        self.running: Dict[int, Request] = {}
        self.prefilled: List[int] = []   # rids past their prefill, in admission order
        self.finished: List[Request] = []
        self.use_graphs = use_graphs
        self.graph_sizes = sorted(graph_sizes)
        self._graphs: Dict[int, tuple] = {}
        self.stats = dict(steps=0, extend_tokens=0, decode_tokens=0, prompt_tokens=0, cached_tokens=0,
                          tree_s=0.0, gpu_ms=0.0, wall_s=0.0, evicted=0)
        self._next_token = 1 << 24       # generated token ids never collide with prompt ids below 2^24
        self.tags: Dict[int, object] = {}  # caller's label per request id

    # ------------------------------------------------------------------ slots
    def _alloc(self, n: int) -> np.ndarray:
        if n == 0:
            return np.zeros(0, np.int32)
        s = self.pool.alloc(n)
        if s is None:
            t0 = time.perf_counter()
            self.stats["evicted"] += self.cache.evict(n - self.pool.available())
            self.stats["tree_s"] += time.perf_counter() - t0
            s = self.pool.alloc(n)
            if s is None:
                raise RuntimeError(f"pool exhausted: {n} slots wanted, {self.pool.available()} free after eviction")
        return s

    def _randn(self, shape) -> torch.Tensor:
        return torch.randn(shape, generator=self.gen, device=self.dev).to(torch.bfloat16)

    def _i32(self, a) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(self.dev, non_blocking=True)

    # ------------------------------------------------------------------ decode graphs
    def _graph(self, bs: int):
        if bs in self._graphs:
            return self._graphs[bs]
        bf = torch.bfloat16
        buf = dict(q=torch.zeros((bs, self.hq, self.d), dtype=bf, device=self.dev),
                   k_new=torch.zeros((bs, self.hkv, self.d), dtype=bf, device=self.dev),
                   v_new=torch.zeros((bs, self.hkv, self.d), dtype=bf, device=self.dev),
                   loc=torch.zeros(bs, dtype=torch.int32, device=self.dev),
                   rpi=torch.full((bs,), self.pad_row, dtype=torch.int32, device=self.dev),
                   lens=torch.ones(bs, dtype=torch.int32, device=self.dev))
        buf["o"] = torch.empty_like(buf["q"])
        buf["ws"] = torch.empty(ra_decode_workspace_bytes(bs, self.hq, self.hkv, self.d, self.max_len),
                                dtype=torch.uint8, device=self.dev)

        def run():
            ra_kv_store(self.k_pool, self.v_pool, buf["k_new"], buf["v_new"], buf["loc"], device_error=self.err)
            ra_decode_attention(self.k_pool, self.v_pool, buf["q"], buf["o"], self.table, buf["rpi"], buf["lens"],
                                max_seq_len=self.max_len, sm_scale=self.scale, workspace=buf["ws"],
                                device_error=self.err)
        g = None
        if self.use_graphs:
            run()  # first-call set-up outside the capture
            torch.cuda.synchronize(self.dev)
            stream = torch.cuda.Stream(self.dev)
            stream.wait_stream(torch.cuda.current_stream(self.dev))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    run()
            torch.cuda.current_stream(self.dev).wait_stream(stream)
            torch.cuda.synchronize(self.dev)
        self._graphs[bs] = (g, buf, run)
        return self._graphs[bs]

    # ------------------------------------------------------------------ one step
    def step(self, arrivals: Sequence[Tuple[int, np.ndarray, int]]) -> Dict[str, float]:
        """Admit `arrivals` (rid, prompt tokens, tokens to generate), prefill them, decode one token for
        every request past its prefill, retire finished turns."""
        wall0 = time.perf_counter()
        tree = 0.0
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # ---- admission
        admitted: List[Request] = []
        deferred = []
        reserved = sum(r.out_len - len(r.generated) for r in self.running.values())
        for rid, prompt, out_len in arrivals:
            prompt = np.asarray(prompt, dtype=np.int32)
            if len(prompt) + out_len > self.max_len:
                raise ValueError(f"request {rid}: {len(prompt)} + {out_len} tokens exceed max_len {self.max_len}")
            if not self.free_rows:
                deferred.append((rid, prompt, out_len))
                continue
            t0 = time.perf_counter()
            hit, node = self.cache.match_prefix(prompt)
            self.cache.lock(node)
            hit = hit[:len(prompt) - 1]  # at least one token is prefilled (its query yields the first output)
            need = len(prompt) - hit.size + out_len
            fits = self.pool.available() + self.cache.evictable_size - reserved >= need
            if not fits:
                self.cache.unlock(node)
            tree += time.perf_counter() - t0
            if not fits:
                if not self.running and not admitted:
                    raise RuntimeError(f"request {rid} needs {need} slots; the pool cannot supply them")
                deferred.append((rid, prompt, out_len))
                continue
            reserved += out_len
            slots = np.concatenate([hit, self._alloc(len(prompt) - hit.size)]).astype(np.int32)
            row = self.free_rows.pop()
            self.table[row, :slots.size] = self._i32(slots)
            req = Request(rid, prompt, out_len, slots, row, node, int(hit.size))
            self.running[rid] = req
            admitted.append(req)
            self.stats["prompt_tokens"] += len(prompt)
            self.stats["cached_tokens"] += int(hit.size)
        ev0.record()
        # ---- prefill of the admitted suffixes
        if admitted:
            ext = np.array([len(r.prompt) - r.cached for r in admitted], np.int32)
            pre = np.array([r.cached for r in admitted], np.int32)
            total = int(ext.sum())
            loc = np.concatenate([r.slots[r.cached:] for r in admitted])
            q = self._randn((total, self.hq, self.d))
            ra_kv_store(self.k_pool, self.v_pool, self._randn((total, self.hkv, self.d)),
                        self._randn((total, self.hkv, self.d)), self._i32(loc), device_error=self.err)
            ws = torch.empty(ra_extend_workspace_bytes(len(admitted), total, self.hq, self.hkv), dtype=torch.uint8,
                             device=self.dev)
            ra_extend_attention(self.k_pool, self.v_pool, q, torch.empty_like(q), self.table,
                                self._i32([r.row for r in admitted]), self._i32(pre), self._i32(ext),
                                self._i32(np.concatenate([[0], np.cumsum(ext)])), max_extend_len=int(ext.max()),
                                max_prefix_len=int(pre.max()), sm_scale=self.scale, workspace=ws,
                                device_error=self.err)
            self.stats["extend_tokens"] += total
        # ---- one decode token for every request past its prefill
        dec = [self.running[rid] for rid in self.prefilled]
        if dec:
            n = len(dec)
            bs = next((s for s in self.graph_sizes if s >= n), n)
            g, buf, run = self._graph(bs)
            new = self._alloc(n)
            lens = np.empty(n, np.int32)
            for k, r in enumerate(dec):
                r.slots = np.concatenate([r.slots, new[k:k + 1]])
                lens[k] = r.slots.size
            rows = self._i32([r.row for r in dec])
            self.table[rows.long(), self._i32(lens - 1).long()] = self._i32(new)
            buf["q"][:n] = self._randn((n, self.hq, self.d))
            buf["k_new"][:n] = self._randn((n, self.hkv, self.d))
            buf["v_new"][:n] = self._randn((n, self.hkv, self.d))
            buf["loc"][:n] = self._i32(new)
            buf["loc"][n:] = 0
            buf["rpi"][:n] = rows
            buf["rpi"][n:] = self.pad_row
            buf["lens"][:n] = self._i32(lens)
            buf["lens"][n:] = 1
            if g is not None:
                g.replay()
            else:
                run()
            for r in dec:
                r.generated.append(self._next_token)
                self._next_token += 1
            self.stats["decode_tokens"] += n
        ev1.record()
        self.prefilled += [r.rid for r in admitted]
        # ---- retire finished turns: their whole sequence enters the tree
        done = [r for r in dec if len(r.generated) >= r.out_len]
        for r in done:
            seq = np.concatenate([r.prompt, np.asarray(r.generated, np.int32)])
            t0 = time.perf_counter()
            kept = self.cache.insert(seq, r.slots)
            self.cache.unlock(r.node)
            tree += time.perf_counter() - t0
            if kept > r.cached:  # positions another request cached first: our copies go back to the pool
                self.pool.free(r.slots[r.cached:kept])
            self.free_rows.append(r.row)
            del self.running[r.rid]
            self.prefilled.remove(r.rid)
            self.finished.append(r)
        ev1.synchronize()
        gpu_ms = ev0.elapsed_time(ev1)
        wall = time.perf_counter() - wall0
        self.stats["steps"] += 1
        self.stats["tree_s"] += tree
        self.stats["gpu_ms"] += gpu_ms
        self.stats["wall_s"] += wall
        return dict(gpu_ms=gpu_ms, tree_ms=tree * 1e3, wall_ms=wall * 1e3, decode=len(dec), admitted=len(admitted),
                    finished=len(done), deferred=deferred)

    def hit_ratio(self) -> float:
        return self.stats["cached_tokens"] / max(self.stats["prompt_tokens"], 1)


def multiturn_chat(num_convs: int, turns: int, seed: int = 0, system_prompts: int = 4, system_len: int = 512,
                   user_len: Tuple[int, int] = (32, 256), out_len: Tuple[int, int] = (16, 64)):
    """Synthetic multi-turn chats: each conversation starts from one of a few shared system prompts;
    turn t's prompt is the previous turn's prompt and output followed by new user tokens.  Yields,
    per conversation, the token generator the replay loop drives (the outputs are the replay's own)."""
    rng = np.random.default_rng(seed)
    sys_prompts = [rng.integers(1, 1 << 20, size=system_len, dtype=np.int32) for _ in range(system_prompts)]
    convs = []
    for c in range(num_convs):
        users = [rng.integers(1, 1 << 20, size=int(rng.integers(user_len[0], user_len[1] + 1)), dtype=np.int32)
                 for _ in range(turns)]
        outs = [int(rng.integers(out_len[0], out_len[1] + 1)) for _ in range(turns)]
        convs.append(dict(system=sys_prompts[c % system_prompts], users=users, outs=outs))
    return convs


def run_chat(replay: ServingReplay, convs, max_steps: int, arrivals_per_step: int = 16,
             rid0: int = 0) -> Dict[str, float]:
    """Drive `replay` through the conversations of `multiturn_chat`: each step admits up to
    `arrivals_per_step` pending turns (a conversation's next turn becomes pending when its previous
    turn finishes, its prompt being that turn's prompt and output plus the new user tokens)."""
    from collections import deque
    pending = deque((c, 0) for c in range(len(convs)))
    history = {c: convs[c]["system"] for c in range(len(convs))}
    meta = {}
    rid = rid0
    seen = len(replay.finished)
    for _ in range(max_steps):
        arrivals = []
        while pending and len(arrivals) < arrivals_per_step and \
                len(replay.running) + len(arrivals) < replay.max_running:
            c, t = pending.popleft()
            prompt = np.concatenate([history[c], convs[c]["users"][t]])
            arrivals.append((rid, prompt, convs[c]["outs"][t]))
            meta[rid] = (c, t)
            replay.tags[rid] = (c, t)
            rid += 1
        if not arrivals and not replay.running:
            break
        res = replay.step(arrivals)
        for a in reversed(res["deferred"]):  # back to the front of the queue, in order
            pending.appendleft(meta[a[0]])
        for r in replay.finished[seen:]:
            c, t = meta[r.rid]
            history[c] = np.concatenate([r.prompt, np.asarray(r.generated, np.int32)])
            if t + 1 < len(convs[c]["users"]):
                pending.append((c, t + 1))
        seen = len(replay.finished)
    return dict(replay.stats, hit_ratio=replay.hit_ratio(),
                tree_overhead=replay.stats["tree_s"] / max(replay.stats["wall_s"], 1e-9))
