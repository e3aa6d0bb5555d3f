#!/usr/bin/env python3
"""Benchmark of the RadixAttention hot path on GB300 (one JSON line on stdout).

One step = one pass of the whole path over one batch of the multi-turn chat
workload (70B attention heads: 64 q / 8 kv, head_dim 128; 256 requests with
lognormal contexts sharing prefixes through a radix tree at a ~70% token
hit ratio; 32 extend requests + 224 decode requests; 2M-slot pool):
  ra_kv_store (this step's 9.4K new tokens)  ->  ra_extend_attention  ->
  ra_decode_attention.
value = attention tokens (extend suffix tokens + decode tokens) per second
with inputs resident in HBM; L2 is flushed between steps (a 256 MB write, then a 256 MB read).
Extra objects: per-kernel roofline (decode KV GB/s vs measured HBM copy
bandwidth, extend TFLOP/s vs measured dense BF16), e2e through the public API
with host buffers, the CPU oracle as baseline, SM clocks during the timed
region, and the same kernels on the decode (Llama-3-8B shape, system-prompt
groups), few-shot extend and forked-decode workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-extra]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn tokens/s; decode KV GB/s and extend TFLOP/s as % of GB300 roofline"
UNIT = "tokens/s"
WORKLOAD = ("multi-turn chat mix, 70B heads (64 q / 8 kv, head_dim 128, bf16): 256 requests, lognormal "
            "contexts (median 2048, clipped 16..32768), radix-tree prefix sharing at 70% token hit ratio; "
            "32 extend (suffix 64..512) + 224 decode in the tree's depth-first order (cascade groups of >= 4 "
            "members from the radix tree); pool 2M slots")
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Between timed steps: write one 256 MB buffer (evicts every line the last step left in L2), then read
    another (evicts the first buffer's dirty lines, so their write-back happens here and not inside the next
    step's kernels).  The step then starts with an L2 that holds none of its data and nothing dirty, as an
    ncu capture with cache control does; a write-only flush charged the decode call ~10 us of write-backs."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.acc = torch.zeros(1, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.acc.copy_(self.r.sum().view(1))
# Before each timed step the stream runs a ~0.5 ms GPU delay (after the L2 flush, outside the timed region), so
# the host has enqueued the whole step before its first kernel starts and the events time the GPU's work, not
# the Python binding's launch latency (serving replays its decode step from a CUDA graph for the same reason).
HOST_LEAD_CYCLES = 1_000_000
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s the problem statement quotes for GB300's HBM3e (context beside the measured peak)
KV_BYTES_PER_TOKEN_HEAD = 2 * 128 * 2  # K + V row of one kv head, bf16


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- algorithmic work
def extend_flops(b) -> float:
    e = b.ext_extend_lens.astype(np.float64)
    p = b.ext_prefix_lens.astype(np.float64)
    return float(np.sum(b.num_q_heads * (e * p + e * (e + 1) / 2) * 4 * b.head_dim))


def decode_bytes(b, cascade: bool = False) -> dict:
    """Algorithmic decode bytes: every distinct K/V row the batch's contexts reference
    (a row shared by several requests counts once), plus q, o and table entries.
    `logical` counts every request's rows separately."""
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    uniq = np.unique(np.concatenate(rows)).size if rows else 0
    logical = int(np.sum(b.dec_seq_lens))
    kv_row = b.num_kv_heads * b.head_dim * 2 * 2
    qo = 2 * b.n_decode * b.num_q_heads * b.head_dim * 2
    idx = logical * 4
    return {"unique_tokens": int(uniq), "logical_tokens": logical,
            "algorithmic": uniq * kv_row + qo + idx, "logical": logical * kv_row + qo + idx}


def store_bytes(b) -> int:
    return 2 * 2 * b.num_new_tokens * b.num_kv_heads * b.head_dim * 2  # read + write, K and V


# ----------------------------------------------------------------------------- ncu traffic
def source_digest() -> str:
    """Digest of the CUDA sources and the C header: ties a recorded ncu traffic figure to the code."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "prefix_shared_kv_ra_gb300", "csrc", "*"))) + \
        [os.path.join(ROOT, "include", "ra.h")]
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) recorded from an ncu capture in
    profiles/traffic.json, or None when absent or captured on other sources (the record names the source
    digest it was taken on).  A recorded figure, not one measured by this run: the line says so."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_digest") != source_digest():
        return None
    for e in rec.get("launches", []):
        if e.get("kernel") == kernel and e.get("workload") == workload:
            return float(e["dram_bytes"])
    return None


TRAFFIC_NOTE = ("recorded, not measured by this run: DRAM bytes per launch from a one-pass ncu capture of the same "
                "workload (profiles/traffic.json), used only while its source digest equals this build's")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["uuid", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.out = os.path.join("/tmp", f"ra_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out):
            return None
        by_gpu = {}
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                by_gpu.setdefault(parts[0], []).append((float(parts[1]), float(parts[2]), parts[5:]))
            except ValueError:
                continue
        if not by_gpu:
            return None
        # this process's GPU by UUID; with one visible GPU its rows are the only ones
        rows = by_gpu.get(self.uuid) or next(iter(by_gpu.values()))
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, v in zip(names, flags) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def schedule_decode_dfs(b):
    """The batch with its decode requests in the radix tree's depth-first order (radix.dfs_order), as a
    cache-aware scheduler runs it: requests that share slots beyond their group's prefix are adjacent, so
    the decode kernel's items read those slots close together in time.  Queries, lengths, table rows and
    the requests' new-token rows (store inputs) are permuted together; the extend part is unchanged."""
    import copy
    from prefix_shared_kv_ra_gb300.radix import dfs_order
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    order = dfs_order(rows)
    c = copy.copy(b)
    c.dec_rpi, c.dec_seq_lens, c.dec_q = b.dec_rpi[order], b.dec_seq_lens[order], b.dec_q[order]
    n0 = b.total_q_extend  # new tokens: the extend suffixes, then one per decode request
    perm = np.concatenate([np.arange(n0), n0 + order])
    c.out_cache_loc, c.k_new, c.v_new = b.out_cache_loc[perm], b.k_new[perm], b.v_new[perm]
    c.casc_group_indptr = c.casc_group_reqs = c.casc_group_prefix_len = None
    c.casc_group_start = c.casc_group_level = None
    c.casc_levels = 1
    return c


def mix_step_batch(seed: int = 5):
    """The benchmark's batch: the multi-turn mix with its decode requests in the tree's depth-first order
    and the one-level cascade groups the tree derives from them (at least 4 members sharing >= 256
    tokens: with the depth-first order, smaller groups' shared slots are cheaper to read through L2 in the
    plain decode than to run through the tensor-core prefix pass -- decode call 217 / 216 / 214 / 216 us
    for groups of >= 2 / 3 / 4 / 6 members, same box)."""
    import workloads as W
    return with_tree_groups(schedule_decode_dfs(W.multiturn_mix_70b(seed=seed)), min_members=4)


def with_tree_groups(b, min_prefix: int = 256, multilevel: bool = False, min_members: int = 2):
    """Attach the cascade groups the radix tree derives from the batch's decode table rows: one level
    (per subtree of the root, >= min_members requests sharing >= min_prefix tokens) or one group per
    shared node."""
    from prefix_shared_kv_ra_gb300.radix import cascade_groups, cascade_groups_multilevel
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    if multilevel:
        (b.casc_group_indptr, b.casc_group_reqs, b.casc_group_start, b.casc_group_prefix_len, b.casc_group_level,
         b.casc_levels) = cascade_groups_multilevel(rows, min_members=min_members, min_range=min_prefix)
    else:
        b.casc_group_indptr, b.casc_group_reqs, b.casc_group_prefix_len = cascade_groups(
            rows, min_prefix=min_prefix, min_members=min_members)
        b.casc_group_start, b.casc_group_level, b.casc_levels = None, None, 1
    return b


# ----------------------------------------------------------------------------- GPU arm
class Step:
    """The hot path on one batch, resident on the device."""

    def __init__(self, b, dev, cascade: bool = False, fused_store: bool = False):
        import torch
        import prefix_shared_kv_ra_gb300 as ra
        self.torch, self.ra, self.b, self.dev = torch, ra, b, dev
        self.cascade = cascade and b.has_cascade()
        # decode-only batch: the store of its new tokens fused into the decode call (one launch fewer)
        self.fused_store = fused_store and b.n_extend == 0 and b.n_decode > 0

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        S, hkv, d = b.num_slots, b.num_kv_heads, b.head_dim
        self.k_pool = torch.zeros((S, hkv, d), dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.zeros((S, hkv, d), dtype=torch.bfloat16, device=dev)
        idx = torch.from_numpy(b.pool_slots.astype(np.int64)).to(dev)
        self.k_pool.index_copy_(0, idx, bf16(b.pool_k))
        self.v_pool.index_copy_(0, idx, bf16(b.pool_v))
        self.host = {  # per-step inputs (pinned host copies for the e2e measurement)
            "k_new": b.k_new, "v_new": b.v_new, "loc": b.out_cache_loc.astype(np.int32),
            "ext_q": b.ext_q, "ext_rpi": b.ext_rpi, "ext_prefix": b.ext_prefix_lens, "ext_len": b.ext_extend_lens,
            "ext_qo": b.ext_qo_indptr, "dec_q": b.dec_q, "dec_rpi": b.dec_rpi, "dec_lens": b.dec_seq_lens}
        self.d = {k: (bf16(v) if v.dtype == np.uint16 else i32(v)) for k, v in self.host.items()}
        self.table = i32(b.req_to_token)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ext_o = torch.empty_like(self.d["ext_q"])
        self.dec_o = torch.empty_like(self.d["dec_q"])
        self.casc = {}
        if self.cascade:
            self.casc = dict(group_indptr=i32(b.casc_group_indptr), group_reqs=i32(b.casc_group_reqs),
                             group_prefix_len=i32(b.casc_group_prefix_len),
                             max_group_prefix_len=int(b.casc_group_prefix_len.max()),
                             max_group_size=int(np.diff(b.casc_group_indptr).max()),
                             group_prefix_start=None if b.casc_group_start is None else i32(b.casc_group_start),
                             group_level=None if b.casc_group_level is None else i32(b.casc_group_level),
                             max_group_levels=int(b.casc_levels))
        ng = b.casc_group_indptr.size - 1 if self.cascade else 0
        nws = ra.ra_decode_workspace_bytes(max(b.n_decode, 1), b.num_q_heads, hkv, d, max(b.max_seq_len, 1), ng,
                                           self.casc.get("max_group_prefix_len", 0),
                                           self.casc.get("max_group_size", 0), self.casc.get("max_group_levels", 1))
        self.ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
        self.ext_ws = torch.empty(max(ra.ra_extend_workspace_bytes(b.n_extend, b.total_q_extend, b.num_q_heads, hkv),
                                      256), dtype=torch.uint8, device=dev)
        # kernel launches per step: store, [work-list plan, extend,] [[set-up, prefix pass,] decode plan, decode,
        # combine]
        self.launches = 1 + (2 if b.n_extend else 0) + ((3 + (2 if self.cascade else 0)) if b.n_decode else 0)
        if self.fused_store:
            self.launches -= 1

    def run(self, d=None, events=None, outs=None):
        ra, b = self.ra, self.b
        d = d or self.d
        ext_o, dec_o = outs or (self.ext_o, self.dec_o)
        ev = events or [None] * 4
        if ev[0] is not None:
            ev[0].record()
        if self.fused_store:
            ra.ra_decode_attention_store(self.k_pool, self.v_pool, d["k_new"], d["v_new"], d["loc"], d["dec_q"],
                                         dec_o, self.table, d["dec_rpi"], d["dec_lens"], max_seq_len=b.max_seq_len,
                                         sm_scale=b.sm_scale, workspace=self.ws, device_error=self.err, **self.casc)
            for e in ev[1:]:
                if e is not None:
                    e.record()
            return
        ra.ra_kv_store(self.k_pool, self.v_pool, d["k_new"], d["v_new"], d["loc"], device_error=self.err)
        if ev[1] is not None:
            ev[1].record()
        if b.n_extend:
            ra.ra_extend_attention(self.k_pool, self.v_pool, d["ext_q"], ext_o, self.table, d["ext_rpi"],
                                   d["ext_prefix"], d["ext_len"], d["ext_qo"], max_extend_len=b.max_extend_len,
                                   max_prefix_len=b.max_prefix_len, sm_scale=b.sm_scale, workspace=self.ext_ws,
                                   device_error=self.err)
        if ev[2] is not None:
            ev[2].record()
        if b.n_decode:
            ra.ra_decode_attention(self.k_pool, self.v_pool, d["dec_q"], dec_o, self.table, d["dec_rpi"],
                                   d["dec_lens"], max_seq_len=b.max_seq_len, sm_scale=b.sm_scale,
                                   workspace=self.ws, device_error=self.err, **self.casc)
        if ev[3] is not None:
            ev[3].record()


def time_steps(step, steps: int, warmup: int, flush, sample_clocks_uuid=None, breakdown: bool = True):
    """Headline pass: events around each whole step only (the kernels of a step may overlap through
    programmatic dependent launch).  Breakdown pass: events between the three calls as well (which
    serialises them) for the per-kernel times the roofline uses.  Each step starts after the L2 flush and a
    GPU delay that lets the host enqueue the whole step first (HOST_LEAD_CYCLES)."""
    torch = step.torch
    for _ in range(warmup):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        step.run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    sampler = ClockSampler(sample_clocks_uuid) if sample_clocks_uuid is not None else None
    if sampler:
        sampler.__enter__()
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            flush()
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            step.run(events=[evs[k][0], None, None, evs[k][1]])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
    total = np.array([e[0].elapsed_time(e[1]) for e in evs])
    out = {"step_ms": total, "wall_s": wall, "clocks": sampler.summary() if sampler else None}
    if breakdown:
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for k in range(steps):
            flush()
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            step.run(events=evb[k])
        torch.cuda.synchronize()
        per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evb])  # store, extend, decode
        out.update(store_ms=per[:, 0], extend_ms=per[:, 1], decode_ms=per[:, 2])
    out["device_error"] = int(step.err.item())
    return out


def e2e_steps(step, steps: int, warmup: int, flush):
    """Same step through the public API with host buffers, as a serving loop runs it: every step
    copies its inputs from pinned host memory and reads both outputs back, on copy streams that
    overlap the neighbouring steps' compute (inputs and outputs double-buffered on the device; step
    k's compute waits for its inputs and for step k-2's outputs to be read back).  The timed region
    spans the first input copy to the last output copy; L2 is flushed before every step's compute."""
    torch = step.torch
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16
                                  else np.ascontiguousarray(v, dtype=np.int32)).pin_memory()
              for k, v in step.host.items()}
    dev_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=step.dev) for k, v in pinned.items()} for _ in range(2)]
    dev_out = [(torch.empty_like(step.ext_o), torch.empty_like(step.dec_o)) for _ in range(2)]
    host_out = [(torch.empty(step.ext_o.shape, dtype=torch.int16).pin_memory(),
                 torch.empty(step.dec_o.shape, dtype=torch.int16).pin_memory()) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = host_out[0][0].numel() * 2 + host_out[0][1].numel() * 2
    comp = torch.cuda.current_stream(step.dev)
    s_in, s_out = torch.cuda.Stream(step.dev), torch.cuda.Stream(step.dev)

    def run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for k in range(n):
            i = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_comp[k - 2])  # step k-2 has consumed input buffer i
                for name, v in pinned.items():
                    dev_in[i][name].copy_(v, non_blocking=True)
                ev_in[k].record(s_in)
            comp.wait_event(ev_in[k])
            if k >= 2:
                comp.wait_event(ev_out[k - 2])  # step k-2's outputs are back on the host
            flush()
            d = {name: (v.view(torch.bfloat16) if v.dtype == torch.int16 else v) for name, v in dev_in[i].items()}
            step.run(d=d, outs=dev_out[i])
            ev_comp[k].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k])
                host_out[i][0].copy_(dev_out[i][0].view(torch.int16), non_blocking=True)
                host_out[i][1].copy_(dev_out[i][1].view(torch.int16), non_blocking=True)
                ev_out[k].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    run(max(warmup, 2))
    ms = run(steps)
    # the last step's outputs, as read back, equal the device-resident step bit for bit
    last = host_out[(steps - 1) % 2]
    step.run()
    torch.cuda.synchronize()
    same = bool(torch.equal(last[0], step.ext_o.view(torch.int16).cpu()) and
                torch.equal(last[1], step.dec_o.view(torch.int16).cpu()))
    return ms, h2d, d2h, same


def extra_kernels(dev, flush, peaks, reps: int = 20, with_oracle: bool = True):
    """The same kernels on the other workloads (parity-tested elsewhere): per-kernel roofline."""
    import workloads as W
    out = {}
    specs = [("decode_8b_system_prompts", W.decode_8b_system_prompts, (False, True)),
             ("decode_8b_system_prompts_page16", lambda: W.decode_8b_system_prompts(page_size=16), (False,)),
             ("extend_fewshot_3000", W.fewshot_extend, (False,)),
             ("decode_70b_forked_8192", W.forked_decode_70b, (False, True))]
    for name, fn, modes in specs:
        b = fn()
        for casc in modes:
            st = Step(b, dev, cascade=casc)
            st.run()  # store once: the pool then holds this step's tokens
            r = time_steps(st, reps, 3, flush)
            key = name + ("_cascade" if casc else "")
            if b.n_extend:
                ms = float(np.median(r["extend_ms"]))
                fl = extend_flops(b)
                out[key] = {"kernel": "extend (tcgen05)", "ms": ms, "tokens_per_s": b.total_q_extend / ms * 1e3,
                            "tflops": fl / ms / 1e9, "frac_of_measured_bf16": fl / ms / 1e9 / peaks["bf16_tflops"]}
            else:
                ms = float(np.median(r["decode_ms"]))
                db = decode_bytes(b)
                gbs = db["algorithmic"] / ms / 1e6
                out[key] = {"kernel": "decode" + (" + cascade prefix pass" if casc else ""), "ms": ms,
                            "tokens_per_s": b.n_decode / ms * 1e3, "algorithmic_bytes": db["algorithmic"],
                            "gbs": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
                            "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                            "effective_gbs": db["logical"] / ms / 1e6}
            out[key]["device_error"] = r["device_error"]
            del st
        if with_oracle and not name.endswith("_page16"):
            # the oracle on the same batch, the whole call's rows, timed on the host cores
            o = oracle_step(b)
            for casc in modes:
                out[name + ("_cascade" if casc else "")]["oracle"] = {
                    "tokens_per_s": o["tokens_per_s"], "seconds": o["seconds"], "cores": o["cores"],
                    "rows": o["rows"], "kind": "fp64 oracle, every query row of the call, measured"}
    # the decode step's store fused into the decode call, against the two calls (whole steps, no events
    # between the calls, so the programmatic launch chain is kept in both)
    b = W.decode_8b_system_prompts()
    steps = {}
    for fused in (False, True):
        st = Step(b, dev, fused_store=fused)
        st.run()
        r = time_steps(st, reps, 3, flush, breakdown=False)
        steps[fused] = (float(np.median(r["step_ms"])), r["device_error"])
        del st
    nbytes = decode_bytes(b)["algorithmic"] + store_bytes(b)
    ms = steps[True][0]
    out["decode_8b_system_prompts_store_fused"] = {
        "kernel": "store + decode in one call (ra_decode_attention_store)", "ms": ms,
        "separate_store_then_decode_ms": steps[False][0], "tokens_per_s": b.n_decode / ms * 1e3,
        "algorithmic_bytes": nbytes, "gbs": nbytes / ms / 1e6,
        "frac_of_measured_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"],
        "frac_of_nominal_8tbs": nbytes / ms / 1e6 / NOMINAL_HBM_GBS,
        "device_error": steps[True][1] | steps[False][1]}
    return out


def serving_replay(dev, convs: int = 192, turns: int = 4):
    """The radix cache driving the hot path over many steps (multi-turn chats, 70B heads, CUDA-graph
    decode): tokens/s of the whole loop and the share of its wall time spent in the tree."""
    from prefix_shared_kv_ra_gb300.serving import ServingReplay, multiturn_chat, run_chat
    rp = ServingReplay(num_slots=1 << 20, num_q_heads=64, num_kv_heads=8, head_dim=128, max_len=4096,
                       max_running=256, device=dev, seed=11)
    chats = multiturn_chat(convs, turns, seed=11, system_prompts=8, system_len=1024, user_len=(32, 256),
                           out_len=(16, 64))
    st = run_chat(rp, chats, max_steps=100000, arrivals_per_step=32)
    toks = st["extend_tokens"] + st["decode_tokens"]
    return {"workload": f"{convs} chats x {turns} turns, 8 shared 1024-token system prompts, user 32..256, "
                        f"output 16..64 tokens, 64 q / 8 kv heads, head_dim 128; CUDA-graph decode",
            "steps": st["steps"], "extend_tokens": st["extend_tokens"], "decode_tokens": st["decode_tokens"],
            "hit_ratio": round(st["hit_ratio"], 4), "tokens_per_s": toks / st["wall_s"],
            "gpu_ms_per_step": st["gpu_ms"] / st["steps"], "wall_ms_per_step": st["wall_s"] * 1e3 / st["steps"],
            "tree_overhead_of_wall": st["tree_overhead"], "device_error": int(rp.err.item())}


# ----------------------------------------------------------------------------- CPU oracle arm
def bench_config(b, world: int = 1) -> dict:
    """The `config` of the bench line: the same dict for the GPU arm and the oracle (reference) arm."""
    return {"workload": WORKLOAD, "global_batch": 256 * world, "replica_extend_tokens": b.total_q_extend,
            "replica_decode_tokens": b.n_decode,
            "l2": "GPU: flushed between steps (256 MB write, then 256 MB read: no step data, no dirty lines); "
                  "oracle: its 8 GiB pool exceeds every CPU cache",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "hit_ratio": round(b.meta["construction_hit_ratio"], 4)}


def oracle_step(b, pool=None, fraction: float = 1.0) -> dict:
    """One step of the fp64 oracle on the host cores, timed: every extend and decode query row of the batch
    (or, with fraction < 1, every round(1/fraction)-th (token, head) row of each part).  tokens = rows / Hq."""
    import oracle
    pool = pool or oracle.pool_after_store(b)
    hq = b.num_q_heads
    n_e, n_d = b.total_q_extend * hq, b.n_decode * hq
    stride = max(1, int(round(1.0 / fraction))) if fraction < 1.0 else 1
    se = None if stride == 1 else np.arange(0, n_e, stride, dtype=np.int64)
    sd = None if stride == 1 else np.arange(0, n_d, stride, dtype=np.int64)
    t0 = time.perf_counter()
    if n_e:
        oracle.extend_batch(b, sel=se, pool=pool)
    if n_d:
        oracle.decode_batch(b, sel=sd, pool=pool)
    dt = time.perf_counter() - t0
    rows = (n_e if se is None else se.size) + (n_d if sd is None else sd.size)
    return {"seconds": dt, "tokens": rows / hq, "tokens_per_s": rows / hq / dt, "cores": oracle.num_threads(),
            "rows": int(rows), "all_rows": stride == 1}


def oracle_baseline(b, fraction: float = 1.0) -> dict:
    """cpu_baseline of the GPU line: the oracle as it stands on one step of the same batch, measured."""
    r = oracle_step(b, fraction=fraction)
    what = ("the whole step" if r["all_rows"] else f"every {int(round(1 / fraction))}-th query row of the step")
    return {"value": r["tokens_per_s"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
            "sample": f"{what}: {r['rows']} (token, q head) rows of extend and decode attention in fp64, "
                      f"{r['seconds']:.1f} s on {r['cores']} host threads, no extrapolation",
            "seconds": r["seconds"]}


def run_reference(args):
    """The reference arm: the fp64 oracle (the only implementation the pages allow to be written from
    them) on the GPU arm's workload, one whole step per timed step on the host cores."""
    import workloads as W
    import oracle
    b = mix_step_batch(seed=5)
    pool = oracle.pool_after_store(b)
    for _ in range(args.warmup):  # the CPU has nothing to warm beyond its first pass: short warm-up steps
        oracle_step(b, pool, fraction=min(args.ref_fraction, 1.0 / 16))
    timed = [oracle_step(b, pool, fraction=args.ref_fraction) for _ in range(args.steps)]
    secs = float(np.mean([r["seconds"] for r in timed]))
    val = timed[0]["tokens"] / secs
    what = "whole step" if timed[0]["all_rows"] else f"every {int(round(1 / args.ref_fraction))}-th query row"
    sample = (f"{what}: {timed[0]['rows']} (token, q head) rows per timed step, fp64, {timed[0]['cores']} host "
              f"threads, {secs:.2f} s per step measured (warm-up steps: 1/16 of the rows)")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(b, args.gpus),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": timed[0]["cores"], "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------------------- ncu cases
PROFILE_CASES = {
    "extend_fewshot": ("fewshot_extend", False),
    "multiturn_mix_cascade": ("multiturn_mix_70b", True),
    "decode_8b": ("decode_8b_system_prompts", False),
    "decode_8b_cascade": ("decode_8b_system_prompts", True),
    "decode_70b_forked_cascade": ("forked_decode_70b", True),
    "multiturn_mix": ("multiturn_mix_70b", False),
}


def run_profile_case(name: str, steps: int):
    """Run `steps` passes (store, extend, decode) of one workload, untimed, for a profiler."""
    import torch
    import prefix_shared_kv_ra_gb300 as ra
    import workloads as W
    ra.load()
    cfg, cascade = PROFILE_CASES[name]
    dev = torch.device("cuda:0")
    if cfg == "multiturn_mix_70b":
        b = mix_step_batch()  # the benchmark's own batch (its groups are used only with the cascade)
    else:
        b = W.WORKLOADS[cfg]()
        if cascade and not b.has_cascade():
            b = with_tree_groups(b)
    st = Step(b, dev, cascade=cascade)
    for _ in range(steps):
        st.run()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, "steps": steps, "launches_per_step": st.launches,
                      "device_error": int(st.err.item())}))


# ----------------------------------------------------------------------------- ranks
def reduce_over_ranks(dist, device, step_ms: float, e2e_ms: float, tokens: int):
    """Whole-job figures of independent replicas: the slowest rank's step and end-to-end times and the
    tokens all ranks processed (each rank draws its own batch).  dist None = one process."""
    if dist is None:
        return step_ms, e2e_ms, tokens
    import torch
    t = torch.tensor([step_ms, e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t[0].item()), float(t[1].item()), int(n.item())


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the per-kernel runs on the other workloads")
    ap.add_argument("--cpu-fraction", type=float, default=1.0,
                    help="share of the step's query rows the cpu_baseline oracle runs (1 = the whole step)")
    ap.add_argument("--ref-fraction", type=float, default=1.0,
                    help="share of the step's query rows per reference (oracle) step (1 = the whole step)")
    ap.add_argument("--profile", default=None, choices=sorted(PROFILE_CASES),
                    help="untimed: run the hot path of one workload --steps times (for an ncu capture)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.profile:
        return run_profile_case(args.profile, args.steps)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import torch
    import prefix_shared_kv_ra_gb300 as ra
    from prefix_shared_kv_ra_gb300 import _build
    import workloads as W

    if not os.path.exists(_build.LIB):
        _build.build()
    ra.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()

    # independent replicas: each rank draws its own batch of the same workload; the decode requests are
    # grouped by the radix tree (one-level cascade groups over shared prefixes of >= 256 tokens)
    b = mix_step_batch(seed=5 + rank)
    step = Step(b, dev, cascade=True)
    flush = L2Flush(dev)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = ""
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    r = time_steps(step, args.steps, args.warmup, flush, sample_clocks_uuid=uuid)
    step_ms = float(np.mean(r["step_ms"]))
    if dist:
        dist.barrier()
    e2e_ms, h2d, d2h, e2e_same = e2e_steps(step, args.steps, args.warmup, flush)
    tokens = b.total_q_extend + b.n_decode
    step_ms, e2e_ms, job_tokens = reduce_over_ranks(dist, dev, step_ms, e2e_ms, tokens)
    value = job_tokens / step_ms * 1e3
    if rank != 0:
        dist.barrier()
        dist.destroy_process_group()
        return

    ext_ms = float(np.mean(r["extend_ms"]))
    dec_ms = float(np.mean(r["decode_ms"]))
    st_ms = float(np.mean(r["store_ms"]))
    fl = extend_flops(b)
    dbytes = decode_bytes(b)
    ext_tf = fl / ext_ms / 1e9
    dec_gbs = dbytes["algorithmic"] / dec_ms / 1e6
    # dominant kernel of the step: the one with the larger share of the step time
    if ext_ms >= dec_ms:
        roof = {"kernel": "attn_tc_kernel<extend>", "bound": "tensor", "achieved": ext_tf,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ext_tf / peaks["bf16_tflops"],
                "traffic": recorded_traffic("attn_tc_kernel<extend>", "multiturn_mix"),
                "traffic_source": TRAFFIC_NOTE,
                "peak_source": peaks["source"] + " bf16 burst",
                "per_launch": {"flops": fl, "ms": ext_ms}}
    else:
        roof = {"kernel": "decode_kernel + decode_combine_kernel", "bound": "hbm", "achieved": dec_gbs,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                "traffic": recorded_traffic("decode_kernel", "multiturn_mix"),
                "traffic_source": TRAFFIC_NOTE,
                "peak_source": peaks["source"] + " HBM copy",
                "per_launch": {"bytes": dbytes["algorithmic"], "ms": dec_ms}}
    extra = {} if args.no_extra else extra_kernels(dev, flush, peaks)
    replay = {} if args.no_extra else serving_replay(dev)
    cpu = oracle_baseline(b, args.cpu_fraction)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(b, world),
        "tokens_per_step": job_tokens,
        "roofline": roof,
        "kernels": {
            "step_breakdown_ms": {"kv_store": st_ms, "extend": ext_ms, "decode": dec_ms},
            "extend": {"tflops": ext_tf, "frac_of_measured_bf16": ext_tf / peaks["bf16_tflops"],
                       "flops": fl},
            "decode": {"gbs": dec_gbs, "frac_of_measured_hbm": dec_gbs / peaks["hbm_gbs"],
                       "frac_of_nominal_8tbs": dec_gbs / NOMINAL_HBM_GBS,
                       "effective_gbs": dbytes["logical"] / dec_ms / 1e6, "unique_tokens": dbytes["unique_tokens"],
                       "logical_tokens": dbytes["logical_tokens"]},
            "kv_store": {"gbs": store_bytes(b) / st_ms / 1e6},
            "other_workloads": extra,
        },
        "serving_replay": replay,
        "cpu_baseline": {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": job_tokens / e2e_ms * 1e3, "unit": UNIT, "ms_per_step": e2e_ms,
                "outputs_match_device_run": e2e_same,
                "pipeline": "per-step H2D / D2H on copy streams overlapping neighbouring steps' compute",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches * args.steps,
        "source_digest": source_digest(),
        "clocks": r["clocks"],
        "device_error": r["device_error"],
        "peaks": peaks,
    }
    print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
