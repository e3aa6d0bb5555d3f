"""Seeded synthetic inputs for the RadixAttention hot path.

This module only *draws inputs*: token sequences that share prefixes the way a
radix-tree prefix cache shares them, the KV-pool slot that every token lives
in, the ``req_to_token`` table that maps (request, position) to a slot, and
bf16 Q/K/V values.  It holds none of the attention or store arithmetic; both
the CUDA path (through its Python binding) and the CPU oracle consume what it
returns, and neither side imports the other.

Sharing model (SGLang paper summary, §3 "Efficient KV Cache Reuse with
RadixAttention": KV depends only on the prefix tokens, so a request that
shares a prefix with an earlier one reuses its KV slots; the yaopepe.com
explainer, §04, walks the same insert/split picture).  Every sequence below is
``SeqSpec``: its first ``fork`` positions use the slots of an earlier sequence
(its parent), the rest get fresh slots drawn from a seeded permutation of
``[1, num_slots)``.  Slot 0 is never assigned: it is the dummy slot that
padded CUDA-graph requests write to (anrans handbook, "v0.2：不到四千行的调度
核心跑出 3.1 倍", 来源一: CUDA Graph replay pads with ``out_cache_loc = 0``).

Values are N(0, 1) float32 rounded to bf16 (round to nearest even) and kept
as raw ``uint16`` bit patterns, so that no consumer can disagree about them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "SeqSpec", "Batch", "build_batch", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "tiny_extend_decode", "decode_8b_system_prompts", "fewshot_extend", "forked_decode_70b",
    "multiturn_mix_70b", "random_mixed", "WORKLOADS",
]

NO_SLOT = -1  # unused req_to_token entries; a kernel that reads one has a bug


# ----------------------------------------------------------------------------
# bf16 bit patterns
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape: Tuple[int, ...], chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# sequence specs and the batch record
# ----------------------------------------------------------------------------
@dataclass
class SeqSpec:
    """One token sequence of the prefix cache.

    total_len  L: context length once this step's new tokens are stored.
    cached_len C: tokens whose K/V are already in the pool before this step.
    parent/fork: positions [0, fork) share the parent's slots (fork <= parent's C).
    kind: "extend" (new tokens C..L-1 are a prefill suffix), "decode" (exactly one
          new token, L = C + 1) or "cached" (a tree-only sequence, e.g. a system
          prompt, that is in the pool but not in this batch; L = C).
    """
    total_len: int
    cached_len: int
    kind: str
    parent: int = -1
    fork: int = 0


@dataclass
class Batch:
    name: str
    num_slots: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    sm_scale: float
    # pool contents before this step (rows of the slots listed)
    pool_slots: np.ndarray          # int64 [U]
    pool_k: np.ndarray              # uint16 [U, Hkv, D]
    pool_v: np.ndarray              # uint16 [U, Hkv, D]
    # this step's new tokens: extend suffixes first, then one token per decode request
    out_cache_loc: np.ndarray       # int32 [N]
    k_new: np.ndarray               # uint16 [N, Hkv, D]
    v_new: np.ndarray               # uint16 [N, Hkv, D]
    # request table (already holds this step's slots, as the caller writes it before attention)
    req_to_token: np.ndarray        # int32 [R, Lmax]
    # extend part
    ext_rpi: np.ndarray             # int32 [Be]
    ext_prefix_lens: np.ndarray     # int32 [Be]
    ext_extend_lens: np.ndarray     # int32 [Be]
    ext_qo_indptr: np.ndarray       # int32 [Be + 1]
    ext_q: np.ndarray               # uint16 [sum E, Hq, D]
    # decode part
    dec_rpi: np.ndarray             # int32 [Bd]
    dec_seq_lens: np.ndarray        # int32 [Bd] (includes the new token)
    dec_q: np.ndarray               # uint16 [Bd, Hq, D]
    # optional cascade over decode requests: group g covers positions [start, prefix_len) of its members
    casc_group_indptr: Optional[np.ndarray] = None   # int32 [NG + 1]
    casc_group_reqs: Optional[np.ndarray] = None     # int32 [sum members] (decode batch indices)
    casc_group_prefix_len: Optional[np.ndarray] = None  # int32 [NG] (range end)
    casc_group_start: Optional[np.ndarray] = None    # int32 [NG]; None = all 0 (one level)
    casc_group_level: Optional[np.ndarray] = None    # int32 [NG]; None = all 0
    casc_levels: int = 1
    # cached token ids of every sequence in build order (for hit-ratio checks)
    tokens: List[np.ndarray] = field(default_factory=list)
    specs: List[SeqSpec] = field(default_factory=list)
    meta: Dict = field(default_factory=dict)

    # ---- derived sizes ----
    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def n_extend(self) -> int:
        return int(self.ext_rpi.shape[0])

    @property
    def n_decode(self) -> int:
        return int(self.dec_rpi.shape[0])

    @property
    def total_q_extend(self) -> int:
        return int(self.ext_qo_indptr[-1]) if self.ext_qo_indptr.size else 0

    @property
    def max_extend_len(self) -> int:
        return int(self.ext_extend_lens.max()) if self.n_extend else 0

    @property
    def max_prefix_len(self) -> int:
        return int(self.ext_prefix_lens.max()) if self.n_extend else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.dec_seq_lens.max()) if self.n_decode else 0

    @property
    def num_new_tokens(self) -> int:
        return int(self.out_cache_loc.shape[0])

    def dense_pool(self) -> Tuple[np.ndarray, np.ndarray]:
        """Full [S, Hkv, D] pools before the store (zeros where unused). Small S only."""
        shape = (self.num_slots, self.num_kv_heads, self.head_dim)
        k = np.zeros(shape, np.uint16)
        v = np.zeros(shape, np.uint16)
        k[self.pool_slots] = self.pool_k
        v[self.pool_slots] = self.pool_v
        return k, v

    def has_cascade(self) -> bool:
        return self.casc_group_indptr is not None and self.casc_group_indptr.size > 1


def build_batch(name: str, specs: Sequence[SeqSpec], *, num_slots: int, num_q_heads: int,
                num_kv_heads: int, head_dim: int, seed: int,
                cascade: Optional[Sequence[Tuple[Sequence[int], int]]] = None,
                spare_rows: int = 3, sm_scale: Optional[float] = None,
                meta: Optional[Dict] = None, page_size: int = 1) -> Batch:
    """Assign slots and draw values for ``specs``.

    ``cascade``: optional list of (spec indices of decode members, prefix_len);
    the first member is the group leader whose table row holds the prefix.
    ``page_size`` > 1: slots come in pages of that many consecutive slots (page 0
    reserved); a sequence's own tokens fill fresh pages in order, and sharing
    with a parent is page-granular (every fork a multiple of the page size).
    """
    specs = list(specs)
    rng = np.random.Generator(np.random.PCG64(seed))
    for r, s in enumerate(specs):
        assert s.kind in ("extend", "decode", "cached"), s.kind
        assert 0 <= s.cached_len <= s.total_len, s
        if s.kind == "decode":
            assert s.total_len == s.cached_len + 1, s
        if s.kind == "cached":
            assert s.total_len == s.cached_len, s
        if s.parent >= 0:
            assert s.parent < r and 0 <= s.fork <= specs[s.parent].cached_len, (r, s)
            assert s.fork <= s.cached_len, (r, s)
        else:
            assert s.fork == 0, s

    n_unique = sum(s.total_len - s.fork for s in specs)
    if page_size == 1:
        assert n_unique <= num_slots - 1, (n_unique, num_slots)
        fresh = (rng.permutation(num_slots - 1)[:n_unique] + 1).astype(np.int32)
    else:
        assert page_size > 1 and num_slots % page_size == 0, (page_size, num_slots)
        assert all(s.fork % page_size == 0 for s in specs), "forks must be page-aligned"
        n_pages = sum(-(-(s.total_len - s.fork) // page_size) for s in specs)
        assert n_pages <= num_slots // page_size - 1, (n_pages, num_slots // page_size)
        pages = rng.permutation(num_slots // page_size - 1)[:n_pages] + 1
        runs, k = [], 0
        for s in specs:  # each sequence's own tokens: its pages' slots in order
            own = s.total_len - s.fork
            npg = -(-own // page_size)
            pg = pages[k:k + npg]
            k += npg
            runs.append((pg[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)[:own])
        fresh = (np.concatenate(runs) if runs else np.zeros(0, np.int64)).astype(np.int32)

    slots: List[np.ndarray] = []
    tokens: List[np.ndarray] = []
    next_tok = 0
    pos = 0
    cached_slots: List[np.ndarray] = []
    for r, s in enumerate(specs):
        own = fresh[pos:pos + s.total_len - s.fork]
        pos += s.total_len - s.fork
        if s.parent >= 0:
            row = np.concatenate([slots[s.parent][:s.fork], own])
            tk = np.concatenate([tokens[s.parent][:s.fork],
                                 np.arange(next_tok, next_tok + s.cached_len - s.fork, dtype=np.int32)])
        else:
            row = own
            tk = np.arange(next_tok, next_tok + s.cached_len, dtype=np.int32)
        next_tok += s.cached_len - s.fork
        slots.append(row.astype(np.int32))
        tokens.append(tk.astype(np.int32))
        cached_slots.append(row[s.fork:s.cached_len])

    pool_slots = np.concatenate(cached_slots).astype(np.int64) if cached_slots else np.zeros(0, np.int64)
    ext_ids = [r for r, s in enumerate(specs) if s.kind == "extend"]
    dec_ids = [r for r, s in enumerate(specs) if s.kind == "decode"]
    batch_ids = ext_ids + dec_ids

    n_rows = len(batch_ids) + spare_rows
    rows = rng.permutation(n_rows)[:len(batch_ids)].astype(np.int32)
    lmax = max([specs[r].total_len for r in batch_ids] + [1])
    table = np.full((n_rows, lmax), NO_SLOT, dtype=np.int32)
    for k, r in enumerate(batch_ids):
        table[rows[k], :specs[r].total_len] = slots[r]
    ext_rpi = rows[:len(ext_ids)]
    dec_rpi = rows[len(ext_ids):]

    ext_prefix = np.array([specs[r].cached_len for r in ext_ids], np.int32)
    ext_len = np.array([specs[r].total_len - specs[r].cached_len for r in ext_ids], np.int32)
    qo = np.zeros(len(ext_ids) + 1, np.int32)
    qo[1:] = np.cumsum(ext_len)
    dec_lens = np.array([specs[r].total_len for r in dec_ids], np.int32)

    new_loc = [slots[r][specs[r].cached_len:] for r in ext_ids] + [slots[r][-1:] for r in dec_ids]
    out_cache_loc = np.concatenate(new_loc).astype(np.int32) if new_loc else np.zeros(0, np.int32)

    hkv, d, hq = num_kv_heads, head_dim, num_q_heads
    pool_k = _normal_bf16(rng, (pool_slots.size, hkv, d))
    pool_v = _normal_bf16(rng, (pool_slots.size, hkv, d))
    k_new = _normal_bf16(rng, (out_cache_loc.size, hkv, d))
    v_new = _normal_bf16(rng, (out_cache_loc.size, hkv, d))
    ext_q = _normal_bf16(rng, (int(qo[-1]), hq, d))
    dec_q = _normal_bf16(rng, (len(dec_ids), hq, d))

    gi = gr = gp = None
    if cascade:
        dec_pos = {r: k for k, r in enumerate(dec_ids)}
        gi = [0]
        gr, gp = [], []
        for members, plen in cascade:
            for m in members:
                assert specs[m].kind == "decode"
                assert np.array_equal(slots[m][:plen], slots[members[0]][:plen]), "members must share the prefix"
                assert plen <= specs[m].total_len
                gr.append(dec_pos[m])
            gi.append(len(gr))
            gp.append(plen)
        gi, gr, gp = (np.array(x, np.int32) for x in (gi, gr, gp))

    return Batch(
        name=name, num_slots=num_slots, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
        sm_scale=float(np.float32(1.0 / math.sqrt(d))) if sm_scale is None else float(np.float32(sm_scale)),
        pool_slots=pool_slots, pool_k=pool_k, pool_v=pool_v,
        out_cache_loc=out_cache_loc, k_new=k_new, v_new=v_new, req_to_token=table,
        ext_rpi=ext_rpi, ext_prefix_lens=ext_prefix, ext_extend_lens=ext_len, ext_qo_indptr=qo, ext_q=ext_q,
        dec_rpi=dec_rpi, dec_seq_lens=dec_lens, dec_q=dec_q,
        casc_group_indptr=gi, casc_group_reqs=gr, casc_group_prefix_len=gp,
        tokens=tokens, specs=specs, meta=dict(meta or {}, seed=seed))


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def tiny_extend_decode(seed: int = 1) -> Tuple[Batch, Batch]:
    """Tiny correctness case: 4 requests share a 32-token cached prefix, suffixes
    of 8/12/16/24 tokens, 8 q heads / 2 kv heads, head_dim 64, 512 slots.

    Returns (extend step, decode step).  The decode step continues the same
    requests: its pool holds the prefix and the stored suffixes (same slots and
    values), and each request adds one token (L = 32 + E + 1).  96 slots used.
    """
    suffix = [8, 12, 16, 24]
    specs = [SeqSpec(32, 32, "cached")] + [SeqSpec(32 + e, 32, "extend", parent=0, fork=32) for e in suffix]
    ext = build_batch("tiny_extend", specs, num_slots=512, num_q_heads=8, num_kv_heads=2,
                      head_dim=64, seed=seed)
    # decode step: same slots for the first 32+E positions, one new slot each
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    used = set(ext.pool_slots.tolist()) | set(ext.out_cache_loc.tolist())
    free = np.array(sorted(set(range(1, 512)) - used), np.int64)
    new_slots = rng.permutation(free)[:4].astype(np.int32)
    pool_slots = np.concatenate([ext.pool_slots, ext.out_cache_loc.astype(np.int64)])
    pool_k = np.concatenate([ext.pool_k, ext.k_new])
    pool_v = np.concatenate([ext.pool_v, ext.v_new])
    table = ext.req_to_token.copy()
    lmax = 32 + max(suffix) + 1
    table = np.concatenate([table, np.full((table.shape[0], lmax - table.shape[1]), NO_SLOT, np.int32)], axis=1)
    seq_lens = np.array([32 + e + 1 for e in suffix], np.int32)
    for k in range(4):
        table[ext.ext_rpi[k], seq_lens[k] - 1] = new_slots[k]
    dec = Batch(
        name="tiny_decode", num_slots=512, num_q_heads=8, num_kv_heads=2, head_dim=64,
        sm_scale=ext.sm_scale, pool_slots=pool_slots, pool_k=pool_k, pool_v=pool_v,
        out_cache_loc=new_slots, k_new=_normal_bf16(rng, (4, 2, 64)), v_new=_normal_bf16(rng, (4, 2, 64)),
        req_to_token=table,
        ext_rpi=np.zeros(0, np.int32), ext_prefix_lens=np.zeros(0, np.int32),
        ext_extend_lens=np.zeros(0, np.int32), ext_qo_indptr=np.zeros(1, np.int32),
        ext_q=np.zeros((0, 8, 64), np.uint16),
        dec_rpi=ext.ext_rpi.copy(), dec_seq_lens=seq_lens, dec_q=_normal_bf16(rng, (4, 8, 64)),
        casc_group_indptr=np.array([0, 4], np.int32), casc_group_reqs=np.arange(4, dtype=np.int32),
        casc_group_prefix_len=np.array([32], np.int32),
        tokens=ext.tokens, specs=ext.specs, meta={"seed": seed})
    return ext, dec


def decode_8b_system_prompts(seed: int = 2, page_size: int = 1) -> Batch:
    """Decode, Llama-3-8B attention shape: batch 64, 32 q / 8 kv heads, head_dim 128.
    Context lengths (including the new token) uniform in 512..4096; 8 groups of 8
    requests share a 1024-token system prompt (same slots); pool of 512K slots.
    A request whose context is shorter than prompt + 1 shares L - 1 prompt tokens.
    The cascade groups list, per system prompt, the members holding all 1024."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    specs: List[SeqSpec] = [SeqSpec(1024, 1024, "cached") for _ in range(8)]
    groups = []
    for g in range(8):
        members = []
        for i in range(8):
            L = int(lens[g * 8 + i])
            f = min(1024, L - 1) // page_size * page_size
            specs.append(SeqSpec(L, L - 1, "decode", parent=g, fork=f))
            if f == 1024:
                members.append(len(specs) - 1)
        if len(members) >= 2:
            groups.append((members, 1024))
    name = "decode_8b_system_prompts" if page_size == 1 else f"decode_8b_system_prompts_page{page_size}"
    return build_batch(name, specs, num_slots=512 * 1024, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed + 1,
                       cascade=groups, page_size=page_size)


def fewshot_extend(seed: int = 3) -> Batch:
    """Few-shot extend: 16 requests share a cached 3000-token prefix, each with
    200..400 new suffix tokens; 32 q / 8 kv heads, head_dim 128, scale 1/sqrt(128)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ext = rng.integers(200, 400, size=16, endpoint=True)
    specs = [SeqSpec(3000, 3000, "cached")] + [
        SeqSpec(3000 + int(e), 3000, "extend", parent=0, fork=3000) for e in ext]
    return build_batch("fewshot_extend", specs, num_slots=64 * 1024, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, seed=seed + 1)


def forked_decode_70b(seed: int = 4) -> Batch:
    """Forked-branch decode, Llama-3-70B attention shape (64 q / 8 kv heads, D 128):
    one 8192-token shared prefix, 64 sibling branches with 0..256 private tokens
    each, then one decode token per branch (L = 8192 + p + 1).  One cascade group."""
    rng = np.random.Generator(np.random.PCG64(seed))
    priv = rng.integers(0, 256, size=64, endpoint=True)
    specs = [SeqSpec(8192, 8192, "cached")]
    for p in priv:
        L = 8192 + int(p) + 1
        specs.append(SeqSpec(L, L - 1, "decode", parent=0, fork=8192))
    return build_batch("forked_decode_70b", specs, num_slots=64 * 1024, num_q_heads=64, num_kv_heads=8,
                       head_dim=128, seed=seed + 1, cascade=[(list(range(1, 65)), 8192)])


def _multiturn_mix_specs(lens: np.ndarray, is_ext: np.ndarray, ext_len: np.ndarray, u: np.ndarray,
                pick: np.ndarray, alpha: float, window: int) -> Tuple[List[SeqSpec], float]:
    specs: List[SeqSpec] = []
    num = den = 0
    for r in range(lens.size):
        L = int(lens[r])
        C = L - int(ext_len[r]) if is_ext[r] else L - 1
        kind = "extend" if is_ext[r] else "decode"
        parent, fork = -1, 0
        if r > 0 and u[r] < alpha:
            parent = r - 1 - int(pick[r] % min(window, r))
            fork = min(specs[parent].cached_len, C)
            if fork == 0:
                parent = -1
        specs.append(SeqSpec(L, C, kind, parent=parent, fork=fork))
        num += fork
        den += C
    return specs, (num / den if den else 0.0)


def multiturn_mix_70b(seed: int = 5, target_hit: float = 0.70, num_slots: int = 2 * 1024 * 1024) -> Batch:
    """Multi-turn chat mix, 70B heads (64 / 8, D 128): 256 requests, contexts
    lognormal(median 2048, sigma 1) clipped to [16, 32768].  Sequences are generated
    in ascending length; with probability alpha a request continues or forks one of
    the 8 sequences generated just before it (sharing as much of that sequence's
    cached prefix as it can), otherwise it starts fresh.  alpha is bisected so the
    token-weighted prefix hit ratio of the construction is target_hit +- 0.01.
    32 requests (seeded choice) are extend with suffix 64..512 (at most L), the
    other 224 are decode.  Pool of 2M slots, one per tree token."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.clip(np.round(rng.lognormal(mean=math.log(2048.0), sigma=1.0, size=256)), 16, 32768).astype(np.int64)
    lens.sort()
    is_ext = np.zeros(256, bool)
    is_ext[rng.permutation(256)[:32]] = True
    ext_len = np.minimum(rng.integers(64, 512, size=256, endpoint=True), lens)
    ext_len = np.where(is_ext, ext_len, 1)
    u = rng.random(256)
    pick = rng.integers(0, 1 << 30, size=256)
    lo, hi = 0.0, 1.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        _, h = _multiturn_mix_specs(lens, is_ext, ext_len, u, pick, mid, 8)
        if h < target_hit:
            lo = mid
        else:
            hi = mid
    alpha = hi
    specs, hit = _multiturn_mix_specs(lens, is_ext, ext_len, u, pick, alpha, 8)
    assert abs(hit - target_hit) <= 0.01, hit
    return build_batch("multiturn_mix_70b", specs, num_slots=num_slots, num_q_heads=64, num_kv_heads=8,
                       head_dim=128, seed=seed + 1,
                       meta={"alpha": alpha, "construction_hit_ratio": hit})


def random_mixed(seed: int, *, n_extend: int, n_decode: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, max_len: int, num_slots: Optional[int] = None,
                 share_prob: float = 0.6, min_len: int = 1, with_cascade: bool = False,
                 ext_lens: Optional[Sequence[int]] = None, page_size: int = 1) -> Batch:
    """A ragged mixed batch for parity tests: random lengths in [min_len, max_len],
    random forks of earlier sequences (multi-level sharing), extend suffixes of
    random length (prefix 0 allowed), optional cascade groups of decode requests
    that share a common prefix of at least 1 token."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = n_extend + n_decode
    kinds = ["extend"] * n_extend + ["decode"] * n_decode
    kinds = [kinds[i] for i in rng.permutation(n)]
    specs: List[SeqSpec] = []
    for r in range(n):
        L = int(rng.integers(min_len, max_len, endpoint=True))
        if kinds[r] == "extend":
            E = int(ext_lens[len([s for s in specs if s.kind == 'extend'])]) if ext_lens is not None \
                else int(rng.integers(1, L, endpoint=True))
            E = max(1, min(E, L))
            C = L - E
        else:
            L = max(L, 1)
            C = L - 1
        parent, fork = -1, 0
        if specs and rng.random() < share_prob:
            parent = int(rng.integers(0, len(specs)))
            fork = int(rng.integers(0, min(specs[parent].cached_len, C), endpoint=True))
            fork = fork // page_size * page_size  # page-granular sharing
            if fork == 0:
                parent = -1
        specs.append(SeqSpec(L, C, kinds[r], parent=parent, fork=fork))
    cascade = None
    if with_cascade:
        # group decode requests by (root ancestor) when they share >= 1 token with it
        dec = [r for r, s in enumerate(specs) if s.kind == "decode"]
        by_root: Dict[int, List[int]] = {}
        for r in dec:
            a = r
            while specs[a].parent >= 0:
                a = specs[a].parent
            by_root.setdefault(a, []).append(r)
        cascade = []
        for root, members in by_root.items():
            # common prefix length: walk each member's fork chain down to the root
            def shared_with_root(m: int) -> int:
                f = specs[m].total_len
                a = m
                while specs[a].parent >= 0:
                    f = min(f, specs[a].fork)
                    a = specs[a].parent
                return f if a == root else 0
            plen = min(shared_with_root(m) for m in members)
            if root in members and len(members) >= 1:
                plen = min(plen, specs[root].total_len - 1)
            if len(members) >= 2 and plen >= 1:
                cascade.append((members, plen))
    if page_size == 1:
        total_unique = sum(s.total_len - s.fork for s in specs)
        S = num_slots or max(64, 2 * total_unique + 8)
    else:
        pages = sum(-(-(s.total_len - s.fork) // page_size) for s in specs)
        S = num_slots or page_size * (2 * pages + 8)
    return build_batch(f"random_mixed_{seed}" + (f"_page{page_size}" if page_size > 1 else ""), specs,
                       num_slots=S, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                       seed=seed + 7919, cascade=cascade, page_size=page_size)


WORKLOADS = {
    "decode_8b_system_prompts": decode_8b_system_prompts,
    "fewshot_extend": fewshot_extend,
    "forked_decode_70b": forked_decode_70b,
    "multiturn_mix_70b": multiturn_mix_70b,
}
