"""Host radix-tree prefix cache (no GPU): the pages' worked example with eviction, the hit
ratio against the oracle's definition, reference-count protection, LRU order, slot reuse,
and the cascade groups it derives for a decode batch."""
import os

import numpy as np
import pytest

from oracle import hit_ratio as H
from prefix_shared_kv_ra_gb300.radix import RadixCache, SlotPool, cascade_groups
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_steps():
    out = []
    for line in open(os.path.join(GOLDEN, "radix_worked_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        step, op, toks, matched, edges = line.split("|")
        edge_set = set()
        for e in edges.split(";"):
            parent, edge = e.split(":")
            edge_set.add((tuple(int(x) for x in parent.split()), tuple(int(x) for x in edge.split())))
        out.append((op, [int(x) for x in toks.split()], matched, edge_set))
    return out


def test_worked_example_insert_split_evict():
    pool = SlotPool(64)
    cache = RadixCache(pool)
    running = {}
    for op, toks, matched, edges in _golden_steps():
        if op == "insert":
            got, node = cache.match_prefix(toks)
            assert got.size == int(matched)
            slots = np.concatenate([got, pool.alloc(len(toks) - got.size)])
            cache.insert(toks, slots)
            # the newest request is running; the earlier ones are finished
            for n in running.values():
                cache.unlock(n)
            running = {tuple(toks): cache.path(toks)[-1]}
            cache.lock(running[tuple(toks)])
        else:
            # A is the least recently used unreferenced leaf; B (running) is protected
            freed = cache.evict(len(toks) - 4)
            assert freed == len(toks) - 4
        assert set(cache.edges()) == edges


def test_unbounded_cache_matches_hit_ratio_definition():
    b = W.random_mixed(3, n_extend=3, n_decode=20, num_q_heads=2, num_kv_heads=1, head_dim=8, max_len=200)
    pool = SlotPool(1 << 16)
    cache = RadixCache(pool)
    matched = []
    for toks in b.tokens:
        got, _ = cache.match_prefix(toks)
        matched.append(int(got.size))
        cache.insert(toks, np.concatenate([got, pool.alloc(len(toks) - got.size)]))
    assert matched == H.cached_prefix_lengths(b.tokens)
    total = sum(len(t) for t in b.tokens)
    assert cache.total_tokens() == H.c_dfs(b.tokens)
    assert sum(matched) / total == pytest.approx(H.hit_ratio(b.tokens), abs=1e-15)


def test_eviction_respects_locks_lru_and_returns_slots():
    pool = SlotPool(100)
    cache = RadixCache(pool)
    seqs = [[1, 2, 3, 4], [1, 2, 5, 6], [1, 2, 7], [9, 9]]
    for s in seqs:
        got, _ = cache.match_prefix(s)
        cache.insert(s, np.concatenate([got, pool.alloc(len(s) - got.size)]))
    before = pool.available()
    locked = cache.path([1, 2, 5, 6])[-1]
    cache.lock(locked)
    # LRU leaves: [3,4] (oldest), then [7], then [9,9] ... [5,6] is locked
    assert cache.evict(1) == 2 and pool.available() == before + 2
    assert ((1, 2), (3, 4)) not in set(cache.edges())
    freed = cache.evict(100)  # everything unlocked goes; [1,2] stays (ancestor of a locked leaf)
    assert set(cache.edges()) == {((), (1, 2)), ((1, 2), (5, 6))}
    assert pool.available() == before + 2 + freed
    cache.unlock(locked)
    cache.evict(100)
    assert cache.edges() == [] and pool.available() == 99


def test_cascade_groups_share_their_prefix_slots():
    b = W.cfg2_decode_8b()
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    gi, gr, gp = cascade_groups(rows)
    assert gi.size - 1 == 8  # one group per system prompt
    for g in range(gi.size - 1):
        mem = gr[gi[g]:gi[g + 1]]
        lead = rows[mem[0]][:gp[g]]
        for m in mem:
            assert gp[g] <= rows[m].size - 1
            np.testing.assert_array_equal(rows[m][:gp[g]], lead)
        # the group prefix is the shortest member's context minus its own new token, at most the prompt
        assert gp[g] == min(1024, min(rows[m].size - 1 for m in mem))
