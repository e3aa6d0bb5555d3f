"""Pins for the hit-ratio oracle (no GPU): the pages' worked example, Theorem 3.1's
identity for an unbounded cache, and a brute-force cache-of-prefixes simulation."""
import os

import numpy as np
import pytest

from oracle import hit_ratio as H
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _worked_example():
    steps = []
    for line in open(os.path.join(GOLDEN, "radix_worked_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        step, op, toks, matched, edges = line.split("|")
        steps.append((op, np.array([int(x) for x in toks.split()], np.int32), matched))
    return steps


def test_worked_example_matched_lengths_and_ratio():
    # unbounded cache (no eviction): the inserts of the worked example
    seqs = [t for op, t, _ in _worked_example() if op == "insert"]
    assert H.cached_prefix_lengths(seqs) == [0, 4, 4]
    # token weighted: (0 + 4 + 4) / (6 + 7 + 5)
    assert H.hit_ratio(seqs) == pytest.approx(8 / 18, abs=0)
    # C_DFS: distinct prefixes = |S + A| + |B| + |C| = 6 + 3 + 1
    assert H.c_dfs(seqs) == 10
    assert H.optimal_hit_ratio(seqs) == pytest.approx(1 - 10 / 18, abs=1e-15)


def _brute_cache_of_prefixes(seqs):
    cache = set()
    hits = 0
    for s in seqs:
        t = tuple(int(x) for x in s)
        k = max([j for j in range(len(t) + 1) if t[:j] in cache or j == 0])
        hits += k
        for j in range(1, len(t) + 1):
            cache.add(t[:j])
    return hits


@pytest.mark.parametrize("seed", range(8))
def test_unbounded_cache_reaches_c_dfs_in_any_order(seed):
    rng = np.random.default_rng(seed)
    # small alphabet so prefixes collide often
    seqs = [rng.integers(0, 3, size=rng.integers(1, 9)).astype(np.int32) for _ in range(12)]
    total = sum(s.size for s in seqs)
    for order in (range(12), rng.permutation(12)):
        ordered = [seqs[i] for i in order]
        hits = sum(H.cached_prefix_lengths(ordered))
        assert hits == _brute_cache_of_prefixes(ordered)
        assert total - hits == H.c_dfs(ordered)
        assert H.hit_ratio(ordered) == pytest.approx(H.optimal_hit_ratio(ordered), abs=1e-15)


def test_generator_construction_ratio_matches_definition_small():
    b = W.random_mixed(5, n_extend=4, n_decode=8, num_q_heads=2, num_kv_heads=1, head_dim=8, max_len=60)
    # generator: sequence r shares exactly its fork with its parent; fresh tokens are unique
    cached = H.cached_prefix_lengths(b.tokens)
    assert cached == [s.fork for s in b.specs]


def test_multiturn_mix_hit_ratio_is_seventy_percent():
    b = W.multiturn_mix_70b()
    hr = H.hit_ratio(b.tokens)
    assert abs(hr - 0.70) <= 0.01
    assert hr == pytest.approx(b.meta["construction_hit_ratio"], abs=1e-12)
