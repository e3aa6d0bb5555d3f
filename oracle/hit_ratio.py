"""Token-weighted prefix-cache hit ratio -- TEST INFRASTRUCTURE ONLY.

Definitions followed (yaopepe.com explainer of the SGLang paper, §04
"RadixAttention：以树管理跨请求缓存"):
  * hit ratio = sum_r cached_prefill_tokens(r) / sum_r prefill_tokens(r),
    weighted by tokens, not by requests;
  * for a request set with radix tree T, the prefill tokens any schedule must
    compute are at least C_DFS = sum over edges e of |e|, and the optimal hit
    ratio is 1 - C_DFS / sum_r prefill_tokens(r) (Theorem 3.1, also in the
    SGLang paper summary, appendix A.3).

``cached_prefix_lengths`` is the plain definition under an unbounded cache
with no eviction: request r, processed after requests 0..r-1, finds cached the
longest prefix it shares with any earlier request.  ``c_dfs`` counts the
distinct non-empty prefixes of the request set, which is the total edge length
of its (compressed or not) prefix tree.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np


def _lcp(a: np.ndarray, b: np.ndarray) -> int:
    n = min(a.size, b.size)
    if n == 0:
        return 0
    diff = np.nonzero(a[:n] != b[:n])[0]
    return int(diff[0]) if diff.size else n


def cached_prefix_lengths(seqs: Sequence[np.ndarray]) -> List[int]:
    out = []
    for r, s in enumerate(seqs):
        best = 0
        for p in range(r):
            best = max(best, _lcp(np.asarray(s), np.asarray(seqs[p])))
        out.append(best)
    return out


def hit_ratio(seqs: Sequence[np.ndarray]) -> float:
    cached = cached_prefix_lengths(seqs)
    total = sum(int(np.asarray(s).size) for s in seqs)
    return sum(cached) / total if total else 0.0


def c_dfs(seqs: Sequence[np.ndarray]) -> int:
    """Number of distinct non-empty prefixes = sum of the prefix tree's edge lengths."""
    seen = set()
    for s in seqs:
        t = tuple(int(x) for x in np.asarray(s).tolist())
        for k in range(1, len(t) + 1):
            seen.add(t[:k])
    return len(seen)


def optimal_hit_ratio(seqs: Sequence[np.ndarray]) -> float:
    total = sum(int(np.asarray(s).size) for s in seqs)
    return 1.0 - c_dfs(seqs) / total if total else 0.0
