"""Host-side radix-tree prefix cache over the token-granular KV pool.

The cache maps token sequences to the pool slots that hold their K/V, so a
new request reuses the slots of the longest cached prefix and only computes
its suffix (SGLang paper summary, §3 "Efficient KV Cache Reuse with
RadixAttention"; the yaopepe.com explainer, §04):

* a node's edge is a run of tokens with the slots of those tokens;
* matching walks from the root edge by edge; a match that ends inside an
  edge splits it, so the shared part becomes a common ancestor (the
  explainer's figure: S+A and S+B become S with children A and B);
* running requests hold a reference on every node of their path; only
  unreferenced leaves may be evicted, least recently used first, and a parent
  that becomes an unreferenced leaf becomes a candidate in turn;
* evicted slots go back to the slot pool for reuse;
* with pages of P > 1 slots (P consecutive slots per page), the cache shares
  whole pages only: matches and inserts are cut to a multiple of P, so every
  edge starts and ends on a page boundary and eviction frees whole pages.

This is support code for the attention path: it produces the
``req_to_token`` rows, the cascade groups and the hit ratio the kernels and
the benchmarks use.  It holds no attention arithmetic.
"""
from __future__ import annotations

import heapq
import itertools
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

__all__ = ["SlotPool", "RadixCache", "cascade_groups"]


class SlotPool:
    """Free list of token slots in pages of `page_size` consecutive slots; page 0 (holding slot 0,
    the dummy slot padded requests write) is never handed out.  The free pages form a stack: the
    lowest pages go out first at the start, and freed pages are handed out again before older ones.
    Freeing a page that is already free raises (it would be handed out twice)."""

    def __init__(self, num_slots: int, page_size: int = 1):
        if page_size < 1 or num_slots % page_size:
            raise ValueError("num_slots must be a multiple of page_size")
        self.num_slots = int(num_slots)
        self.page_size = int(page_size)
        n_pages = self.num_slots // page_size
        self._stack = np.arange(n_pages - 1, 0, -1, dtype=np.int64)  # free pages; the top is handed out first
        self._top = self._stack.size
        self._is_free = np.ones(n_pages, dtype=bool)
        self._is_free[0] = False

    def available(self) -> int:
        """Free slots (whole pages)."""
        return self._top * self.page_size

    def free_pages(self) -> np.ndarray:
        """The free pages, the next one to be handed out last."""
        return self._stack[:self._top].copy()

    def alloc(self, n: int) -> Optional[np.ndarray]:
        """Slots for n new tokens, in order: the first n slots of ceil(n / page_size) fresh pages (the rest
        of the last page stays with the caller until freed)."""
        pages = -(-n // self.page_size)
        if pages > self._top:
            return None
        out = self._stack[self._top - pages:self._top][::-1].copy()
        self._top -= pages
        self._is_free[out] = False
        slots = (out[:, None] * self.page_size + np.arange(self.page_size)[None, :]).reshape(-1)[:n]
        return slots.astype(np.int32)

    def free(self, slots: Sequence[int]) -> None:
        """Return the pages holding these slots."""
        s = np.asarray(slots, dtype=np.int64)
        if s.size == 0:
            return
        if s.min() < self.page_size or s.max() >= self.num_slots:
            raise ValueError("slot out of range")
        pages = np.unique(s // self.page_size)
        if self._is_free[pages].any():
            raise ValueError("a page freed twice")
        self._stack[self._top:self._top + pages.size] = pages
        self._top += pages.size
        self._is_free[pages] = True


class _Node:
    __slots__ = ("key", "value", "children", "parent", "lock_ref", "last_access", "uid")
    _ids = itertools.count()

    def __init__(self, key: np.ndarray, value: np.ndarray, parent: Optional["_Node"]):
        self.key = key          # int32 tokens of the edge into this node
        self.value = value      # int32 slots of those tokens
        self.children: Dict[int, "_Node"] = {}
        self.parent = parent
        self.lock_ref = 0
        self.last_access = 0
        self.uid = next(_Node._ids)


def _common_len(a: np.ndarray, b: np.ndarray) -> int:
    n = min(a.size, b.size)
    if n == 0:
        return 0
    neq = a[:n] != b[:n]
    i = int(neq.argmax())  # the first mismatch (argmax of a boolean array stops at the first True)
    return i if neq[i] else n


class RadixCache:
    def __init__(self, pool: SlotPool):
        self.pool = pool
        self.page = pool.page_size
        self.root = _Node(np.zeros(0, np.int32), np.zeros(0, np.int32), None)
        self.root.lock_ref = 1  # never evicted
        self._clock = 0
        self.evictable_size = 0  # tokens in nodes no running request references (all can be evicted)

    # ------------------------------------------------------------------ queries
    def _child_key(self, key: np.ndarray):
        """A child is found by the first page of its edge: siblings may share leading tokens within
        a page (an edge is split on page boundaries only), never a whole first page."""
        return int(key[0]) if self.page == 1 else tuple(key[:self.page].tolist())

    def _tick(self) -> int:
        self._clock += 1
        return self._clock

    def match_prefix(self, tokens: Sequence[int]) -> Tuple[np.ndarray, _Node]:
        """Slots of the longest cached prefix of `tokens` (whole pages) and the node where it ends
        (an edge matched part-way is split there)."""
        key = np.asarray(tokens, dtype=np.int32)
        node, pos, slots = self.root, 0, []
        now = self._tick()
        node.last_access = now
        while pos < key.size:
            child = node.children.get(self._child_key(key[pos:]))
            if child is None:
                break
            k = _common_len(child.key, key[pos:]) // self.page * self.page
            if k == 0:
                break
            child.last_access = now
            if k < child.key.size:
                child = self._split(child, k)
                slots.append(child.value)
                node = child
                pos += k
                break
            slots.append(child.value)
            node = child
            pos += k
        value = np.concatenate(slots) if slots else np.zeros(0, np.int32)  # a fresh array either way
        return value.astype(np.int32, copy=False), node

    def _split(self, child: _Node, k: int) -> _Node:
        """Make the first k tokens of child's edge a new node between child and its parent."""
        parent = child.parent
        mid = _Node(child.key[:k].copy(), child.value[:k].copy(), parent)
        mid.lock_ref = child.lock_ref
        mid.last_access = child.last_access
        parent.children[self._child_key(mid.key)] = mid
        child.key, child.value = child.key[k:].copy(), child.value[k:].copy()
        child.parent = mid
        mid.children[self._child_key(child.key)] = child
        return mid

    def insert(self, tokens: Sequence[int], slots: Sequence[int]) -> int:
        """Insert tokens with their slots (their whole pages only); returns how many leading tokens
        were already cached (the caller frees its duplicate slots for those positions)."""
        key = np.asarray(tokens, dtype=np.int32)
        val = np.asarray(slots, dtype=np.int32)
        assert key.size == val.size
        n = key.size // self.page * self.page
        key, val = key[:n], val[:n]
        matched, node = self.match_prefix(key)
        k = matched.size
        if k < key.size:
            leaf = _Node(key[k:].copy(), val[k:].copy(), node)
            leaf.last_access = self._tick()
            node.children[self._child_key(leaf.key)] = leaf
            self.evictable_size += leaf.key.size
        return k

    def path(self, tokens: Sequence[int]) -> List[_Node]:
        """Nodes along the cached prefix of tokens (after splitting at its end)."""
        _, node = self.match_prefix(tokens)
        out = []
        while node is not self.root:
            out.append(node)
            node = node.parent
        return out[::-1]

    # ------------------------------------------------------------------ references
    def lock(self, node: _Node) -> None:
        while node is not None:
            if node.lock_ref == 0:
                self.evictable_size -= node.key.size
            node.lock_ref += 1
            node = node.parent

    def unlock(self, node: _Node) -> None:
        while node is not None:
            node.lock_ref -= 1
            assert node.lock_ref >= 0
            if node.lock_ref == 0:
                self.evictable_size += node.key.size
            node = node.parent

    # ------------------------------------------------------------------ eviction
    def _leaves(self) -> List[_Node]:
        out, stack = [], [self.root]
        while stack:
            n = stack.pop()
            if not n.children and n is not self.root:
                out.append(n)
            stack.extend(n.children.values())
        return out

    def evict(self, num_tokens: int) -> int:
        """Free at least num_tokens slots by removing unreferenced leaves, least recently used first.
        Returns the number of slots freed (less if everything left is referenced)."""
        heap = [(n.last_access, n.uid, n) for n in self._leaves() if n.lock_ref == 0]
        heapq.heapify(heap)
        freed = 0
        while freed < num_tokens and heap:
            _, _, leaf = heapq.heappop(heap)
            self.pool.free(leaf.value)
            freed += leaf.value.size
            self.evictable_size -= leaf.key.size
            parent = leaf.parent
            del parent.children[self._child_key(leaf.key)]
            if parent is not self.root and not parent.children and parent.lock_ref == 0:
                heapq.heappush(heap, (parent.last_access, parent.uid, parent))
        return freed

    # ------------------------------------------------------------------ sizes
    def total_tokens(self) -> int:
        total, stack = 0, [self.root]
        while stack:
            n = stack.pop()
            total += n.key.size
            stack.extend(n.children.values())
        return total

    def edges(self) -> List[Tuple[Tuple[int, ...], Tuple[int, ...]]]:
        """(tokens of the parent path, tokens of the edge) for every node: a canonical view of the tree."""
        out, stack = [], [(self.root, ())]
        while stack:
            n, prefix = stack.pop()
            for c in n.children.values():
                e = tuple(int(x) for x in c.key.tolist())
                out.append((prefix, e))
                stack.append((c, prefix + e))
        return sorted(out)


def dfs_order(paths: Sequence[Sequence[int]]) -> np.ndarray:
    """The order in which a depth-first walk of the radix tree of these slot rows meets the requests:
    requests sorted lexicographically by their slot rows (a node's children are visited by their first
    slot, a request that ends at a node before the requests below it).  A scheduler that runs a batch in
    this order keeps requests that share a node next to each other, so their shared slots are read
    close together in time.  The SGLang paper summary (§3, cache-aware scheduling; A.3, proof of
    Theorem 3.1) schedules longest shared prefix first and shows that order equivalent to a depth-first
    walk of the radix tree."""
    return np.asarray(sorted(range(len(paths)), key=lambda b: tuple(int(x) for x in paths[b])), np.int64)


def cascade_groups(paths: Sequence[Sequence[int]], min_prefix: int = 1,
                   min_members: int = 2) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One-level cascade groups for a decode batch from its table rows.

    paths[b] is request b's slot row (context order).  Requests are grouped by
    their first slot (the subtree under the root they belong to); a group's
    prefix is the longest run of slots all its members share, capped so that
    every member keeps its last (new) token private.  Groups below min_members
    or min_prefix are dropped.  Returns (group_indptr, group_reqs,
    group_prefix_len) for ra_decode_attention.
    """
    by_first: Dict[int, List[int]] = {}
    for b, row in enumerate(paths):
        if len(row):
            by_first.setdefault(int(row[0]), []).append(b)
    indptr, reqs, plens = [0], [], []
    for _, members in sorted(by_first.items()):
        if len(members) < min_members:
            continue
        rows = [np.asarray(paths[b]) for b in members]
        plen = min(r.size - 1 for r in rows)
        lead = rows[0]
        for r in rows[1:]:
            plen = min(plen, _common_len(lead, r))
        if plen < min_prefix:
            continue
        reqs.extend(members)
        indptr.append(len(reqs))
        plens.append(plen)
    return (np.asarray(indptr, np.int32), np.asarray(reqs, np.int32), np.asarray(plens, np.int32))


def cascade_groups_multilevel(paths: Sequence[Sequence[int]], min_members: int = 2, min_range: int = 1):
    """Multi-level cascade groups for a decode batch: groups over the nodes of the tree of the requests'
    slot rows (each cut one token short, so every request keeps its newest token private) that at
    least `min_members` requests pass through.  A group covers positions [start, end) of its members,
    where end is its node's end and start the end of the group above it (0 at the top); a node whose
    range so far is shorter than `min_range` forms no group, and its positions go to the groups below
    it (its members that end there read them privately).  A group's level is the number of groups
    above it, so each request's groups cover positions 0 .. (its deepest end) - 1 without gaps.

    Returns (group_indptr, group_reqs, group_start, group_end, group_level, max_levels)."""
    root = {"key": np.zeros(0, np.int64), "children": {}, "reqs": []}
    for b, row in enumerate(paths):
        seq = np.asarray(row, dtype=np.int64)[:max(len(row) - 1, 0)]
        node, pos = root, 0
        while pos < seq.size:
            child = node["children"].get(int(seq[pos]))
            if child is None:
                leaf = {"key": seq[pos:].copy(), "children": {}, "reqs": [b]}
                node["children"][int(seq[pos])] = leaf
                pos = seq.size
                break
            k = _common_len(child["key"], seq[pos:])
            if k < child["key"].size:  # split the edge at k
                mid = {"key": child["key"][:k].copy(), "children": {}, "reqs": list(child["reqs"])}
                child["key"] = child["key"][k:].copy()
                mid["children"][int(child["key"][0])] = child
                node["children"][int(mid["key"][0])] = mid
                child = mid
            child["reqs"].append(b)
            node = child
            pos += k
    indptr, reqs, starts, ends, levels = [0], [], [], [], []
    max_levels = 0
    stack = [(root, 0, 0, 0)]  # node, depth at its start, start of its pending range, groups above it
    while stack:
        node, depth, pending, lvl = stack.pop()
        end = depth + node["key"].size
        is_group = node is not root and len(node["reqs"]) >= min_members and end - pending >= min_range
        if is_group:
            reqs.extend(sorted(node["reqs"]))
            indptr.append(len(reqs))
            starts.append(pending)
            ends.append(end)
            levels.append(lvl)
            max_levels = max(max_levels, lvl + 1)
        for c in node["children"].values():
            if len(c["reqs"]) >= min_members:  # only shared nodes can hold groups
                stack.append((c, end, end if is_group else pending, lvl + (1 if is_group else 0)))
    a = lambda x: np.asarray(x, np.int32)
    return a(indptr), a(reqs), a(starts), a(ends), a(levels), max_levels
