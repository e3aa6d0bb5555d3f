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
    b = W.decode_8b_system_prompts()
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


def test_paged_pool_hands_out_whole_pages_in_order():
    pool = SlotPool(64, page_size=16)
    assert pool.available() == 48  # page 0 (slots 0-15, the padding slot's page) is reserved
    a = pool.alloc(20)
    assert a.size == 20 and np.array_equal(a[:16], np.arange(16, 32)) and np.array_equal(a[16:], np.arange(32, 36))
    assert pool.available() == 16 and pool.alloc(17) is None
    pool.free(a)
    assert pool.available() == 48


def test_paged_cache_shares_whole_pages_only():
    P = 4
    pool = SlotPool(256, page_size=P)
    cache = RadixCache(pool)
    seq = list(range(100, 114))                      # 14 tokens: 3 whole pages cached
    slots = pool.alloc(len(seq))
    assert cache.insert(seq, slots) == 0
    assert cache.total_tokens() == 12
    got, _ = cache.match_prefix(seq)
    assert np.array_equal(got, slots[:12])
    other = seq[:9] + [7, 7, 7]                      # shares 9 tokens: 2 whole pages
    got, node = cache.match_prefix(other)
    assert got.size == 8 and np.array_equal(got, slots[:8])
    assert all(len(e) % P == 0 for _, e in cache.edges())  # the split fell on a page boundary
    assert cache.match_prefix(seq[:3])[0].size == 0        # less than a page: no hit


def test_paged_eviction_frees_whole_pages():
    P = 8
    pool = SlotPool(128, page_size=P)
    cache = RadixCache(pool)
    a = list(range(32))
    b = a[:16] + list(range(500, 516))
    sa = pool.alloc(32)
    cache.insert(a, sa)
    hit, _ = cache.match_prefix(b)
    assert hit.size == 16
    sb = np.concatenate([hit, pool.alloc(16)])
    cache.insert(b, sb)
    free0 = pool.available()
    assert cache.evict(1) == 16                      # one whole leaf (two pages)
    assert pool.available() == free0 + 16
    assert cache.evict(100) == 32                    # the other leaf, then the shared parent
    assert pool.available() == 120


def test_evictable_size_tracks_locks_inserts_and_evictions():
    rng = np.random.default_rng(5)
    pool = SlotPool(4096)
    cache = RadixCache(pool)
    locked = []

    def brute():
        out, stack = 0, [cache.root]
        while stack:
            n = stack.pop()
            if n is not cache.root and n.lock_ref == 0:
                out += n.key.size
            stack.extend(n.children.values())
        return out

    for step in range(300):
        op = rng.integers(0, 4)
        if op <= 1:  # a request: match, lock, insert its sequence
            base = [int(x) for x in rng.integers(0, 4, size=int(rng.integers(1, 4)))]
            seq = base + [int(x) for x in rng.integers(0, 50, size=int(rng.integers(1, 20)))]
            hit, node = cache.match_prefix(seq)
            cache.lock(node)
            locked.append(node)
            slots = pool.alloc(len(seq) - hit.size)
            if slots is None:
                cache.unlock(locked.pop())
                continue
            kept = cache.insert(seq, np.concatenate([hit, slots]))
            if kept > hit.size:
                pool.free(slots[:kept - hit.size])
        elif op == 2 and locked:
            cache.unlock(locked.pop(int(rng.integers(0, len(locked)))))
        else:
            cache.evict(int(rng.integers(1, 40)))
        assert cache.evictable_size == brute(), step


def test_multilevel_groups_are_the_shared_nodes_of_the_rows():
    # rows (slot sequences): a, b share 0..5; c shares 0..2 with them; d is alone
    base = list(range(100, 106))
    rows = [base + [1, 2, 3], base + [7, 8], base[:3] + [40, 41, 42, 43], [900, 901, 902]]
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    indptr, reqs, start, end, level, nl = cascade_groups_multilevel(rows)
    groups = {(int(s), int(e), int(l)): sorted(reqs[indptr[g]:indptr[g + 1]].tolist())
              for g, (s, e, l) in enumerate(zip(start, end, level))}
    assert groups == {(0, 3, 0): [0, 1, 2], (3, 6, 1): [0, 1]} and nl == 2
    # every request's groups cover 0 .. (deepest end) - 1 without gaps, members share the slots, and the
    # newest token stays private
    for b, row in enumerate(rows):
        mine = sorted((s, e) for (s, e, l), m in groups.items() if b in m)
        pos = 0
        for s, e in mine:
            assert s == pos
            pos = e
        assert pos <= len(row) - 1
    for (s, e, l), m in groups.items():
        for b in m:
            assert rows[b][s:e] == rows[m[0]][s:e]


def test_multilevel_groups_on_a_generated_batch():
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    b = W.multiturn_mix_70b()
    rows = [b.req_to_token[r, :L] for r, L in zip(b.dec_rpi, b.dec_seq_lens)]
    indptr, reqs, start, end, level, nl = cascade_groups_multilevel(rows)
    assert nl >= 2 and len(start) > 0
    cover = {}
    for g in range(len(start)):
        for m in reqs[indptr[g]:indptr[g + 1]]:
            cover.setdefault(int(m), []).append((int(start[g]), int(end[g]), int(level[g])))
            assert np.array_equal(rows[m][start[g]:end[g]], rows[reqs[indptr[g]]][start[g]:end[g]])
    for m, rng in cover.items():
        rng.sort()
        assert [l for _, _, l in rng] == list(range(len(rng)))   # one group per level, in depth order
        assert rng[0][0] == 0 and all(rng[i][1] == rng[i + 1][0] for i in range(len(rng) - 1))
        assert rng[-1][1] <= len(rows[m]) - 1


def test_multilevel_short_nodes_fold_into_the_groups_below():
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    base = list(range(100, 106))
    rows = [base + [1, 2, 3], base + [7, 8], base[:3] + [40, 41, 42, 43], [900, 901, 902]]
    indptr, reqs, start, end, level, nl = cascade_groups_multilevel(rows, min_range=4)
    groups = {(int(s), int(e), int(l)): sorted(reqs[indptr[g]:indptr[g + 1]].tolist())
              for g, (s, e, l) in enumerate(zip(start, end, level))}
    # the 3-token node shared by rows 0-2 is too short: its positions join the node below (rows 0, 1)
    assert groups == {(0, 6, 0): [0, 1]} and nl == 1



def _tree_pages(cache):
    """Every cached page as (tokens from the root to the end of the page) -> (its slots), read from
    the nodes.  With pages of one token this is every cached position and its slot."""
    out, stack, P = {}, [(cache.root, ())], cache.page
    while stack:
        node, pre = stack.pop()
        for c in node.children.values():
            key, val = c.key.tolist(), c.value.tolist()
            assert len(key) % P == 0 and len(key) > 0
            p = pre
            for j in range(0, len(key), P):
                p = p + tuple(key[j:j + P])
                out[p] = tuple(val[j:j + P])
            stack.append((c, p))
    return out


@pytest.mark.parametrize("page", [1, 4])
def test_random_operations_against_a_page_set_model(page):
    """Seeded random requests, finishes and evictions against a plain model of the cache: the set of
    cached pages, each named by the tokens from the root to its end (prefix-closed) and holding its
    slots.  Two requests that differ inside a page own a page each.  A request matches its longest
    cached run of whole pages, locks it, evicts if the pool is short, inserts its whole pages and
    holds them until it finishes.  Checked after every operation: the match and the slots it returns,
    the tree's pages and slots against the model, eviction only of unlocked pages (the least
    recently used unlocked leaf first, everything left locked when it frees too little), slots freed
    back to the pool exactly once, and the evictable-token count."""
    rng = np.random.default_rng(7 + page)
    pool = SlotPool(96, page_size=page)
    cache = RadixCache(pool)
    model = {}        # page path -> slots of the page
    live = []         # (cached tokens of a running request, its locked node)
    seen = []         # earlier requests, to fork from

    def locked_pages():
        return {tuple(toks[:j + page]) for toks, _ in live for j in range(0, len(toks), page)}

    def check_state():
        assert _tree_pages(cache) == model
        assert cache.total_tokens() == page * len(model)
        assert cache.evictable_size == page * (len(model) - len(locked_pages()))
        slots = np.asarray(sorted(s for v in model.values() for s in v), dtype=np.int64)
        assert np.unique(slots).size == slots.size                    # one token per slot
        free_pages = set(pool.free_pages().tolist())
        assert not any(s // page in free_pages for s in slots.tolist())  # none on a free page
        assert slots.size == 0 or slots.min() >= page                 # never the reserved page 0
        assert pool.available() + slots.size == pool.num_slots - page  # nothing leaks
        for p in model:                                               # prefix-closed
            assert len(p) == page or p[:-page] in model

    def evict(want):
        before = _tree_pages(cache)
        freed = cache.evict(want)
        after = _tree_pages(cache)
        removed = set(before) - set(after)
        assert set(after) <= set(before) and all(after[p] == before[p] for p in after)
        assert freed == page * len(removed)
        assert not (removed & locked_pages())
        for p in removed:
            del model[p]
        return freed, removed, after

    for step in range(2500):
        op = rng.random()
        if op < 0.55:                                                  # a new request
            if seen and rng.random() < 0.7:
                base = seen[int(rng.integers(len(seen)))]
                base = base[:int(rng.integers(0, len(base) + 1))]
            else:
                base = []
            toks = base + rng.integers(0, 3, size=int(rng.integers(1, 10))).tolist()
            got, node = cache.match_prefix(toks)
            L = 0
            while L + page <= len(toks) and tuple(toks[:L + page]) in model:
                L += page
            assert got.tolist() == [s for j in range(0, L, page) for s in model[tuple(toks[:j + page])]]
            cache.lock(node)                                           # protect the hit while evicting
            need = len(toks) - L
            short = -(-need // page) * page - pool.available()
            if short > 0:
                evict(short)
            new = pool.alloc(need)
            if new is None:                  # everything left is locked: by running requests or this hit
                assert set(model) == locked_pages() | {tuple(toks[:j + page]) for j in range(0, L, page)}
                cache.unlock(node)
                check_state()
                continue
            slots = np.concatenate([got, new]).astype(np.int32)
            assert cache.insert(toks, slots) == L
            n = len(toks) // page * page
            if n < len(toks):
                pool.free(slots[n:])                                   # the partial last page is the caller's
            for j in range(L, n, page):
                model[tuple(toks[:j + page])] = tuple(int(x) for x in slots[j:j + page])
            cache.unlock(node)
            if n > 0:
                live.append((toks[:n], cache.path(toks[:n])[-1]))
                cache.lock(live[-1][1])
            seen.append(toks)
        elif op < 0.85 and live:                                       # a request finishes
            _, node = live.pop(int(rng.integers(len(live))))
            cache.unlock(node)
        else:                                                          # the scheduler evicts
            want = int(rng.integers(1, 40))
            leaves = [n for n in cache._leaves() if n.lock_ref == 0]
            oldest_key = None
            if leaves:
                n = min(leaves, key=lambda x: (x.last_access, x.uid))
                path = []
                while n is not cache.root:
                    path = n.key.tolist() + path
                    n = n.parent
                oldest_key = tuple(path)
            avail = pool.available()
            freed, removed, after = evict(want)
            assert pool.available() == avail + freed
            if freed < want:
                assert len(after) == len(locked_pages())               # only locked pages are left
            if freed > 0:
                assert oldest_key in removed                          # least recently used leaf first
        check_state()
    assert len(seen) > 500


def _random_tree_rows(rng, n):
    """Slot rows of n requests with radix sharing: each row copies a prefix of an earlier row (or
    nothing) and continues with fresh slots, so equal slots at a position mean an equal prefix."""
    rows, fresh = [], iter(range(1000, 10 ** 6))
    for _ in range(n):
        row = []
        if rows and rng.random() < 0.8:
            parent = rows[int(rng.integers(len(rows)))]
            row = parent[:int(rng.integers(0, len(parent) + 1))]
        row = row + [next(fresh) for _ in range(int(rng.integers(1, 6)))]
        rows.append(row)
    return rows


def _brute_force_shared_nodes(rows):
    """The multi-level groups with min_range 1, from their definition by enumeration: every prefix p
    of the rows cut one token short that at least two requests hold, and at which those requests do
    not all continue with one same slot, ends a node; its group covers [end of the nearest such
    prefix above it, len(p)) and its level counts those above it."""
    seqs = [tuple(r[:len(r) - 1]) for r in rows]
    members = {}
    for b, s in enumerate(seqs):
        for d in range(1, len(s) + 1):
            members.setdefault(s[:d], set()).add(b)
    ends = set()
    for p, m in members.items():
        if len(m) < 2:
            continue
        nxt = {seqs[b][len(p)] if len(seqs[b]) > len(p) else None for b in m}
        if len(nxt) > 1 or None in nxt:
            ends.add(p)
    out = set()
    for p in ends:
        above = [len(q) for q in ends if len(q) < len(p) and p[:len(q)] == q]
        out.add((max(above, default=0), len(p), len(above), tuple(sorted(members[p]))))
    return out


@pytest.mark.parametrize("seed", range(40))
def test_multilevel_groups_against_brute_force(seed):
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    rng = np.random.default_rng(300 + seed)
    rows = _random_tree_rows(rng, int(rng.integers(2, 14)))
    indptr, reqs, start, end, level, nl = cascade_groups_multilevel(rows)
    got = {(int(start[g]), int(end[g]), int(level[g]), tuple(sorted(reqs[indptr[g]:indptr[g + 1]].tolist())))
           for g in range(len(start))}
    want = _brute_force_shared_nodes(rows)
    assert got == want
    assert nl == (1 + max(l for _, _, l, _ in want) if want else 0)


@pytest.mark.parametrize("seed", range(30))
def test_group_builders_hold_their_invariants_on_random_trees(seed):
    """Any min_range: each request's groups tile 0 .. (deepest end) - 1 one level after another, the
    members of a group hold the same slots over its range, and the newest token stays private.  The
    one-level builder: a group's prefix is shared by all its members and is maximal (it stops where
    the shortest member's newest token begins, or where two members differ)."""
    from prefix_shared_kv_ra_gb300.radix import cascade_groups_multilevel
    rng = np.random.default_rng(500 + seed)
    rows = _random_tree_rows(rng, int(rng.integers(2, 16)))
    min_range = int(rng.integers(1, 6))
    indptr, reqs, start, end, level, nl = cascade_groups_multilevel(rows, min_range=min_range)
    cover = {}
    for g in range(len(start)):
        mem = reqs[indptr[g]:indptr[g + 1]].tolist()
        assert len(mem) >= 2 and end[g] > start[g]
        for m in mem:
            assert rows[m][start[g]:end[g]] == rows[mem[0]][start[g]:end[g]]
            cover.setdefault(m, []).append((int(start[g]), int(end[g]), int(level[g])))
    for m, rng_ in cover.items():
        rng_.sort()
        assert [l for _, _, l in rng_] == list(range(len(rng_)))
        assert rng_[0][0] == 0 and all(rng_[i][1] == rng_[i + 1][0] for i in range(len(rng_) - 1))
        assert rng_[-1][1] <= len(rows[m]) - 1
    gi, gr, gp = cascade_groups(rows)
    for g in range(gi.size - 1):
        mem = gr[gi[g]:gi[g + 1]].tolist()
        assert len(mem) >= 2 and gp[g] >= 1
        for m in mem:
            assert rows[m][:gp[g]] == rows[mem[0]][:gp[g]] and gp[g] <= len(rows[m]) - 1
        at_end = gp[g] == min(len(rows[m]) - 1 for m in mem)
        differ = len({rows[m][gp[g]] for m in mem if len(rows[m]) > gp[g]}) > 1
        assert at_end or differ


@pytest.mark.parametrize("page", [1, 4, 16])
def test_slot_pool_against_a_list_model(page):
    """The pool hands out exactly the slots a plain list of free pages would (pop the last; a free
    appends the pages in increasing order), keeps count, and refuses a page freed twice."""
    rng = np.random.default_rng(40 + page)
    pool = SlotPool(64 * page, page_size=page)
    model = list(range(63, 0, -1))
    held = []
    for _ in range(3000):
        if held and rng.random() < 0.45:
            slots = held.pop(int(rng.integers(len(held))))
            pool.free(slots)
            model.extend(np.unique(np.asarray(slots) // page).tolist())
        else:
            n = int(rng.integers(0, 5 * page))
            got = pool.alloc(n)
            pages = -(-n // page)
            if pages > len(model):
                assert got is None
                continue
            want = [model.pop() for _ in range(pages)]
            assert got.tolist() == [pg * page + i for pg in want for i in range(page)][:n]
            if n:
                held.append(got)
        assert pool.available() == len(model) * page
        assert sorted(pool.free_pages().tolist()) == sorted(model)
    if held:
        pool.free(held[0])
        with pytest.raises(ValueError):
            pool.free(held[0])                                         # the same pages again
    with pytest.raises(ValueError):
        pool.free([0])                                                 # the reserved page


# ---------------------------------------------------------------- depth-first order of a batch
def _trie_dfs(paths):
    """Brute force: build a trie of the slot rows, walk it depth first (children by slot, a request that
    ends at a node before the requests below it) and list the requests in the order met."""
    root = {"children": {}, "ends": []}
    for b, row in enumerate(paths):
        node = root
        for x in row:
            node = node["children"].setdefault(int(x), {"children": {}, "ends": []})
        node["ends"].append(b)
    out = []

    def walk(node):
        out.extend(node["ends"])
        for x in sorted(node["children"]):
            walk(node["children"][x])
    walk(root)
    return out


def test_dfs_order_matches_a_trie_walk():
    from prefix_shared_kv_ra_gb300.radix import dfs_order
    rng = np.random.default_rng(7)
    for _ in range(30):
        base = [rng.integers(0, 50, size=rng.integers(1, 12)).tolist() for _ in range(4)]
        paths = []
        for _ in range(int(rng.integers(1, 15))):
            p = list(base[int(rng.integers(0, 4))])[: int(rng.integers(1, 12))]
            p += rng.integers(0, 50, size=int(rng.integers(0, 5))).tolist()
            paths.append(p)
        assert dfs_order(paths).tolist() == _trie_dfs(paths)


def test_dfs_order_puts_sharing_requests_next_to_each_other():
    from prefix_shared_kv_ra_gb300.radix import dfs_order
    paths = [[9, 1, 2], [5, 6], [9, 1, 3], [5, 7], [9, 4]]
    assert dfs_order(paths).tolist() == [1, 3, 0, 2, 4]
