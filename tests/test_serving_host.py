"""Host logic of the serving replay on the CPU: admission by longest cached prefix, prefill and decode
bookkeeping, retiring turns into the radix tree, eviction under a small pool and slot accounting.

The replay's host decisions never depend on what the kernels compute (generated token ids are
counters), so here the store, extend and decode calls and the CUDA events are replaced by no-ops
for the duration of each test; the same loop runs with the real kernels in test_gpu_serving.py."""
import numpy as np
import pytest
import torch

import prefix_shared_kv_ra_gb300.serving as S


class _NoEvent:
    def __init__(self, **kw):
        pass

    def record(self, *a):
        pass

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return 0.0


@pytest.fixture
def host_only(monkeypatch):
    monkeypatch.setattr(torch.cuda, "Event", _NoEvent)
    for name in ("ra_kv_store", "ra_extend_attention", "ra_decode_attention"):
        monkeypatch.setattr(S, name, lambda *a, **k: None)
    monkeypatch.setattr(S, "ra_extend_workspace_bytes", lambda *a, **k: 16)
    monkeypatch.setattr(S, "ra_decode_workspace_bytes", lambda *a, **k: 16)
    monkeypatch.setattr(S.ServingReplay, "_randn", lambda self, shape: torch.empty(shape, dtype=torch.bfloat16))

    def make(num_slots, **kw):
        return S.ServingReplay(num_slots=num_slots, num_q_heads=4, num_kv_heads=2, head_dim=8, max_len=2048,
                               max_running=64, device="cpu", seed=3, graph_sizes=(8, 16, 32, 64), use_graphs=False,
                               **kw)
    return make


def _accounting(rp):
    """Every slot is free, in the tree, or held by a running request beyond its cached prefix."""
    held = sum(r.slots.size - r.cached for r in rp.running.values())
    assert rp.pool.available() + rp.cache.total_tokens() + held == rp.pool.num_slots - 1


def test_later_turns_hit_their_whole_history(host_only):
    rp = host_only(1 << 16)
    convs = S.multiturn_chat(24, 3, seed=1, system_prompts=3, system_len=256, user_len=(16, 64), out_len=(4, 12))
    st = S.run_chat(rp, convs, max_steps=400, arrivals_per_step=8)
    assert len(rp.finished) == 24 * 3 and not rp.running and st["evicted"] == 0
    by_turn = {rp.tags[r.rid]: r for r in rp.finished}
    for (c, turn), r in by_turn.items():
        if turn > 0:   # the previous turn's prompt and output are all cached, nothing more
            prev = by_turn[(c, turn - 1)]
            assert r.cached == len(prev.prompt) + len(prev.generated), (c, turn)
        else:          # a first turn shares at most its system prompt
            assert r.cached <= 256
    assert sum(r.cached for r in rp.finished) == st["cached_tokens"]
    assert st["decode_tokens"] == sum(len(r.generated) for r in rp.finished)
    assert all(len(r.generated) == r.out_len for r in rp.finished)
    _accounting(rp)


def test_small_pool_defers_and_evicts_but_never_loses_a_slot(host_only):
    rp = host_only(8 * 1024)
    convs = S.multiturn_chat(32, 4, seed=2, system_prompts=4, system_len=256, user_len=(32, 96), out_len=(8, 24))
    seen_running = 0
    orig_step = rp.step

    def step(arrivals):
        nonlocal seen_running
        out = orig_step(arrivals)
        _accounting(rp)                                   # after every step, not only at the end
        seen_running = max(seen_running, len(rp.running))
        free = set(rp.pool.free_pages().tolist())         # no running request's slot is on a free page
        for r in rp.running.values():
            assert not (set(r.slots.tolist()) & free)
        return out
    rp.step = step
    st = S.run_chat(rp, convs, max_steps=2000, arrivals_per_step=8)
    assert len(rp.finished) == 32 * 4 and st["evicted"] > 0 and not rp.running
    assert seen_running <= rp.max_running
    assert 0.0 < st["hit_ratio"] < 1.0
    for r in rp.finished:                                 # one slot per position of prompt and output
        assert r.slots.size == len(r.prompt) + len(r.generated)


def test_a_request_larger_than_the_pool_is_refused(host_only):
    rp = host_only(512)
    with pytest.raises(RuntimeError):
        rp.step([(0, np.arange(1, 600, dtype=np.int32), 4)])
