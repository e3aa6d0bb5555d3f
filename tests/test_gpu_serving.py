"""The host radix cache driving the hot path across steps: multi-turn chats admitted by longest
cached prefix, prefilled, decoded from CUDA graphs, retired into the tree; eviction under a small
pool.  Checks the device error word, the pool's slot accounting, the hit ratio against the
oracle's definition, and one decode step against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from prefix_shared_kv_ra_gb300.serving import ServingReplay, multiturn_chat, run_chat
from helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu


def _replay(num_slots, **kw):
    return ServingReplay(num_slots=num_slots, num_q_heads=16, num_kv_heads=4, head_dim=128, max_len=2048,
                         max_running=64, device="cuda:0", seed=3, graph_sizes=(8, 16, 32, 64), **kw)


def test_chat_replay_hit_ratio_and_decode_parity():
    rp = _replay(1 << 16)
    convs = multiturn_chat(24, 3, seed=1, system_prompts=3, system_len=256, user_len=(16, 64), out_len=(4, 12))
    st = run_chat(rp, convs, max_steps=400, arrivals_per_step=8)
    torch.cuda.synchronize()
    assert int(rp.err.item()) == 0
    assert len(rp.finished) == 24 * 3 and not rp.running and st["evicted"] == 0
    # a later turn's prompt is the previous turn's sequence plus new user tokens: with no eviction, the
    # tree serves exactly that sequence (user tokens are random and generated ids unique)
    by_turn = {rp.tags[r.rid]: r for r in rp.finished}
    for (c, turn), r in by_turn.items():
        if turn > 0:
            prev = by_turn[(c, turn - 1)]
            assert r.cached == len(prev.prompt) + len(prev.generated), (c, turn)
    assert sum(r.cached for r in rp.finished) == st["cached_tokens"]
    assert 0.5 < st["hit_ratio"] < 1.0
    # pool accounting: every slot is free, in the tree, or reserved
    assert rp.pool.available() + rp.cache.total_tokens() == rp.pool.num_slots - 1

    # one more decode step, checked against the oracle on the device pool's rows
    convs2 = multiturn_chat(6, 1, seed=9, system_prompts=2, system_len=128, user_len=(8, 16), out_len=(3, 3))
    run_chat(rp, convs2, max_steps=2, arrivals_per_step=6, rid0=10_000)  # admit + prefill, one decode
    assert rp.prefilled, "requests should be decoding"
    g, buf, run = rp._graph(next(s for s in rp.graph_sizes if s >= len(rp.prefilled)))
    n = len(rp.prefilled)
    torch.cuda.synchronize()
    rows = buf["rpi"][:n].cpu().numpy()
    lens = buf["lens"][:n].cpu().numpy()
    table = rp.table.cpu().numpy()
    used = np.unique(np.concatenate([table[r, :l] for r, l in zip(rows, lens)])).astype(np.int64)
    idx = torch.from_numpy(used).to(rp.dev)
    kp = rp.k_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    vp = rp.v_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    pool = oracle.CompactPool(rp.pool.num_slots, used, kp, vp)
    q = buf["q"][:n].view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.decode(pool, q, table, rows, lens, rp.scale)
    got = to_f64(buf["o"][:n]).reshape(-1, rp.d)
    assert_close(got, ref, "graph decode in the replay")


def test_small_pool_evicts_and_keeps_accounting():
    rp = _replay(8 * 1024)  # ~11.3K unique tokens: the tree must give slots back
    convs = multiturn_chat(32, 4, seed=2, system_prompts=4, system_len=256, user_len=(32, 96), out_len=(8, 24))
    st = run_chat(rp, convs, max_steps=2000, arrivals_per_step=8)
    torch.cuda.synchronize()
    assert int(rp.err.item()) == 0
    assert len(rp.finished) == 32 * 4 and st["evicted"] > 0
    assert rp.pool.available() + rp.cache.total_tokens() == rp.pool.num_slots - 1
