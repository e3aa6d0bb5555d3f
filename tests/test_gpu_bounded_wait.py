"""A wait inside a kernel that runs out returns instead of hanging.  ra_selftest_bounded_wait runs one CTA
whose waits -- on an mbarrier no thread arrives at and on a counter no thread raises -- use the bounded-wait
primitives of every kernel of the library, with a deadline of about a millisecond.  Both waits must run
out, flag RA_DEVERR_TIMEOUT and return; the context stays usable (a decode afterwards matches the oracle).
Nothing faults, traps or hangs: the deadline, not an external kill, ends the waits."""
import time

import pytest
import torch

import oracle
import prefix_shared_kv_ra_gb300 as ra
import workloads as W
from helpers import DeviceBatch, assert_close, to_f64

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_flags_timeout_and_returns():
    dev = torch.device("cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ra.ra_selftest_bounded_wait(2_000_000, err)  # ~1 ms at GB300's SM clock
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(err.item()) & ra.DEVERR_TIMEOUT
    # the context still computes correct results
    b = W.random_mixed(71, n_extend=0, n_decode=6, num_q_heads=16, num_kv_heads=4, head_dim=128, max_len=700)
    db = DeviceBatch(b)
    db.store()
    db.decode()
    torch.cuda.synchronize()
    assert int(db.err.item()) == 0
    assert_close(to_f64(db.dec_o).reshape(-1, b.head_dim), oracle.decode_batch(b), "decode after a timed-out wait")
