"""GPU parity on paged slot layouts (pages of 16 consecutive slots, page-granular sharing): the
table still lists token slots, so store, extend, decode and the cascade decode run unchanged and
must match the oracle exactly as on token-granular layouts."""
import numpy as np
import pytest

import workloads as W
from helpers import DeviceBatch, check_store
from test_gpu_extend import check_cascade, check_extend
from test_gpu_store_decode import check_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,hq,hkv,d", [(41, 32, 8, 128), (42, 16, 2, 64)])
def test_paged_store_extend_decode(seed, hq, hkv, d):
    b = W.random_mixed(seed, n_extend=5, n_decode=6, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, max_len=700,
                       min_len=100, share_prob=0.8, page_size=16)
    assert any(s.fork > 0 for s in b.specs) and all(s.fork % 16 == 0 for s in b.specs)
    db = DeviceBatch(b)
    check_store(db)
    check_extend(db)
    check_decode(db)


def test_paged_decode_8b_cascade():
    b = W.decode_8b_system_prompts(page_size=16)
    assert b.has_cascade()
    db = DeviceBatch(b)
    db.store()
    check_cascade(db)
