"""Host side of the cache runtime (cache.py), on CPU: the flush planner's host
mirror, its behaviour when the page pool is exhausted, and the serving step's
look-ahead planning, which must resume where an allocation failed instead of
planning a layer twice.  The device calls are not made here."""

import numpy as np
import pytest
import torch

from mixed_precision_bit_gb300 import kitty
from mixed_precision_bit_gb300.cache import PAGE, LayerCache, ServingStep


def _cache(B=4, max_pages=6, pool_pages=64):
    cfg = kitty.Config(num_kv_heads=2, num_q_heads=8, n_hi=32, in_dtype=kitty.BF16)
    return LayerCache(cfg, B, max_pages, pool_pages, device="cpu")


def test_plan_flush_follows_the_tails():
    lc = _cache()
    lc.h_tail[:] = [31, 0, 30, 5]
    lc.h_pages[:] = [2, 0, 6, 1]  # sequence 2's table is full
    seen = set()
    for step in range(70):
        before_t, before_p = lc.h_tail.copy(), lc.h_pages.copy()
        fl = lc.plan_flush()
        for b in range(4):
            fills = before_t[b] + 1 == PAGE
            if fills and before_p[b] < lc.max_pages:
                assert fl[b] >= 0 and int(fl[b]) not in seen
                seen.add(int(fl[b]))
                assert lc.h_tail[b] == 0 and lc.h_pages[b] == before_p[b] + 1
            else:
                assert fl[b] == -1
                assert lc.h_pages[b] == before_p[b]
                if not fills:
                    assert lc.h_tail[b] == before_t[b] + 1
    # sequence 0 fills at steps 0, 32 and 64; sequence 1 at 31; sequence 3 at 26
    assert lc.h_pages.tolist() == [5, 2, 6, 3]
    assert len(seen) == 3 + 2 + 2


def test_plan_flush_out_of_pages_leaves_the_mirror():
    lc = _cache(B=2, pool_pages=1)
    lc.h_tail[:] = [31, 31]
    with pytest.raises(kitty.KittyError):
        lc.plan_flush()  # two pages wanted, one free
    assert lc.h_tail.tolist() == [31, 31] and lc.h_pages.tolist() == [0, 0]
    lc.h_tail[:] = [31, 3]
    fl = lc.plan_flush()
    assert fl.tolist() == [0, -1] and lc.h_tail.tolist() == [0, 4]


class _Layer:
    """Stands in for a LayerCache: plan_flush fails the first `fail` times."""

    def __init__(self, B, fail=0):
        self.B, self.calls, self.fail = B, 0, fail

    def plan_flush(self):
        if self.fail:
            self.fail -= 1
            raise kitty.KittyError("kitty_alloc_pages", -5)  # KITTY_ERR_OOM
        self.calls += 1
        return np.full(self.B, self.calls, np.int32)


def test_lookahead_planning_resumes_at_the_failed_layer():
    B = 3
    srv = object.__new__(ServingStep)  # the planning state only; no device buffers
    srv.layers = [_Layer(B), _Layer(B, fail=1), _Layer(B)]
    srv.h_fl = [torch.zeros((3, B), dtype=torch.int32) for _ in range(2)]
    srv._planned = 0
    with pytest.raises(kitty.KittyError):
        srv._plan(1)
    assert srv._planned == 1 and [x.calls for x in srv.layers] == [1, 0, 0]
    srv._plan(1)  # resumes at layer 1; layer 0 is not planned twice
    assert srv._planned == 3 and [x.calls for x in srv.layers] == [1, 1, 1]
    assert srv.h_fl[1].tolist() == [[1] * B] * 3
    srv._plan(1)  # nothing pending
    assert [x.calls for x in srv.layers] == [1, 1, 1]
