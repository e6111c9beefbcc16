"""Host step planner: token budget, decode-first, chunking, page growth.

Pins from niuwancheng.cn "11. chunked prefill and unified scheduling": a 30,000-token
input with a 2048-token budget is done in 15 chunks; decodes get 1 token each and come
first; prefill gets min(remaining input, remaining budget); a step never exceeds the budget.
"""
import numpy as np
import pytest

from paged_kv_cache_token_gb300 import workloads as W
from paged_kv_cache_token_gb300.scheduler import (OutOfPages, PagePool, Scheduler, pages_for,
                                                  scheduler_for)


def test_thirty_thousand_tokens_fifteen_chunks():
    w = W.mixed()
    s = scheduler_for(w)
    hist = s.history_plan()
    assert hist.num_reqs == 30 and np.all(hist.context_lens == 0)
    steps = s.all_steps()
    assert len(steps) == 15
    chunk = [int(p.q_lens[-1]) for p in steps]
    assert chunk[:14] == [2018] * 14 and chunk[14] == 30000 - 14 * 2018 == 1748
    for p in steps:
        assert p.total_q_tokens <= 2048
        assert np.all(p.q_lens[:30] == 1)                 # decodes first, one token each
        assert p.rids[-1] == 30
    # the prompt's context grows chunk by chunk
    assert [int(p.context_lens[-1]) for p in steps] == [2018 * i for i in range(15)]


def test_tiny_schedule_table():
    w = W.tiny()
    steps = scheduler_for(w).all_steps()
    got = [(p.rids, p.q_lens.tolist(), p.context_lens.tolist()) for p in steps]
    assert got == [([0, 1], [37, 64], [0, 0]),
                   ([0, 1], [1, 36], [37, 64]),
                   ([0, 1], [1, 1], [38, 100]),
                   ([0, 1], [1, 1], [39, 101]),
                   ([0, 1], [1, 1], [40, 102]),
                   ([0, 1], [1, 1], [41, 103]),
                   ([1], [1], [104])]


def test_block_tables_cover_every_position_and_pages_are_unique():
    for w in (W.tiny(), W.mha_skew(), W.mixed(steps=3, prompt=5000)):
        s = scheduler_for(w)
        plans = [s.history_plan()] + s.all_steps()
        for p in plans:
            if p is None:
                continue
            for i in range(p.num_reqs):
                need = pages_for(int(p.context_lens[i] + p.q_lens[i]))
                row = p.block_table[i]
                assert np.all(row[:need] >= 0) and np.all(row[:need] < w.num_pages)
                assert np.all(row[need:] == -1)
        final = [st.pages for st in s.reqs]
        flat = [x for pages in final for x in pages]
        assert len(flat) == len(set(flat))


def test_interleaved_history_pages_round_robin():
    w = W.mha_skew()
    s = scheduler_for(w)
    h = s.history_plan()
    # page 0 to request 0, page 1 to request 1, ... while every request still needs pages
    first = [int(h.block_table[i, 0]) for i in range(h.num_reqs)]
    assert first == list(range(h.num_reqs))


def test_budget_respected_with_many_prefills():
    class R:
        def __init__(self, rid, prompt, dec):
            self.rid, self.history, self.prompt, self.decodes = rid, 0, prompt, dec
    reqs = [R(0, 300, 2), R(1, 50, 3), R(2, 1000, 1)]
    s = Scheduler(reqs, PagePool(range(200)), budget=256)
    steps = s.all_steps()
    for p in steps:
        assert 0 < p.total_q_tokens <= 256
    total = sum(p.total_q_tokens for p in steps)
    assert total == 300 + 2 + 50 + 3 + 1000 + 1


def test_pool_exhaustion_raises():
    class R:
        rid, history, prompt, decodes = 0, 0, 40, 0
    with pytest.raises(OutOfPages):
        Scheduler([R()], PagePool(range(2)), budget=64).next_step()


def test_zero_budget_rejected():
    with pytest.raises(ValueError):
        Scheduler([], PagePool([]), budget=0)
