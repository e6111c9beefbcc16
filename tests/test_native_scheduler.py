"""The native step planner and page allocator (include/pkv_sched.h) against the Python
planner, which the scheduler tests pin to the pages' worked numbers: identical plans on
every workload, plus the native-only behaviour (page release, all-or-nothing steps)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_token_gb300 import binding, build
from paged_kv_cache_token_gb300 import workloads as W
from paged_kv_cache_token_gb300.native_scheduler import NativeScheduler, native_scheduler_for
from paged_kv_cache_token_gb300.scheduler import PagePool, Scheduler, scheduler_for


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def same_plan(a, b):
    assert (a is None) == (b is None)
    if a is None:
        return
    assert list(a.rids) == list(b.rids)
    for name in ("q_lens", "context_lens", "q_offsets", "block_table"):
        x, y = getattr(a, name), getattr(b, name)
        assert x.dtype == y.dtype == np.int32, name
        assert np.array_equal(x, y), name


def same_run(py, nat):
    same_plan(py.history_plan(), nat.history_plan())
    steps = 0
    while True:
        p, n = py.next_step(), nat.next_step()
        same_plan(p, n)
        if p is None:
            return steps
        steps += 1


@pytest.mark.parametrize("make", [W.tiny, W.decode_only, W.prefill,
                                  lambda: W.prefill(chunk=2048), W.mixed, W.mha_skew])
def test_workloads_identical_plans(make):
    w = make()
    assert same_run(scheduler_for(w), native_scheduler_for(w)) > 0


@pytest.mark.parametrize("seed", range(12))
def test_random_batches_identical_plans(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 12))
    reqs = [W.RequestSpec(i, int(g.integers(0, 300)), int(g.integers(0, 300)),
                          int(g.integers(0, 20))) for i in range(n)]
    reqs = [r for r in reqs if r.total > 0] or [W.RequestSpec(0, 0, 5, 1)]
    pages = sum(-(-r.total // 16) for r in reqs) + 4
    order = g.permutation(pages).astype(np.int32)
    budget = int(g.integers(1, 400))
    cap = int(g.integers(1, 64)) if seed % 3 == 0 else None
    inter = bool(seed % 2)
    py = Scheduler(reqs, PagePool(order), budget, cap, inter)
    nat = NativeScheduler(reqs, order, budget, cap, inter)
    same_run(py, nat)
    assert nat.num_free == py.pool.num_free


def test_release_returns_pages_fifo():
    reqs = [W.RequestSpec(0, 0, 20, 1), W.RequestSpec(1, 0, 40, 1)]
    nat = NativeScheduler(reqs, np.arange(10, dtype=np.int32), 1000)
    steps = nat.all_steps()
    assert len(steps) == 2 and nat.num_free == 10 - 2 - 3
    held = list(steps[-1].block_table[0][steps[-1].block_table[0] >= 0])
    nat.release(0)
    assert nat.num_free == 10 - 3
    with pytest.raises(binding.PkvError):
        nat.release(0)            # forgotten after release
    # released pages join the end of the free list: a new request gets the untouched pages
    # first, then the released ones in their order
    nat.add_request(7, 0, 16 * 7, 0)
    p = nat.next_step()
    assert list(p.block_table[0]) == [5, 6, 7, 8, 9] + held


def test_release_refuses_unfinished():
    nat = NativeScheduler([W.RequestSpec(0, 0, 40, 3)], np.arange(8, dtype=np.int32), 16)
    nat.next_step()
    with pytest.raises(binding.PkvError):
        nat.release(0)


def test_out_of_pages_changes_nothing():
    reqs = [W.RequestSpec(0, 0, 40, 0), W.RequestSpec(1, 0, 40, 0)]
    nat = NativeScheduler(reqs, np.arange(4, dtype=np.int32), 1000)   # needs 6 pages
    with pytest.raises(binding.PkvError) as e:
        nat.next_step()
    assert e.value.status == -7 and nat.num_free == 4
    # the failed step took no page; with a third request the step needs 8 pages and is
    # refused the same way, still taking nothing
    nat.add_request(2, 0, 20, 0)
    with pytest.raises(binding.PkvError):
        nat.next_step()
    assert nat.num_free == 4


def test_small_output_arrays_change_nothing():
    reqs = [W.RequestSpec(i, 0, 30, 1) for i in range(3)]
    order = np.arange(20, dtype=np.int32)
    nat, py = NativeScheduler(reqs, order, 1000), Scheduler(reqs, PagePool(order), 1000)
    real_max = nat.max_reqs
    nat.max_reqs = 2                               # arrays for 2 of the 3 requests
    with pytest.raises(binding.PkvError) as e:
        nat.next_step()
    assert e.value.status == -3 and nat.num_free == 20
    nat.max_reqs = real_max
    same_run(py, nat)


# ---------------------------------------------------------------- sort by prompt length
def _pair(reqs, pages, budget, cap=None):
    order = np.arange(pages, dtype=np.int32)
    return (Scheduler(reqs, PagePool(order), budget, cap),
            NativeScheduler(reqs, order, budget, cap))


@pytest.mark.parametrize("seed", range(8))
def test_sort_by_length_identical_plans_mid_run(seed):
    # sort a batch, run a few steps, add requests, sort again (started requests keep their
    # place at the front), then run to the end: the native and Python planners agree
    g = np.random.default_rng(100 + seed)
    mk = lambda i: W.RequestSpec(i, int(g.integers(0, 100)), int(g.integers(0, 400)),
                                 int(g.integers(0, 6)))
    first = [mk(i) for i in range(int(g.integers(2, 9)))]
    later = [mk(i) for i in range(len(first), len(first) + int(g.integers(1, 6)))]
    pages = sum(-(-r.total // 16) for r in first + later) + 4
    budget = int(g.integers(16, 300))
    py, nat = _pair(first, pages, budget, 64 if seed % 2 else None)
    py.sort_by_length()
    nat.sort_by_length()
    same_plan(py.history_plan(), nat.history_plan())
    for _ in range(int(g.integers(1, 4))):
        same_plan(py.next_step(), nat.next_step())
    for r in later:
        py.add_request(r)
        nat.add_request(r.rid, r.history, r.prompt, r.decodes)
    py.sort_by_length()
    nat.sort_by_length()
    same_plan(py.history_plan(), nat.history_plan())
    while True:
        p, n = py.next_step(), nat.next_step()
        same_plan(p, n)
        if p is None:
            break


def test_sort_by_length_order():
    # prompts 300, 20, 300, 5, 20: shortest first, equal lengths in arrival order
    reqs = [W.RequestSpec(i, 0, n, 1) for i, n in enumerate([300, 20, 300, 5, 20])]
    py, nat = _pair(reqs, 200, 4096)
    py.sort_by_length()
    nat.sort_by_length()
    p, n = py.next_step(), nat.next_step()
    same_plan(p, n)
    assert list(n.rids) == [3, 1, 4, 0, 2]
    # a reused prefix counts as not started; its key is the prompt left to compute
    s = NativeScheduler([], np.arange(64, dtype=np.int32), 4096)
    a = np.arange(100, dtype=np.int32)
    s.add_prompt(0, a, 0)
    s.next_step()
    s.add_prompt(1, np.arange(40, dtype=np.int32) + 1000, 0)   # 40 new tokens
    assert s.add_prompt(2, a, 0) == 96                          # 4 tokens left
    s.sort_by_length()
    assert list(s.next_step().rids) == [2, 1]


def test_sort_by_length_keeps_pages_together():
    # lshu.cn/news/11576 §2.2: with prompts of mixed lengths, prefilling in arrival order
    # leaves short requests' pages between long ones; sorted, each request's pages form
    # fewer separate runs of the pool, and every short prompt prefills in the first step
    lens = [1800, 32, 2048, 2048, 1800, 48, 1500, 48, 32, 64, 32, 48, 2048, 2048, 32, 1800]
    reqs = [W.RequestSpec(i, 0, n, 2) for i, n in enumerate(lens)]
    runs = lambda pages: 1 + sum(1 for a, b in zip(pages, pages[1:]) if b != a + 1)
    total = {}
    for srt in (False, True):
        s = NativeScheduler(reqs, np.arange(4000, dtype=np.int32), 512)
        if srt:
            s.sort_by_length()
        steps = s.all_steps()
        first = {r: i for i, p in reversed(list(enumerate(steps))) for r in p.rids}
        last = steps[-1]
        tables = {}
        for p in steps:
            for j, r in enumerate(p.rids):
                row = p.block_table[j]
                tables[r] = [int(x) for x in row[row >= 0]]
        total[srt] = sum(runs(t) for t in tables.values())
        if srt:
            assert all(first[i] == 0 for i, n in enumerate(lens) if n <= 64)
    assert total[True] < total[False]
