"""The attention step for callers that cannot allocate device memory at call time (for
example code run from a plugin or callback that must not synchronise the device, or a
runtime that hands out all device memory at start-up): its scratch is a fixed array inside
the library instead of a caller workspace.  Its output must match the regular entry point
on the same inputs, on consecutive calls that reuse the array.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_token_gb300 import binding, build, runner
from paged_kv_cache_token_gb300 import workloads as W
from paged_kv_cache_token_gb300.scheduler import scheduler_for

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _workload(index, specs, budget=1 << 30):
    reqs = [W.RequestSpec(i, *s) for i, s in enumerate(specs)]
    need = sum(-(-r.total // 16) for r in reqs) + 8
    order = torch.randperm(need, generator=torch.Generator().manual_seed(77 + index)).numpy()
    return W.Workload(index, "no-alloc", 32, 8, 128, W.BF16, reqs, order.astype(np.int32), need,
                      budget=budget)


def _prepared_steps(w):
    """Device state after the history load plus the inputs of every planned step."""
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    steps = []
    for plan in s.all_steps():
        q, k, v = runner.step_host_inputs(w, plan)
        ds = kv.upload(plan)
        kv.append(ds, runner.bits_to_tensor(k, w.dtype), runner.bits_to_tensor(v, w.dtype))
        steps.append((ds, runner.bits_to_tensor(q, w.dtype)))
    return kv, steps


def _compare(a: torch.Tensor, b: torch.Tensor):
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a.double()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, \
        (err.max().item(), err.mean().item())


def test_static_workspace_matches_regular_entry_point_on_two_calls():
    # decode rows split over several work items, plus prefill rows, in separate steps
    w = _workload(1, [(3000, 0, 2), (700, 0, 2), (33, 0, 2), (0, 150, 0), (1500, 0, 2)],
                  budget=100)
    kv, steps = _prepared_steps(w)
    assert len(steps) >= 2
    for ds, q in steps[:2]:                 # two calls in a row share the array
        shape = (ds.plan.total_q_tokens, w.num_q_heads, w.head_dim)
        ref = kv.attention(ds, q, w.scale)  # regular entry point, caller workspace
        got = torch.full(shape, float("nan"), dtype=kv.dtype, device="cuda")
        binding.paged_attention_step_static_ws(ds.desc, q, kv.k_cache, kv.v_cache, got,
                                               w.scale, kv.err)
        torch.cuda.synchronize()
        _compare(got, ref)
    assert kv.read_error() == 0


def test_static_workspace_repeated_call_same_step():
    w = _workload(2, [(c, 0, 1) for c in (4000, 100, 2500, 16, 900, 0)])
    kv, steps = _prepared_steps(w)
    ds, q = steps[0]
    ref = kv.attention(ds, q, w.scale)
    outs = []
    for _ in range(2):
        got = torch.empty_like(ref)
        binding.paged_attention_step_static_ws(ds.desc, q, kv.k_cache, kv.v_cache, got, w.scale,
                                               kv.err)
        outs.append(got)
    torch.cuda.synchronize()
    for got in outs:
        _compare(got, ref)
    assert kv.read_error() == 0


def _big_desc(num_pages):
    # 4,096 decode rows over 100,000-token contexts: the split-KV scratch this needs does
    # not depend on the pool size, only on the rows, heads and context lengths
    n, ctx = 4096, 100_000
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    desc = binding.make_desc(num_reqs=n, num_q_heads=32, num_kv_heads=8, head_dim=128,
                             num_pages=num_pages, max_pages_per_req=ctx // 16 + 1,
                             total_q_tokens=n, max_q_len=1, max_context_len=ctx, dtype=W.BF16,
                             q_lens=dummy, q_offsets=dummy, context_lens=dummy,
                             block_table=dummy)
    return desc, dummy


def test_static_workspace_rejects_steps_beyond_its_size():
    # more scratch than the 32 MiB array holds: refused on the host, nothing launched
    desc, dummy = _big_desc(num_pages=1024)
    assert binding.attention_workspace_bytes(desc) > binding.STATIC_WORKSPACE_BYTES
    rc = binding.paged_attention_step_static_ws(desc, dummy, dummy, dummy, dummy, 1.0,
                                                check=False)
    assert rc == -4  # PKV_ERR_WORKSPACE


def test_static_workspace_passes_description_errors_through():
    # a pool of 2^31 (page, KV head, token) rows is not supported by either entry point
    desc, dummy = _big_desc(num_pages=1 << 24)
    assert binding.attention_workspace_bytes(desc) == 0
    rc = binding.paged_attention_step_static_ws(desc, dummy, dummy, dummy, dummy, 1.0,
                                                check=False)
    assert rc == -2  # PKV_ERR_UNSUPPORTED
