"""Helpers shared by the GPU parity tests: run steps through the C ABI, compute the
oracle's rows for the same step, compare under the attention tolerance."""
import numpy as np
import torch

import oracle
from paged_kv_cache_token_gb300 import runner
from paged_kv_cache_token_gb300.scheduler import make_plan

# bf16/fp16 attention outputs against the fp64 oracle (fp32 accumulation on the GPU)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def oracle_rows(workload, plan, rows=None):
    """fp64 expected outputs for the step's query rows (all rows, or the given step-row
    indices), from the contiguous sequences -- the oracle never sees pages."""
    out = np.zeros((plan.total_q_tokens if rows is None else len(rows), workload.num_q_heads,
                    workload.head_dim))
    want = None if rows is None else {int(t): i for i, t in enumerate(rows)}
    for j, rid in enumerate(plan.rids):
        c, n, o = (int(plan.context_lens[j]), int(plan.q_lens[j]), int(plan.q_offsets[j]))
        req = workload.requests[rid]
        sel = list(range(n)) if want is None else [i for i in range(n) if o + i in want]
        if not sel:
            continue
        k, v = workload.kv(rid)
        qrows = workload.q(rid)[[c - req.history + i for i in sel]]
        pos = np.array([c + i for i in sel], np.int32)
        res = oracle.attention_rows(workload.dtype, qrows, pos, k[:c + n], v[:c + n],
                                    workload.scale)
        for a, i in enumerate(sel):
            out[(o + i) if want is None else want[o + i]] = res[a]
    return out


def gpu_as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def assert_close(got: np.ndarray, ref: np.ndarray, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite output " + what
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, "%s max_abs=%.3g mean_abs=%.3g" % (what, mx, mean)
    return mx, mean


def pool_bits(kv: runner.PagedKV):
    return runner.tensor_to_bits(kv.k_cache), runner.tensor_to_bits(kv.v_cache)


def request_codes(workload, rid):
    """The oracle's INT8 codes of a request's whole K and V sequence."""
    key = ("codes", rid)
    if key not in workload._cache:
        ks, vs = workload.int8_scales()
        k, v = workload.kv(rid)
        workload._cache[key] = (oracle.quantize_int8(workload.dtype, k, ks),
                                oracle.quantize_int8(workload.dtype, v, vs))
    return workload._cache[key]


def oracle_rows_int8(workload, plan, rows=None):
    """As :func:`oracle_rows` over an INT8 cache: the oracle quantises each request's K/V
    with the workload's per-channel scales and attends over the values the codes stand
    for."""
    ks, vs = workload.int8_scales()
    out = np.zeros((plan.total_q_tokens if rows is None else len(rows), workload.num_q_heads,
                    workload.head_dim))
    want = None if rows is None else {int(t): i for i, t in enumerate(rows)}
    for j, rid in enumerate(plan.rids):
        c, n, o = (int(plan.context_lens[j]), int(plan.q_lens[j]), int(plan.q_offsets[j]))
        req = workload.requests[rid]
        sel = list(range(n)) if want is None else [i for i in range(n) if o + i in want]
        if not sel:
            continue
        kc, vc = request_codes(workload, rid)
        qrows = workload.q(rid)[[c - req.history + i for i in sel]]
        pos = np.array([c + i for i in sel], np.int32)
        res = oracle.attention_rows_int8(workload.dtype, qrows, pos, kc[:c + n], vc[:c + n], ks,
                                         vs, workload.scale)
        for a, i in enumerate(sel):
            out[(o + i) if want is None else want[o + i]] = res[a]
    return out
