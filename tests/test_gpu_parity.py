"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs.  kv_append, page contents and slot ids must be bit-exact; attention outputs must be
within max-abs 2e-2 and mean-abs 2e-3 of the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_token_gb300 import binding, build, runner
from paged_kv_cache_token_gb300 import workloads as W
from paged_kv_cache_token_gb300.scheduler import PagePool, Scheduler, make_plan, scheduler_for

from gpu_common import assert_close, gpu_as_f64, oracle_rows, oracle_rows_int8, pool_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def custom(index, hq, hkv, d, dtype, specs, budget=1 << 30, chunk_cap=None, extra_pages=8,
           interleave=False):
    reqs = [W.RequestSpec(i, *s) for i, s in enumerate(specs)]
    need = sum(-(-r.total // 16) for r in reqs) + extra_pages
    g = torch.Generator().manual_seed(9000 + index)
    order = torch.randperm(need, generator=g).numpy().astype(np.int32)
    return W.Workload(index, "custom", hq, hkv, d, dtype, reqs, order, need, budget=budget,
                      chunk_cap=chunk_cap, interleave_history=interleave)


def run_all(w, check_rows=None, every_step=True):
    """Run a workload's history load and every step; compare each step with the oracle."""
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    worst = (0.0, 0.0)
    outs = []
    for i, plan in enumerate(s.all_steps()):
        out = runner.run_step(kv, w, plan)
        if every_step or i == 0:
            rows = None if check_rows is None else check_rows(plan)
            ref = oracle_rows(w, plan, rows)
            got = gpu_as_f64(out) if rows is None else gpu_as_f64(out[torch.as_tensor(rows)])
            assert kv.read_error() == 0
            mx, mean = assert_close(got, ref, "%s step %d" % (w.name, i))
            worst = (max(worst[0], mx), max(worst[1], mean))
        outs.append(out)
    assert kv.read_error() == 0
    return worst, outs, kv


# ------------------------------------------------------------------------------ kv_append
def test_append_tiny_bit_exact():
    w = W.tiny()
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    shape = (w.num_pages, w.num_kv_heads, 16, w.head_dim)
    ref_k = np.full(shape, 0xFFFF, np.uint16)
    ref_v = ref_k.copy()
    for plan in s.all_steps():
        _, k, v = runner.step_host_inputs(w, plan)
        ds = kv.upload(plan)
        slots = torch.full((plan.total_q_tokens,), -7, dtype=torch.int64, device="cuda")
        kv.append(ds, runner.bits_to_tensor(k, w.dtype), runner.bits_to_tensor(v, w.dtype), slots)
        ref_k, ref_v, ref_slots = oracle.kv_append(plan.q_lens, plan.context_lens,
                                                   plan.block_table, w.num_pages, k, v, ref_k,
                                                   ref_v)
        gk, gv = pool_bits(kv)
        assert np.array_equal(gk, ref_k) and np.array_equal(gv, ref_v)
        assert np.array_equal(slots.cpu().numpy(), ref_slots)
    assert kv.read_error() == 0


@pytest.mark.parametrize("d,hkv,dtype", [(64, 2, 0), (128, 8, 0), (128, 3, 1), (64, 1, 1)])
def test_append_page_boundaries_bit_exact(d, hkv, dtype):
    rng = np.random.default_rng(d + hkv)
    ctx = [0, 15, 16, 31, 32, 1023, 1024, 5, 0]
    ql = [1, 1, 16, 17, 33, 1, 16, 0, 64]
    need = [-(-(c + q) // 16) for c, q in zip(ctx, ql)]
    npages = sum(need) + 5
    order = rng.permutation(npages).astype(np.int32)
    tables, used = [], 0
    for n in need:
        tables.append(order[used:used + n].tolist())
        used += n
    plan = make_plan(list(range(len(ctx))), ql, ctx, tables)
    T = plan.total_q_tokens
    k = rng.integers(0, 0xFFFF, size=(T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 0xFFFF, size=(T, hkv, d), dtype=np.uint16)
    kv = runner.PagedKV(npages, hkv, hkv, d, dtype)
    ds = kv.upload(plan)
    slots = torch.empty((T,), dtype=torch.int64, device="cuda")
    kv.append(ds, runner.bits_to_tensor(k, dtype), runner.bits_to_tensor(v, dtype), slots)
    sent = np.full((npages, hkv, 16, d), 0xFFFF, np.uint16)
    rk, rv, rs = oracle.kv_append(plan.q_lens, plan.context_lens, plan.block_table, npages, k, v,
                                  sent, sent)
    gk, gv = pool_bits(kv)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    assert np.array_equal(slots.cpu().numpy(), rs)
    assert kv.read_error() == 0


def test_append_bad_page_sets_flag_and_skips():
    plan = make_plan([0, 1], [3, 2], [0, 0], [[0], [7]])   # page 7 outside a 4-page pool
    kv = runner.PagedKV(4, 1, 1, 64, 0)
    ds = kv.upload(plan)
    k = torch.zeros((5, 1, 64), dtype=torch.bfloat16, device="cuda")
    kv.append(ds, k, k)
    assert kv.read_error() & binding.DEVERR_PAGE_RANGE
    gk, _ = pool_bits(kv)
    assert np.all(gk[0, 0, :3] == 0) and np.all(gk[0, 0, 3:] == 0xFFFF)
    assert np.all(gk[1:] == 0xFFFF)


def test_append_negative_offsets_flagged_and_skipped():
    # q_offsets = [0, -1, 0]: request 0's length disagrees with its offsets, and request 1
    # starts at token row -1 although its own length (1) matches.  Both must be refused:
    # the flag gets the token bit and no page slot or slot id changes.
    plan = make_plan([0, 1], [1, 1], [0, 0], [[0], [1]])
    kv = runner.PagedKV(4, 1, 1, 64, 0)
    ds = kv.upload(plan)
    qo = torch.tensor([0, -1, 0], dtype=torch.int32, device="cuda")
    desc = binding.make_desc(num_reqs=2, num_q_heads=1, num_kv_heads=1, head_dim=64,
                             num_pages=4, max_pages_per_req=plan.max_pages, total_q_tokens=2,
                             max_q_len=1, max_context_len=0, dtype=0, q_lens=ds.tensors[0],
                             q_offsets=qo, context_lens=ds.tensors[2],
                             block_table=ds.tensors[3])
    k = torch.zeros((2, 1, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.full((2,), -7, dtype=torch.int64, device="cuda")
    kv.append_desc(desc, k, k, slots)
    assert kv.read_error() & binding.DEVERR_TOKENS
    gk, gv = pool_bits(kv)
    assert np.all(gk == 0xFFFF) and np.all(gv == 0xFFFF)
    assert slots.cpu().tolist() == [-7, -7]


# ------------------------------------------------------------------------------ attention
def test_tiny_all_steps():
    run_all(W.tiny())


@pytest.mark.parametrize("hq,hkv,d,dtype", [(4, 2, 64, 0), (32, 8, 128, 0), (8, 8, 128, 1),
                                            (16, 2, 128, 1), (8, 1, 64, 0), (6, 3, 64, 1)])
def test_decode_batches(hq, hkv, d, dtype):
    ctx = [0, 1, 15, 16, 17, 100, 255, 256, 1000, 3000]  # one key, page edges, multi-split
    w = custom(100 + hq + d, hq, hkv, d, dtype, [(c, 0, 2) for c in ctx])
    run_all(w)


def _steps_both_ways(w, kv_int8=False):
    """Every step of w through pkv_append_attention(_int8) and through the two separate
    calls, on fresh pools: (outputs, slot ids, pool bits) of each, and the plans."""
    res = {}
    for fused in (True, False):
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w, kv_int8=kv_int8)
        runner.load_history(kv, w, s.history_plan())
        outs, slots, plans = [], [], []
        for plan in s.all_steps():
            sl = torch.full((plan.total_q_tokens,), -7, dtype=torch.int64, device="cuda")
            if fused:
                out = runner.run_step_fused(kv, w, plan, sl)
            else:
                q, k, v = runner.step_host_inputs(w, plan)
                ds = kv.upload(plan)
                kv.append(ds, runner.bits_to_tensor(k, w.dtype), runner.bits_to_tensor(v, w.dtype),
                          sl)
                out = kv.attention(ds, runner.bits_to_tensor(q, w.dtype), w.scale)
            outs.append(out)
            slots.append(sl)
            plans.append(plan)
        assert kv.read_error() == 0
        res[fused] = (outs, slots, pool_bits(kv))
    return res, plans


@pytest.mark.parametrize("hq,hkv,d,dtype", [(32, 8, 128, 0), (8, 8, 128, 1), (16, 2, 64, 1),
                                            (64, 8, 128, 0), (8, 1, 64, 0)])
def test_fused_append_attention_decode_steps(hq, hkv, d, dtype):
    # decode steps through pkv_append_attention: the warp streaming a (request, KV head)'s
    # last page writes the new row first.  Outputs, slot ids and every pool byte equal the
    # separate kv_append + attention calls, and every row matches the oracle.
    ctx = [0, 1, 15, 16, 17, 100, 255, 256, 1000, 3000]
    w = custom(1800 + hq + d, hq, hkv, d, dtype, [(c, 0, 3) for c in ctx])
    res, plans = _steps_both_ways(w)
    (fo, fs, fp), (so, ss, sp) = res[True], res[False]
    for i, plan in enumerate(plans):
        assert torch.equal(fo[i].view(torch.int16), so[i].view(torch.int16)), i
        assert torch.equal(fs[i], ss[i]), i
        assert_close(gpu_as_f64(fo[i]), oracle_rows(w, plan), "fused step %d" % i)
    assert all(np.array_equal(a, b) for a, b in zip(fp, sp))


@pytest.mark.parametrize("hq,hkv,d,dtype", [(32, 8, 128, 0), (8, 8, 128, 1), (16, 2, 64, 1),
                                            (8, 1, 64, 0)])
def test_fused_append_attention_int8_decode_steps(hq, hkv, d, dtype):
    # decode steps through pkv_append_attention_int8: the warp streaming a (request, KV
    # head)'s last page quantises the new row (the INT8 append's arithmetic) into it first.
    # Outputs, slot ids and every pool byte equal the separate kv_append_int8 + attention
    # calls, and every row matches the INT8 oracle.
    ctx = [0, 1, 15, 16, 17, 100, 255, 256, 1000, 3000]
    w = custom(1850 + hq + d, hq, hkv, d, dtype, [(c, 0, 3) for c in ctx])
    res, plans = _steps_both_ways(w, kv_int8=True)
    (fo, fs, fp), (so, ss, sp) = res[True], res[False]
    for i, plan in enumerate(plans):
        assert torch.equal(fo[i].view(torch.int16), so[i].view(torch.int16)), i
        assert torch.equal(fs[i], ss[i]), i
        assert_close(gpu_as_f64(fo[i]), oracle_rows_int8(w, plan), "fused INT8 step %d" % i)
    assert all(np.array_equal(a, b) for a, b in zip(fp, sp))


def test_fused_append_attention_other_steps_fall_back():
    # steps with prefill chunks (and more than 256 requests) take the append kernel, then
    # the attention step: same bits as the separate calls
    specs = [(300, 40, 1), (0, 200, 0), (17, 0, 2)] + [(5, 0, 1)] * 260
    w = custom(1900, 8, 2, 128, 0, specs, budget=512)
    res, plans = _steps_both_ways(w)
    assert any(p.max_q_len > 1 for p in plans) and plans[0].num_reqs > 256
    for i, plan in enumerate(plans):
        assert torch.equal(res[True][0][i].view(torch.int16), res[False][0][i].view(torch.int16))
        assert torch.equal(res[True][1][i], res[False][1][i])
    assert all(np.array_equal(a, b) for a, b in zip(res[True][2], res[False][2]))


def test_fused_append_attention_bad_page_flagged():
    w = custom(1950, 4, 2, 64, 0, [(20, 0, 1), (40, 0, 1)])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    plan.block_table[1, 2] = w.num_pages + 5   # the page the second request appends into
    runner.run_step_fused(kv, w, plan)
    assert kv.read_error() & binding.DEVERR_PAGE_RANGE


def test_decode_literal_skeleton_scale_one():
    # hotelren.com/news/6181127 §5.1 writes softmax(q @ K_all.T) with no scale: scale = 1.0
    w = custom(200, 4, 2, 64, 0, [(40, 0, 1), (3, 0, 1)])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    q, k, v = runner.step_host_inputs(w, plan)
    ds = kv.upload(plan)
    kv.append(ds, runner.bits_to_tensor(k, 0), runner.bits_to_tensor(v, 0))
    out = kv.attention(ds, runner.bits_to_tensor(q, 0), 1.0)
    w.scale_override = 1.0
    ref = np.concatenate([oracle.attention_rows(0, w.q(r)[:1], np.array([c], np.int32),
                                                w.kv(r)[0][:c + 1], w.kv(r)[1][:c + 1], 1.0)
                          for r, c in zip(plan.rids, plan.context_lens.tolist())])
    assert_close(gpu_as_f64(out), ref, "scale 1")


@pytest.mark.parametrize("hq,hkv,d,dtype", [(4, 2, 64, 0), (32, 8, 128, 0), (8, 8, 128, 1),
                                            (8, 2, 128, 1), (16, 2, 64, 1), (4, 4, 128, 0)])
def test_prefill_chunks_small(hq, hkv, d, dtype):
    # prompts around the 128-row tile and 16-token page edges, chunked by a small budget
    specs = [(0, 1, 1), (0, 2, 0), (0, 127, 1), (0, 128, 0), (0, 129, 2), (0, 300, 1),
             (20, 33, 0)]
    run_all(custom(300 + hq + d, hq, hkv, d, dtype, specs, budget=160, chunk_cap=96))


def test_step_staging_bitwise_identical():
    # the packed one-copy staging (inputs in one pinned buffer, device views into one
    # device buffer), alone and as the two-staging pipeline whose copies run on their own
    # streams beside the neighbouring steps, gives the same output bits and pool bytes as
    # separate uploads, over decode steps, prefill chunks and mixed steps
    w = custom(500, 8, 2, 128, 0, [(40, 0, 3), (0, 70, 1), (300, 0, 2), (0, 20, 2)],
               budget=48)
    results = []
    for mode in ("separate", "staged", "pipelined"):
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w)
        runner.load_history(kv, w, s.history_plan())
        stg = runner.StepStaging(kv)
        pipe = runner.StepPipeline(kv)
        outs = []
        plans = s.all_steps()
        for i, plan in enumerate(plans):
            if mode == "staged":
                stg.stage(plan, *runner.step_host_inputs(w, plan))
                stg.upload()
                stg.run(w.scale)
                stg.download()
                torch.cuda.synchronize()
                # the pinned output buffer is reused by the next step: keep a copy
                outs.append(runner.tensor_to_bits(stg.out_host).copy())
            elif mode == "pipelined":
                pipe.stage(i % 2, plan, *runner.step_host_inputs(w, plan))
                pipe.launch(i % 2, w.scale)
                if i > 0:  # the previous step's output, before its staging is reused
                    outs.append(runner.tensor_to_bits(pipe.result((i - 1) % 2)).copy())
            else:
                outs.append(runner.tensor_to_bits(runner.run_step(kv, w, plan)))
        if mode == "pipelined":
            outs.append(runner.tensor_to_bits(pipe.result((len(plans) - 1) % 2)).copy())
        torch.cuda.synchronize()
        assert kv.read_error() == 0
        results.append((outs, pool_bits(kv)))
    for other in results[1:]:
        assert len(results[0][0]) == len(other[0]) > 2
        for a, b in zip(results[0][0], other[0]):
            assert np.array_equal(a, b)
        assert all(np.array_equal(a, b) for a, b in zip(results[0][1], other[1]))


@pytest.mark.parametrize("kv_int8", [False, True])
def test_ragged_step_with_idle_requests(kv_int8):
    # one launch mixing requests that do not advance (q_len 0, with and without cached
    # keys) with rows on both sides of the decode/prefill switch (15 rows stay on the
    # streaming path, 16 and 17 take the tensor-core tiles), two-row decodes and a decode
    # at a page edge: every row against the oracle; no page of an idle request changes
    specs = [(50, 0, 0), (33, 15, 0), (0, 16, 0), (16, 1, 0), (0, 0, 0), (127, 17, 0),
             (31, 0, 0), (200, 2, 0)]
    w = custom(640, 8, 2, 128, 0, specs)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=kv_int8)
    runner.load_history(kv, w, s.history_plan())
    step = s.next_step()
    got = {int(r): j for j, r in enumerate(step.rids)}
    rids, q_lens, ctx, tables = [], [], [], []
    for r, spec in enumerate(specs):
        rids.append(r)
        if r in got:
            j = got[r]
            q_lens.append(int(step.q_lens[j]))
            ctx.append(int(step.context_lens[j]))
            tables.append([p for p in step.block_table[j].tolist() if p >= 0])
        else:
            q_lens.append(0)
            ctx.append(spec[0])
            tables.append(list(s.reqs[r].pages))
    assert q_lens == [0, 15, 16, 1, 0, 17, 0, 2]
    plan = make_plan(rids, q_lens, ctx, tables)
    idle_pages = [p for r in (0, 6) for p in tables[r]]
    before = [b[idle_pages].copy() for b in pool_bits(kv)]
    out = runner.run_step(kv, w, plan)
    assert kv.read_error() == 0
    assert all(np.array_equal(b[idle_pages], a) for b, a in zip(pool_bits(kv), before))
    ref = oracle_rows_int8(w, plan) if kv_int8 else oracle_rows(w, plan)
    assert out.shape[0] == sum(q_lens)
    assert_close(gpu_as_f64(out), ref, "ragged step")


@pytest.mark.parametrize("kv_int8", [False, True])
def test_decode_step_with_idle_requests(kv_int8):
    # a decode step (every row q_len <= 1, so the self-planned decode grid) in which some
    # requests do not advance: q_len 0 with cached keys, and q_len 0 with none.  They give
    # zero-length segments to the in-kernel plan; every row matches the oracle, the fused
    # and the separate calls give the same bits, and no page of an idle request changes.
    specs = [(50, 0, 0), (33, 0, 1), (0, 0, 0), (16, 0, 1), (300, 0, 0), (127, 0, 1),
             (31, 0, 0), (1000, 0, 1), (15, 0, 1)]
    w = custom(660 + kv_int8, 8, 2, 128, 0, specs)
    results = []
    for fused in (True, False):
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w, kv_int8=kv_int8)
        runner.load_history(kv, w, s.history_plan())
        step = s.next_step()
        got = {int(r): j for j, r in enumerate(step.rids)}
        rids, q_lens, ctx, tables = [], [], [], []
        for r, spec in enumerate(specs):
            rids.append(r)
            if r in got:
                j = got[r]
                q_lens.append(int(step.q_lens[j]))
                ctx.append(int(step.context_lens[j]))
                tables.append([p for p in step.block_table[j].tolist() if p >= 0])
            else:
                q_lens.append(0)
                ctx.append(spec[0])
                tables.append(list(s.reqs[r].pages))
        assert q_lens == [0, 1, 0, 1, 0, 1, 0, 1, 1]
        plan = make_plan(rids, q_lens, ctx, tables)
        idle_pages = [p for r in (0, 4, 6) for p in tables[r]]
        before = [b[idle_pages].copy() for b in pool_bits(kv)]
        sl = torch.full((plan.total_q_tokens,), -7, dtype=torch.int64, device="cuda")
        if fused:
            out = runner.run_step_fused(kv, w, plan, sl)
        else:
            q, k, v = runner.step_host_inputs(w, plan)
            ds = kv.upload(plan)
            kv.append(ds, runner.bits_to_tensor(k, w.dtype), runner.bits_to_tensor(v, w.dtype),
                      sl)
            out = kv.attention(ds, runner.bits_to_tensor(q, w.dtype), w.scale)
        assert kv.read_error() == 0
        assert all(np.array_equal(b[idle_pages], a) for b, a in zip(pool_bits(kv), before))
        ref = oracle_rows_int8(w, plan) if kv_int8 else oracle_rows(w, plan)
        assert out.shape[0] == 5
        assert_close(gpu_as_f64(out), ref, "decode step with idle requests")
        results.append((out, sl, pool_bits(kv)))
    (fo, fs, fp), (so, ss, sp) = results
    assert torch.equal(fo.view(torch.int16), so.view(torch.int16))
    assert torch.equal(fs, ss)
    assert all(np.array_equal(a, b) for a, b in zip(fp, sp))


@pytest.mark.parametrize("kv_int8", [False, True])
def test_host_resident_decode_steps(kv_int8):
    # decode steps whose Q, new K/V, metadata and output stay in pinned host memory, read
    # and written in place by the kernels: the same output bits and pool bytes as the
    # copy-engine pipeline over device buffers, and every row against the oracle
    ctx = [0, 1, 15, 16, 17, 100, 255, 256, 1000, 3000]
    w = custom(2100 + kv_int8, 32, 8, 128, 0, [(c, 0, 3) for c in ctx])
    res = {}
    for host in (True, False):
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w, kv_int8=kv_int8)
        runner.load_history(kv, w, s.history_plan())
        pipe = runner.HostPipeline(kv) if host else runner.StepPipeline(kv)
        outs, plans = [], []
        for i, plan in enumerate(s.all_steps()):
            q, k, v = runner.step_host_inputs(w, plan)
            pipe.stage(i % 2, plan, q, k, v)
            pipe.launch(i % 2, w.scale)
            outs.append(pipe.result(i % 2).clone())
            plans.append(plan)
        torch.cuda.synchronize()
        assert kv.read_error() == 0
        res[host] = (outs, pool_bits(kv))
    (ho, hp), (do, dp) = res[True], res[False]
    assert len(ho) == len(do) == 3
    for i, plan in enumerate(plans):
        assert torch.equal(ho[i].view(torch.int16), do[i].view(torch.int16)), i
        ref = oracle_rows_int8(w, plan) if kv_int8 else oracle_rows(w, plan)
        assert_close(gpu_as_f64(ho[i]), ref, "host-resident step %d" % i)
    assert all(np.array_equal(a, b) for a, b in zip(hp, dp))


def test_host_q_refused_on_prefill_steps():
    # a step with a 40-token prefill reads Q with tensor-memory-accelerator copies: a Q in
    # pinned host memory is refused on the host, before anything is launched
    w = custom(2150, 8, 2, 128, 0, [(0, 40, 0), (20, 0, 1)])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    plan = s.next_step()
    assert plan.max_q_len >= 16
    q, _, _ = runner.step_host_inputs(w, plan)
    ds = kv.upload(plan)
    out = torch.full((plan.total_q_tokens, w.num_q_heads, w.head_dim), 7.0,
                     dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.PkvError) as e:
        kv.attention_desc(ds.desc, runner.bits_to_tensor(q, w.dtype, "cpu", pin=True), out,
                          w.scale, kv.workspace(ds.desc))
    assert e.value.status == -1  # PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    with pytest.raises(ValueError):
        runner.HostPipeline(kv).stage(0, plan, q, q, q)


def test_long_contexts():
    # maximum-size rows: a decode row over 131,071 cached tokens (8,192 pages, about 900
    # splits per (row, KV head); with up to 45 decode rows possible in this step the combine
    # runs one CTA of eight thread groups per (row, KV head)), one over 40,000,
    # and a 300-token prefill chunk on a 70,000-token history (about 550 key tiles per query
    # tile); every row is checked against the oracle
    worst, _, _ = run_all(custom(600, 32, 8, 128, 0, [(131071, 0, 1), (40000, 0, 1),
                                                      (70000, 300, 0)]))
    assert worst[0] < 2e-2


_LONG_SPECS = {
    "one_long_row": [(131071, 0, 1)],
    "long_among_short": [(60000, 0, 1)] + [(16 + (37 * i) % 600, 0, 1) for i in range(63)],
    "four_equal_rows": [(8191, 0, 1)] * 4,
}


@pytest.mark.parametrize("kv_int8,fused", [(False, True), (False, False), (True, True),
                                           (True, False)])
@pytest.mark.parametrize("case", sorted(_LONG_SPECS))
def test_decode_step_long_pairs(case, kv_int8, fused):
    # decode-only steps whose (request, KV head) pairs span many more work units than one
    # CTA folds at once: their pieces are folded in chunks on different CTAs and merged by
    # whichever arrives last.  Every row against the oracle; a second run of the same step
    # gives the same bits (the merge order does not depend on the arrival order).
    w = custom(700 + len(case) + 2 * kv_int8 + fused, 32, 8, 128, 0, _LONG_SPECS[case])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=kv_int8)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    assert plan.max_q_len == 1
    if fused:
        out = runner.run_step_fused(kv, w, plan)
        again = runner.run_step_fused(kv, w, plan)   # re-appends the same rows
    else:
        out = runner.run_step(kv, w, plan)
        q, _, _ = runner.step_host_inputs(w, plan)
        again = kv.attention(kv.upload(plan), runner.bits_to_tensor(q, w.dtype), w.scale)
    assert kv.read_error() == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    ref = oracle_rows_int8(w, plan) if kv_int8 else oracle_rows(w, plan)
    assert_close(gpu_as_f64(out), ref, "long pairs %s" % case)


@pytest.mark.parametrize("hq,hkv,d,dtype,case", [(32, 32, 128, 1, "four_equal_rows"),
                                                 (8, 1, 64, 0, "one_long_row"),
                                                 (16, 2, 64, 1, "long_among_short")])
def test_decode_step_long_pairs_head_shapes(hq, hkv, d, dtype, case):
    # the long-pair combine with other group sizes and head dims (thread groups of 32 to
    # 256 threads): fused decode steps against the oracle, repeated runs bit-identical
    w = custom(760 + hq + d, hq, hkv, d, dtype, _LONG_SPECS[case])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    out = runner.run_step_fused(kv, w, plan)
    again = runner.run_step_fused(kv, w, plan)
    assert kv.read_error() == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert_close(gpu_as_f64(out), oracle_rows(w, plan), "long pairs %s %d/%d" % (case, hq, hkv))


def test_long_row_two_pass_combine():
    # three decode rows, two self-planned steps: 131,071 cached keys (its 8 KV-head segments
    # span thousands of work units: folded in chunks on many CTAs, then merged), 3,000 keys
    # (a few dozen pieces per segment, folded by one CTA) and 100 keys (7 pages per segment:
    # mostly inside one unit, written by the decode kernel).  The long row's second token
    # opens page 8,192.
    worst, _, _ = run_all(custom(610, 32, 8, 128, 0, [(131071, 0, 2), (3000, 0, 2),
                                                      (100, 0, 2)]))
    assert worst[0] < 2e-2


def _tile_rows(plan, per_tile, seed=5):
    """Rows of every 128-row query tile of every request (its first and last row plus
    per_tile - 2 seeded picks), so each prefill unit of the step is checked."""
    rng = np.random.default_rng(seed)
    pick = set()
    for j in range(plan.num_reqs):
        o, n = int(plan.q_offsets[j]), int(plan.q_lens[j])
        for t0 in range(0, n, 128):
            t1 = min(n, t0 + 128)
            pick |= {o + t0, o + t1 - 1}
            pick |= set((o + rng.integers(t0, t1, size=per_tile - 2)).tolist())
    return sorted(pick)


@pytest.mark.parametrize("hq,hkv,d,dtype,specs", [
    (32, 8, 128, 0, [(12000, 2018, 0)]),
    (32, 32, 64, 1, [(12000, 2018, 0)]),
    (32, 4, 128, 0, [(9000, 1024, 0), (14000, 1024, 0), (3000, 0, 1)]),
])
def test_prefill_chunks_on_long_contexts(hq, hkv, d, dtype, specs):
    # 2K-row chunks over 9K-14K cached keys: 256 prefill CTAs of ~100 key tiles each (GQA
    # head pairs, MHA query-tile pairs, and two requests beside a decode row).  Sampled rows
    # of every 128-row query tile against the oracle; a second run gives the same bits.
    w = custom(620 + hkv + d, hq, hkv, d, dtype, specs)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    out = runner.run_step(kv, w, plan)
    again = runner.run_step(kv, w, plan)
    assert kv.read_error() == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    rows = _tile_rows(plan, 6)
    mx, mean = assert_close(gpu_as_f64(out[torch.as_tensor(rows)]), oracle_rows(w, plan, rows),
                            "long-context chunk")
    print("long-context chunk", hq, hkv, d, dtype, "worst", mx, mean)


def test_decode_loop_and_graph_bitwise_identical():
    # the MHA-skew workload's 64 decode steps (16 requests, fp16, page boundaries crossed
    # mid-run) as 64 separate steps, as one device-side loop (lengths advanced on the
    # device, the last step's block table) and as one CUDA graph replay: same output bits
    # and pool bytes
    w = W.mha_skew()

    def fresh():
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w)
        runner.load_history(kv, w, s.history_plan())
        return s, kv

    s, kv = fresh()
    plans = s.all_steps()
    ref = torch.stack([runner.run_step(kv, w, p) for p in plans])
    ref_pool = pool_bits(kv)
    for mode in ("loop", "graph"):
        s, kv = fresh()
        loop = runner.DecodeLoop(kv, w, plans)
        if mode == "loop":
            out = loop.run()
        else:
            loop.capture()
            kv.k_cache.view(torch.int16).fill_(-1)  # replay must rewrite every appended slot
            kv.v_cache.view(torch.int16).fill_(-1)
            runner.load_history(kv, w, scheduler_for(w).history_plan())
            out = loop.replay()
        torch.cuda.synchronize()
        assert kv.read_error() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), mode
        assert all(np.array_equal(a, b) for a, b in zip(pool_bits(kv), ref_pool)), mode
        # and against the oracle directly, at the first, a middle and the last step
        for i in (0, 31, 63):
            assert_close(gpu_as_f64(out[i]), oracle_rows(w, plans[i]), "%s step %d" % (mode, i))


def _layer_of(w, layer):
    """Layer ``layer`` of a model step over workload ``w``: the same requests, lengths and
    pages, its own Q/K/V values (another seed)."""
    import dataclasses
    return dataclasses.replace(w, index=w.index + 100 * layer, _cache={})


def test_shared_plan_layers_match_per_layer_steps_and_oracle():
    # two layers of the MHA-skew run's 64 decode steps: one plan per step shared by both
    # layers (pkv_plan_attention + pkv_paged_attention_run) gives the same bits as every
    # layer planning its own step, and both layers match the oracle
    w0 = W.mha_skew()
    w1 = _layer_of(w0, 1)

    def fresh():
        pools = []
        for lw in (w0, w1):
            kv = runner.paged_kv_for(lw)
            runner.load_history(kv, lw, scheduler_for(lw).history_plan())
            pools.append(kv)
        return pools

    s = scheduler_for(w0)
    s.history_plan()
    plans = s.all_steps()
    outs = {}
    for shared in (False, True):
        kv0, kv1 = fresh()
        kv1.err = kv0.err
        loop = runner.DecodeLoop(kv0, w0, plans, layers=[(kv1, w1)], shared_plan=shared)
        if shared:
            loop.capture()
            loop.replay()
        else:
            loop.run()
        torch.cuda.synchronize()
        assert kv0.read_error() == 0
        outs[shared] = [o.clone() for o in loop.outs]
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for lw, o in zip((w0, w1), outs[True]):
        for i in (0, 31, 63):
            assert_close(gpu_as_f64(o[i]), oracle_rows(lw, plans[i]), "layer step %d" % i)


def _first_step(w):
    """The first step after the workload's cached history is loaded."""
    s = scheduler_for(w)
    s.history_plan()
    return s.next_step()


def test_shared_plan_mixed_step_two_layers():
    # a step with decode rows and prefill chunks (both kernels, prefill first): plan once,
    # then two layers' append + run; each layer's output equals a full step on its pools
    specs = [(3000, 0, 1), (0, 700, 0), (40, 0, 1), (900, 300, 0), (5, 0, 1)]
    w0 = custom(1600, 32, 8, 128, 0, specs)
    w1 = _layer_of(w0, 1)
    full, planned = [], []
    for mode in ("full", "planned"):
        pools = []
        for lw in (w0, w1):
            kv = runner.paged_kv_for(lw)
            runner.load_history(kv, lw, scheduler_for(lw).history_plan())
            pools.append(kv)
        plan = _first_step(w0)
        assert plan.max_q_len >= 16 and int((plan.q_lens == 1).sum()) == 3
        ds = pools[0].upload(plan)
        ws = pools[0].workspace(ds.desc)
        if mode == "planned":
            binding.plan_attention(ds.desc, ws, pools[0].err)
        for kv, lw in zip(pools, (w0, w1)):
            q, k, v = runner.step_host_inputs(lw, plan)
            kv.append(ds, runner.bits_to_tensor(k, 0), runner.bits_to_tensor(v, 0))
            out = torch.empty((plan.total_q_tokens, 32, 128), dtype=torch.bfloat16, device="cuda")
            qd = runner.bits_to_tensor(q, 0)
            if mode == "planned":
                kv.run_desc(ds.desc, qd, out, lw.scale, ws)
            else:
                kv.attention_desc(ds.desc, qd, out, lw.scale, ws)
            (full if mode == "full" else planned).append(out)
            assert kv.read_error() == 0
    for a, b in zip(full, planned):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_close(gpu_as_f64(planned[1]), oracle_rows(w1, plan), "planned layer 1")


def test_prefix_cache_reuse_matches_oracle():
    # prefix caching (hotelren.com/news/6181127 §4.3) through the native planner: requests
    # sharing a 100-token system prompt reuse the full prompt blocks the first one already
    # computed, continue at the reused position, and every row they compute must match the
    # oracle over their whole token sequence.  K, V and Q are functions of (position, token
    # id), as a model's are, so equal prefixes really hold equal K/V; the pool must hold
    # exactly that K/V in every slot any request's block table reaches.
    from paged_kv_cache_token_gb300.native_scheduler import NativeScheduler
    hq, hkv, d, vocab, P = 8, 2, 128, 40, 256
    g = torch.Generator().manual_seed(77)
    tab = lambda h: torch.randn(P, vocab, h, d, generator=g).to(torch.bfloat16)
    ktab, vtab, qtab = tab(hkv), tab(hkv), tab(hq)
    rng = np.random.default_rng(5)
    system = rng.integers(0, vocab, 100)
    prompts = [np.concatenate([system, rng.integers(0, vocab, n)]) for n in (30, 50, 12)]
    prompts.append(rng.integers(0, vocab, 80))
    decodes = [3, 2, 4, 2]
    seqs = [np.concatenate([p, rng.integers(0, vocab, n)]) for p, n in zip(prompts, decodes)]
    specs = [W.RequestSpec(r, 0, len(p), n) for r, (p, n) in enumerate(zip(prompts, decodes))]
    pages = sum(-(-len(x) // 16) for x in seqs) + 4
    w = W.Workload(900, "prefix", hq, hkv, d, 0, specs, np.arange(pages, dtype=np.int32), pages)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    for r, x in enumerate(seqs):
        pos = torch.arange(len(x))
        tok = torch.as_tensor(x)
        w._cache[("kv", r)] = (bits(ktab[pos, tok]), bits(vtab[pos, tok]))
        w._cache[("q", r)] = bits(qtab[pos, tok])
    s = NativeScheduler([], w.page_order, 64)  # 64-token budget: chunked prefills too
    kv = runner.paged_kv_for(w)
    assert s.add_prompt(0, prompts[0], decodes[0]) == 0
    tables = {}
    reused = None
    while True:
        plan = s.next_step()
        if plan is None:
            break
        out = runner.run_step(kv, w, plan)
        assert kv.read_error() == 0
        assert_close(gpu_as_f64(out), oracle_rows(w, plan), "prefix step")
        for j, rid in enumerate(plan.rids):
            tables[rid] = plan.block_table[j]
        if reused is None:  # after the first step the system prompt's first blocks exist
            reused = [s.add_prompt(r, prompts[r], decodes[r]) for r in (1, 2, 3)]
    assert reused[0] > 0 and reused[1] > 0 and reused[2] == 0
    shared = set(tables[0][:reused[0] // 16]) & set(tables[1][:reused[0] // 16])
    assert len(shared) == reused[0] // 16
    kc, vc = pool_bits(kv)
    for r, x in enumerate(seqs):
        k, v = w.kv(r)
        for p_ in range(len(x)):
            page = tables[r][p_ // 16]
            assert np.array_equal(kc[page, :, p_ % 16], k[p_]), (r, p_)
            assert np.array_equal(vc[page, :, p_ % 16], v[p_]), (r, p_)


def test_forked_requests_copy_the_shared_partial_page_on_write():
    # parallel samples of one prompt (pkv_sched_fork): a 100-token prompt leaves 4 tokens in
    # its 7th page; two forks share every page with it, and the three then decode 20 tokens
    # each, diverging inside that page.  The first writers get copies of the shared page
    # (pkv_copy_pages before the step's append), the last holder writes in place.  Every row
    # must match the oracle over the request's own sequence (the shared 100 prompt tokens,
    # then its own tokens), and every slot of every request's pages must hold its K/V.
    from paged_kv_cache_token_gb300.native_scheduler import NativeScheduler
    hq, hkv, d, P, n_dec = 8, 2, 128, 100, 20
    rng = np.random.default_rng(31)
    draw = lambda *shape: runner.tensor_to_bits(
        torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16))
    kp, vp, qp = draw(P, hkv, d), draw(P, hkv, d), draw(P, hq, d)
    specs = [W.RequestSpec(r, 0, P, n_dec) for r in range(3)]
    pages = 3 * -(-(P + n_dec) // 16) + 4
    w = W.Workload(910, "fork", hq, hkv, d, 0, specs, np.arange(pages, dtype=np.int32), pages)
    for r in range(3):
        k = np.concatenate([kp, draw(n_dec, hkv, d)])
        v = np.concatenate([vp, draw(n_dec, hkv, d)])
        w._cache[("kv", r)] = (k, v)
        w._cache[("q", r)] = np.concatenate([qp, draw(n_dec, hq, d)])
    s = NativeScheduler([], w.page_order, 256)
    s.add_request(0, 0, P, n_dec)
    kv = runner.paged_kv_for(w)
    plan = s.next_step()                      # the prompt, one chunk
    out = runner.run_step(kv, w, plan)
    assert_close(gpu_as_f64(out), oracle_rows(w, plan), "prompt")
    s.fork(0, 1, n_dec)
    s.fork(0, 2, n_dec)
    tables, copied = {}, 0
    while True:
        plan = s.next_step()
        if plan is None:
            break
        copied += 0 if plan.copies is None else len(plan.copies)
        out = runner.run_step(kv, w, plan)
        assert kv.read_error() == 0
        assert_close(gpu_as_f64(out), oracle_rows(w, plan), "forked decode step")
        for j, rid in enumerate(plan.rids):
            tables[rid] = plan.block_table[j].copy()
    assert copied == 2
    assert len({int(tables[r][6]) for r in range(3)}) == 3    # the partial page diverged
    assert len({tuple(tables[r][:6]) for r in range(3)}) == 1  # full pages still shared
    kc, vc = pool_bits(kv)
    for r in range(3):
        k, v = w.kv(r)
        for pos in range(P + n_dec):
            page = tables[r][pos // 16]
            assert np.array_equal(kc[page, :, pos % 16], k[pos]), (r, pos)
            assert np.array_equal(vc[page, :, pos % 16], v[pos]), (r, pos)


def test_copy_pages_bit_exact_and_bad_ids_flagged():
    # whole-page copies in both pool kinds, bit for bit; an out-of-range id is flagged and
    # its copy skipped
    for kv_int8 in (False, True):
        sc = np.full((4, 64), 0.03, np.float32) if kv_int8 else None
        kv = runner.PagedKV(10, 8, 4, 64, 1, k_scale=sc, v_scale=sc)
        g = torch.Generator(device="cuda").manual_seed(3)
        kb, vb = kv.k_cache.view(torch.uint8), kv.v_cache.view(torch.uint8)
        for t in (kb, vb):
            t.copy_(torch.randint(0, 256, t.shape, generator=g, device="cuda",
                                  dtype=torch.uint8))
        k0, v0 = kb.clone(), vb.clone()
        plan = make_plan([0], [1], [0], [[0]])
        ds = kv.upload(plan)
        src = torch.tensor([1, 4, 7, 2], dtype=torch.int32, device="cuda")
        dst = torch.tensor([5, 9, 0, 12], dtype=torch.int32, device="cuda")  # 12: out of pool
        binding.copy_pages(ds.desc, src, dst, kv.k_cache, kv.v_cache, kv_int8, kv.err)
        assert kv.read_error() & binding.DEVERR_PAGE_RANGE
        ek, ev = k0.clone(), v0.clone()
        for a, b in ((1, 5), (4, 9), (7, 0)):
            ek[b], ev[b] = k0[a], v0[a]
        assert torch.equal(kb, ek) and torch.equal(vb, ev)


def test_block_table_permutation_bitwise_identical():
    base = custom(400, 32, 8, 128, 0, [(c, 0, 1) for c in (50, 700, 2100, 16)])
    outs = []
    for seed in (1, 2):
        w = custom(400, 32, 8, 128, 0, [(c, 0, 1) for c in (50, 700, 2100, 16)])
        g = torch.Generator().manual_seed(seed)
        w.page_order = torch.randperm(base.num_pages, generator=g).numpy().astype(np.int32)
        _, o, _ = run_all(w, every_step=False)
        outs.append(runner.tensor_to_bits(o[0]))
    assert np.array_equal(outs[0], outs[1])


def test_attention_bad_page_sets_flag():
    w = custom(500, 4, 2, 64, 0, [(20, 0, 1)])
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    plan.block_table[0, 0] = w.num_pages + 3
    q, k, v = runner.step_host_inputs(w, plan)
    ds = kv.upload(plan)
    kv.attention(ds, runner.bits_to_tensor(q, 0), w.scale)
    assert kv.read_error() & binding.DEVERR_PAGE_RANGE


# ------------------------------------------------------------------------------ full configs
def test_config_decode_only_full():
    """64 requests, ctx U[512, 4096], 32/8 heads, d=128, bf16, 70k-page permuted pool:
    every output row against the oracle."""
    worst, _, _ = run_all(W.decode_only())
    print("decode-only worst max/mean abs", worst)


def test_config_mha_skew_all_64_steps():
    worst, _, _ = run_all(W.mha_skew())
    print("mha-skew worst max/mean abs", worst)


def _sample_rows(plan, n=24, seed=0):
    T = plan.total_q_tokens
    rng = np.random.default_rng(seed + T)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pick |= {0, T - 1}
    # every request's first and last row (decodes, chunk edges)
    for j in range(plan.num_reqs):
        if plan.q_lens[j]:
            pick |= {int(plan.q_offsets[j]), int(plan.q_offsets[j + 1]) - 1}
    return sorted(pick)


def test_config_prefill_one_shot_and_chunked():
    # every 128-row query tile of every step has oracle-checked rows (all 32 heads)
    one = W.prefill()
    w1, o1, _ = run_all(one, check_rows=lambda p: _tile_rows(p, 6))
    ch = W.prefill(chunk=2048)
    w2, o2, _ = run_all(ch, check_rows=lambda p: _tile_rows(p, 6))
    chunked = torch.cat(o2)
    diff = (chunked.float() - o1[0].float()).abs().max().item()
    print("prefill one-shot", w1, "chunked", w2, "gpu chunked-vs-one-shot max diff", diff)
    assert diff <= 2 * 2e-2


def test_config_mixed_chunked_matches_oracle_and_one_shot():
    # every decode row and rows of every 128-row query tile of each chunk, every step
    w = W.mixed()
    worst, outs, _ = run_all(w, check_rows=lambda p: _tile_rows(p, 4))
    print("mixed worst", worst)
    # the prompt's chunked rows against a one-shot run of the same prompt
    prompt = w.requests[-1]
    npages = (prompt.prompt + 15) // 16 + 8
    order = torch.randperm(npages, generator=torch.Generator().manual_seed(11)).numpy()
    one = W.Workload(w.index, "one-shot", 32, 8, 128, 0, [W.RequestSpec(0, 0, prompt.prompt, 0)],
                     order.astype(np.int32), npages, budget=prompt.prompt)
    one._cache[("kv", 0)] = w.kv(prompt.rid)
    one._cache[("q", 0)] = w.q(prompt.rid)
    _, o1, _ = run_all(one, check_rows=lambda p: _sample_rows(p, 16))
    chunked = torch.cat([o[-int(len_):] for o, len_ in
                         zip(outs, [2018] * 14 + [1748])])
    diff = (chunked.float() - o1[0].float()).abs().max().item()
    print("mixed: gpu chunked-vs-one-shot max diff", diff)
    assert diff <= 2 * 2e-2


def test_sorted_native_plans_match_oracle():
    # steps planned by the native planner after sorting the batch by prompt length
    # (lshu.cn/news/11576 §2.2): launch order and page placement change, the rows do not
    from paged_kv_cache_token_gb300.native_scheduler import native_scheduler_for
    w = custom(520, 8, 2, 128, 0, [(0, n, 2) for n in (300, 20, 150, 5, 64, 17)], budget=128)
    s = native_scheduler_for(w)
    s.sort_by_length()
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    steps = s.all_steps()
    assert list(steps[0].rids[:3]) == [3, 5, 1]
    for i, plan in enumerate(steps):
        out = runner.run_step(kv, w, plan)
        assert_close(gpu_as_f64(out), oracle_rows(w, plan), "sorted step %d" % i)
    assert kv.read_error() == 0


@pytest.mark.parametrize("hq,d,dtype", [(8, 64, 1), (4, 128, 0), (2, 128, 1)])
def test_mha_prefill_tile_pairs(hq, d, dtype):
    # one query head per KV head: a prefill CTA takes query tiles 2u and 2u + 1 of one
    # head; odd tile counts leave its second chain without rows, and the first chain sees
    # the second tile's extra keys fully masked
    specs = [(0, 1, 0), (0, 127, 0), (0, 128, 0), (0, 129, 1), (0, 256, 0), (0, 257, 0),
             (300, 383, 0), (40, 640, 1)]
    run_all(custom(1100 + hq + d, hq, hq, d, dtype, specs))


def test_mha_prefill_8k_one_shot_sampled():
    """An 8,192-token causal prefill with 32 query heads each on its own KV head (MHA):
    sampled rows against the oracle."""
    w = W.prefill()
    w.num_kv_heads = 32
    w.num_pages = w.pages_needed() + 8
    w.page_order = torch.randperm(w.num_pages,
                                  generator=torch.Generator().manual_seed(77)).numpy().astype(np.int32)
    worst, _, _ = run_all(w, check_rows=lambda p: _tile_rows(p, 4))
    print("mha prefill 8k worst", worst)


def test_many_requests_cross_plan_chunks():
    # 2,500 requests in one step: the device planner works through them 1,024 at a time,
    # carrying its row, item and tile counts from chunk to chunk; decodes and short
    # prefill chunks are interleaved so every chunk holds both kinds
    rng = np.random.default_rng(2500)
    specs = []
    for i in range(2500):
        if i % 7 == 3:
            specs.append((int(rng.integers(0, 60)), int(rng.integers(16, 40)), 0))
        else:
            specs.append((int(rng.integers(0, 90)), 0, 1))
    w = custom(1300, 4, 2, 64, 0, specs, extra_pages=16)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    assert plan.num_reqs == 2500 and plan.max_q_len >= 16
    out = runner.run_step(kv, w, plan)
    assert kv.read_error() == 0
    rows = _sample_rows(plan, 400)
    assert_close(gpu_as_f64(out[torch.as_tensor(rows)]), oracle_rows(w, plan, rows), "2500 reqs")


def test_gqa8_prefill_4k_and_decode_sampled():
    """Eight query heads per KV head (64/8, d=128, bf16): a 4,096-token one-shot prefill in
    the pair kernel, then 4 decode steps, sampled rows against the oracle."""
    w = custom(1400, 64, 8, 128, 0, [(0, 4096, 4)])
    worst, _, _ = run_all(w, check_rows=lambda p: _tile_rows(p, 4))
    print("gqa8 worst", worst)


def test_fp16_prefill_8k_one_shot_sampled():
    """The 8,192-token one-shot prefill with fp16 Q/K/V (32/8 heads, d=128)."""
    w = W.prefill()
    w.dtype = W.FP16
    w._cache.clear()
    worst, _, _ = run_all(w, check_rows=lambda p: _tile_rows(p, 4))
    print("fp16 prefill worst", worst)


def test_d64_decode_long_contexts():
    """Head dim 64 (16/4 heads, fp16): decode rows over 20k-60k cached tokens, many splits."""
    w = custom(1500, 16, 4, 64, 1, [(60000, 0, 2), (20000, 0, 2), (33333, 0, 2)])
    worst, _, _ = run_all(w)
    assert worst[0] < 2e-2
