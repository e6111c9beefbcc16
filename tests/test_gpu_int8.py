"""GPU parity of the INT8 KV cache (wmrh.cn/news/64708 §4.3, §5.4) through the C ABI: the
codes kv_append writes must equal the oracle's quantiser bit for bit, in the slots the
block table names; attention over the codes must be within max-abs 2e-2 and mean-abs 2e-3
of the oracle's fp64 attention over the values the codes stand for."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_token_gb300 import binding, build, runner
from paged_kv_cache_token_gb300 import workloads as W
from paged_kv_cache_token_gb300.scheduler import scheduler_for

from gpu_common import assert_close, gpu_as_f64, oracle_rows_int8, request_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def custom(index, hq, hkv, d, dtype, specs, budget=1 << 30, chunk_cap=None, extra_pages=8):
    reqs = [W.RequestSpec(i, *s) for i, s in enumerate(specs)]
    need = sum(-(-r.total // 16) for r in reqs) + extra_pages
    g = torch.Generator().manual_seed(9000 + index)
    order = torch.randperm(need, generator=g).numpy().astype(np.int32)
    return W.Workload(index, "custom-int8", hq, hkv, d, dtype, reqs, order, need, budget=budget,
                      chunk_cap=chunk_cap)


def run_all_int8(w, check_rows=None):
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=True)
    runner.load_history(kv, w, s.history_plan())
    worst, outs = (0.0, 0.0), []
    for i, plan in enumerate(s.all_steps()):
        out = runner.run_step(kv, w, plan)
        rows = None if check_rows is None else check_rows(plan)
        ref = oracle_rows_int8(w, plan, rows)
        got = gpu_as_f64(out) if rows is None else gpu_as_f64(out[torch.as_tensor(rows)])
        assert kv.read_error() == 0
        mx, mean = assert_close(got, ref, "%s int8 step %d" % (w.name, i))
        worst = (max(worst[0], mx), max(worst[1], mean))
        outs.append(out)
    assert kv.read_error() == 0
    return worst, outs, kv


def expected_pools(w, kv_steps):
    """Pools the oracle writes: its codes (as bytes in uint16 cells) placed by its append,
    the value pool in the library's dim-major page order."""
    shape = (w.num_pages, w.num_kv_heads, 16, w.head_dim)
    kp = np.full(shape, 0x80, np.uint16)   # INT8 sentinel -128 as a byte
    vp = kp.copy()
    slots = []
    for plan in kv_steps:
        kc = np.concatenate([request_codes(w, r)[0][c:c + n] for r, c, n in
                             zip(plan.rids, plan.context_lens.tolist(), plan.q_lens.tolist())])
        vc = np.concatenate([request_codes(w, r)[1][c:c + n] for r, c, n in
                             zip(plan.rids, plan.context_lens.tolist(), plan.q_lens.tolist())])
        as_u16 = lambda x: x.view(np.uint8).astype(np.uint16)
        kp, vp, sl = oracle.kv_append(plan.q_lens, plan.context_lens, plan.block_table,
                                      w.num_pages, as_u16(kc), as_u16(vc), kp, vp)
        slots.append(sl)
    to_i8 = lambda p: p.astype(np.uint8).view(np.int8)
    # value pages are stored dim-major ([page][head][dim][slot])
    return to_i8(kp), np.ascontiguousarray(np.swapaxes(to_i8(vp), 2, 3)), slots


# ------------------------------------------------------------------------------ kv_append
@pytest.mark.parametrize("hq,hkv,d,dtype", [(4, 2, 64, 0), (32, 8, 128, 0), (6, 3, 128, 1),
                                            (8, 1, 64, 1)])
def test_int8_append_codes_bit_exact(hq, hkv, d, dtype):
    # histories and prompts across page edges, then decode steps; every pool byte and every
    # slot id must equal the oracle's
    specs = [(0, 1, 2), (15, 1, 1), (16, 17, 1), (31, 0, 3), (100, 40, 0), (0, 0, 2)]
    w = custom(700 + hq + d + dtype, hq, hkv, d, dtype, specs, budget=64)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=True)
    steps = [p for p in [s.history_plan()] + s.all_steps() if p is not None]
    got_slots = []
    for plan in steps:
        _, k, v = runner.step_host_inputs(w, plan)
        ds = kv.upload(plan)
        slots = torch.full((plan.total_q_tokens,), -7, dtype=torch.int64, device="cuda")
        kv.append(ds, runner.bits_to_tensor(k, w.dtype), runner.bits_to_tensor(v, w.dtype),
                  slots)
        got_slots.append(slots.cpu().numpy())
    ref_k, ref_v, ref_slots = expected_pools(w, steps)
    assert kv.read_error() == 0
    assert np.array_equal(kv.k_cache.cpu().numpy(), ref_k)
    assert np.array_equal(kv.v_cache.cpu().numpy(), ref_v)
    assert all(np.array_equal(a, b) for a, b in zip(got_slots, ref_slots))


def test_int8_append_ties_and_clamps_exact():
    # K/V values placed on code ties (k + 0.5) * s and past the +-127 range: the kernel's
    # rounding (ties to even) and clamping must equal the oracle's
    w = custom(750, 4, 2, 64, 0, [(0, 40, 0)])
    ks, vs = w.int8_scales()
    rng = np.random.default_rng(5)
    codes = rng.integers(-140, 141, size=(40, 2, 64)).astype(np.float32)
    # channels 0..31: s = 2^-5 and |2c + 1| <= 127, so bf16 holds x = (c + 0.5) * s exactly
    # and x / s is an exact tie; channels 32..63 keep the drawn scales and reach past +-127
    codes[:, :, :32] = rng.integers(-64, 64, size=(40, 2, 32))
    ks = ks.copy()
    ks[:, :32] = 2.0 ** -5
    vs = ks.copy()
    x = (codes + 0.5) * ks[None]
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w._cache[("kv", 0)] = (bits, bits.copy())
    w._cache[("int8_scales",)] = (ks, vs)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=True)
    plan = s.next_step()
    _, k, v = runner.step_host_inputs(w, plan)
    ds = kv.upload(plan)
    kv.append(ds, runner.bits_to_tensor(k, 0), runner.bits_to_tensor(v, 0))
    ref_k, ref_v, _ = expected_pools(w, [plan])
    assert kv.read_error() == 0
    got = kv.k_cache.cpu().numpy()
    assert np.array_equal(got, ref_k) and np.array_equal(kv.v_cache.cpu().numpy(), ref_v)
    # the case really has ties and clamps
    ref_codes = request_codes(w, 0)[0]
    assert (np.abs(ref_codes) == 127).sum() > 100
    assert (ref_codes[:, :, :32] % 2 == 0).all()    # exact ties round to the even code


def test_int8_append_rejects_missing_or_unaligned_scales():
    w = custom(760, 4, 2, 64, 0, [(0, 3, 0)])
    kv = runner.paged_kv_for(w, kv_int8=True)
    plan = scheduler_for(w).next_step()
    _, k, v = runner.step_host_inputs(w, plan)
    ds = kv.upload(plan)
    kt, vt = runner.bits_to_tensor(k, 0), runner.bits_to_tensor(v, 0)
    rc = binding.kv_append_int8(ds.desc, kt, vt, None, kv.v_scale, kv.k_cache, kv.v_cache,
                                check=False)
    assert rc == -1
    off = torch.empty(2 * 64 + 1, dtype=torch.float32, device="cuda")[1:]
    rc = binding.kv_append_int8(ds.desc, kt, vt, off, kv.v_scale, kv.k_cache, kv.v_cache,
                                check=False)
    assert rc == -1
    torch.cuda.synchronize()


# ------------------------------------------------------------------------------ attention
def test_int8_tiny_all_steps():
    run_all_int8(W.tiny())


@pytest.mark.parametrize("hq,hkv,d,dtype", [(4, 2, 64, 0), (32, 8, 128, 0), (8, 8, 128, 1),
                                            (16, 2, 128, 1), (8, 1, 64, 0), (6, 3, 64, 1)])
def test_int8_decode_batches(hq, hkv, d, dtype):
    ctx = [0, 1, 15, 16, 17, 100, 255, 256, 1000, 3000]  # one key, page edges, multi-split
    run_all_int8(custom(800 + hq + d, hq, hkv, d, dtype, [(c, 0, 2) for c in ctx]))


@pytest.mark.parametrize("hq,hkv,d,dtype", [(4, 2, 64, 0), (32, 8, 128, 0), (8, 2, 128, 1),
                                            (16, 2, 64, 1), (8, 8, 64, 0), (4, 4, 128, 1)])
def test_int8_prefill_chunks(hq, hkv, d, dtype):
    # chunks of up to 96 rows over histories, around the 128-row tile and 16-token page
    # edges: an even KV group takes the tensor-core prefill over INT8 pages; with one query
    # head per KV head every row streams
    specs = [(0, 1, 1), (0, 127, 1), (0, 129, 2), (0, 300, 1), (20, 33, 0), (500, 64, 1)]
    run_all_int8(custom(900 + hq + d, hq, hkv, d, dtype, specs, budget=160, chunk_cap=96))


def test_int8_prefill_tiles_cross_pages_and_tiles():
    # one-shot prompts of 1..300 tokens over histories of 0..1000: ragged last pages and
    # tiles, diagonal tiles at every offset, pages past the end of a tile zero-filled
    specs = [(0, 16, 0), (0, 17, 0), (15, 113, 0), (1000, 300, 0), (130, 255, 1), (7, 129, 0)]
    run_all_int8(custom(960, 8, 2, 128, 0, specs))


def test_int8_prefill_scale_extremes():
    # Q' = Q * k_scale is rescaled by a power of two into fp16 range: queries of 1e-5 and
    # of 3e4 (far outside fp16 once multiplied out) give the oracle's rows
    for mag in (1e-5, 3e4):
        w = custom(970 + int(mag > 1), 4, 2, 64, 0, [(40, 200, 0)])
        q = w.q(0)
        x = (torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).float() * mag)
        w._cache[("q", 0)] = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        run_all_int8(w)


def test_int8_prefill_8k_one_shot_sampled():
    """The 8,192-token one-shot prefill (32/8 heads, d=128, bf16) over INT8 pages: sampled
    rows (every tile's first and last, ragged spots) against the oracle."""
    w = W.prefill()
    rng = np.random.default_rng(3)
    rows = lambda p: sorted(set(rng.choice(p.total_q_tokens, 40, replace=False).tolist()) |
                            {0, 127, 128, 4095, 8191})
    worst, _, _ = run_all_int8(w, check_rows=rows)
    print("int8 prefill 8k worst", worst)


def test_int8_long_rows():
    # a decode row over 131,071 cached tokens (thousands of splits per KV head) and a
    # 700-row prefill chunk in one step: rows many 32-row groups long in the work-list fill
    worst, _, _ = run_all_int8(custom(950, 32, 8, 128, 0, [(131071, 0, 1), (3000, 700, 0)]))
    assert worst[0] < 2e-2


def test_int8_mha_skew_all_64_steps():
    worst, _, _ = run_all_int8(W.mha_skew())
    print("int8 mha-skew worst", worst)


def test_int8_decode_only_full_sampled():
    """The decode batch (64 requests, ctx U[512, 4096], 32/8 heads, d=128, bf16): every
    request's row against the oracle."""
    worst, _, _ = run_all_int8(W.decode_only())
    print("int8 decode-only worst", worst)


def test_int8_decode_loop_graph_bitwise_identical():
    w = W.mha_skew()

    def fresh():
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w, kv_int8=True)
        runner.load_history(kv, w, s.history_plan())
        return s, kv

    s, kv = fresh()
    plans = s.all_steps()
    ref = torch.stack([runner.run_step(kv, w, p) for p in plans])
    ref_pool = (kv.k_cache.clone(), kv.v_cache.clone())
    s, kv = fresh()
    loop = runner.DecodeLoop(kv, w, plans)
    loop.capture()
    kv.k_cache.fill_(runner.INT8_SENTINEL)
    kv.v_cache.fill_(runner.INT8_SENTINEL)
    runner.load_history(kv, w, scheduler_for(w).history_plan())
    out = loop.replay()
    torch.cuda.synchronize()
    assert kv.read_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kv.k_cache, ref_pool[0]) and torch.equal(kv.v_cache, ref_pool[1])
    for i in (0, 31, 63):  # the replayed steps against the oracle directly
        assert_close(gpu_as_f64(out[i]), oracle_rows_int8(w, plans[i]), "graph step %d" % i)
    # the device loop launched call by call, against the oracle too
    s, kv = fresh()
    out = runner.DecodeLoop(kv, w, plans).run()
    torch.cuda.synchronize()
    assert kv.read_error() == 0
    for i in (0, 31, 63):
        assert_close(gpu_as_f64(out[i]), oracle_rows_int8(w, plans[i]), "loop step %d" % i)


def test_int8_mha_prefill_tile_pairs():
    # INT8 pages with one query head per KV head: tile pairs of one head on the tensor cores
    specs = [(0, 1, 0), (0, 129, 1), (0, 256, 0), (0, 257, 0), (300, 383, 0), (40, 640, 1)]
    run_all_int8(custom(1200, 8, 8, 128, 0, specs))


def test_int8_many_requests_cross_plan_chunks():
    rng = np.random.default_rng(2501)
    specs = [((int(rng.integers(0, 60)), int(rng.integers(16, 40)), 0) if i % 7 == 3
              else (int(rng.integers(0, 90)), 0, 1)) for i in range(2500)]
    w = custom(1301, 8, 2, 128, 0, specs, extra_pages=16)
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, kv_int8=True)
    runner.load_history(kv, w, s.history_plan())
    plan = s.next_step()
    assert plan.num_reqs == 2500
    out = runner.run_step(kv, w, plan)
    assert kv.read_error() == 0
    T = plan.total_q_tokens
    rows = sorted(set(np.random.default_rng(5).choice(T, 300, replace=False).tolist()) | {0, T - 1})
    got = gpu_as_f64(out[torch.as_tensor(rows)])
    assert_close(got, oracle_rows_int8(w, plan, rows), "int8 2500 reqs")


def test_int8_bad_pages_set_flags_and_skip():
    # a page id outside the pool: the append skips that token (nothing else written) and
    # flags it; attention through the same table flags it too and never faults
    from paged_kv_cache_token_gb300.scheduler import make_plan
    plan = make_plan([0, 1], [3, 2], [0, 0], [[0], [7]])   # page 7 outside a 4-page pool
    scales = np.full((1, 64), 0.05, np.float32)
    kv = runner.PagedKV(4, 1, 1, 64, 0, k_scale=scales, v_scale=scales)
    ds = kv.upload(plan)
    k = torch.full((5, 1, 64), 1.0, dtype=torch.bfloat16, device="cuda")   # code 20
    kv.append(ds, k, k)
    assert kv.read_error() & binding.DEVERR_PAGE_RANGE
    kc = kv.k_cache.cpu().numpy()
    assert np.all(kc[0, 0, :3] == 20) and np.all(kc[0, 0, 3:] == runner.INT8_SENTINEL)
    assert np.all(kc[1:] == runner.INT8_SENTINEL)
    kv.err.zero_()
    q = torch.zeros((5, 1, 64), dtype=torch.bfloat16, device="cuda")
    kv.attention(ds, q, 0.125)
    assert kv.read_error() & binding.DEVERR_PAGE_RANGE


def test_int8_append_negative_offsets_flagged_and_skipped():
    # request 1 starts at token row -1 with a length that matches its offsets: refused like
    # request 0, whose length disagrees; no code or slot id is written
    from paged_kv_cache_token_gb300.scheduler import make_plan
    plan = make_plan([0, 1], [1, 1], [0, 0], [[0], [1]])
    sc = np.full((1, 64), 0.03, np.float32)
    kv = runner.PagedKV(4, 1, 1, 64, 0, k_scale=sc, v_scale=sc)
    ds = kv.upload(plan)
    qo = torch.tensor([0, -1, 0], dtype=torch.int32, device="cuda")
    desc = binding.make_desc(num_reqs=2, num_q_heads=1, num_kv_heads=1, head_dim=64,
                             num_pages=4, max_pages_per_req=plan.max_pages, total_q_tokens=2,
                             max_q_len=1, max_context_len=0, dtype=0, q_lens=ds.tensors[0],
                             q_offsets=qo, context_lens=ds.tensors[2],
                             block_table=ds.tensors[3])
    k = torch.ones((2, 1, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.full((2,), -7, dtype=torch.int64, device="cuda")
    kv.append_desc(desc, k, k, slots)
    assert kv.read_error() & binding.DEVERR_TOKENS
    assert bool((kv.k_cache == runner.INT8_SENTINEL).all())
    assert bool((kv.v_cache == runner.INT8_SENTINEL).all())
    assert slots.cpu().tolist() == [-7, -7]


def _first_step(w):
    """The first step after the workload's cached history is loaded."""
    s = scheduler_for(w)
    s.history_plan()
    return s.next_step()


def test_int8_shared_plan_two_layers():
    # INT8 pools: one plan, two layers' runs (pkv_paged_attention_run_int8), each layer
    # against the oracle over its own codes
    import dataclasses
    specs = [(2000, 0, 1), (0, 300, 0), (100, 0, 1)]
    w0 = custom(1700, 32, 8, 128, 0, specs)
    w1 = dataclasses.replace(w0, index=w0.index + 100, _cache={})
    plan = _first_step(w0)
    pools = []
    for lw in (w0, w1):
        kv = runner.paged_kv_for(lw, kv_int8=True)
        runner.load_history(kv, lw, scheduler_for(lw).history_plan())
        pools.append(kv)
    ds = pools[0].upload(plan)
    ws = pools[0].workspace(ds.desc)
    binding.plan_attention(ds.desc, ws, pools[0].err)
    for kv, lw in zip(pools, (w0, w1)):
        q, k, v = runner.step_host_inputs(lw, plan)
        kv.append(ds, runner.bits_to_tensor(k, 0), runner.bits_to_tensor(v, 0))
        out = torch.empty((plan.total_q_tokens, 32, 128), dtype=torch.bfloat16, device="cuda")
        kv.run_desc(ds.desc, runner.bits_to_tensor(q, 0), out, lw.scale, ws)
        assert kv.read_error() == 0
        assert_close(gpu_as_f64(out), oracle_rows_int8(lw, plan), "int8 planned layer")
