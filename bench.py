"""Benchmark of the paged-KV attention step on GB300.

Default workload (the headline metric): decode-only step with Llama-3-8B attention shapes --
64 requests, cached contexts uniform in [512, 4096], 32 query / 8 KV heads, head dim 128,
bf16, 16-token pages scattered over a 70,000-page pool.  One step = kv_append of the 64 new
tokens + paged_attention_step (plan, decode stream, split combine).  The metric is KV GB/s:
algorithmic bytes of the step (K/V read by attention, Q read, output write, append read +
write, block-table reads) divided by the step time.  The secondary object "prefill_chunk"
times the tensor-core-bound workload: one-shot causal prefill of 8,192 tokens (32/8 heads,
d=128) and the same prompt as 4 x 2,048-token chunks, in TFLOP/s of causal attention FLOPs.
The object "decode_loop" times 64 consecutive decode steps of the MHA-skew workload as
separate steps, as one device-side loop and as one CUDA graph replay (per-step overhead).
The object "int8_kv" times the decode step over INT8 pages (per-channel scales): half the
K/V bytes of the bf16 step.  The object "mixed_step" times the 15 unified steps of the
mixed workload (30 decodes plus a 2,018-token prefill chunk per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 the script runs under torch.distributed.run, one rank per GPU; every rank runs
its own copy of the workload (requests are independent, no collective on the data path),
timing is max over ranks and ``value`` counts the bytes of all ranks (weak scaling).
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
import argparse
import gc
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_token_gb300 import workloads as W  # noqa: E402
from paged_kv_cache_token_gb300.scheduler import scheduler_for  # noqa: E402

METRIC = "paged-attn decode KV GB/s and prefill-chunk TFLOPS, % of GB300 peak"
L2_BYTES = 129 * 2 ** 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------------------ accounting
def step_bytes(w, plan, kv_esz=2):
    """Algorithmic bytes of one step: every byte the definition has to touch once.  With
    kv_esz = 1 (INT8 pages) the pages hold one byte per element and the per-channel K and V
    scales are read once by each kernel."""
    esz = 2
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    T = plan.total_q_tokens
    kv_tokens = int((plan.context_lens.astype(np.int64) + plan.q_lens).sum())
    scales = 0 if kv_esz == 2 else 2 * hkv * d * 4
    attn_kv = kv_tokens * hkv * d * kv_esz * 2 + scales  # K and V read once per KV head
    q_out = T * hq * d * esz * 2                       # Q read, output written
    append = T * hkv * d * (esz + kv_esz) * 2 + scales  # K_new, V_new read, pages written
    pages = int(((plan.context_lens + plan.q_lens + 15) // 16).sum())
    meta = pages * 4 + plan.num_reqs * 12
    return dict(attention=attn_kv + q_out + meta, append=append,
                step=attn_kv + q_out + meta + append, kv=attn_kv)


def causal_flops(w, plan):
    """4 * D * Hq * (number of (query, key) pairs with key <= query)."""
    pairs = 0
    for c, n in zip(plan.context_lens.tolist(), plan.q_lens.tolist()):
        pairs += n * c + n * (n + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * pairs


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""
        else:
            self.out = ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unavailable"]}
        # samples under load: the upper half of the run is the timed kernels
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ our arm
# DRAM traffic per launch from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum),
# kept in profiles/dram_traffic.json with a digest of the kernel's sources at capture time;
# reported only while the sources still match, else null.
KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "common.cuh", "launch.h"],
    "decode_kernel_int8": ["decode.cu", "common.cuh", "launch.h"],
    "prefill_q8_kernel": ["prefill_q8.cu", "prefill_tile.cuh", "tc.cuh", "common.cuh",
                          "launch.h"],
    "prefill_pair_kernel": ["prefill_pair.cu", "prefill_tile.cuh", "tc.cuh", "common.cuh",
                            "launch.h"],
}


def kernel_source_digest(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def captured_traffic(kernel, scale=1.0):
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_digest(kernel):
        return None
    return rec["bytes_per_launch"] * scale


def lib_event():
    """A timing event whose CUDA handle exists (torch creates it on first record), so the
    library can record it on its own stream."""
    e = torch.cuda.Event(enable_timing=True)
    e.record()
    return e


def build_decode_state(device, pool_pages=70000):
    from paged_kv_cache_token_gb300 import runner
    w = W.decode_only(num_pages=pool_pages)
    s = scheduler_for(w)
    hist = s.history_plan()
    plan = s.next_step()
    kv = runner.paged_kv_for(w, device=device, fill_sentinel=False)
    runner.load_history(kv, w, hist)
    q, k, v = runner.step_host_inputs(w, plan)
    return w, plan, kv, (q, k, v)


def settle():
    """Collects garbage before a timed section.  The cyclic collector stays off while the
    bench runs (main): a collection landing in a timed loop of one or two milliseconds adds
    its whole pause to the steps (measured: the INT8 decode step read 0.084 instead of
    0.063 ms once the earlier sections had left enough live objects)."""
    gc.collect()


def time_decode(device, steps, warmup, dist_ctx, pool_pages=70000):
    settle()
    from paged_kv_cache_token_gb300 import binding, runner
    w, plan, kv, (qh, kh, vh) = build_decode_state(device, pool_pages)
    dt = w.dtype
    q = runner.bits_to_tensor(qh, dt, device)
    k_new = runner.bits_to_tensor(kh, dt, device)
    v_new = runner.bits_to_tensor(vh, dt, device)
    ds = kv.upload(plan)
    out = torch.empty((plan.total_q_tokens, w.num_q_heads, w.head_dim), dtype=kv.dtype,
                      device=device)
    ws = kv.workspace(ds.desc)
    stream = torch.cuda.current_stream()
    # a second, disjoint copy of the pools: consecutive steps alternate between the two, so
    # no step finds the previous step's K/V (613 MB, about 5x L2) in L2 -- the same effect as
    # flushing L2 between steps, without a flush kernel inside the timed region
    kv2 = runner.PagedKV(kv.num_pages, kv.hq, kv.hkv, kv.d, kv.dtype_code, device,
                         fill_sentinel=False)
    kv2.k_cache.copy_(kv.k_cache)
    kv2.v_cache.copy_(kv.v_cache)
    kv2.err = kv.err
    pools = (kv, kv2)
    parity = [0]

    def one_step():
        # kv_append + paged_attention_step as one call (pkv_append_attention: one fused
        # decode grid plus the combine for this decode step)
        p = pools[parity[0]]
        parity[0] ^= 1
        binding.append_attention(ds.desc, k_new, v_new, p.k_cache, p.v_cache, q, out, w.scale,
                                 ws, None, kv.err, stream)

    for _ in range(max(3, warmup)):
        one_step()
    torch.cuda.synchronize()
    assert kv.read_error() == 0

    kstart = [lib_event() for _ in range(steps)]
    kstop = [lib_event() for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    dist_ctx.barrier()
    torch.cuda.synchronize()
    with clocks:
        # repeat the timed region so the clock sampler sees >= ~1 s of load.  Each round
        # times `steps` plain steps (the step rate), then `steps` steps with events around
        # the decode kernel (its per-launch time): an event recorded between two launches
        # ends their programmatic overlap, so the plain steps carry none.
        reps = 0
        wall0 = time.time()
        while True:
            t0.record(stream)
            for i in range(steps):
                one_step()
            t1.record(stream)
            for i in range(steps):
                binding.set_kernel_events(0, kstart[i], kstop[i])
                one_step()
            binding.set_kernel_events(0, None, None)
            torch.cuda.synchronize()
            reps += 1
            if time.time() - wall0 > 1.0 or reps >= 50:
                break
    dist_ctx.barrier()
    ms_total = t0.elapsed_time(t1)          # last round's plain steps: exactly `steps`
    ms_kernel = float(np.mean([a.elapsed_time(b) for a, b in zip(kstart, kstop)]))
    ms_step = dist_ctx.max(ms_total / steps)
    assert kv.read_error() == 0
    acct = step_bytes(w, plan)

    # ---- end to end through the C ABI with host buffers (transfers inside the timed region).
    #      Each step's inputs sit packed in pinned host memory and its output lands there.
    #      Primary form (runner.HostPipeline): the decode kernels read Q, the new K/V and the
    #      step's metadata from the pinned buffer and write the output rows into pinned
    #      memory over the CPU-GPU link -- one library call per step on one stream.  Second
    #      form (runner.StepPipeline): one H2D copy, the call, one D2H copy, on copy streams
    #      with events; its event waits end the programmatic overlap between steps.  Both
    #      alternate two buffers (and the two pools).  A run with packing also packs every
    #      step's inputs from the caller's numpy arrays inside the timed region.
    def e2e_run(pipe, pack):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        pack_s = 0.0
        e0.record(stream)
        if hasattr(pipe, "start_after"):
            pipe.start_after(e0)
        for i in range(steps):
            if pack:
                h0 = time.perf_counter()
                pipe.stage(i % 2, plan, qh, kh, vh)
                pack_s += time.perf_counter() - h0
            pipe.launch(i % 2, w.scale)
        if hasattr(pipe, "join"):
            pipe.join()
        e1.record(stream)
        torch.cuda.synchronize()
        dist_ctx.barrier()
        return dist_ctx.max(e0.elapsed_time(e1) / steps), pack_s * 1e3 / steps

    e2e = {}
    for kind, cls in (("host", runner.HostPipeline), ("copy_engine", runner.StepPipeline)):
        pipe = cls(kv, stream, kv_alt=kv2)
        for slot in range(2):
            pipe.stage(slot, plan, qh, kh, vh)
        for i in range(4):
            pipe.launch(i % 2, w.scale)
        if hasattr(pipe, "join"):
            pipe.join()
        torch.cuda.synchronize()
        ms, _ = e2e_run(pipe, False)
        ms_pack, pack_ms = e2e_run(pipe, True)
        e2e[kind] = dict(ms=ms, ms_pack=ms_pack, host_pack_ms=pack_ms,
                         h2d=pipe.stg[0].h2d_bytes, d2h=pipe.stg[0].d2h_bytes)
        del pipe
    assert kv.read_error() == 0
    del kv2
    h2d, d2h = e2e["host"]["h2d"], e2e["host"]["d2h"]
    ms_e2e, ms_e2e_pack = e2e["host"]["ms"], e2e["host"]["ms_pack"]
    host_pack_ms = e2e["host"]["host_pack_ms"]
    return dict(w=w, plan=plan, acct=acct, ms_step=ms_step, ms_kernel=ms_kernel, ms_e2e=ms_e2e,
                h2d=h2d, d2h=d2h, clocks=clocks.summary(), launches=2 * steps,
                host_pack_ms=host_pack_ms, ms_e2e_pack=ms_e2e_pack,
                ms_e2e_copy=e2e["copy_engine"]["ms"])


def time_decode_int8(device, steps, pool_pages=70000):
    """The decode step over INT8 pages (same requests and shapes; per-channel scales), one
    pkv_append_attention_int8 call: step time, decode-kernel time (the grid that also
    appends the new rows) and their algorithmic bytes."""
    settle()
    from paged_kv_cache_token_gb300 import binding, runner
    w = W.decode_only(num_pages=pool_pages)
    s = scheduler_for(w)
    hist, plan = s.history_plan(), s.next_step()
    kv = runner.paged_kv_for(w, device=device, fill_sentinel=False, kv_int8=True)
    runner.load_history(kv, w, hist)
    qh, kh, vh = runner.step_host_inputs(w, plan)
    q, k_new, v_new = (runner.bits_to_tensor(x, w.dtype, device) for x in (qh, kh, vh))
    ds = kv.upload(plan)
    out = torch.empty((plan.total_q_tokens, w.num_q_heads, w.head_dim), dtype=kv.dtype,
                      device=device)
    ws = kv.workspace(ds.desc)
    stream = torch.cuda.current_stream()

    def one_step():
        # pkv_append_attention_int8: one decode grid quantises the new rows into their pages
        # and attends, then the combine
        kv.append_attention_desc(ds.desc, k_new, v_new, q, out, w.scale, ws, None, stream)

    for _ in range(3):
        one_step()
    torch.cuda.synchronize()
    assert kv.read_error() == 0
    kstart = [lib_event() for _ in range(steps)]
    kstop = [lib_event() for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # plain steps for the step rate, then as many with events around the decode kernel
    t0.record(stream)
    for i in range(steps):
        one_step()
    t1.record(stream)
    for i in range(steps):
        binding.set_kernel_events(0, kstart[i], kstop[i])
        one_step()
    binding.set_kernel_events(0, None, None)
    torch.cuda.synchronize()
    assert kv.read_error() == 0
    ms_step = t0.elapsed_time(t1) / steps
    ms_kernel = float(np.mean([a.elapsed_time(b) for a, b in zip(kstart, kstop)]))
    acct = step_bytes(w, plan, kv_esz=1)
    res = dict(ms_step=ms_step, ms_kernel=ms_kernel, step_bytes=acct["step"],
               kernel_bytes=acct["attention"] + acct["append"],
               step_GBps=acct["step"] / (ms_step * 1e-3) / 1e9,
               kernel_GBps=(acct["attention"] + acct["append"]) / (ms_kernel * 1e-3) / 1e9)
    del kv
    torch.cuda.empty_cache()
    return res


def time_prefill(device, reps=5, kv_int8=False):
    """Attention-kernel time of the 8K one-shot prefill and of the 4 x 2048 chunks (over
    INT8 pages with ``kv_int8``)."""
    settle()
    from paged_kv_cache_token_gb300 import binding, runner
    res = {}
    for label, chunk in (("one_shot_8192", None), ("chunks_4x2048", 2048)):
        w = W.prefill(chunk=chunk)
        s = scheduler_for(w)
        kv = runner.paged_kv_for(w, device=device, fill_sentinel=False, kv_int8=kv_int8)
        plans = s.all_steps()
        flops = sum(causal_flops(w, p) for p in plans)
        total_ms = 0.0
        main_ms = 0.0
        for p in plans:
            qh, kh, vh = runner.step_host_inputs(w, p)
            ds = kv.upload(p)
            q = runner.bits_to_tensor(qh, w.dtype, device)
            kv.append(ds, runner.bits_to_tensor(kh, w.dtype, device),
                      runner.bits_to_tensor(vh, w.dtype, device))
            out = torch.empty((p.total_q_tokens, w.num_q_heads, w.head_dim), dtype=kv.dtype,
                              device=device)
            kv.attention(ds, q, w.scale, out)          # warm-up
            torch.cuda.synchronize()
            # `reps` identical steps queued back to back between the events, so the host's
            # launch latency overlaps device work as it does in a stream of steps; then one
            # more step with events around its main kernel (kept out of the timed steps: an
            # event between two launches ends their programmatic overlap)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ka, kb = lib_event(), lib_event()
            a.record()
            for _ in range(reps):
                kv.attention(ds, q, w.scale, out)
            b.record()
            binding.set_kernel_events(0, ka, kb)
            binding.set_kernel_events(1, ka, kb)
            kv.attention(ds, q, w.scale, out)
            binding.set_kernel_events(0, None, None)
            binding.set_kernel_events(1, None, None)
            torch.cuda.synchronize()
            total_ms += a.elapsed_time(b) / reps
            main_ms += ka.elapsed_time(kb)
        assert kv.read_error() == 0
        res[label] = dict(ms=total_ms, tflops=flops / total_ms / 1e9, flops=flops,
                          main_kernel_ms=main_ms)
        del kv
        torch.cuda.empty_cache()
    return res


def time_mixed(device, reps=3):
    """The mixed workload's 15 unified steps (30 decodes + a 2,018-token chunk of a
    30,000-token prompt, token budget 2048): every step's append + attention, each step
    repeated `reps` times back to back between events (the repeats rewrite the same pages
    with the same values and recompute the same outputs)."""
    settle()
    from paged_kv_cache_token_gb300 import runner
    w = W.mixed()
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, device=device, fill_sentinel=False)
    runner.load_history(kv, w, s.history_plan())
    plans = s.all_steps()
    flops = sum(causal_flops(w, p) for p in plans)
    nbytes = sum(step_bytes(w, p)["step"] for p in plans)
    total = 0.0
    per_step = []
    for p in plans:
        qh, kh, vh = runner.step_host_inputs(w, p)
        ds = kv.upload(p)
        q, k, v = (runner.bits_to_tensor(x, w.dtype, device) for x in (qh, kh, vh))
        out = torch.empty((p.total_q_tokens, w.num_q_heads, w.head_dim), dtype=kv.dtype,
                          device=device)
        kv.append(ds, k, v)
        kv.attention(ds, q, w.scale, out)   # warm-up
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            kv.append(ds, k, v)
            kv.attention(ds, q, w.scale, out)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        per_step.append(ms)
        total += ms
    assert kv.read_error() == 0
    del kv
    torch.cuda.empty_cache()
    return {"steps": len(plans), "ms_total": total,
            "ms_per_step_first_last": [per_step[0], per_step[-1]],
            "tflops": flops / total / 1e9, "flops": flops, "step_bytes_total": nbytes}


def time_decode_loop(device, reps=5):
    """64 consecutive decode steps of the MHA-skew workload (16 requests, 32 heads, fp16):
    per-step time as separate steps (metadata of every step already on the device, append +
    attention launched from the host), as one device-side loop (lengths advanced on the
    device) and as one CUDA graph replay of all 64 steps."""
    settle()
    from paged_kv_cache_token_gb300 import binding, runner
    w = W.mha_skew()
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, device=device, fill_sentinel=False)
    runner.load_history(kv, w, s.history_plan())
    plans = s.all_steps()
    nbytes = sum(step_bytes(w, p)["step"] for p in plans)
    loop = runner.DecodeLoop(kv, w, plans)
    loop.capture()
    dsteps = [kv.upload(p) for p in plans]
    ws = kv.workspace(loop.desc)
    for ds in dsteps:
        ws = kv.workspace(ds.desc)
    stream = torch.cuda.current_stream()

    def separate():
        for i, ds in enumerate(dsteps):
            binding.kv_append(ds.desc, loop.k_new[i], loop.v_new[i], kv.k_cache, kv.v_cache,
                              None, kv.err, stream)
            binding.paged_attention_step(ds.desc, loop.q[i], kv.k_cache, kv.v_cache,
                                         loop.out[i], w.scale, ws, kv.err, stream)

    res = {}
    for name, fn in (("separate_steps", separate), ("device_loop", loop.run),
                     ("graph", loop.replay)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b))
        ms = float(np.median(t))
        res[name] = {"us_per_step": ms * 1e3 / len(plans), "GBps": nbytes / (ms * 1e-3) / 1e9}
    assert kv.read_error() == 0
    res["steps"] = len(plans)
    res["bytes_per_step"] = nbytes / len(plans)
    return res


def time_decode_loop_layers(device, n_layers=4, reps=5):
    """The MHA-skew workload's 64 decode steps over ``n_layers`` layers, each layer with its
    own page pools (one layer's cache is ~93 MB, so four of them do not fit in the 129 MB
    L2): per step, every layer's append + attention, then the lengths advance on the device;
    the whole sequence is one CUDA graph, so per-layer steps read their K/V from HBM.  Timed
    twice: every layer planning its own step (pkv_paged_attention_step), and one plan per
    step shared by the layers (pkv_plan_attention + pkv_paged_attention_run)."""
    settle()
    from paged_kv_cache_token_gb300 import runner
    w = W.mha_skew()
    s = scheduler_for(w)
    kv = runner.paged_kv_for(w, device=device, fill_sentinel=False)
    runner.load_history(kv, w, s.history_plan())
    plans = s.all_steps()
    nbytes = sum(step_bytes(w, p)["step"] for p in plans)
    extra = []
    for _ in range(n_layers - 1):
        p = runner.PagedKV(kv.num_pages, kv.hq, kv.hkv, kv.d, kv.dtype_code, device,
                           fill_sentinel=False)
        p.k_cache.copy_(kv.k_cache)
        p.v_cache.copy_(kv.v_cache)
        p.err = kv.err
        extra.append((p, w))
    stream = torch.cuda.current_stream()
    res = {"layers": n_layers, "steps": len(plans), "bytes_per_layer_step": nbytes / len(plans)}
    for name, shared in (("plan_per_layer", False), ("shared_plan", True)):
        loop = runner.DecodeLoop(kv, w, plans, layers=extra, shared_plan=shared)
        loop.capture()
        for _ in range(2):
            loop.replay()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            loop.replay()
            b.record(stream)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b))
        ms = float(np.median(t))
        res[name] = {"us_per_layer_step": ms * 1e3 / (len(plans) * n_layers),
                     "GBps": nbytes * n_layers / (ms * 1e-3) / 1e9}
        del loop
    assert kv.read_error() == 0
    del extra, kv
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------ oracle arm
def oracle_decode_sample(n_req, min_seconds=0.0):
    """Time the fp64 oracle on the first n_req decode rows of the decode workload (all 32
    heads each), repeating the pass until at least ``min_seconds`` of CPU work."""
    import oracle
    w = W.decode_only()
    s = scheduler_for(w)
    s.history_plan()
    plan = s.next_step()
    sel = list(range(n_req))
    data = [(w.q(r)[:1], w.kv(r)) for r in sel]
    kv_tokens = int(sum(int(plan.context_lens[j]) + 1 for j in sel))
    nbytes = kv_tokens * w.num_kv_heads * w.head_dim * 2 * 2 + n_req * w.num_q_heads * \
        w.head_dim * 2 * 2
    passes, t0 = 0, time.time()
    while True:
        for j, r in enumerate(sel):
            c = int(plan.context_lens[j])
            k, v = data[j][1]
            oracle.attention_rows(w.dtype, data[j][0], np.array([c], np.int32), k[:c + 1],
                                  v[:c + 1], w.scale)
        passes += 1
        if time.time() - t0 >= min_seconds:
            break
    secs = time.time() - t0
    return secs, nbytes * passes, oracle.num_threads(), passes


# ------------------------------------------------------------------------------ dist glue
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def run_reference(args, dist_ctx):
    if dist_ctx.rank != 0:
        return
    n_req = 16  # a quarter of the 64 decode rows per step
    for _ in range(args.warmup):
        oracle_decode_sample(2)
    total_s, total_b, cores = 0.0, 0, 1
    for _ in range(args.steps):
        s, b, cores, _ = oracle_decode_sample(n_req)
        total_s += s
        total_b += b
    value = total_b / total_s / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "decode-only, 32q/8kv heads, d=128, bf16 inputs, ctx "
                                   "U[512,4096], 64 requests (oracle sample: 16 rows/step)",
                       "parallelism": "host cores (OpenMP)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "first 16 of 64 decode rows per step, all 32 heads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode-loop", action="store_true")
    ap.add_argument("--no-int8", action="store_true")
    ap.add_argument("--only", choices=["prefill", "decode-loop", "int8", "int8-prefill", "mixed"],
                    default=None,
                    help="time only the prefill workload (one-shot 8K and 4 x 2K) and print "
                         "its JSON object; used for focused profiler captures")
    ap.add_argument("--pool-pages", type=int, default=70000,
                    help="page-pool size (the step touches the same bytes at any size; a "
                         "smaller pool keeps profiler captures small)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    dist_ctx = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist_ctx)
            return
        from paged_kv_cache_token_gb300 import binding, build
        # one process per node compiles (ranks share the in-tree build); the rest wait
        if dist_ctx.local == 0:
            build.build()
        dist_ctx.barrier()
        binding.load()
        gc.disable()  # sections collect before their timed regions (settle)
        device = torch.device("cuda", dist_ctx.local if dist_ctx.world > 1 else 0)
        torch.cuda.set_device(device)
        hbm, bf16, bf16_sus, peak_src = peaks()
        if args.only == "prefill":
            if dist_ctx.rank == 0:
                pf = time_prefill(device)
                print(json.dumps({"prefill_chunk": pf, "peak_tflops": bf16}))
            return
        if args.only == "mixed":
            if dist_ctx.rank == 0:
                print(json.dumps({"mixed_step": time_mixed(device), "peak_tflops": bf16}))
            return
        if args.only == "int8":
            if dist_ctx.rank == 0:
                print(json.dumps({"int8_kv": time_decode_int8(device, args.steps,
                                                              args.pool_pages)}))
            return
        if args.only == "int8-prefill":
            if dist_ctx.rank == 0:
                print(json.dumps({"int8_prefill": time_prefill(device, kv_int8=True),
                                  "peak_tflops": bf16}))
            return
        if args.only == "decode-loop":
            if dist_ctx.rank == 0:
                print(json.dumps({"decode_loop": time_decode_loop(device),
                                  "layers_from_hbm": time_decode_loop_layers(device)}))
            return
        r = time_decode(device, args.steps, args.warmup, dist_ctx, args.pool_pages)
        acct = r["acct"]
        value = acct["step"] * dist_ctx.world / (r["ms_step"] * 1e-3) / 1e9
        # the decode kernel of this step also appends the new rows (pkv_append_attention)
        kernel_bytes = acct["attention"] + acct["append"]
        achieved = kernel_bytes / (r["ms_kernel"] * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist_ctx.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "decode-only step: 64 requests, cached ctx U[512,4096], 32 q /"
                                   " 8 kv heads, d_head 128, bf16, 16-token pages over a "
                                   "%d-page permuted pool (kv_append + paged_attention_step "
                                   "through pkv_append_attention)"
                                   % args.pool_pages,
                       "kv_bytes_per_step": acct["kv"], "step_bytes": acct["step"],
                       "l2": "steps alternate between two disjoint page pools: each step's "
                             "%.0f MB of K/V was last read two steps (1.2 GB of K/V) earlier, "
                             "vs 129 MB of L2" % (acct["kv"] / 1e6),
                       "l2_flush": True,
                       "parallelism": "independent replica per GPU" if dist_ctx.world > 1
                       else "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": peak_src + " hbm_gbs",
                         "kernel": "decode_kernel", "bytes_per_launch": kernel_bytes,
                         "ms_per_launch": r["ms_kernel"],
                         "traffic": captured_traffic("decode_kernel")},
            "e2e": {"value": acct["step"] * dist_ctx.world / (r["ms_e2e"] * 1e-3) / 1e9,
                    "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["ms_e2e"],
                    "copies": "inputs already packed in pinned host buffers (Q, new K/V and "
                              "the step's metadata); the decode kernels read them there and "
                              "write the output rows into pinned host memory over the CPU-GPU "
                              "link, one library call per step on one stream (runner."
                              "HostPipeline); two buffers alternate",
                    "copy_engine": {
                        "value": acct["step"] * dist_ctx.world / (r["ms_e2e_copy"] * 1e-3) / 1e9,
                        "unit": "GB/s", "ms_per_step": r["ms_e2e_copy"],
                        "note": "the same steps with one H2D copy of the packed inputs and one "
                                "D2H copy of the output per step on copy streams, ordered by "
                                "events (runner.StepPipeline)"},
                    "with_host_pack": {
                        "value": acct["step"] * dist_ctx.world / (r["ms_e2e_pack"] * 1e-3) / 1e9,
                        "unit": "GB/s", "ms_per_step": r["ms_e2e_pack"],
                        "host_pack_ms": r["host_pack_ms"],
                        "note": "the same loop with every step's inputs also packed from the "
                                "caller's numpy arrays into the pinned buffer inside the "
                                "timed region (host-bound when packing plus launch exceed the "
                                "GPU step)"}},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        if not args.no_prefill and dist_ctx.rank == 0:
            pf = time_prefill(device)
            one = pf["one_shot_8192"]
            ch = pf["chunks_4x2048"]
            kern_tflops = one["flops"] / one["main_kernel_ms"] / 1e9
            line["prefill_chunk"] = {
                "workload": "causal prefill S=8192, 32 q / 8 kv heads, d 128, bf16, pages; "
                            "one shot and 4 x 2048 chunks",
                "one_shot_tflops": one["tflops"], "chunked_tflops": ch["tflops"],
                "one_shot_ms": one["ms"], "chunked_ms": ch["ms"],
                "flops": one["flops"], "peak_tflops": bf16, "frac": one["tflops"] / bf16,
                "peak_source": peak_src + " bf16_tflops (burst)",
                "roofline": {"bound": "tensor", "kernel": "prefill_pair_kernel",
                             "achieved": kern_tflops, "peak": bf16, "unit": "TFLOP/s",
                             "frac": kern_tflops / bf16, "ms_per_launch": one["main_kernel_ms"],
                             "flops_per_launch": one["flops"],
                             "traffic": captured_traffic("prefill_pair_kernel"),
                             "chunked_kernel_tflops": ch["flops"] / ch["main_kernel_ms"] / 1e9}}
        if not args.no_decode_loop and dist_ctx.rank == 0:
            dl = time_decode_loop(device)
            line["decode_loop"] = {
                "workload": "64 consecutive decode steps, 16 requests, ctx log-uniform 32-2048, "
                            "32 q / 32 kv heads, d 128, fp16, pages handed out round-robin",
                "note": "one layer's cache (~%.0f MB) is re-read every step and stays largely "
                        "in L2, so GB/s here is not an HBM rate; the comparison is between "
                        "launch modes" % (dl["bytes_per_step"] / 1e6),
                **dl}
            ml = time_decode_loop_layers(device)
            line["decode_loop"]["layers_from_hbm"] = {
                "workload": "the same 64 steps over %d layers with separate page pools (%.0f MB "
                            "of cache in all, above L2), all layers' append + attention in one "
                            "CUDA graph" % (ml["layers"], ml["layers"] *
                                            ml["bytes_per_layer_step"] / 1e6),
                **ml, "frac_of_hbm": max(ml["plan_per_layer"]["GBps"],
                                         ml["shared_plan"]["GBps"]) / hbm}
        if not args.no_prefill and dist_ctx.rank == 0:
            mx = time_mixed(device)
            line["mixed_step"] = {
                "workload": "15 unified steps, token budget 2048: 30 decode requests (ctx "
                            "U[1k,8k]) + a 30,000-token prompt in 2,018-token chunks, 32/8 "
                            "heads, d 128, bf16 (append + attention per step)",
                **mx, "frac_of_bf16_peak": mx["tflops"] / bf16}
        if not args.no_int8 and dist_ctx.rank == 0:
            q8 = time_decode_int8(device, args.steps, args.pool_pages)
            line["int8_kv"] = {
                "workload": "the decode-only step over INT8 pages (per-channel K and V "
                            "scales; Q, new K/V and output bf16), one "
                            "pkv_append_attention_int8 call per step",
                **q8, "speedup_vs_bf16_step": r["ms_step"] / q8["ms_step"],
                "roofline": {"bound": "hbm", "kernel": "decode_kernel (INT8 pages)",
                             "achieved": q8["kernel_GBps"], "peak": hbm, "unit": "GB/s",
                             "frac": q8["kernel_GBps"] / hbm,
                             "peak_source": peak_src + " hbm_gbs",
                             "traffic": captured_traffic("decode_kernel_int8")}}
            if not args.no_prefill:
                pq = time_prefill(device, kv_int8=True)
                one, ch = pq["one_shot_8192"], pq["chunks_4x2048"]
                kt = one["flops"] / one["main_kernel_ms"] / 1e9
                line["int8_kv"]["prefill"] = {
                    "workload": "the 8192-token causal prefill over INT8 pages, one shot and "
                                "4 x 2048 chunks (prefill_q8_kernel)",
                    "one_shot_tflops": one["tflops"], "chunked_tflops": ch["tflops"],
                    "one_shot_ms": one["ms"], "kernel_ms": one["main_kernel_ms"],
                    "roofline": {"bound": "tensor", "kernel": "prefill_q8_kernel",
                                 "achieved": kt, "peak": bf16, "unit": "TFLOP/s",
                                 "frac": kt / bf16,
                                 "peak_source": peak_src + " bf16_tflops (burst; fp16 has "
                                                           "the same nominal dense rate)",
                                 "traffic": captured_traffic("prefill_q8_kernel")}}
        if not args.no_cpu_baseline and dist_ctx.rank == 0:
            secs, nbytes, cores, passes = oracle_decode_sample(64, min_seconds=10.0)
            line["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": cores,
                                    "kind": "oracle",
                                    "sample": "fp64 oracle on the whole decode step (64 rows x 32 "
                                              "heads), repeated %d times: %.1f s" % (passes, secs)}
        if dist_ctx.rank == 0:
            print(json.dumps(line))
    finally:
        dist_ctx.close()


if __name__ == "__main__":
    main()
