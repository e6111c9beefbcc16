"""Device-side driver for a sequence of steps: page pools, per-step metadata upload and
the two C-ABI calls (append, then attention), all through :mod:`binding`.

* :class:`PagedKV` -- the page pools (16-bit or INT8), the error flag and the workspace;
* :class:`StepStaging` -- a step's inputs packed into one pinned buffer, one copy each way;
* :class:`StepPipeline` -- two stagings alternating, copies on their own streams, so a
  step's transfers overlap its neighbours' computation;
* :class:`DecodeLoop` -- consecutive decode steps advanced on the device, one CUDA graph.

This is host plumbing around the library (allocation, copies, streams), the same thing a
serving engine does around its attention backend.  It holds no attention arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding
from .scheduler import StepPlan

SENTINEL = 0xFFFF  # NaN in both bf16 and fp16: slots never written stay recognisable
TORCH_DTYPE = {binding.BF16: torch.bfloat16, binding.FP16: torch.float16}


def bits_to_tensor(bits: np.ndarray, dtype_code: int, device="cuda", pin=False) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DTYPE[dtype_code])
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device, non_blocking=False)


def tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class DeviceStep:
    """Device copies of one step's metadata plus the matching StepDesc."""
    plan: StepPlan
    desc: binding.StepDesc
    tensors: tuple


INT8_SENTINEL = -128  # a code the quantiser never writes (it clamps to +-127)


class PagedKV:
    """Two page pools [num_pages, Hkv, 16, D] on one device plus an error flag.

    With ``k_scale``/``v_scale`` (float32 [Hkv, D], one fixed scale per KV head and channel)
    the pools hold INT8 codes and every call goes through the library's INT8 entry points;
    Q, the new K/V and the output keep the 16-bit dtype either way.
    """

    def __init__(self, num_pages: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 dtype_code: int, device="cuda", fill_sentinel: bool = True,
                 k_scale=None, v_scale=None):
        self.num_pages, self.hq, self.hkv, self.d = num_pages, num_q_heads, num_kv_heads, head_dim
        self.dtype_code = dtype_code
        self.dtype = TORCH_DTYPE[dtype_code]
        self.device = torch.device(device)
        self.kv_int8 = k_scale is not None
        shape = (num_pages, num_kv_heads, 16, head_dim)
        pool_dtype = torch.int8 if self.kv_int8 else self.dtype
        self.k_cache = torch.empty(shape, dtype=pool_dtype, device=self.device)
        # INT8 value pages are dim-major: [num_pages, Hkv, D, 16]
        vshape = (num_pages, num_kv_heads, head_dim, 16) if self.kv_int8 else shape
        self.v_cache = torch.empty(vshape, dtype=pool_dtype, device=self.device)
        if self.kv_int8:
            as_dev = lambda x: torch.as_tensor(np.asarray(x, np.float32)).reshape(
                num_kv_heads, head_dim).to(self.device).contiguous()
            self.k_scale, self.v_scale = as_dev(k_scale), as_dev(v_scale)
            if fill_sentinel:
                self.k_cache.fill_(INT8_SENTINEL)
                self.v_cache.fill_(INT8_SENTINEL)
        elif fill_sentinel:
            self.k_cache.view(torch.int16).fill_(-1)
            self.v_cache.view(torch.int16).fill_(-1)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._ws = None

    # ------------------------------------------------------------------ metadata
    def upload(self, plan: StepPlan, stream=None) -> DeviceStep:
        dev = self.device
        ql = torch.from_numpy(plan.q_lens).to(dev)
        qo = torch.from_numpy(plan.q_offsets).to(dev)
        cl = torch.from_numpy(plan.context_lens).to(dev)
        bt = torch.from_numpy(np.ascontiguousarray(plan.block_table)).to(dev)
        desc = binding.make_desc(num_reqs=plan.num_reqs, num_q_heads=self.hq,
                                 num_kv_heads=self.hkv, head_dim=self.d,
                                 num_pages=self.num_pages, max_pages_per_req=plan.max_pages,
                                 total_q_tokens=plan.total_q_tokens, max_q_len=plan.max_q_len,
                                 max_context_len=plan.max_context_len, dtype=self.dtype_code,
                                 q_lens=ql, q_offsets=qo, context_lens=cl, block_table=bt)
        return DeviceStep(plan, desc, (ql, qo, cl, bt))

    def workspace(self, desc) -> torch.Tensor:
        need = binding.attention_workspace_bytes_int8(desc) if self.kv_int8 else \
            binding.attention_workspace_bytes(desc)
        need = max(256, need)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    # ------------------------------------------------------------------ calls
    def append_desc(self, desc, k_new, v_new, slot_mapping=None, stream=None) -> None:
        """kv_append (16-bit or INT8 pools) for a StepDesc whose arrays are on the device."""
        if self.kv_int8:
            binding.kv_append_int8(desc, k_new, v_new, self.k_scale, self.v_scale,
                                   self.k_cache, self.v_cache, slot_mapping, self.err, stream)
        else:
            binding.kv_append(desc, k_new, v_new, self.k_cache, self.v_cache, slot_mapping,
                              self.err, stream)

    def attention_desc(self, desc, q, out, scale: float, ws, stream=None) -> None:
        """The attention step (16-bit or INT8 pools) into ``out``."""
        if self.kv_int8:
            binding.paged_attention_step_int8(desc, q, self.k_cache, self.v_cache, self.k_scale,
                                              self.v_scale, out, scale, ws, self.err, stream)
        else:
            binding.paged_attention_step(desc, q, self.k_cache, self.v_cache, out, scale, ws,
                                         self.err, stream)

    def append_attention_desc(self, desc, k_new, v_new, q, out, scale: float, ws,
                              slot_mapping=None, stream=None) -> None:
        """kv_append then the attention step in one call (fused into one decode grid for
        decode steps), for 16-bit and INT8 pools."""
        if self.kv_int8:
            binding.append_attention_int8(desc, k_new, v_new, self.k_scale, self.v_scale,
                                          self.k_cache, self.v_cache, q, out, scale, ws,
                                          slot_mapping, self.err, stream)
        else:
            binding.append_attention(desc, k_new, v_new, self.k_cache, self.v_cache, q, out,
                                     scale, ws, slot_mapping, self.err, stream)

    def run_desc(self, desc, q, out, scale: float, ws, stream=None) -> None:
        """The attention kernels over the plan already in ``ws`` (see
        binding.plan_attention): one more layer of a planned step."""
        if self.kv_int8:
            binding.paged_attention_run_int8(desc, q, self.k_cache, self.v_cache, self.k_scale,
                                             self.v_scale, out, scale, ws, self.err, stream)
        else:
            binding.paged_attention_run(desc, q, self.k_cache, self.v_cache, out, scale, ws,
                                        self.err, stream)

    def copy_pages(self, ds: DeviceStep, stream=None) -> None:
        """The step's copy-on-write page copies (plan.copies), before its kv_append."""
        c = ds.plan.copies
        if c is None or len(c) == 0:
            return
        cd = torch.from_numpy(np.ascontiguousarray(c.T)).to(self.device)
        binding.copy_pages(ds.desc, cd[0], cd[1], self.k_cache, self.v_cache, self.kv_int8,
                           self.err, stream)

    def append(self, ds: DeviceStep, k_new: torch.Tensor, v_new: torch.Tensor,
               slot_mapping: Optional[torch.Tensor] = None, stream=None) -> None:
        self.append_desc(ds.desc, k_new, v_new, slot_mapping, stream)

    def attention(self, ds: DeviceStep, q: torch.Tensor, scale: float,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((ds.plan.total_q_tokens, self.hq, self.d), dtype=self.dtype,
                              device=self.device)
        self.attention_desc(ds.desc, q, out, scale, self.workspace(ds.desc), stream)
        return out

    def read_error(self) -> int:
        return binding.read_device_error(self.err)


class StepStaging:
    """A step's inputs in one transfer each way.

    Q, K_new, V_new and the four metadata arrays are packed, 256-byte aligned, into one
    pinned host buffer; one asynchronous copy moves them into a device buffer whose views
    are what the library calls take, and one copy brings the output back.  Separate small
    copies would each pay the transfer latency; a decode step's inputs are under a
    megabyte.  Buffers grow on demand and are reused across steps; ``stage`` rewrites the
    pinned buffer, so call it only once the previous ``upload`` has completed (or keep two
    stagings and alternate).
    """

    ALIGN = 256

    def __init__(self, kv: PagedKV):
        self.kv = kv
        self._host = self._dev = None
        self._out_host = self._out_dev = None

    @staticmethod
    def _up(x: int) -> int:
        return (x + StepStaging.ALIGN - 1) // StepStaging.ALIGN * StepStaging.ALIGN

    def _layout(self, plan: StepPlan):
        kv, T, B = self.kv, plan.total_q_tokens, plan.num_reqs
        esz = torch.tensor([], dtype=kv.dtype).element_size()
        parts = [("q", T * kv.hq * kv.d * esz), ("k", T * kv.hkv * kv.d * esz),
                 ("v", T * kv.hkv * kv.d * esz), ("q_lens", B * 4), ("q_offsets", (B + 1) * 4),
                 ("context_lens", B * 4), ("block_table", B * plan.max_pages * 4)]
        offs, off = {}, 0
        for name, nbytes in parts:
            offs[name] = (off, nbytes)
            off = self._up(off + nbytes)
        return offs, off

    def _ensure(self, nbytes: int, out_bytes: int) -> None:
        if self._host is None or self._host.numel() < nbytes:
            self._host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            self._dev = torch.empty(nbytes, dtype=torch.uint8, device=self.kv.device)
        if self._out_host is None or self._out_host.numel() < out_bytes:
            self._out_host = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
            self._out_dev = torch.empty(out_bytes, dtype=torch.uint8, device=self.kv.device)

    def stage(self, plan: StepPlan, q_bits: np.ndarray, k_bits: np.ndarray,
              v_bits: np.ndarray) -> None:
        """Write a step's inputs (16-bit patterns and metadata) into the pinned buffer.  The
        layout, the device views and the step description depend only on the step's shape
        (tokens, requests, block-table width); while it repeats they are reused and staging
        is just the byte copies."""
        kv = self.kv
        key = (plan.total_q_tokens, plan.num_reqs, plan.max_pages, plan.max_q_len,
               plan.max_context_len)
        if getattr(self, "_key", None) != key:
            self._prepare(plan)
            self._key = key
        src = (q_bits, k_bits, v_bits, plan.q_lens, plan.q_offsets, plan.context_lens,
               plan.block_table)
        for dst, a in zip(self._host_views, src):
            np.copyto(dst, a.reshape(dst.shape), casting="no")
        self.plan = plan

    def _prepare(self, plan: StepPlan) -> None:
        kv = self.kv
        offs, total = self._layout(plan)
        out_bytes = self._up(plan.total_q_tokens * kv.hq * kv.d * 2)
        self._ensure(total, out_bytes)
        h = self._host.numpy()
        kinds = {"q": np.uint16, "k": np.uint16, "v": np.uint16, "q_lens": np.int32,
                 "q_offsets": np.int32, "context_lens": np.int32, "block_table": np.int32}
        self._host_views = [h[off:off + nbytes].view(kinds[name])
                            for name, (off, nbytes) in offs.items()]
        self.offs, self.total = offs, total
        T = plan.total_q_tokens
        d = self._dev
        view = lambda name, dt, shape: d[offs[name][0]:offs[name][0] + offs[name][1]].view(dt) \
            .view(shape)
        self.q = view("q", kv.dtype, (T, kv.hq, kv.d))
        self.k_new = view("k", kv.dtype, (T, kv.hkv, kv.d))
        self.v_new = view("v", kv.dtype, (T, kv.hkv, kv.d))
        meta = [view(n, torch.int32, (-1,)) for n in ("q_lens", "q_offsets", "context_lens")]
        bt = view("block_table", torch.int32, (plan.num_reqs, plan.max_pages))
        self.desc = binding.make_desc(
            num_reqs=plan.num_reqs, num_q_heads=kv.hq, num_kv_heads=kv.hkv, head_dim=kv.d,
            num_pages=kv.num_pages, max_pages_per_req=plan.max_pages,
            total_q_tokens=T, max_q_len=plan.max_q_len, max_context_len=plan.max_context_len,
            dtype=kv.dtype_code, q_lens=meta[0], q_offsets=meta[1], context_lens=meta[2],
            block_table=bt)
        self.out = self._out_dev[:T * kv.hq * kv.d * 2].view(kv.dtype).view(T, kv.hq, kv.d)
        self.out_host = self._out_host[:T * kv.hq * kv.d * 2].view(kv.dtype) \
            .view(T, kv.hq, kv.d)
        self._ws = kv.workspace(self.desc)

    @property
    def h2d_bytes(self) -> int:
        return self.total

    @property
    def d2h_bytes(self) -> int:
        return self.out.numel() * self.out.element_size()

    def upload(self) -> None:
        """Host -> device copy of the staged inputs on the current stream."""
        self._dev[:self.total].copy_(self._host[:self.total], non_blocking=True)

    def run(self, scale: float, stream=None) -> None:
        """kv_append then the attention step (one call), on the staged device views."""
        self.kv.append_attention_desc(self.desc, self.k_new, self.v_new, self.q, self.out,
                                      scale, self._ws, None, stream)

    def download(self) -> None:
        """Device -> host copy of the step's output on the current stream."""
        self.out_host.copy_(self.out, non_blocking=True)


class HostStaging(StepStaging):
    """A decode step's inputs and output kept in pinned host memory and used in place.

    Pinned host memory is mapped into the device's address space at the same address, and
    the decode kernels read Q, the new K/V and the step's four metadata arrays from it and
    write the output rows into it: plain loads and stores over the CPU-GPU link (NVLink-C2C
    on GB300).  One library call per step then moves the step's bytes both ways, with no
    copy-engine transfer and no cross-stream event wait between the step's kernels and
    its neighbours' (such a wait ends their programmatic overlap).  Decode steps only: with
    max_q_len >= 16 the library reads Q with tensor-memory-accelerator copies and refuses
    host memory.  ``upload`` and ``download`` do nothing; ``stage`` rewrites the buffer, so
    call it only once the GPU is done with the previous step that used it.
    """

    def _ensure(self, nbytes: int, out_bytes: int) -> None:
        if self._host is None or self._host.numel() < nbytes:
            self._host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            self._dev = self._host
        if self._out_host is None or self._out_host.numel() < out_bytes:
            self._out_host = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
            self._out_dev = self._out_host

    def upload(self) -> None:
        pass

    def download(self) -> None:
        pass


class HostPipeline:
    """Consecutive decode steps on one stream through two HostStaging buffers.

    Step i uses buffer i % 2 (and, with ``kv_alt``, the second set of pools on odd steps).
    ``launch`` is the one library call of the step plus an event; ``stage`` waits for the
    event of the step that last used the buffer before rewriting it; ``result`` waits for
    the step's event and returns the pinned output, valid until the buffer's next launch.
    """

    def __init__(self, kv: PagedKV, stream=None, kv_alt: Optional[PagedKV] = None):
        self.stg = [HostStaging(kv), HostStaging(kv_alt if kv_alt is not None else kv)]
        self.stream = stream or torch.cuda.current_stream(kv.device)
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]

    def stage(self, slot: int, plan: StepPlan, q_bits: np.ndarray, k_bits: np.ndarray,
              v_bits: np.ndarray) -> None:
        if plan.max_q_len >= 16:
            raise ValueError("HostPipeline runs decode steps (max_q_len < 16)")
        if self.used[slot]:
            self.done[slot].synchronize()
        self.stg[slot].stage(plan, q_bits, k_bits, v_bits)

    def launch(self, slot: int, scale: float) -> None:
        self.stg[slot].run(scale, self.stream)
        self.done[slot].record(self.stream)
        self.used[slot] = True

    def result(self, slot: int) -> torch.Tensor:
        self.done[slot].synchronize()
        return self.stg[slot].out_host


class StepPipeline:
    """Consecutive steps through two stagings, with the copies on their own streams.

    Step i uses staging i % 2.  Its upload (on the H2D stream) waits only for the last
    step that read that staging's device inputs, so it runs while the previous step
    computes; its append + attention (on the compute stream) wait for its upload and for
    the staging's previous download; its download (on the D2H stream) waits for its own
    computation and overlaps the next step's.  Every step still moves its whole input up
    and its whole output down.

    ``stage(slot, ...)`` fills a staging's pinned input buffer (waiting first for that
    staging's previous upload), ``launch(slot, scale)`` enqueues the step and ``result(slot)``
    waits for its download and returns the pinned host output, valid until the slot's next
    ``launch``.
    """

    def __init__(self, kv: PagedKV, compute_stream=None, kv_alt: Optional[PagedKV] = None):
        """``kv_alt``: a second set of pools for the odd steps (e.g. another layer's cache);
        by default both stagings use ``kv``."""
        self.kv = kv
        self.stg = [StepStaging(kv), StepStaging(kv_alt if kv_alt is not None else kv)]
        self.compute = compute_stream or torch.cuda.current_stream(kv.device)
        self.h2d = torch.cuda.Stream(device=kv.device)
        self.d2h = torch.cuda.Stream(device=kv.device)
        self.uploaded = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.downloaded = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]

    def stage(self, slot: int, plan: StepPlan, q_bits: np.ndarray, k_bits: np.ndarray,
              v_bits: np.ndarray) -> None:
        if self.used[slot]:
            self.uploaded[slot].synchronize()
        self.stg[slot].stage(plan, q_bits, k_bits, v_bits)

    def start_after(self, event: torch.cuda.Event) -> None:
        """Order the copy streams after ``event`` (e.g. the start of a timed region)."""
        self.h2d.wait_event(event)
        self.d2h.wait_event(event)

    def launch(self, slot: int, scale: float) -> None:
        s = self.stg[slot]
        with torch.cuda.stream(self.h2d):
            if self.used[slot]:
                self.h2d.wait_event(self.computed[slot])
            s.upload()
            self.uploaded[slot].record(self.h2d)
        self.compute.wait_event(self.uploaded[slot])
        if self.used[slot]:
            self.compute.wait_event(self.downloaded[slot])
        s.run(scale, self.compute)
        self.computed[slot].record(self.compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.computed[slot])
            s.download()
            self.downloaded[slot].record(self.d2h)
        self.used[slot] = True

    def join(self) -> None:
        """Make the compute stream wait for every download launched so far."""
        for slot in range(2):
            if self.used[slot]:
                self.compute.wait_event(self.downloaded[slot])

    def result(self, slot: int) -> torch.Tensor:
        self.downloaded[slot].synchronize()
        return self.stg[slot].out_host


class DecodeLoop:
    """Consecutive steps of one batch run as one device-side sequence.

    Every step is kv_append with the attention step (pkv_append_attention: one fused grid
    for decode steps) and pkv_advance_context (context_lens += q_lens), so no metadata
    crosses from the host between steps; the block table is the
    last step's, which already holds every page the earlier steps reach.  Each step's Q,
    K_new, V_new are staged on the device up front and each step's output has its own slot.
    ``capture`` records the whole sequence in one CUDA graph (the lengths are reset at its
    start, so it can be replayed); ``replay`` then runs all steps with one launch.

    ``layers``: more layers of the same model step, each a ``(PagedKV, workload)`` with its
    own pools and its own values for the same requests and pages; every step runs each
    layer's append + attention in turn.  With ``shared_plan`` a step plans once
    (pkv_plan_attention) and every layer runs over that plan (pkv_paged_attention_run)
    instead of planning again.  ``outs[l]`` holds layer l's outputs, ``out`` layer 0's.
    """

    def __init__(self, kv: PagedKV, workload, plans, layers=(), shared_plan: bool = False):
        if not plans:
            raise ValueError("no steps")
        p0, pl = plans[0], plans[-1]
        for i, p in enumerate(plans):
            if (list(p.rids) != list(p0.rids) or not np.array_equal(p.q_lens, p0.q_lens)
                    or not np.array_equal(p.context_lens, p0.context_lens + i * p0.q_lens)):
                raise ValueError("plans are not consecutive steps of one batch")
            for r in range(p.num_reqs):
                n = -(-(int(p.context_lens[r]) + int(p.q_lens[r])) // 16)
                if not np.array_equal(p.block_table[r, :n], pl.block_table[r, :n]):
                    raise ValueError("block tables of the steps disagree")
        self.kv, self.scale, self.steps = kv, workload.scale, len(plans)
        self.shared_plan = shared_plan
        self.layers = [(kv, workload)] + list(layers)
        dev = kv.device
        T = p0.total_q_tokens
        self.io = []
        for lkv, lw in self.layers:
            if (lkv.hq, lkv.hkv, lkv.d, lkv.num_pages) != (kv.hq, kv.hkv, kv.d, kv.num_pages):
                raise ValueError("layers must share the pool geometry")
            ins = [step_host_inputs(lw, p) for p in plans]
            stack = lambda i: bits_to_tensor(np.stack([x[i] for x in ins]), lw.dtype, dev)
            out = torch.empty((self.steps, T, kv.hq, kv.d), dtype=kv.dtype, device=dev)
            self.io.append((stack(0), stack(1), stack(2), out))
        self.q, self.k_new, self.v_new, self.out = self.io[0]
        self.outs = [x[3] for x in self.io]
        self.q_lens = torch.from_numpy(p0.q_lens).to(dev)
        self.q_offsets = torch.from_numpy(p0.q_offsets).to(dev)
        self.ctx0 = torch.from_numpy(p0.context_lens).to(dev)
        self.ctx = self.ctx0.clone()
        self.block_table = torch.from_numpy(np.ascontiguousarray(pl.block_table)).to(dev)
        self.desc = binding.make_desc(
            num_reqs=p0.num_reqs, num_q_heads=kv.hq, num_kv_heads=kv.hkv, head_dim=kv.d,
            num_pages=kv.num_pages, max_pages_per_req=pl.max_pages, total_q_tokens=T,
            max_q_len=p0.max_q_len, max_context_len=pl.max_context_len, dtype=kv.dtype_code,
            q_lens=self.q_lens, q_offsets=self.q_offsets, context_lens=self.ctx,
            block_table=self.block_table)
        self.ws = kv.workspace(self.desc)
        self.graph = None

    def _body(self, stream=None) -> None:
        self.ctx.copy_(self.ctx0, non_blocking=True)
        for s in range(self.steps):
            if self.shared_plan:
                binding.plan_attention(self.desc, self.ws, self.kv.err, stream)
            for (lkv, _), (q, k_new, v_new, out) in zip(self.layers, self.io):
                if self.shared_plan:
                    lkv.append_desc(self.desc, k_new[s], v_new[s], None, stream)
                    lkv.run_desc(self.desc, q[s], out[s], self.scale, self.ws, stream)
                else:
                    lkv.append_attention_desc(self.desc, k_new[s], v_new[s], q[s], out[s],
                                              self.scale, self.ws, None, stream)
            binding.advance_context(self.desc, self.ctx, stream)

    def run(self) -> torch.Tensor:
        """All steps, launched one call at a time on the current stream."""
        self._body()
        return self.out

    def capture(self) -> None:
        """Record all steps in one CUDA graph (after one eager run, which sets up the
        library's per-kernel attributes outside the capture)."""
        self.run()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()
        torch.cuda.synchronize()

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out


# ---------------------------------------------------------------------- workload glue
def step_host_inputs(workload, plan: StepPlan):
    """(q, k_new, v_new) bit arrays for a step, gathered from the workload's sequences."""
    qs, ks, vs = [], [], []
    for rid, c, n in zip(plan.rids, plan.context_lens.tolist(), plan.q_lens.tolist()):
        req = workload.requests[rid]
        k, v = workload.kv(rid)
        ks.append(k[c:c + n])
        vs.append(v[c:c + n])
        if c >= req.history:
            qs.append(workload.q(rid)[c - req.history:c - req.history + n])
        else:  # loading cached history: no queries
            qs.append(np.zeros((n, workload.num_q_heads, workload.head_dim), np.uint16))
    cat = lambda xs, h: (np.concatenate(xs) if xs else
                         np.zeros((0, h, workload.head_dim), np.uint16))
    return cat(qs, workload.num_q_heads), cat(ks, workload.num_kv_heads), \
        cat(vs, workload.num_kv_heads)


def paged_kv_for(workload, device="cuda", fill_sentinel=True, kv_int8=False) -> PagedKV:
    """Pools for a workload; with ``kv_int8`` INT8 pools with the workload's seeded
    per-channel scales."""
    ks, vs = workload.int8_scales() if kv_int8 else (None, None)
    return PagedKV(workload.num_pages, workload.num_q_heads, workload.num_kv_heads,
                   workload.head_dim, workload.dtype, device, fill_sentinel, ks, vs)


def load_history(kv: PagedKV, workload, plan: Optional[StepPlan]) -> None:
    """Append every request's cached history (no attention)."""
    if plan is None:
        return
    _, k, v = step_host_inputs(workload, plan)
    ds = kv.upload(plan)
    kv.append(ds, bits_to_tensor(k, workload.dtype), bits_to_tensor(v, workload.dtype))


def run_step_fused(kv: PagedKV, workload, plan: StepPlan, slot_mapping=None) -> torch.Tensor:
    """As :func:`run_step`, through the one-call pkv_append_attention."""
    q, k, v = step_host_inputs(workload, plan)
    ds = kv.upload(plan)
    kv.copy_pages(ds)
    out = torch.empty((plan.total_q_tokens, kv.hq, kv.d), dtype=kv.dtype, device=kv.device)
    kv.append_attention_desc(ds.desc, bits_to_tensor(k, workload.dtype),
                             bits_to_tensor(v, workload.dtype), bits_to_tensor(q, workload.dtype),
                             out, workload.scale, kv.workspace(ds.desc), slot_mapping)
    return out


def run_step(kv: PagedKV, workload, plan: StepPlan) -> torch.Tensor:
    q, k, v = step_host_inputs(workload, plan)
    ds = kv.upload(plan)
    kv.copy_pages(ds)
    kv.append(ds, bits_to_tensor(k, workload.dtype), bits_to_tensor(v, workload.dtype))
    return kv.attention(ds, bits_to_tensor(q, workload.dtype), workload.scale)
