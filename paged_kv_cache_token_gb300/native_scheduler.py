"""Python face of the native step planner and page allocator (include/pkv_sched.h).

Same interface as :class:`scheduler.Scheduler` (``history_plan``, ``next_step``,
``all_steps``) and the same plans; the planning runs in the library's C++ code.  Adds
``release`` (return a finished request's pages to the free list), ``num_free`` and prefix
caching: ``add_prompt`` takes a request's prompt token ids and reuses the pages of
matching full 16-token prompt blocks other requests computed before.
Host code only: usable without a GPU.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional

import numpy as np

from . import binding
from .scheduler import StepPlan

_I32P = ctypes.POINTER(ctypes.c_int32)


class _Plan(ctypes.Structure):
    """Mirror of ``pkv_plan``."""
    _fields_ = [("max_reqs", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("rids", _I32P), ("q_lens", _I32P), ("context_lens", _I32P),
                ("q_offsets", _I32P), ("block_table", _I32P),
                ("num_reqs", ctypes.c_int32), ("total_q_tokens", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("pages_used", ctypes.c_int32), ("max_copies", ctypes.c_int32),
                ("copy_src", _I32P), ("copy_dst", _I32P), ("num_copies", ctypes.c_int32)]


def _lib():
    lib = binding.load()
    if not getattr(lib, "_pkv_sched_ready", False):
        V = ctypes.c_void_p
        lib.pkv_sched_create.argtypes = [ctypes.c_int32, V, ctypes.c_int32, ctypes.c_int32]
        lib.pkv_sched_create.restype = V
        lib.pkv_sched_destroy.argtypes = [V]
        lib.pkv_sched_destroy.restype = None
        lib.pkv_sched_add_request.argtypes = [V] + [ctypes.c_int32] * 4
        lib.pkv_sched_add_request.restype = ctypes.c_int
        lib.pkv_sched_history_plan.argtypes = [V, ctypes.c_int, ctypes.POINTER(_Plan)]
        lib.pkv_sched_history_plan.restype = ctypes.c_int
        lib.pkv_sched_next_step.argtypes = [V, ctypes.POINTER(_Plan)]
        lib.pkv_sched_next_step.restype = ctypes.c_int
        lib.pkv_sched_release.argtypes = [V, ctypes.c_int32]
        lib.pkv_sched_release.restype = ctypes.c_int
        lib.pkv_sched_free_pages.argtypes = [V]
        lib.pkv_sched_free_pages.restype = ctypes.c_int32
        lib.pkv_sched_add_prompt.argtypes = [V, ctypes.c_int32, V, ctypes.c_int32,
                                             ctypes.c_int32]
        lib.pkv_sched_add_prompt.restype = ctypes.c_int
        lib.pkv_sched_fork.argtypes = [V, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        lib.pkv_sched_fork.restype = ctypes.c_int
        lib.pkv_sched_sort_by_length.argtypes = [V]
        lib.pkv_sched_sort_by_length.restype = ctypes.c_int
        for fn in (lib.pkv_sched_cached_blocks, lib.pkv_sched_evictable_blocks):
            fn.argtypes = [V]
            fn.restype = ctypes.c_int32
        lib._pkv_sched_ready = True
    return lib


class NativeScheduler:
    """Token-budget planner over requests sharing one page pool (C++ implementation)."""

    def __init__(self, requests, page_order, budget: int, chunk_cap: Optional[int] = None,
                 interleave_history: bool = False):
        self._lib = _lib()
        order = np.ascontiguousarray(np.asarray(page_order, dtype=np.int32))
        self._h = self._lib.pkv_sched_create(len(order), order.ctypes.data_as(ctypes.c_void_p),
                                             int(budget), int(chunk_cap or 0))
        if not self._h:
            raise ValueError("bad scheduler arguments")
        self._interleave = interleave_history
        self._total = {}
        self.max_reqs = 0
        self.max_pages = 1
        for r in requests:
            self.add_request(r.rid, r.history, r.prompt, r.decodes)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pkv_sched_destroy(h)

    def add_request(self, rid: int, history: int, prompt: int, decodes: int) -> None:
        rc = self._lib.pkv_sched_add_request(self._h, rid, history, prompt, decodes)
        if rc != binding.OK:
            raise binding.PkvError("pkv_sched_add_request", rc)
        self.max_reqs += 1
        self._total[rid] = history + prompt + decodes
        self.max_pages = max(self.max_pages, -(-self._total[rid] // 16))

    def add_prompt(self, rid: int, tokens, decodes: int) -> int:
        """Add a request with known prompt token ids (prefix caching); returns the number
        of prompt tokens reused from the cache."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        rc = self._lib.pkv_sched_add_prompt(self._h, rid, t.ctypes.data_as(ctypes.c_void_p),
                                            len(t), decodes)
        if rc < 0:
            raise binding.PkvError("pkv_sched_add_prompt", rc)
        self.max_reqs += 1
        self._total[rid] = len(t) + decodes
        self.max_pages = max(self.max_pages, -(-self._total[rid] // 16))
        return rc

    def fork(self, parent_rid: int, rid: int, decodes: int) -> None:
        """Add request ``rid`` continuing from everything ``parent_rid`` has cached, with
        ``decodes`` generated tokens of its own; pages are shared and copied on write."""
        rc = self._lib.pkv_sched_fork(self._h, parent_rid, rid, decodes)
        if rc != binding.OK:
            raise binding.PkvError("pkv_sched_fork", rc)
        self.max_reqs += 1
        # the child holds at most the parent's whole sequence plus its own tokens
        self._total[rid] = self._total[parent_rid] + decodes
        self.max_pages = max(self.max_pages, -(-self._total[rid] // 16))

    def sort_by_length(self) -> None:
        """Order the requests whose prompt has not started by the prompt tokens still to
        compute, shortest first, after the started ones (lshu.cn/news/11576 §2.2)."""
        rc = self._lib.pkv_sched_sort_by_length(self._h)
        if rc != binding.OK:
            raise binding.PkvError("pkv_sched_sort_by_length", rc)

    @property
    def cached_blocks(self) -> int:
        return int(self._lib.pkv_sched_cached_blocks(self._h))

    @property
    def evictable_blocks(self) -> int:
        return int(self._lib.pkv_sched_evictable_blocks(self._h))

    def _call(self, fn, *args) -> Optional[StepPlan]:
        R, P = max(1, self.max_reqs), self.max_pages
        arr = {n: np.zeros(R + (n == "q_offsets"), np.int32)
               for n in ("rids", "q_lens", "context_lens", "q_offsets")}
        bt = np.zeros(R * P, np.int32)
        C = R  # at most one page copy per request and step
        cp = np.zeros((2, C), np.int32)
        ptr = lambda a: a.ctypes.data_as(_I32P)
        plan = _Plan(R, P, ptr(arr["rids"]), ptr(arr["q_lens"]), ptr(arr["context_lens"]),
                     ptr(arr["q_offsets"]), ptr(bt), 0, 0, 0, 0, 0, C, ptr(cp[0]), ptr(cp[1]),
                     0)
        rc = fn(self._h, *args, ctypes.byref(plan))
        if rc < 0:
            raise binding.PkvError(fn.__name__, rc)
        if rc == 0:
            return None
        n, w = plan.num_reqs, max(1, plan.pages_used)
        copies = np.ascontiguousarray(cp[:, :plan.num_copies].T) if plan.num_copies else None
        return StepPlan([int(x) for x in arr["rids"][:n]], arr["q_lens"][:n].copy(),
                        arr["context_lens"][:n].copy(), arr["q_offsets"][:n + 1].copy(),
                        np.ascontiguousarray(bt.reshape(R, P)[:n, :w]), copies)

    def history_plan(self) -> Optional[StepPlan]:
        return self._call(self._lib.pkv_sched_history_plan, 1 if self._interleave else 0)

    def next_step(self) -> Optional[StepPlan]:
        return self._call(self._lib.pkv_sched_next_step)

    def all_steps(self) -> List[StepPlan]:
        out = []
        while True:
            p = self.next_step()
            if p is None:
                return out
            out.append(p)

    def release(self, rid: int) -> None:
        rc = self._lib.pkv_sched_release(self._h, rid)
        if rc != binding.OK:
            raise binding.PkvError("pkv_sched_release", rc)

    @property
    def num_free(self) -> int:
        return int(self._lib.pkv_sched_free_pages(self._h))


def native_scheduler_for(workload) -> NativeScheduler:
    return NativeScheduler(workload.requests, workload.page_order, workload.budget,
                           workload.chunk_cap, workload.interleave_history)
