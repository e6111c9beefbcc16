"""Host-side step planner for a unified prefill/decode scheduler with a paged KV pool.

Follows niuwancheng.cn "11. chunked prefill and unified scheduling", section "token
budget per step": every request records how many of its tokens are already computed
(cached) and how many it needs in total; each step gives a decoding request 1 token and a
prefilling request min(remaining input, remaining budget); the step's total never exceeds
the budget; decodes are scheduled first and the prefill takes what is left.  Pages hold 16
tokens (lshu.cn/news/11576 §2.3) and are taken from a free list as a request's cached
length crosses a page boundary (§2.2: K/V written by page index).

The planner produces exactly the per-request arrays the C ABI consumes:
``q_lens``, ``context_lens`` (tokens cached before the step), ``q_offsets`` (exclusive
prefix sum of q_lens) and ``block_table`` (physical page ids, -1 past the end).
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass
from typing import Iterable, List, Optional, Sequence

import numpy as np

PAGE = 16


def pages_for(tokens: int) -> int:
    return (tokens + PAGE - 1) // PAGE


class OutOfPages(RuntimeError):
    pass


class PagePool:
    """Free list of physical page ids, handed out in the given order (FIFO)."""

    def __init__(self, order: Iterable[int]):
        self._free = deque(int(p) for p in order)
        self.capacity = len(self._free)

    def allocate(self) -> int:
        if not self._free:
            raise OutOfPages("page pool exhausted")
        return self._free.popleft()

    def free(self, pages: Sequence[int]) -> None:
        self._free.extend(int(p) for p in pages)

    @property
    def num_free(self) -> int:
        return len(self._free)


@dataclass
class ReqState:
    rid: int
    prompt_end: int      # history + prompt: positions below this are input, not generated
    total: int           # every position this request will ever hold
    computed: int        # tokens already in the KV cache
    pages: List[int]
    begun: bool = False  # a step has computed some of its prompt

    @property
    def decoding(self) -> bool:
        return self.computed >= self.prompt_end and self.computed < self.total

    @property
    def prefilling(self) -> bool:
        return self.computed < self.prompt_end

    @property
    def done(self) -> bool:
        return self.computed >= self.total


@dataclass
class StepPlan:
    """One step: request ids in launch order plus the C-ABI arrays."""
    rids: List[int]
    q_lens: np.ndarray         # int32 [B]
    context_lens: np.ndarray   # int32 [B]
    q_offsets: np.ndarray      # int32 [B+1]
    block_table: np.ndarray    # int32 [B, max_pages]
    # page copies to run before the step's kv_append (copy-on-write of shared pages):
    # int32 [n, 2] rows (source page, destination page), or None
    copies: Optional[np.ndarray] = None

    @property
    def num_reqs(self) -> int:
        return len(self.rids)

    @property
    def total_q_tokens(self) -> int:
        return int(self.q_offsets[-1])

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if len(self.rids) else 0

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if len(self.rids) else 0

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def make_plan(rids: List[int], q_lens: Sequence[int], ctx: Sequence[int],
              tables: Sequence[Sequence[int]], max_pages: Optional[int] = None) -> StepPlan:
    q = np.asarray(q_lens, dtype=np.int32)
    c = np.asarray(ctx, dtype=np.int32)
    offs = np.zeros(len(rids) + 1, dtype=np.int32)
    np.cumsum(q, out=offs[1:])
    width = max_pages if max_pages is not None else max([len(t) for t in tables] + [1])
    bt = np.full((len(rids), width), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    return StepPlan(list(rids), q, c, offs, bt)


class Scheduler:
    """Token-budget planner over a set of requests sharing one page pool."""

    def __init__(self, requests, pool: PagePool, budget: int, chunk_cap: Optional[int] = None,
                 interleave_history: bool = False):
        """``requests``: objects with ``rid``, ``history``, ``prompt``, ``decodes``."""
        if budget <= 0:
            raise ValueError("token budget must be positive")
        self.pool = pool
        self.budget = budget
        self.chunk_cap = chunk_cap
        self.reqs = [ReqState(r.rid, r.history + r.prompt, r.history + r.prompt + r.decodes, 0,
                              []) for r in requests]
        self._history = [r.history for r in requests]
        self._interleave = interleave_history

    def add_request(self, r) -> None:
        """Append a request (``rid``, ``history``, ``prompt``, ``decodes``) to the batch."""
        self.reqs.append(ReqState(r.rid, r.history + r.prompt, r.history + r.prompt + r.decodes,
                                  0, []))
        self._history.append(r.history)

    def sort_by_length(self) -> None:
        """Order the requests whose prompt has not started by the prompt tokens still to
        compute, shortest first (ties keep arrival order), after every request that has
        started.  lshu.cn/news/11576 §2.2: sorting a batch by prompt length before prefill
        keeps requests of similar length adjacent, so their pages are allocated together
        instead of short requests' pages landing in the gaps between long ones."""
        started = [i for i, st in enumerate(self.reqs) if st.begun]
        waiting = [i for i, st in enumerate(self.reqs) if not st.begun]
        waiting.sort(key=lambda i: self.reqs[i].prompt_end - self.reqs[i].computed)
        order = started + waiting
        self.reqs = [self.reqs[i] for i in order]
        self._history = [self._history[i] for i in order]

    def _grow(self, st: ReqState, upto_tokens: int) -> None:
        while len(st.pages) < pages_for(upto_tokens):
            st.pages.append(self.pool.allocate())

    def history_plan(self) -> Optional[StepPlan]:
        """The append that loads every request's cached history (q_len = history,
        context_len = 0).  Pages are taken per request, or round-robin one page at a time
        across requests when ``interleave_history`` is set.  Marks the history computed."""
        idx = [i for i, h in enumerate(self._history) if h > 0 and self.reqs[i].computed == 0]
        if not idx:
            return None
        if self._interleave:
            need = {i: pages_for(self._history[i]) for i in idx}
            while any(len(self.reqs[i].pages) < need[i] for i in idx):
                for i in idx:
                    if len(self.reqs[i].pages) < need[i]:
                        self.reqs[i].pages.append(self.pool.allocate())
        else:
            for i in idx:
                self._grow(self.reqs[i], self._history[i])
        plan = make_plan([self.reqs[i].rid for i in idx], [self._history[i] for i in idx],
                         [0] * len(idx), [list(self.reqs[i].pages) for i in idx])
        for i in idx:
            self.reqs[i].computed = self._history[i]
        return plan

    def next_step(self) -> Optional[StepPlan]:
        """Plan the next step (decode-first, then prefill chunks within the budget) and
        advance the request states as if it ran.  None when every request is done."""
        left = self.budget
        chosen = []
        for st in self.reqs:                       # decodes first, one token each
            if st.decoding and left > 0:
                chosen.append((st, 1))
                left -= 1
        for st in self.reqs:                       # then prefills take what is left
            if st.prefilling and left > 0:
                n = min(st.prompt_end - st.computed, left)
                if self.chunk_cap is not None:
                    n = min(n, self.chunk_cap)
                chosen.append((st, n))
                left -= n
        if not chosen:
            return None
        for st, n in chosen:
            self._grow(st, st.computed + n)
        plan = make_plan([st.rid for st, _ in chosen], [n for _, n in chosen],
                         [st.computed for st, _ in chosen], [list(st.pages) for st, _ in chosen])
        for st, n in chosen:
            st.computed += n
            st.begun = True
        return plan

    def all_steps(self) -> List[StepPlan]:
        out = []
        while True:
            p = self.next_step()
            if p is None:
                return out
            out.append(p)


def scheduler_for(workload) -> Scheduler:
    return Scheduler(workload.requests, PagePool(workload.page_order), workload.budget,
                     workload.chunk_cap, workload.interleave_history)
