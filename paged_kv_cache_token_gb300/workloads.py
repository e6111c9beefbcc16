"""Seeded synthetic inputs for the paged-KV attention step.

This module holds no attention arithmetic: it only draws random tensors and lays out
request lengths and page orders.  Both the CUDA path (through the binding) and the fp64
oracle consume what it produces; neither is imported here.

Recipe (all values exact, all draws reproducible):

* Every request ``r`` of workload ``w`` owns three independent ``torch.Generator``
  streams seeded ``(1000 + w) * 2**20 + 4 * r + kind`` (kind 0 = Q, 1 = K, 2 = V; kind 3 of
  requests 0 and 1 draws an INT8 cache's K and V per-channel scales).
  Values are fp32 N(0, 1) draws rounded to bf16 / fp16 with round-to-nearest-even
  (torch's ``.to(dtype)``), kept as their 16-bit patterns.
* K and V exist for every position the request will ever hold (cached history plus the
  tokens the schedule will process); Q exists only for processed tokens (the cached
  history was never a query in this step sequence).  Decode tokens are fresh draws: there
  is no model, so a "generated" token's Q/K/V are random like the prompt's.
* Page orders (the free list the allocator pops from) follow the five workloads'
  descriptions: a seeded shuffle, a seeded permutation of a large pool, or a sequential
  pool handed out round-robin one page at a time across requests (fragmented,
  interleaved block tables).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

PAGE = 16
BF16, FP16 = 0, 1
_TORCH_DTYPE = {BF16: torch.bfloat16, FP16: torch.float16}


def _seed(workload: int, req: int, kind: int) -> int:
    return (1000 + workload) * (1 << 20) + 4 * req + kind


def draw_bits(seed: int, shape, dtype: int) -> np.ndarray:
    """fp32 N(0,1) draws rounded RNE to bf16/fp16, returned as uint16 bit patterns."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32).to(_TORCH_DTYPE[dtype])
    return x.view(torch.int16).numpy().view(np.uint16)


@dataclass
class RequestSpec:
    """One request of a workload: ``history`` tokens already cached before the first
    scheduled step, ``prompt`` tokens to prefill, then ``decodes`` single-token steps."""
    rid: int
    history: int
    prompt: int
    decodes: int

    @property
    def total(self) -> int:
        return self.history + self.prompt + self.decodes

    @property
    def processed(self) -> int:
        return self.prompt + self.decodes


@dataclass
class Workload:
    index: int
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: int
    requests: List[RequestSpec]
    page_order: np.ndarray          # free-list order of physical page ids
    num_pages: int
    budget: int = 1 << 30            # token budget per step
    chunk_cap: Optional[int] = None  # per-request cap on a prefill chunk
    interleave_history: bool = False  # hand out history pages round-robin one page at a time
    notes: str = ""
    _cache: dict = field(default_factory=dict, repr=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def kv(self, rid: int):
        """(K, V) bit patterns [total, Hkv, D] of request rid (whole sequence)."""
        key = ("kv", rid)
        if key not in self._cache:
            req = self.requests[rid]
            shape = (req.total, self.num_kv_heads, self.head_dim)
            self._cache[key] = (draw_bits(_seed(self.index, rid, 1), shape, self.dtype),
                                draw_bits(_seed(self.index, rid, 2), shape, self.dtype))
        return self._cache[key]

    def q(self, rid: int) -> np.ndarray:
        """Q bit patterns [processed, Hq, D]; row i is the token at position history + i."""
        key = ("q", rid)
        if key not in self._cache:
            req = self.requests[rid]
            shape = (req.processed, self.num_q_heads, self.head_dim)
            self._cache[key] = draw_bits(_seed(self.index, rid, 0), shape, self.dtype)
        return self._cache[key]

    def int8_scales(self):
        """(k_scale, v_scale) float32 [Hkv, D] for an INT8 cache: one fixed scale per KV head
        and channel, drawn uniform in [0.02, 0.04) (127 codes then span |x| up to 2.5..5.1,
        so the N(0, 1) values are mostly in range and a few clamp)."""
        key = ("int8_scales",)
        if key not in self._cache:
            shape = (self.num_kv_heads, self.head_dim)
            draw = lambda r: (0.02 + 0.02 * torch.rand(
                *shape, generator=torch.Generator().manual_seed(_seed(self.index, r, 3)),
                dtype=torch.float32)).numpy()
            self._cache[key] = (draw(0), draw(1))
        return self._cache[key]

    def drop(self, rid: int) -> None:
        self._cache.pop(("kv", rid), None)
        self._cache.pop(("q", rid), None)

    def pages_needed(self) -> int:
        return sum((r.total + PAGE - 1) // PAGE for r in self.requests)


def _shuffled(n: int, seed: int) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n, generator=g).numpy().astype(np.int32)


def tiny(index: int = 0) -> Workload:
    """2 requests, 4 q / 2 kv heads, d=64, bf16; prompts 37 and 100 prefilled in 64-token
    chunks, then 5 decode steps each; 32-page pool in a seeded shuffled order."""
    reqs = [RequestSpec(0, 0, 37, 5), RequestSpec(1, 0, 100, 5)]
    return Workload(index, "tiny step", 4, 2, 64, BF16, reqs, _shuffled(32, 7000 + index), 32,
                    budget=2048, chunk_cap=64)


def decode_only(index: int = 1, batch: int = 64, lo: int = 512, hi: int = 4096,
                num_pages: int = 70000) -> Workload:
    """Llama-3-8B attention shapes (32 q / 8 kv heads, d=128), bf16, batch 64, cached
    contexts uniform in [512, 4096]; each request's pages are a consecutive slice of a
    seeded random permutation of a 70k-page pool; one decode step."""
    g = torch.Generator().manual_seed(5000 + index)
    ctx = torch.randint(lo, hi + 1, (batch,), generator=g).tolist()
    reqs = [RequestSpec(r, c, 0, 1) for r, c in enumerate(ctx)]
    return Workload(index, "decode-only", 32, 8, 128, BF16, reqs,
                    _shuffled(num_pages, 7000 + index), num_pages)


def prefill(index: int = 2, seq: int = 8192, chunk: Optional[int] = None) -> Workload:
    """One request of S=8192 prompt tokens, 32 q / 8 kv heads, d=128, bf16, 512 shuffled
    pages; ``chunk=None`` is one-shot, ``chunk=2048`` gives the 4 x 2048 schedule."""
    npages = max(512, (seq + PAGE - 1) // PAGE)
    reqs = [RequestSpec(0, 0, seq, 0)]
    return Workload(index, "prefill" if chunk is None else "prefill-chunked", 32, 8, 128, BF16,
                    reqs, _shuffled(npages, 7000 + index), npages,
                    budget=seq if chunk is None else chunk)


def mixed(index: int = 3, n_decode: int = 30, prompt: int = 30000, budget: int = 2048,
          lo: int = 1024, hi: int = 8192, steps: Optional[int] = None) -> Workload:
    """30 decode requests (cached contexts uniform in [1k, 8k]) plus one 30,000-token
    prompt, token budget 2048 (decode-first; the prompt gets the rest: 2018 tokens a step,
    15 steps); 32/8 heads, d=128, bf16.  The decode requests decode once per step for as
    many steps as the prompt needs (``steps`` overrides)."""
    g = torch.Generator().manual_seed(5000 + index)
    ctx = torch.randint(lo, hi + 1, (n_decode,), generator=g).tolist()
    per_step = budget - n_decode
    n_steps = steps if steps is not None else (prompt + per_step - 1) // per_step
    reqs = [RequestSpec(r, c, 0, n_steps) for r, c in enumerate(ctx)]
    reqs.append(RequestSpec(n_decode, 0, prompt, 0))
    need = sum((r.total + PAGE - 1) // PAGE for r in reqs)
    npages = need + 64
    return Workload(index, "mixed", 32, 8, 128, BF16, reqs, _shuffled(npages, 7000 + index),
                    npages, budget=budget)


def mha_skew(index: int = 4, batch: int = 16, steps: int = 64, lo: int = 32,
             hi: int = 2048) -> Workload:
    """MHA 32/32 heads, d=128, fp16; batch 16 with cached contexts round(exp(U(ln 32,
    ln 2048))) (log-uniform, 10x+ skew); a sequential pool handed out round-robin across
    requests one page at a time (fragmented, interleaved tables); 64 decode steps."""
    g = torch.Generator().manual_seed(5000 + index)
    u = torch.rand(batch, generator=g, dtype=torch.float64).numpy()
    ctx = [int(round(math.exp(math.log(lo) + x * (math.log(hi) - math.log(lo))))) for x in u]
    reqs = [RequestSpec(r, c, 0, steps) for r, c in enumerate(ctx)]
    need = sum((r.total + PAGE - 1) // PAGE for r in reqs)
    npages = need + 16
    return Workload(index, "mha-skew", 32, 32, 128, FP16, reqs,
                    np.arange(npages, dtype=np.int32), npages, interleave_history=True)


WORKLOADS = {0: tiny, 1: decode_only, 2: prefill, 3: mixed, 4: mha_skew}
