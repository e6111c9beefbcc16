"""ctypes binding of libpkv.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (without the ``pkv_``
prefix) and forwards raw device pointers taken from torch tensors together with the
caller's current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there
is no fallback of any kind: if the shared library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

OK = 0
STATUS = {0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED",
          -3: "PKV_ERR_CAPACITY", -4: "PKV_ERR_WORKSPACE", -5: "PKV_ERR_CUDA",
          -6: "PKV_ERR_DEVICE", -7: "PKV_ERR_NO_PAGES"}
DEVERR_PAGE_RANGE, DEVERR_TABLE_RANGE, DEVERR_TOKENS, DEVERR_TIMEOUT = 1, 2, 4, 8
BF16, FP16 = 0, 1
DTYPE_CODE = {torch.bfloat16: BF16, torch.float16: FP16}

EXPORTED = ("pkv_kv_append", "pkv_advance_context", "pkv_attention_workspace_bytes",
            "pkv_paged_attention_step", "pkv_kv_append_int8",
            "pkv_attention_workspace_bytes_int8", "pkv_paged_attention_step_int8",
            "pkv_paged_attention_step_static_ws", "pkv_plan_attention",
            "pkv_paged_attention_run", "pkv_paged_attention_run_int8", "pkv_copy_pages",
            "pkv_append_attention", "pkv_append_attention_int8",
            "pkv_read_device_error", "pkv_set_kernel_events", "pkv_status_string",
            "pkv_version")


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s returned %s (%d)" % (fn, STATUS.get(status, "?"), status))
        self.status = status


class StepDesc(ctypes.Structure):
    """Mirror of ``pkv_step_desc`` (include/pkv.h)."""
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32), ("total_q_tokens", ctypes.c_int32),
        ("max_q_len", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("q_lens", ctypes.c_void_p), ("q_offsets", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpkv.so (raises OSError if it is absent: build it with build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError("libpkv.so not found at %s; run paged_kv_cache_token_gb300.build.build()"
                      % p)
    lib = ctypes.CDLL(p)
    V, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.pkv_kv_append.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V, V, V, V]
    lib.pkv_kv_append.restype = ctypes.c_int
    lib.pkv_advance_context.argtypes = [ctypes.POINTER(StepDesc), V, V]
    lib.pkv_advance_context.restype = ctypes.c_int
    lib.pkv_attention_workspace_bytes.argtypes = [ctypes.POINTER(StepDesc)]
    lib.pkv_attention_workspace_bytes.restype = sz
    lib.pkv_paged_attention_step.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V,
                                             ctypes.c_float, V, sz, V, V]
    lib.pkv_paged_attention_step.restype = ctypes.c_int
    lib.pkv_kv_append_int8.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V, V, V, V, V, V]
    lib.pkv_kv_append_int8.restype = ctypes.c_int
    lib.pkv_attention_workspace_bytes_int8.argtypes = [ctypes.POINTER(StepDesc)]
    lib.pkv_attention_workspace_bytes_int8.restype = sz
    lib.pkv_paged_attention_step_int8.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V, V, V,
                                                  ctypes.c_float, V, sz, V, V]
    lib.pkv_paged_attention_step_int8.restype = ctypes.c_int
    lib.pkv_append_attention.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V, V, V, V,
                                         ctypes.c_float, V, sz, V, V]
    lib.pkv_append_attention.restype = ctypes.c_int
    lib.pkv_append_attention_int8.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V, V, V, V,
                                              V, V, ctypes.c_float, V, sz, V, V]
    lib.pkv_append_attention_int8.restype = ctypes.c_int
    lib.pkv_copy_pages.argtypes = [ctypes.POINTER(StepDesc), V, V, ctypes.c_int32, V, V,
                                   ctypes.c_int, V, V]
    lib.pkv_copy_pages.restype = ctypes.c_int
    lib.pkv_plan_attention.argtypes = [ctypes.POINTER(StepDesc), V, sz, V, V]
    lib.pkv_plan_attention.restype = ctypes.c_int
    lib.pkv_paged_attention_run.argtypes = lib.pkv_paged_attention_step.argtypes
    lib.pkv_paged_attention_run.restype = ctypes.c_int
    lib.pkv_paged_attention_run_int8.argtypes = lib.pkv_paged_attention_step_int8.argtypes
    lib.pkv_paged_attention_run_int8.restype = ctypes.c_int
    lib.pkv_paged_attention_step_static_ws.argtypes = [ctypes.POINTER(StepDesc), V, V, V, V,
                                                       ctypes.c_float, V, V]
    lib.pkv_paged_attention_step_static_ws.restype = ctypes.c_int
    lib.pkv_read_device_error.argtypes = [V, ctypes.POINTER(ctypes.c_int32), V]
    lib.pkv_read_device_error.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_set_kernel_events.argtypes = [ctypes.c_int, V, V]
    lib.pkv_set_kernel_events.restype = ctypes.c_int
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_desc(*, num_reqs, num_q_heads, num_kv_heads, head_dim, num_pages, max_pages_per_req,
              total_q_tokens, max_q_len, max_context_len, dtype, q_lens=None, q_offsets=None,
              context_lens=None, block_table=None, page_size=16) -> StepDesc:
    """Fill a StepDesc; the four arrays are int32 CUDA tensors (or raw addresses)."""
    def addr(x):
        if x is None:
            return None
        return x.data_ptr() if isinstance(x, torch.Tensor) else int(x)
    code = DTYPE_CODE.get(dtype, dtype)
    return StepDesc(num_reqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                    max_pages_per_req, total_q_tokens, max_q_len, max_context_len, code,
                    addr(q_lens), addr(q_offsets), addr(context_lens), addr(block_table))


def version() -> int:
    return load().pkv_version()


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def kv_append(desc: StepDesc, k_new, v_new, k_cache, v_cache, slot_mapping=None, err=None,
              stream=None, check: bool = True) -> int:
    rc = load().pkv_kv_append(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                              _ptr(v_cache), _ptr(slot_mapping), _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_kv_append", rc)
    return rc


def advance_context(desc: StepDesc, context_lens, stream=None, check: bool = True) -> int:
    """context_lens[r] += q_lens[r] on the device (context_lens: int32 CUDA tensor)."""
    rc = load().pkv_advance_context(ctypes.byref(desc), _ptr(context_lens), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_advance_context", rc)
    return rc


def attention_workspace_bytes(desc: StepDesc) -> int:
    return int(load().pkv_attention_workspace_bytes(ctypes.byref(desc)))


def paged_attention_step(desc: StepDesc, q, k_cache, v_cache, out, scale: float, workspace,
                         err=None, stream=None, check: bool = True,
                         workspace_bytes: Optional[int] = None) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_paged_attention_step(ctypes.byref(desc), _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(out), float(scale), _ptr(workspace),
                                         nbytes, _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_paged_attention_step", rc)
    return rc


def append_attention(desc: StepDesc, k_new, v_new, k_cache, v_cache, q, out, scale: float,
                     workspace, slot_mapping=None, err=None, stream=None, check: bool = True,
                     workspace_bytes: Optional[int] = None) -> int:
    """kv_append then the attention step in one call (one fused grid for decode steps)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_append_attention(ctypes.byref(desc), _ptr(k_new), _ptr(v_new),
                                     _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), _ptr(q),
                                     _ptr(out), float(scale), _ptr(workspace), nbytes, _ptr(err),
                                     _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_append_attention", rc)
    return rc


def append_attention_int8(desc: StepDesc, k_new, v_new, k_scale, v_scale, k_cache, v_cache, q,
                          out, scale: float, workspace, slot_mapping=None, err=None, stream=None,
                          check: bool = True, workspace_bytes: Optional[int] = None) -> int:
    """kv_append_int8 then the INT8 attention step in one call (one fused grid for decode
    steps)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_append_attention_int8(ctypes.byref(desc), _ptr(k_new), _ptr(v_new),
                                          _ptr(k_scale), _ptr(v_scale), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(slot_mapping), _ptr(q), _ptr(out),
                                          float(scale), _ptr(workspace), nbytes, _ptr(err),
                                          _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_append_attention_int8", rc)
    return rc


def copy_pages(desc: StepDesc, src_pages, dst_pages, k_cache, v_cache, kv_int8: bool = False,
               err=None, stream=None, check: bool = True) -> int:
    """Copy whole pages src_pages[i] -> dst_pages[i] (int32 CUDA tensors) in both pools."""
    n = int(src_pages.numel())
    rc = load().pkv_copy_pages(ctypes.byref(desc), _ptr(src_pages), _ptr(dst_pages), n,
                               _ptr(k_cache), _ptr(v_cache), 1 if kv_int8 else 0, _ptr(err),
                               _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_copy_pages", rc)
    return rc


def plan_attention(desc: StepDesc, workspace, err=None, stream=None, check: bool = True,
                   workspace_bytes: Optional[int] = None) -> int:
    """The plan half of the attention step: the step's work list into ``workspace``."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_plan_attention(ctypes.byref(desc), _ptr(workspace), nbytes, _ptr(err),
                                   _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_plan_attention", rc)
    return rc


def paged_attention_run(desc: StepDesc, q, k_cache, v_cache, out, scale: float, workspace,
                        err=None, stream=None, check: bool = True,
                        workspace_bytes: Optional[int] = None) -> int:
    """The run half: attention over the plan already in ``workspace`` (another layer)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_paged_attention_run(ctypes.byref(desc), _ptr(q), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(out), float(scale), _ptr(workspace),
                                        nbytes, _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_paged_attention_run", rc)
    return rc


def paged_attention_run_int8(desc: StepDesc, q, k_cache, v_cache, k_scale, v_scale, out,
                             scale: float, workspace, err=None, stream=None, check: bool = True,
                             workspace_bytes: Optional[int] = None) -> int:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_paged_attention_run_int8(ctypes.byref(desc), _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                             _ptr(out), float(scale), _ptr(workspace), nbytes,
                                             _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_paged_attention_run_int8", rc)
    return rc


def kv_append_int8(desc: StepDesc, k_new, v_new, k_scale, v_scale, k_cache, v_cache,
                   slot_mapping=None, err=None, stream=None, check: bool = True) -> int:
    """Quantise this step's K/V (desc.dtype) to per-channel INT8 codes in the int8 pools;
    k_scale, v_scale: float32 CUDA tensors [Hkv, D]."""
    rc = load().pkv_kv_append_int8(ctypes.byref(desc), _ptr(k_new), _ptr(v_new),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(slot_mapping), _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_kv_append_int8", rc)
    return rc


def attention_workspace_bytes_int8(desc: StepDesc) -> int:
    return int(load().pkv_attention_workspace_bytes_int8(ctypes.byref(desc)))


def paged_attention_step_int8(desc: StepDesc, q, k_cache, v_cache, k_scale, v_scale, out,
                              scale: float, workspace, err=None, stream=None,
                              check: bool = True, workspace_bytes: Optional[int] = None) -> int:
    """The attention step over int8 pools (codes times the per-channel scales)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None \
        else workspace_bytes
    rc = load().pkv_paged_attention_step_int8(ctypes.byref(desc), _ptr(q), _ptr(k_cache),
                                              _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                              _ptr(out), float(scale), _ptr(workspace), nbytes,
                                              _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_paged_attention_step_int8", rc)
    return rc


STATIC_WORKSPACE_BYTES = 32 << 20


def paged_attention_step_static_ws(desc: StepDesc, q, k_cache, v_cache, out, scale: float,
                                   err=None, stream=None, check: bool = True) -> int:
    """The attention step with the library's built-in scratch array instead of a caller
    workspace (for callers that cannot allocate device memory at call time)."""
    rc = load().pkv_paged_attention_step_static_ws(ctypes.byref(desc), _ptr(q), _ptr(k_cache),
                                                   _ptr(v_cache), _ptr(out), float(scale),
                                                   _ptr(err), _stream(stream))
    if check and rc != OK:
        raise PkvError("pkv_paged_attention_step_static_ws", rc)
    return rc


def set_kernel_events(which: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start``/``stop`` around the main kernel of path ``which``
    (0 decode stream, 1 tensor-core prefill) in later attention calls; None clears."""
    s = ctypes.c_void_p(start.cuda_event) if start is not None else None
    e = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    rc = load().pkv_set_kernel_events(which, s, e)
    if rc != OK:
        raise PkvError("pkv_set_kernel_events", rc)


def read_device_error(err: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the flag value (0 = no device-detected error)."""
    val = ctypes.c_int32(0)
    rc = load().pkv_read_device_error(_ptr(err), ctypes.byref(val), _stream(stream))
    if rc not in (OK, -6):
        raise PkvError("pkv_read_device_error", rc)
    return int(val.value)
