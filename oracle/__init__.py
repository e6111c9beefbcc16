"""fp64 CPU oracle for the paged-KV attention step -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may import
this package.  It shares no code with the CUDA library and never imports it.

Functions (numpy in, numpy out; 16-bit inputs are passed as their uint16 bit patterns):

* :func:`attention_rows` -- causal softmax attention of query rows at given absolute
  positions over a request's contiguous K/V (hotelren.com/news/6181127 §1.1, §2.1,
  §3.1, §5.1; niuwancheng.cn "11. chunked prefill and unified scheduling": chunked
  prefill gives the one-shot result).
* :func:`kv_append` -- the page pool after appending a step's new K/V through the
  block table (lshu.cn/news/11576 §2.2-§2.3: pages of 16 tokens written by page index).
* :func:`kv_bytes_per_token` -- 2 x L x n_kv_heads x d_head x bytes
  (hotelren.com/news/6181127 §2.3).
* :func:`quantize_int8`, :func:`attention_rows_int8` -- codes of a per-channel INT8 KV
  cache and attention over the values they stand for (wmrh.cn/news/64708 §4.3, §5.4).
"""
import ctypes
import os

import numpy as np

from .build_oracle import build_oracle

BF16 = 0
FP16 = 1
PAGE_TOKENS = 16

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_attention_rows.argtypes = [ctypes.c_int, P, P, i32, P, P, i32, i32, i32, i32,
                                              dbl, P]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_kv_append.argtypes = [i32, P, P, P, i32, i32, i32, i32, P, P, P, P, P]
        lib.oracle_kv_append.restype = ctypes.c_int
        lib.oracle_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
        lib.oracle_kv_bytes_per_token.restype = i64
        lib.oracle_widen.argtypes = [ctypes.c_int, P, i64, P]
        lib.oracle_widen.restype = ctypes.c_int
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = dbl
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = dbl
        lib.oracle_quantize_int8.argtypes = [ctypes.c_int, P, i64, i32, i32, P, P]
        lib.oracle_quantize_int8.restype = ctypes.c_int
        lib.oracle_attention_rows_int8.argtypes = [ctypes.c_int, P, P, i32, P, P, P, P, i32,
                                                   i32, i32, i32, dbl, P]
        lib.oracle_attention_rows_int8.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("16-bit inputs are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def widen(dtype: int, bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 (dtype=0) or fp16 (dtype=1) bit patterns to float64."""
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().oracle_widen(dtype, _ptr(bits), bits.size, _ptr(out))
    if rc:
        raise ValueError("oracle_widen: bad dtype")
    return out


def bf16_to_double(x: int) -> float:
    return _load().oracle_bf16_to_double(x)


def fp16_to_double(x: int) -> float:
    return _load().oracle_fp16_to_double(x)


def kv_bytes_per_token(layers: int, n_kv_heads: int, d_head: int, bytes_per_elem: int) -> int:
    return _load().oracle_kv_bytes_per_token(layers, n_kv_heads, d_head, bytes_per_elem)


def attention_rows(dtype: int, q: np.ndarray, pos: np.ndarray, k: np.ndarray, v: np.ndarray,
                   scale: float) -> np.ndarray:
    """q [n, Hq, D], pos [n] int, k/v [n_kv, Hkv, D] (uint16 bits) -> out [n, Hq, D] float64.

    Row i attends keys 0..pos[i] inclusive of its request's contiguous sequence.
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    n, Hq, D = q.shape
    n_kv, Hkv, Dk = k.shape
    if Dk != D or v.shape != k.shape or pos.shape != (n,):
        raise ValueError("shape mismatch")
    out = np.empty((n, Hq, D), dtype=np.float64)
    rc = _load().oracle_attention_rows(dtype, _ptr(q), _ptr(pos), n, _ptr(k), _ptr(v), n_kv, Hq,
                                       Hkv, D, float(scale), _ptr(out))
    if rc:
        raise ValueError("oracle_attention_rows: bad argument (rc=%d)" % rc)
    return out


def quantize_int8(dtype: int, x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x [n, H, D] uint16 bits, scale [H, D] float32 > 0 -> codes [n, H, D] int8:
    clamp(rint(x / scale), -127, 127), the quotient in IEEE fp32, ties to even."""
    x = _u16(x)
    n, H, D = x.shape
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    if scale.shape != (H, D):
        raise ValueError("scale must be [H, D]")
    out = np.empty((n, H, D), dtype=np.int8)
    rc = _load().oracle_quantize_int8(dtype, _ptr(x), n, H, D, _ptr(scale), _ptr(out))
    if rc:
        raise ValueError("oracle_quantize_int8: bad argument")
    return out


def attention_rows_int8(dtype: int, q: np.ndarray, pos: np.ndarray, k_codes: np.ndarray,
                        v_codes: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray,
                        scale: float) -> np.ndarray:
    """As :func:`attention_rows` over an INT8 cache: k/v codes [n_kv, Hkv, D] int8 stand
    for code * scale[Hkv, D] (float32)."""
    q = _u16(q)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    kc = np.ascontiguousarray(k_codes, dtype=np.int8)
    vc = np.ascontiguousarray(v_codes, dtype=np.int8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    n, Hq, D = q.shape
    n_kv, Hkv, Dk = kc.shape
    if Dk != D or vc.shape != kc.shape or pos.shape != (n,) or ks.shape != (Hkv, D) or \
            vs.shape != (Hkv, D):
        raise ValueError("shape mismatch")
    out = np.empty((n, Hq, D), dtype=np.float64)
    rc = _load().oracle_attention_rows_int8(dtype, _ptr(q), _ptr(pos), n, _ptr(kc), _ptr(vc),
                                            _ptr(ks), _ptr(vs), n_kv, Hq, Hkv, D, float(scale),
                                            _ptr(out))
    if rc:
        raise ValueError("oracle_attention_rows_int8: bad argument (rc=%d)" % rc)
    return out


def kv_append(q_lens, context_lens, block_table, num_pages, k_new, v_new, k_pool, v_pool,
              want_slots=True):
    """Append one step's K/V into copies of the pools; returns (k_pool', v_pool', slots).

    block_table [num_reqs, max_pages] int32; k_new/v_new [T, Hkv, D] uint16;
    pools [num_pages, Hkv, 16, D] uint16 (the inputs are not modified).
    """
    q_lens = np.ascontiguousarray(q_lens, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    k_new, v_new = _u16(k_new), _u16(v_new)
    kp, vp = _u16(k_pool).copy(), _u16(v_pool).copy()
    num_reqs = q_lens.shape[0]
    max_pages = block_table.shape[1] if block_table.ndim == 2 else 0
    T, Hkv, D = k_new.shape
    slots = np.empty(T, dtype=np.int64) if want_slots else None
    rc = _load().oracle_kv_append(num_reqs, _ptr(q_lens), _ptr(context_lens), _ptr(block_table),
                                  max_pages, num_pages, Hkv, D, _ptr(k_new), _ptr(v_new), _ptr(kp),
                                  _ptr(vp), _ptr(slots))
    if rc:
        raise ValueError("oracle_kv_append: rc=%d" % rc)
    return kp, vp, slots


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all online cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return os.cpu_count() or 1
