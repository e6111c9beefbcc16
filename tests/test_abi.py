"""The C-ABI library loads and exports every entry point include/*.h declares; host-side
argument checks reject bad descriptions without touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_token_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared(header="pkv.h"):
    text = open(os.path.join(ROOT, "include", header)).read()
    return set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text))


def test_header_declares_the_binding_names():
    assert _declared() >= set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    headers = sorted(os.listdir(os.path.join(ROOT, "include")))
    assert "pkv.h" in headers and "pkv_sched.h" in headers
    for header in headers:
        for name in _declared(header):
            assert hasattr(lib, name), (header, name)
            assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.status_string(code) == name
    assert binding.status_string(-99) == "PKV_UNKNOWN_STATUS"
    assert binding.version() >= 100


def _desc(**kw):
    base = dict(num_reqs=1, num_q_heads=4, num_kv_heads=2, head_dim=64, num_pages=8,
                max_pages_per_req=4, total_q_tokens=1, max_q_len=1, max_context_len=3, dtype=0,
                q_lens=16, q_offsets=32, context_lens=48, block_table=64)
    base.update(kw)
    return binding.make_desc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=32), -1),                 # pages hold 16 tokens
    (dict(head_dim=96), -2),
    (dict(num_q_heads=6, num_kv_heads=4), -2),  # Hq % Hkv != 0
    (dict(num_q_heads=32, num_kv_heads=2), -2),  # group 16 not built
    (dict(dtype=7), -2),
    (dict(num_reqs=-1), -1),
    (dict(num_pages=0), -1),
    (dict(num_reqs=0, total_q_tokens=5), -1),
    (dict(max_q_len=100, total_q_tokens=100), -3),  # 100 tokens > 4 pages x 16
    (dict(q_lens=None), -1),
    (dict(num_pages=1 << 26), -2),             # 2^26 pages x 2 heads x 16 = 2^31 pool rows
])
def test_host_validation_rejects_before_launch(lib, kw, code):
    d = _desc(**kw)
    rc = lib.pkv_kv_append(ctypes.byref(d), None, None, None, None, None, None, None)
    assert rc == code
    rc = lib.pkv_paged_attention_step(ctypes.byref(d), None, None, None, None, 1.0, None, 0, None,
                                      None)
    assert rc == code
    assert lib.pkv_attention_workspace_bytes(ctypes.byref(d)) == 0
    # the plan and run halves, the one-call append + attention and the built-in-scratch
    # entry point report description errors the same way
    assert lib.pkv_append_attention(ctypes.byref(d), None, None, None, None, None, None, None,
                                    1.0, None, 0, None, None) == code
    assert lib.pkv_plan_attention(ctypes.byref(d), None, 0, None, None) == code
    assert lib.pkv_paged_attention_run(ctypes.byref(d), None, None, None, None, 1.0, None, 0,
                                       None, None) == code
    rc = lib.pkv_paged_attention_step_static_ws(ctypes.byref(d), None, None, None, None, 1.0,
                                                None, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), -2),
    (dict(num_q_heads=32, num_kv_heads=2), -2),
    (dict(num_pages=0), -1),
    (dict(max_q_len=100, total_q_tokens=100), -3),
])
def test_int8_host_validation_rejects_before_launch(lib, kw, code):
    d = _desc(**kw)
    s = ctypes.c_void_p(0x2000)
    rc = lib.pkv_kv_append_int8(ctypes.byref(d), None, None, s, s, None, None, None, None, None)
    assert rc == code
    rc = lib.pkv_paged_attention_step_int8(ctypes.byref(d), None, None, None, s, s, None, 1.0,
                                           None, 0, None, None)
    assert rc == code
    assert lib.pkv_attention_workspace_bytes_int8(ctypes.byref(d)) == 0


def test_int8_scales_required_and_aligned(lib):
    # every tensor 16-byte aligned (never dereferenced: the checks fail first)
    d = _desc()
    t = ctypes.c_void_p(0x1000)
    good, odd = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x2004)
    for ks, vs in ((None, good), (good, None), (odd, good), (good, odd)):
        assert lib.pkv_kv_append_int8(ctypes.byref(d), t, t, ks, vs, t, t, None, None,
                                      None) == -1
        assert lib.pkv_paged_attention_step_int8(ctypes.byref(d), t, t, t, ks, vs, t, 1.0, t,
                                                 1 << 30, None, None) == -1


def test_int8_empty_step_is_a_no_op(lib):
    d = _desc(num_reqs=0, total_q_tokens=0, max_q_len=0, max_context_len=0, q_lens=None,
              q_offsets=None, context_lens=None, block_table=None)
    s = ctypes.c_void_p(0x2000)
    assert lib.pkv_kv_append_int8(ctypes.byref(d), None, None, s, s, None, None, None, None,
                                  None) == 0
    assert lib.pkv_paged_attention_step_int8(ctypes.byref(d), None, None, None, s, s, None, 1.0,
                                             None, 0, None, None) == 0


def test_null_tensors_rejected(lib):
    d = _desc()
    assert lib.pkv_kv_append(ctypes.byref(d), None, None, None, None, None, None, None) == -1
    assert lib.pkv_paged_attention_step(ctypes.byref(d), None, None, None, None, 1.0, None, 0,
                                        None, None) == -1


def test_misaligned_tensors_rejected(lib):
    d = _desc()
    p = ctypes.c_void_p(0x1008)
    assert lib.pkv_kv_append(ctypes.byref(d), p, p, p, p, None, None, None) == -1


def test_empty_step_is_a_no_op(lib):
    d = _desc(num_reqs=0, total_q_tokens=0, max_q_len=0, max_context_len=0, q_lens=None,
              q_offsets=None, context_lens=None, block_table=None)
    assert lib.pkv_kv_append(ctypes.byref(d), None, None, None, None, None, None, None) == 0
    assert lib.pkv_paged_attention_step(ctypes.byref(d), None, None, None, None, 1.0, None, 0,
                                        None, None) == 0


def test_read_device_error_rejects_null(lib):
    v = ctypes.c_int32(0)
    assert lib.pkv_read_device_error(None, ctypes.byref(v), None) == -1


def test_plan_and_run_argument_checks(lib):
    d = _desc()
    t = ctypes.c_void_p(0x1000)
    # the run needs the tensors (checked before any device query)
    assert lib.pkv_paged_attention_run(ctypes.byref(d), None, None, None, None, 1.0, t, 1 << 30,
                                       None, None) == -1
    assert lib.pkv_paged_attention_run_int8(ctypes.byref(d), t, t, t, None, t, t, 1.0, t,
                                            1 << 30, None, None) == -1
    e = _desc(num_reqs=0, total_q_tokens=0, max_q_len=0, max_context_len=0, q_lens=None,
              q_offsets=None, context_lens=None, block_table=None)
    assert lib.pkv_plan_attention(ctypes.byref(e), None, 0, None, None) == 0
    assert lib.pkv_paged_attention_run(ctypes.byref(e), None, None, None, None, 1.0, None, 0,
                                       None, None) == 0


def test_append_attention_argument_checks(lib):
    d = _desc()
    t, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008)
    # new rows missing or misaligned, a misaligned slot-id array (before any device query)
    assert lib.pkv_append_attention(ctypes.byref(d), None, t, t, t, None, t, t, 1.0, t, 1 << 30,
                                    None, None) == -1
    assert lib.pkv_append_attention(ctypes.byref(d), odd, t, t, t, None, t, t, 1.0, t, 1 << 30,
                                    None, None) == -1
    assert lib.pkv_append_attention(ctypes.byref(d), t, t, t, t, ctypes.c_void_p(0x1004), t, t,
                                    1.0, t, 1 << 30, None, None) == -1
    e = _desc(num_reqs=0, total_q_tokens=0, max_q_len=0, max_context_len=0, q_lens=None,
              q_offsets=None, context_lens=None, block_table=None)
    assert lib.pkv_append_attention(ctypes.byref(e), None, None, None, None, None, None, None,
                                    1.0, None, 0, None, None) == 0


def test_append_attention_int8_argument_checks(lib):
    d = _desc()
    t, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008)
    call = lambda *a: lib.pkv_append_attention_int8(ctypes.byref(d), *a)
    # args: k_new, v_new, k_scale, v_scale, k_cache, v_cache, slot_mapping, q, out, scale,
    # workspace, bytes, err, stream -- refused on the host before any device query
    assert call(None, t, t, t, t, t, None, t, t, 1.0, t, 1 << 30, None, None) == -1
    assert call(t, odd, t, t, t, t, None, t, t, 1.0, t, 1 << 30, None, None) == -1
    assert call(t, t, None, t, t, t, None, t, t, 1.0, t, 1 << 30, None, None) == -1   # no scales
    assert call(t, t, t, odd, t, t, None, t, t, 1.0, t, 1 << 30, None, None) == -1
    assert call(t, t, t, t, t, t, ctypes.c_void_p(0x1004), t, t, 1.0, t, 1 << 30, None,
                None) == -1
    e = _desc(num_reqs=0, total_q_tokens=0, max_q_len=0, max_context_len=0, q_lens=None,
              q_offsets=None, context_lens=None, block_table=None)
    assert lib.pkv_append_attention_int8(ctypes.byref(e), None, None, None, None, None, None,
                                         None, None, None, 1.0, None, 0, None, None) == 0
