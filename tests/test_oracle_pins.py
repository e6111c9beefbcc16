"""Pins for the fp64 oracle: it is checked against what the pages and mathematics fix,
never against itself or the CUDA path.

* KV byte counts printed on hotelren.com/news/6181127 §2.3 and §6.3 (golden file).
* Exact widening of every bf16 / fp16 pattern against numpy's and torch's converters.
* Brute force on tiny inputs: an independent 60-digit mpmath evaluation of softmax
  attention written directly from the definition (no max subtraction).
* Closed forms: q = 0 or scale = 0 gives the mean of V[0..p]; one key gives V[0]; equal
  keys give uniform weights; one-hot V columns turn the output into the softmax weights.
* The paging oracle against an independent gather through the block table.
* Mutation checks: plausible mistakes (dropped scale, transposed GQA mapping, mask off
  by one) planted in a copy of the definition are caught by the same pins.
"""
import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
mpmath.mp.dps = 60


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def _bits(x, dtype):
    t = torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16 if dtype == oracle.BF16 else
                                                   torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bits(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return _bits(torch.randn(*shape, generator=g), dtype)


# --------------------------------------------------------------------------- byte formula
def test_kv_bytes_golden():
    rows = _golden_rows("kv_bytes.txt")
    assert len(rows) >= 6
    for r in rows:
        L, hkv, d, b, tokens, batch, expected = map(int, r[:7])
        assert oracle.kv_bytes_per_token(L, hkv, d, b) * tokens * batch == expected, r


def test_kv_bytes_linear_in_each_factor():
    base = oracle.kv_bytes_per_token(1, 1, 1, 1)
    assert base == 2  # K and V
    for args in [(3, 1, 1, 1), (1, 5, 1, 1), (1, 1, 7, 1), (1, 1, 1, 4)]:
        assert oracle.kv_bytes_per_token(*args) == 2 * math.prod(args)


# --------------------------------------------------------------------------- widening
def test_widen_fp16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.widen(oracle.FP16, bits)
    ref = bits.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def test_widen_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.widen(oracle.BF16, bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133  # smallest subnormal
    assert oracle.fp16_to_double(0x0001) == 2.0 ** -24


# --------------------------------------------------------------------------- brute force
def _mp_attention(qd, kd, vd, pos, scale, group):
    """60-digit softmax attention straight from the definition: weights exp(s_j) / sum exp."""
    n, hq, d = qd.shape
    out = np.zeros((n, hq, d))
    for i in range(n):
        for h in range(hq):
            g = h // group
            s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(qd[i, h, c])) *
                                                 mpmath.mpf(float(kd[j, g, c])) for c in range(d))
                 for j in range(pos[i] + 1)]
            e = [mpmath.exp(x) for x in s]
            z = mpmath.fsum(e)
            for c in range(d):
                out[i, h, c] = float(mpmath.fsum(e[j] * mpmath.mpf(float(vd[j, g, c]))
                                                 for j in range(pos[i] + 1)) / z)
    return out


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("hq,hkv,d,n_kv,seed", [(1, 1, 1, 1, 1), (2, 1, 3, 5, 2), (4, 2, 4, 8, 3),
                                                 (3, 3, 2, 6, 4), (4, 1, 4, 7, 5)])
def test_brute_force_tiny(dtype, hq, hkv, d, n_kv, seed):
    q = _rand_bits((n_kv, hq, d), dtype, seed)
    k = _rand_bits((n_kv, hkv, d), dtype, seed + 100)
    v = _rand_bits((n_kv, hkv, d), dtype, seed + 200)
    pos = np.arange(n_kv, dtype=np.int32)
    for scale in (1.0, 1.0 / math.sqrt(d), 2.5):
        got = oracle.attention_rows(dtype, q, pos, k, v, scale)
        ref = _mp_attention(oracle.widen(dtype, q), oracle.widen(dtype, k), oracle.widen(dtype, v),
                            pos, scale, hq // hkv)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_brute_force_large_logits_no_overflow():
    # logits around 300: exp overflows a naive fp64 evaluation; the oracle subtracts the max
    d = 4
    q = _bits(np.full((3, 1, d), 8.0), oracle.BF16)
    k = _bits(np.array([[[9.0, 9.5, 10.0, 9.0]], [[9.5, 9.5, 9.0, 10.0]], [[8.0, 8.0, 8.0, 8.0]]]),
              oracle.BF16)
    v = _rand_bits((3, 1, d), oracle.BF16, 9)
    pos = np.arange(3, dtype=np.int32)
    got = oracle.attention_rows(oracle.BF16, q, pos, k, v, 1.0)
    ref = _mp_attention(oracle.widen(0, q), oracle.widen(0, k), oracle.widen(0, v), pos, 1.0, 1)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("variant", ["q_zero", "scale_zero"])
def test_zero_logits_give_prefix_mean(variant):
    n, hq, hkv, d = 9, 4, 2, 8
    q = np.zeros((n, hq, d), np.uint16) if variant == "q_zero" else _rand_bits((n, hq, d), 0, 11)
    k = _rand_bits((n, hkv, d), 0, 12)
    v = _rand_bits((n, hkv, d), 0, 13)
    pos = np.arange(n, dtype=np.int32)
    got = oracle.attention_rows(0, q, pos, k, v, 0.0 if variant == "scale_zero" else 0.7)
    vd = oracle.widen(0, v)
    for i in range(n):
        for h in range(hq):
            np.testing.assert_allclose(got[i, h], vd[:i + 1, h // 2].mean(axis=0), rtol=1e-13,
                                       atol=1e-15)


def test_single_key_returns_v0():
    q = _rand_bits((1, 8, 16), 1, 21)
    k = _rand_bits((1, 2, 16), 1, 22)
    v = _rand_bits((1, 2, 16), 1, 23)
    got = oracle.attention_rows(1, q, np.array([0], np.int32), k, v, 3.0)
    vd = oracle.widen(1, v)
    for h in range(8):
        assert np.array_equal(got[0, h], vd[0, h // 4])


def test_equal_keys_uniform_weights():
    n, d = 6, 8
    q = _rand_bits((n, 2, d), 0, 31)
    k = np.repeat(_rand_bits((1, 1, d), 0, 32), n, axis=0)
    v = _rand_bits((n, 1, d), 0, 33)
    got = oracle.attention_rows(0, q, np.arange(n, dtype=np.int32), k, v, 1.3)
    vd = oracle.widen(0, v)
    for i in range(n):
        np.testing.assert_allclose(got[i, 0], vd[:i + 1, 0].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_one_hot_v_gives_softmax_weights():
    n, d = 5, 5   # V[j] = e_j: column j of the output is the weight of key j
    q = _rand_bits((n, 1, d), 0, 41)
    k = _rand_bits((n, 1, d), 0, 42)
    v = _bits(np.eye(n).reshape(n, 1, d), 0)
    pos = np.arange(n, dtype=np.int32)
    got = oracle.attention_rows(0, q, pos, k, v, 0.9)
    qd, kd = oracle.widen(0, q), oracle.widen(0, k)
    for i in range(n):
        w = got[i, 0]
        assert abs(w.sum() - 1.0) < 1e-14
        assert np.all(w[i + 1:] == 0.0)               # causal: no weight past the row
        s = [0.9 * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in
                               zip(qd[i, 0], kd[j, 0])) for j in range(i + 1)]
        e = [mpmath.exp(x) for x in s]
        z = mpmath.fsum(e)
        np.testing.assert_allclose(w[:i + 1], [float(x / z) for x in e], rtol=1e-13)


# --------------------------------------------------------------------------- equivalences
def test_chunked_rows_equal_one_shot_and_decode_equals_last_prefill_row():
    """niuwancheng.cn "11. chunked prefill...": a chunk reads the earlier chunks' K/V and the
    result equals one-shot prefill; hotelren.com/news/6181127 §3.1: a decode step attends
    the whole cache including the token it appended -> the last row of a prefill."""
    n, hq, hkv, d = 40, 4, 2, 16
    q = _rand_bits((n, hq, d), 0, 51)
    k = _rand_bits((n, hkv, d), 0, 52)
    v = _rand_bits((n, hkv, d), 0, 53)
    pos = np.arange(n, dtype=np.int32)
    one = oracle.attention_rows(0, q, pos, k, v, 0.25)
    parts = [oracle.attention_rows(0, q[a:b], pos[a:b], k[:b], v[:b], 0.25)
             for a, b in [(0, 13), (13, 29), (29, 40)]]
    assert np.abs(np.concatenate(parts) - one).max() <= 1e-12 * np.abs(one).max()
    dec = oracle.attention_rows(0, q[n - 1:], pos[n - 1:], k, v, 0.25)
    assert np.abs(dec[0] - one[n - 1]).max() <= 1e-12


def test_rejects_bad_positions():
    q = _rand_bits((2, 1, 4), 0, 1)
    k = _rand_bits((3, 1, 4), 0, 2)
    with pytest.raises(ValueError):
        oracle.attention_rows(0, q, np.array([0, 3], np.int32), k, k, 1.0)


# --------------------------------------------------------------------------- paging
def test_page_counts_golden():
    for r in _golden_rows("page_counts.txt"):
        tokens, pages = int(r[0]), int(r[1])
        assert -(-tokens // oracle.PAGE_TOKENS) == pages, r


def _random_tables(rng, ctx, qlens, num_pages):
    order = rng.permutation(num_pages).astype(np.int32)
    need = [-(-(c + q) // 16) for c, q in zip(ctx, qlens)]
    width = max(need)
    bt = np.full((len(ctx), width), -1, np.int32)
    used = 0
    for r, n in enumerate(need):
        bt[r, :n] = order[used:used + n]
        used += n
    return bt


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_kv_append_against_block_table_gather(seed):
    rng = np.random.default_rng(seed)
    hkv, d, num_pages = 3, 8, 64
    ctx = [0, 15, 16, 31, 5]          # page-boundary cases
    qlens = [16, 1, 17, 33, 0]
    bt = _random_tables(rng, ctx, qlens, num_pages)
    T = sum(qlens)
    k_new = rng.integers(0, 0xFFFE, size=(T, hkv, d), dtype=np.uint16)
    v_new = rng.integers(0, 0xFFFE, size=(T, hkv, d), dtype=np.uint16)
    sentinel = np.full((num_pages, hkv, 16, d), 0xFFFF, np.uint16)
    kp, vp, slots = oracle.kv_append(qlens, ctx, bt, num_pages, k_new, v_new, sentinel, sentinel)
    # independent reading: gather token t back from its page / slot with fancy indexing
    t = 0
    written = np.zeros((num_pages, 16), bool)
    for r in range(len(ctx)):
        for i in range(qlens[r]):
            p = ctx[r] + i
            page, slot = bt[r, p // 16], p % 16
            assert slots[t] == page * 16 + slot
            assert np.array_equal(kp[page, :, slot, :], k_new[t])
            assert np.array_equal(vp[page, :, slot, :], v_new[t])
            written[page, slot] = True
            t += 1
    assert len(set(slots.tolist())) == T                      # no two tokens share a slot
    untouched = ~written[:, None, :, None] & np.ones(kp.shape, bool)
    assert np.all(kp[untouched] == 0xFFFF) and np.all(vp[untouched] == 0xFFFF)
    assert np.all(sentinel == 0xFFFF)                         # inputs untouched


def test_kv_append_rejects_out_of_range():
    bt = np.array([[0, 99]], np.int32)
    pool = np.zeros((4, 1, 16, 2), np.uint16)
    kn = np.zeros((20, 1, 2), np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_append([20], [0], bt, 4, kn, kn, pool, pool)      # page 99 outside pool
    with pytest.raises(ValueError):
        oracle.kv_append([20], [20], bt, 4, kn, kn, pool, pool)     # runs past the table


# --------------------------------------------------------------------------- mutations
def _py_attention(qd, kd, vd, pos, scale, group, mutate=None):
    n, hq, d = qd.shape
    out = np.zeros((n, hq, d))
    hkv = kd.shape[1]
    for i in range(n):
        for h in range(hq):
            g = h // group if mutate != "gqa_modulo" else h % hkv
            last = pos[i] + (0 if mutate != "mask_exclusive" else -1)
            last = max(last, 0)
            sc = 1.0 if mutate == "drop_scale" else scale
            s = np.array([sc * np.dot(qd[i, h], kd[j, g]) for j in range(last + 1)])
            w = np.exp(s - s.max())
            vv = vd[:last + 1, g] if mutate != "v_transposed" else vd[:last + 1, (g + 1) % hkv]
            out[i, h] = (w[:, None] * vv).sum(0) / w.sum()
    return out


@pytest.mark.parametrize("mutate", ["gqa_modulo", "mask_exclusive", "drop_scale", "v_transposed"])
def test_pins_catch_planted_mistakes(mutate):
    n, hq, hkv, d = 6, 4, 2, 4
    q = _rand_bits((n, hq, d), 0, 61)
    k = _rand_bits((n, hkv, d), 0, 62)
    v = _rand_bits((n, hkv, d), 0, 63)
    pos = np.arange(n, dtype=np.int32)
    qd, kd, vd = (oracle.widen(0, a) for a in (q, k, v))
    ref = _mp_attention(qd, kd, vd, pos, 0.5, hq // hkv)
    good = _py_attention(qd, kd, vd, pos, 0.5, hq // hkv)
    np.testing.assert_allclose(good, ref, rtol=1e-10, atol=1e-12)
    bad = _py_attention(qd, kd, vd, pos, 0.5, hq // hkv, mutate)
    assert np.abs(bad - ref).max() > 1e-3


# ------------------------------------------------------------------ INT8 KV cache
# wmrh.cn/news/64708 §4.3 (KV cache in INT8) and §5.4 (calibrated per channel): the code of
# x in channel (h, d) is clamp(rint(x / s[h, d]), -127, 127) and stands for code * s.

def _bf16_bits(vals):
    return torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_int8_codes_of_exact_multiples():
    # x = k * s with s a power of two is exact in bf16, so the code is k itself
    k = np.arange(-127, 128, dtype=np.int64)
    for s in (1.0, 0.5, 2.0 ** -7, 8.0):
        x = _bf16_bits((k * s).reshape(-1, 1, 1))
        codes = oracle.quantize_int8(oracle.BF16, x, np.full((1, 1), s, np.float32))
        assert np.array_equal(codes.reshape(-1), k.astype(np.int8))


def test_int8_ties_to_even_and_clamp():
    vals = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.5, -127.5, 200.0, -300.0, 1e30]
    want = [0, 2, 2, 0, -2, -2, 126, 127, -127, 127, -127, 127]
    x = _bf16_bits(np.array(vals).reshape(-1, 1, 1))
    back = oracle.widen(oracle.BF16, x).reshape(-1)
    assert np.array_equal(back[:9], vals[:9])  # the tie cases are exact in bf16
    codes = oracle.quantize_int8(oracle.BF16, x, np.ones((1, 1), np.float32))
    assert codes.reshape(-1).tolist() == want


def test_int8_scale_per_channel():
    # every channel (h, d) gets its own power-of-two scale; the same value 1.0 in each
    # channel must come out as 1 / s[h, d]
    H, D = 3, 8
    e = (np.arange(H)[:, None] + np.arange(D)[None, :]) % 7
    scale = (2.0 ** -e).astype(np.float32)
    x = _bf16_bits(np.ones((2, H, D)))
    codes = oracle.quantize_int8(oracle.BF16, x, scale)
    assert np.array_equal(codes[0], (2 ** e).astype(np.int8)) and np.array_equal(codes[1],
                                                                               codes[0])


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_int8_attention_equals_plain_attention_on_exact_codes(dtype):
    # K and V values that are integers in [-127, 127] times per-channel power-of-two scales
    # are exact in both 16-bit formats, so quantising them loses nothing: attention over
    # the codes must equal attention over the 16-bit values bit for bit
    g = np.random.default_rng(3)
    n, Hq, Hkv, D = 40, 4, 2, 16
    e = g.integers(0, 6, (Hkv, D))
    ks, vs = (2.0 ** -e).astype(np.float32), (2.0 ** -((e + 3) % 6)).astype(np.float32)
    kc = g.integers(-127, 128, (n, Hkv, D))
    vc = g.integers(-127, 128, (n, Hkv, D))
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    bits = lambda a: torch.tensor(a, dtype=torch.float32).to(tdt).view(torch.int16).numpy() \
        .view(np.uint16)
    k, v = bits(kc * ks), bits(vc * vs)
    assert np.array_equal(oracle.quantize_int8(dtype, k, ks), kc.astype(np.int8))
    assert np.array_equal(oracle.quantize_int8(dtype, v, vs), vc.astype(np.int8))
    q = bits(g.standard_normal((7, Hq, D)))
    pos = np.array([0, 1, 5, 17, 30, 38, 39], np.int32)
    got = oracle.attention_rows_int8(dtype, q, pos, kc, vc, ks, vs, 0.3)
    want = oracle.attention_rows(dtype, q, pos, k, v, 0.3)
    assert np.array_equal(got, want)
