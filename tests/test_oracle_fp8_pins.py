"""Pins of the fp8 (e4m3) oracle against what the format's definition and a
library conversion fix."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_fp8


def test_e4m3_closed_forms():
    vals = [1.0, -2.0, 448.0, 500.0, 1e30, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875,
            -0.0, 0.0, 2.0 ** -6, 0.875 * 2.0 ** -6, 240.0, 464.0, np.nan]
    want = [0x38, 0xC0, 0x7E, 0x7E, 0x7E, 0x01, 0x00, 0x02, 0x38, 0x3A,
            0x80, 0x00, 0x08, 0x07, 0x77, 0x7E, 0x7F]
    assert kv_fp8.e4m3_encode(np.array(vals, dtype=np.float32)).tolist() == want
    # the decoded values of the same codes
    got = kv_fp8.e4m3_decode(np.array([0x38, 0xC0, 0x7E, 0x01, 0x08, 0x07, 0x77], dtype=np.uint8))
    assert got.tolist() == [1.0, -2.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, 240.0]
    assert np.isnan(kv_fp8.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    v = kv_fp8.e4m3_decode(codes)
    ok = ~np.isnan(v)
    assert ok.sum() == 254
    assert np.array_equal(kv_fp8.e4m3_encode(v[ok].astype(np.float32)), codes[ok])
    # the grid is symmetric and strictly increasing over the positive codes
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0) and np.array_equal(-pos, v[0x80:0xFF])


def test_e4m3_matches_library_conversion_in_range():
    rng = np.random.RandomState(60)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (1e-3, 0.1, 1.0, 30.0, 150.0)])
    mids = (kv_fp8.e4m3_decode(np.arange(1, 0x7E)) + kv_fp8.e4m3_decode(np.arange(2, 0x7F))) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)      # exact ties between neighbours
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kv_fp8.e4m3_encode(x), ref)


def test_quantize_is_fp32_division_then_rounding():
    rng = np.random.RandomState(61)
    x = rng.standard_normal(5000).astype(np.float32)
    for scale in (1.0, 0.05, 3.0):
        q = kv_fp8.quantize(x, scale)
        exp = kv_fp8.e4m3_encode(x / np.float32(scale))
        assert np.array_equal(q, exp)
        # dequantised values are within half a grid step of x / scale
        back = kv_fp8.e4m3_decode(q)
        assert np.all(np.abs(back - x.astype(np.float64) / np.float32(scale)) <=
                      np.maximum(np.abs(back) / 16.0, 2.0 ** -10) + 1e-12)


def test_fp8_append_scatters_codes():
    rng = np.random.RandomState(62)
    P, ps, hkv, d = 5, 4, 2, 8
    kc = rng.randint(0, 256, size=(P, ps, hkv, d)).astype(np.uint8)
    vc = rng.randint(0, 256, size=(P, ps, hkv, d)).astype(np.uint8)
    key = rng.standard_normal((3, hkv, d)).astype(np.float32)
    value = rng.standard_normal((3, hkv, d)).astype(np.float32)
    slots = np.array([7, -1, 13])
    k2, v2 = kv_fp8.paged_kv_append_fp8(kc, vc, key, value, slots, 0.5, 2.0)
    assert np.array_equal(k2.reshape(P * ps, hkv, d)[7], kv_fp8.quantize(key[0], 0.5))
    assert np.array_equal(v2.reshape(P * ps, hkv, d)[13], kv_fp8.quantize(value[2], 2.0))
    mask = np.ones(P * ps, dtype=bool)
    mask[[7, 13]] = False
    assert np.array_equal(k2.reshape(P * ps, hkv, d)[mask], kc.reshape(P * ps, hkv, d)[mask])


def test_fp8_decode_is_decode_of_dequantised_pools():
    rng = np.random.RandomState(63)
    P, ps, hkv, d, hq = 6, 4, 2, 8, 4
    kc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), 0.25)
    vc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), 0.5)
    bt = np.array([[3, 1, 4], [0, 5, 2]])
    lens = [10, 7]
    q = rng.standard_normal((2, hq, d))
    got = kv_fp8.paged_attention_decode_fp8(kc, vc, 0.25, 0.5, q, bt, lens, 0.35)
    K = kv_fp8.e4m3_decode(kc) * 0.25
    V = kv_fp8.e4m3_decode(vc) * 0.5
    # the scales pull out: S = scale * k_scale * q.e4m3(K), O = v_scale * softmax(S) e4m3(V)
    K1, V1 = kv_fp8.e4m3_decode(kc), kv_fp8.e4m3_decode(vc)
    alt = oracle.paged_attention_decode(K1, V1, q, bt, lens, 0.35 * 0.25) * 0.5
    np.testing.assert_allclose(got, oracle.paged_attention_decode(K, V, q, bt, lens, 0.35), rtol=0, atol=0)
    np.testing.assert_allclose(got, alt, rtol=1e-12, atol=1e-13)


def test_quantize_matches_library_division_and_conversion():
    """quantize(x, s) against torch's own fp32 division and e4m3 conversion,
    independent of the oracle's encoder.  The inputs include values x whose
    fp32 quotient x / s falls on or next to a midpoint between two e4m3
    neighbours, where a division done in fp64 instead of fp32 (or a multiply
    by 1/s) rounds the other way."""
    rng = np.random.RandomState(64)
    grid = kv_fp8.e4m3_decode(np.arange(0, 0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    for s in (0.02, 0.03, 0.05, 0.3, 1.0, 3.0, 7.0 / 3.0):
        s32 = np.float32(s)
        near = (mids * np.float64(s32)).astype(np.float32)           # x / s lands on or by a tie
        x = np.concatenate([near, np.nextafter(near, np.float32(np.inf)),
                            np.nextafter(near, np.float32(-np.inf)),
                            rng.standard_normal(20000).astype(np.float32) * np.float32(40.0) * s32])
        x = np.concatenate([x, -x])
        x = x[np.abs(x / s32) <= 448.0]
        ref = (torch.from_numpy(x) / torch.tensor(s32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kv_fp8.quantize(x, s), ref), f"scale {s}"


def test_fp8_prefill_brute_force_on_codes():
    """Prefill over e4m3 pools against pure-Python loops that read every key's
    codes straight from the pools through block_table, decode them with the
    format's definition (sign, exponent bias 7, three mantissa bits) and scale
    them: no gather, no vectorised softmax."""
    rng = np.random.RandomState(65)
    P, ps, hkv, d, hq = 7, 4, 2, 4, 4
    ks, vs, scale = 0.125, 0.75, 0.6
    kc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), ks)
    vc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), vs)
    bt = np.array([[5, 2, 6], [1, 3, 0]])
    lens, new = [11, 6], [3, 6]
    qsl = np.array([0, 3, 9])
    q = rng.standard_normal((9, hq, d))
    got = kv_fp8.paged_attention_prefill_fp8(kc, vc, ks, vs, q, qsl, bt, lens, scale)

    def val(c):
        c = int(c)
        e, m = (c >> 3) & 0xF, c & 7
        mag = m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        return -mag if c & 0x80 else mag

    G = hq // hkv
    for b in range(2):
        for i in range(new[b]):
            r, pos = qsl[b] + i, lens[b] - new[b] + i
            for h in range(hq):
                s = []
                for j in range(pos + 1):
                    page, off = bt[b][j // ps], j % ps
                    s.append(scale * sum(q[r, h, x] * val(kc[page, off, h // G, x]) * ks for x in range(d)))
                mx = max(s)
                w = [np.exp(v - mx) for v in s]
                for x in range(d):
                    o = sum(w[j] * val(vc[bt[b][j // ps], j % ps, h // G, x]) * vs
                            for j in range(pos + 1)) / sum(w)
                    assert abs(got[r, h, x] - o) < 1e-12


def test_fp8_prefill_last_row_is_the_decode_and_scales_pull_out():
    """The newest token of a prefill sees every key: its row equals the fp8
    decode of that query; and k_scale / v_scale act as a scale on the softmax
    argument and on the output."""
    rng = np.random.RandomState(66)
    P, ps, hkv, d, hq = 8, 4, 1, 8, 4
    kc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), 0.5)
    vc = kv_fp8.quantize(rng.standard_normal((P, ps, hkv, d)), 0.25)
    bt = np.array([[7, 0, 4, 2]])
    q = rng.standard_normal((5, hq, d))
    qsl = np.array([0, 5])
    pre = kv_fp8.paged_attention_prefill_fp8(kc, vc, 0.5, 0.25, q, qsl, bt, [14], 0.3)
    dec = kv_fp8.paged_attention_decode_fp8(kc, vc, 0.5, 0.25, q[4:5], bt, [14], 0.3)
    np.testing.assert_allclose(pre[4], dec[0], rtol=0, atol=1e-15)
    alt = oracle.paged_attention_prefill(kv_fp8.e4m3_decode(kc), kv_fp8.e4m3_decode(vc), q, qsl, bt, [14],
                                         0.3 * 0.5) * 0.25
    np.testing.assert_allclose(pre, alt, rtol=1e-12, atol=1e-13)
