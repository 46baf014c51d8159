"""FP8 (e4m3) KV pools, stated plainly (test oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Imports: numpy.

The pages name an fp8 KV cache (the fp8-kv-cache build feature of
onnxruntime/mobius PR #395 "Add paged / block-table KV cache export", and the
fp8 element sizes of the pool-sizing table of ROCm/maxtext PR #93 "[Draft] kv
paged kernels") without fixing a scheme.  Readings taken here, the
plainest that fit the rest of the pages:

1. Element format: OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits
   (bias 7), 3 mantissa bits, no infinities, 0x7F / 0xFF are NaN, largest
   finite magnitude 448.
2. One scale per pool and tensor (k_scale, v_scale): a stored code c stands
   for e4m3(c) * scale.
3. Append quantises each new element x (given as bf16) as
   code = e4m3_rn_satfinite(float32(x) / float32(scale)): the division in
   fp32 (IEEE, correctly rounded), then round to nearest even onto the e4m3
   grid, magnitudes past 448 saturating to 448, NaN staying NaN.
4. Attention reads K = e4m3(code) * k_scale and V = e4m3(code) * v_scale and
   is otherwise the attention of paged_attention.py.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import paged_attention_decode, paged_attention_prefill

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Value of each e4m3 code (uint8) as fp64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** -9                                  # e == 0: subnormal m/8 * 2^-6
    nrm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    v = np.where(e == 0, sub, nrm) * sign
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def e4m3_encode(x):
    """Round fp32 values onto the e4m3 grid (nearest, ties to even), saturating
    finite magnitudes above 448 to 448; NaN -> 0x7F.  Returns uint8 codes."""
    a32 = np.asarray(x, dtype=np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        return _e4m3_encode(a32.astype(np.float64))      # fp32 -> fp64 is exact


def _e4m3_encode(v):
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.int64)
    a = np.abs(v)
    code = np.zeros(v.shape, dtype=np.int64)
    # normal range: a = f * 2^E with f in [0.5, 1): exponent e = E - 1, quantum 2^(e-3)
    f, E = np.frexp(np.where(a > 0, a, 1.0))
    e = E.astype(np.int64) - 1
    normal = a >= 2.0 ** -6
    q_exp = np.where(normal, e - 3, -9)                  # subnormals share the quantum 2^-9
    n = np.rint(a / np.exp2(q_exp.astype(np.float64)))   # np.rint: ties to even
    n = np.where(np.isfinite(n), n, 0).astype(np.int64)
    # normal: n in [8, 16]; 16 means the next binade
    e_n = np.where(n >= 16, e + 1, e)
    n_n = np.where(n >= 16, 8, n)
    normal_code = ((e_n + 7) << 3) | (n_n - 8)
    # subnormal: n in [0, 8]; 8 is the smallest normal, whose code is 0x08 as well
    code = np.where(normal, normal_code, n)
    code = np.where(a > E4M3_MAX, 0x7E, code)
    code = code | sign
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def quantize(x, scale):
    """Codes of x (any float array) on a pool with the given scale: fp32
    division by the scale, then e4m3 rounding (reading 3 above)."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q)


def dequantize(codes, scale):
    """fp64 values a pool's codes stand for (reading 2)."""
    return e4m3_decode(codes) * float(scale)


def paged_kv_append_fp8(key_codes, value_codes, key, value, slot_mapping, k_scale, v_scale):
    """ScatterND of the quantised new rows into uint8 pools (copies returned):
    the append of mobius PR #395 ("How it works", step 1) with the element
    conversion of reading 3."""
    key_codes = np.asarray(key_codes, dtype=np.uint8)
    value_codes = np.asarray(value_codes, dtype=np.uint8)
    P, ps, hkv, d = key_codes.shape
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    kq = quantize(np.asarray(key, dtype=np.float32).reshape(slots.shape[0], hkv, d), k_scale)
    vq = quantize(np.asarray(value, dtype=np.float32).reshape(slots.shape[0], hkv, d), v_scale)
    live = slots[slots >= 0]
    if np.any(live >= P * ps):
        raise ValueError("slot_mapping entry out of range")
    if np.unique(live).shape[0] != live.shape[0]:
        raise ValueError("duplicate slot in one append")
    kc = key_codes.copy()
    vc = value_codes.copy()
    kf = kc.reshape(P * ps, hkv, d)
    vf = vc.reshape(P * ps, hkv, d)
    for t in range(slots.shape[0]):
        if slots[t] >= 0:
            kf[slots[t]] = kq[t]
            vf[slots[t]] = vq[t]
    return kc, vc


def paged_attention_decode_fp8(key_codes, value_codes, k_scale, v_scale, q, block_table, seq_lens,
                               scale, seqs=None):
    """Decode over e4m3 pools: the plain decode on the values the codes stand for."""
    return paged_attention_decode(dequantize(key_codes, k_scale), dequantize(value_codes, v_scale), q,
                                  block_table, seq_lens, scale, seqs=seqs)


def paged_attention_prefill_fp8(key_codes, value_codes, k_scale, v_scale, q, query_start_loc, block_table,
                                seq_lens, scale, rows=None):
    """Varlen causal prefill over e4m3 pools: the plain prefill (token i of
    sequence b at position L_b - n_b + i sees keys 0..that position) on the
    values the codes stand for (reading 4)."""
    return paged_attention_prefill(dequantize(key_codes, k_scale), dequantize(value_codes, v_scale), q,
                                   query_start_loc, block_table, seq_lens, scale, rows=rows)


def paged_attention_decode_append_fp8(key_codes, value_codes, key, value, slot_mapping, k_scale, v_scale,
                                      q, block_table, seq_lens, scale, seqs=None):
    """One decode step on e4m3 pools as one call: the quantising append of
    this step's rows, then decode over the values the codes stand for.
    Returns ``(key_codes', value_codes', out)``."""
    kc, vc = paged_kv_append_fp8(key_codes, value_codes, key, value, slot_mapping, k_scale, v_scale)
    return kc, vc, paged_attention_decode_fp8(kc, vc, k_scale, v_scale, q, block_table, seq_lens, scale,
                                              seqs=seqs)
