"""Pins of the oracle's one-call decode step (append, then decode).

onnxruntime/mobius PR #395 "Add paged / block-table KV cache export", "How it
works (per attention layer)": step 1 writes this step's K/V rows into the
pool at slot_mapping, step 2 attends.  ``oracle.paged_attention_decode_append``
states that order.  The checks below do not go through the oracle's own
append or gather: a single-key closed form on a NaN pool (any stale read or
attending before appending gives NaN or the wrong row), pure-Python loops
over dense per-sequence keys in which the new key exists only in the step's
input, and the no-new-token case.
"""
import math

import numpy as np

import oracle
from oracle import kv_fp8


def _case(rng, lens, hq, hkv, d, ps, extra_pages=3):
    """Pools holding keys 0 .. L-2 of each sequence (row L-1 left NaN), the
    dense keys 0 .. L-1, block tables and the slot of each last key."""
    B = len(lens)
    need = [(L + ps - 1) // ps for L in lens]
    P = sum(need) + extra_pages
    perm = rng.permutation(P)
    kp = np.full((P, ps, hkv, d), np.nan)
    vp = np.full((P, ps, hkv, d), np.nan)
    bt = np.full((B, max(max(need), 1)), -1, dtype=np.int64)
    K, V, slots = [], [], []
    cur = 0
    for b, L in enumerate(lens):
        Kb = rng.standard_normal((L, hkv, d))
        Vb = rng.standard_normal((L, hkv, d))
        K.append(Kb)
        V.append(Vb)
        for m in range(need[b]):
            bt[b, m] = perm[cur]
            cur += 1
        for j in range(L - 1):
            kp[bt[b, j // ps], j % ps] = Kb[j]
            vp[bt[b, j // ps], j % ps] = Vb[j]
        slots.append(int(bt[b, (L - 1) // ps]) * ps + (L - 1) % ps)
    new_k = np.stack([Kb[-1] for Kb in K])
    new_v = np.stack([Vb[-1] for Vb in V])
    return kp, vp, bt, K, V, new_k, new_v, np.array(slots, dtype=np.int64)


def _dense_brute(q, K, V, scale, hkv):
    """Softmax attention of one query row set over dense keys, in loops."""
    hq, d = len(q), len(q[0])
    G = hq // hkv
    out = [[0.0] * d for _ in range(hq)]
    for h in range(hq):
        hk = h // G
        ss = [scale * sum(float(q[h][e]) * float(K[j][hk][e]) for e in range(d)) for j in range(len(K))]
        mx = max(ss)
        ws = [math.exp(s - mx) for s in ss]
        tot = sum(ws)
        for e in range(d):
            out[h][e] = sum(w * float(V[j][hk][e]) for j, w in enumerate(ws)) / tot
    return np.array(out)


def test_fused_single_key_is_the_new_value():
    rng = np.random.RandomState(31)
    lens = [1, 1, 1]
    kp, vp, bt, K, V, nk, nv, slots = _case(rng, lens, 4, 2, 8, 4)
    q = rng.standard_normal((3, 4, 8))
    kp2, vp2, out = oracle.paged_attention_decode_append(kp, vp, nk, nv, slots, q, bt, lens, 0.7)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(out[b, h], nv[b, h // 2])
        page, off = divmod(int(slots[b]), 4)
        assert np.array_equal(kp2[page, off], nk[b]) and np.array_equal(vp2[page, off], nv[b])
    assert np.isnan(kp).sum() - np.isnan(kp2).sum() == nk.size  # exactly the new rows were written


def test_fused_bruteforce_new_key_only_in_the_input():
    rng = np.random.RandomState(32)
    lens = [1, 5, 8, 13]
    hq, hkv, d, ps = 6, 3, 5, 4
    kp, vp, bt, K, V, nk, nv, slots = _case(rng, lens, hq, hkv, d, ps)
    q = rng.standard_normal((len(lens), hq, d))
    _, _, out = oracle.paged_attention_decode_append(kp, vp, nk, nv, slots, q, bt, lens, 0.41)
    for b in range(len(lens)):
        np.testing.assert_allclose(out[b], _dense_brute(q[b], K[b], V[b], 0.41, hkv), rtol=1e-12, atol=1e-12)


def test_fused_without_new_token_leaves_pool_and_attends_existing_keys():
    rng = np.random.RandomState(33)
    lens = [4, 9]
    kp, vp, bt, K, V, nk, nv, slots = _case(rng, lens, 2, 1, 4, 4)
    q = rng.standard_normal((2, 2, 4))
    slots_none = np.array([-1, slots[1]], dtype=np.int64)
    lens_none = [lens[0] - 1, lens[1]]  # sequence 0 has no new token: its keys are 0 .. L-2
    kp2, vp2, out = oracle.paged_attention_decode_append(kp, vp, nk, nv, slots_none, q, bt, lens_none, 0.5)
    page, off = divmod(int(slots[0]), 4)
    assert np.all(np.isnan(kp2[page, off]))  # not written
    np.testing.assert_allclose(out[0], _dense_brute(q[0], K[0][:-1], V[0][:-1], 0.5, 1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[1], _dense_brute(q[1], K[1], V[1], 0.5, 1), rtol=1e-12, atol=1e-12)


def test_fused_fp8_single_key_is_the_quantised_new_value():
    rng = np.random.RandomState(34)
    P, ps, hkv, d = 6, 4, 2, 8
    kc = np.full((P, ps, hkv, d), 0x7F, dtype=np.uint8)  # every stale code is NaN
    vc = np.full((P, ps, hkv, d), 0x7F, dtype=np.uint8)
    nk = rng.standard_normal((2, hkv, d)).astype(np.float32)
    nv = rng.standard_normal((2, hkv, d)).astype(np.float32)
    bt = np.array([[3], [1]], dtype=np.int64)
    slots = np.array([3 * ps, 1 * ps], dtype=np.int64)
    q = rng.standard_normal((2, 4, d))
    ks, vs = 0.02, 0.03
    _, _, out = kv_fp8.paged_attention_decode_append_fp8(kc, vc, nk, nv, slots, ks, vs, q, bt, [1, 1], 0.9)
    # the closed form, with the e4m3 grid written out: code = RNE(x / s) on the
    # e4m3 grid, value = code * s
    for b in range(2):
        for h in range(4):
            x = nv[b, h // 2].astype(np.float32) / np.float32(vs)
            exp = kv_fp8.e4m3_decode(kv_fp8.e4m3_encode(x)) * vs
            assert np.array_equal(out[b, h], exp)
