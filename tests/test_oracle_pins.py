"""Pins for the fp64 oracle against things other than itself.

* append: a pure-Python walk that addresses the pool as (page, offset)
  instead of the oracle's flat view; bit patterns compared, NaN payloads
  included.
* attention: pure-Python brute force that reads keys straight from the pool
  through block_table (no gather step), with math.exp.
* dense equivalence: torch's scaled_dot_product_attention (a library
  routine) in fp64 on the same tokens laid out contiguously, GQA through
  repeat_interleave, an explicit bottom-right causal mask.
* closed forms: one visible key, q = 0, constant V, two keys, scale = 0.
* invariants: physical page permutation, shared prefix pages == duplicated
  pages, NaN/Inf in dead slots, split + merge == whole.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import workloads as wl


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _paged_case(rng, lens, hq, hkv, d, ps, extra_pages=3, poison=np.nan):
    """Dense per-sequence K/V scattered into a permuted page pool by hand."""
    B = len(lens)
    need = [(L + ps - 1) // ps for L in lens]
    P = sum(need) + extra_pages
    perm = rng.permutation(P)
    kp = np.full((P, ps, hkv, d), poison)
    vp = np.full((P, ps, hkv, d), poison)
    mb = max(need) if need else 1
    bt = np.full((B, max(mb, 1)), -1, dtype=np.int64)
    dense_k, dense_v = [], []
    cur = 0
    for b, L in enumerate(lens):
        K = _rand(rng, L, hkv, d)
        V = _rand(rng, L, hkv, d)
        dense_k.append(K)
        dense_v.append(V)
        for m in range(need[b]):
            bt[b, m] = perm[cur]
            cur += 1
        for j in range(L):
            page, off = bt[b, j // ps], j % ps
            kp[page, off] = K[j]
            vp[page, off] = V[j]
    return kp, vp, bt, dense_k, dense_v


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

def _append_brute(kpool, vpool, key, value, slots):
    P, ps, hkv, d = kpool.shape
    kp = kpool.copy()
    vp = vpool.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        page, off = divmod(int(s), ps)
        for h in range(hkv):
            for e in range(d):
                kp[page, off, h, e] = key[t, h, e]
                vp[page, off, h, e] = value[t, h, e]
    return kp, vp


@pytest.mark.parametrize("dtype", [np.uint16, np.float32, np.float64])
def test_append_matches_page_offset_walk(dtype):
    rng = np.random.RandomState(11)
    P, ps, hkv, d = 9, 4, 3, 5
    kpool = (rng.randint(0, 60000, size=(P, ps, hkv, d))).astype(dtype)
    vpool = (rng.randint(0, 60000, size=(P, ps, hkv, d))).astype(dtype)
    if dtype != np.uint16:
        kpool[0, 1] = np.nan   # poisoned slots must survive untouched
    T = 13
    slots = rng.choice(P * ps, T, replace=False).astype(np.int64)
    slots[3] = -1          # padding token
    key = rng.randint(0, 60000, size=(T, hkv, d)).astype(dtype)
    value = rng.randint(0, 60000, size=(T, hkv, d)).astype(dtype)
    got_k, got_v = oracle.paged_kv_append(kpool, vpool, key, value, slots)
    exp_k, exp_v = _append_brute(kpool, vpool, key, value, slots)
    assert got_k.tobytes() == exp_k.tobytes()
    assert got_v.tobytes() == exp_v.tobytes()
    # the inputs are not modified
    assert not np.shares_memory(got_k, kpool)


def test_append_rejects_bad_slots():
    kp = np.zeros((2, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle.paged_kv_append(kp, kp, np.zeros((1, 1, 2)), np.zeros((1, 1, 2)), [8])
    with pytest.raises(ValueError):
        oracle.paged_kv_append(kp, kp, np.zeros((2, 1, 2)), np.zeros((2, 1, 2)), [3, 3])


# ---------------------------------------------------------------------------
# attention: brute force straight from the pool
# ---------------------------------------------------------------------------

def _attn_brute(kpool, vpool, q_rows, bt_row, L, n_new, scale, hkv):
    """Pure-Python loops; reads key j at pool[bt[j // ps], j % ps]."""
    ps = len(kpool[0])
    n, hq, d = len(q_rows), len(q_rows[0]), len(q_rows[0][0])
    G = hq // hkv
    out = [[[0.0] * d for _ in range(hq)] for _ in range(n)]
    for i in range(n):
        p = L - n_new + i
        for h in range(hq):
            hk = h // G
            ss = []
            for j in range(0, p + 1):
                page, off = int(bt_row[j // ps]), j % ps
                s = 0.0
                for e in range(d):
                    s += float(q_rows[i][h][e]) * float(kpool[page][off][hk][e])
                ss.append(scale * s)
            if not ss:
                continue
            mx = max(ss)
            ws = [math.exp(s - mx) for s in ss]
            tot = sum(ws)
            for e in range(d):
                acc = 0.0
                for j, w in enumerate(ws):
                    page, off = int(bt_row[j // ps]), j % ps
                    acc += w * float(vpool[page][off][hk][e])
                out[i][h][e] = acc / tot
    return np.array(out)


@pytest.mark.parametrize("hq,hkv", [(4, 2), (4, 4), (6, 1)])
def test_decode_bruteforce(hq, hkv):
    rng = np.random.RandomState(5)
    lens = [1, 7, 16, 23]
    ps, d = 4, 6
    kp, vp, bt, _, _ = _paged_case(rng, lens, hq, hkv, d, ps)
    q = _rand(rng, len(lens), hq, d)
    scale = 0.37
    got = oracle.paged_attention_decode(kp, vp, q, bt, lens, scale)
    for b, L in enumerate(lens):
        exp = _attn_brute(kp, vp, q[b:b + 1], bt[b], L, 1, scale, hkv)[0]
        np.testing.assert_allclose(got[b], exp, rtol=1e-12, atol=1e-12)


def test_prefill_bruteforce_with_cached_context():
    rng = np.random.RandomState(6)
    cached = [0, 5, 9]
    new = [3, 4, 1]
    lens = [c + n for c, n in zip(cached, new)]
    hq, hkv, d, ps = 4, 2, 5, 4
    kp, vp, bt, _, _ = _paged_case(rng, lens, hq, hkv, d, ps)
    qsl = np.concatenate([[0], np.cumsum(new)])
    q = _rand(rng, int(qsl[-1]), hq, d)
    got = oracle.paged_attention_prefill(kp, vp, q, qsl, bt, lens, 0.5)
    for b in range(3):
        rows = q[qsl[b]:qsl[b + 1]]
        exp = _attn_brute(kp, vp, rows, bt[b], lens[b], new[b], 0.5, hkv)
        np.testing.assert_allclose(got[qsl[b]:qsl[b + 1]], exp, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# dense equivalence against torch SDPA (fp64)
# ---------------------------------------------------------------------------

def _sdpa_dense(q_rows, K, V, n_new, scale):
    """torch SDPA over the contiguous tokens; bottom-right causal bool mask."""
    n, hq, d = q_rows.shape
    L, hkv, _ = K.shape
    G = hq // hkv
    qt = torch.from_numpy(q_rows).permute(1, 0, 2)                      # [Hq, n, D]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, L, D]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    pos = torch.arange(n) + (L - n_new)
    mask = torch.arange(L)[None, :] <= pos[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv,ps", [(8, 2, 16), (8, 1, 4), (3, 3, 8)])
def test_prefill_equals_dense_sdpa(hq, hkv, ps):
    rng = np.random.RandomState(7)
    cached = [0, 17, 40, 3]
    new = [9, 30, 1, 16]
    lens = [c + n for c, n in zip(cached, new)]
    d = 16
    kp, vp, bt, DK, DV = _paged_case(rng, lens, hq, hkv, d, ps)
    qsl = np.concatenate([[0], np.cumsum(new)])
    q = _rand(rng, int(qsl[-1]), hq, d)
    got = oracle.paged_attention_prefill(kp, vp, q, qsl, bt, lens, 0.29)
    for b in range(len(lens)):
        exp = _sdpa_dense(q[qsl[b]:qsl[b + 1]], DK[b], DV[b], new[b], 0.29)
        np.testing.assert_allclose(got[qsl[b]:qsl[b + 1]], exp, rtol=1e-10, atol=1e-12)


def test_decode_equals_dense_sdpa():
    rng = np.random.RandomState(8)
    lens = [1, 2, 33, 64, 100]
    hq, hkv, d, ps = 8, 2, 32, 16
    kp, vp, bt, DK, DV = _paged_case(rng, lens, hq, hkv, d, ps)
    q = _rand(rng, len(lens), hq, d)
    got = oracle.paged_attention_decode(kp, vp, q, bt, lens, 1 / math.sqrt(d))
    for b in range(len(lens)):
        exp = _sdpa_dense(q[b:b + 1], DK[b], DV[b], 1, 1 / math.sqrt(d))[0]
        np.testing.assert_allclose(got[b], exp, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_single_key_returns_its_value():
    rng = np.random.RandomState(9)
    kp, vp, bt, DK, DV = _paged_case(rng, [1], 4, 2, 8, 4)
    q = _rand(rng, 1, 4, 8)
    out = oracle.paged_attention_decode(kp, vp, q, bt, [1], 0.8)
    for h in range(4):
        assert np.array_equal(out[0, h], DV[0][0, h // 2])


def test_zero_query_is_mean_of_visible_values():
    rng = np.random.RandomState(10)
    lens = [13]
    kp, vp, bt, DK, DV = _paged_case(rng, lens, 2, 1, 4, 4)
    q = np.zeros((4, 2, 4))
    qsl = np.array([0, 4])
    out = oracle.paged_attention_prefill(kp, vp, q, qsl, bt, lens, 1.0)
    for i in range(4):
        p = 13 - 4 + i
        np.testing.assert_allclose(out[i, 0], DV[0][: p + 1, 0].mean(axis=0), rtol=1e-13)


def test_constant_values_and_scale_zero():
    rng = np.random.RandomState(12)
    kp, vp, bt, DK, DV = _paged_case(rng, [21], 2, 1, 3, 8)
    q = _rand(rng, 1, 2, 3)
    vconst = vp.copy()
    live = ~np.isnan(vconst)
    vconst[live] = 2.5
    out = oracle.paged_attention_decode(kp, vconst, q, bt, [21], 0.9)
    np.testing.assert_allclose(out, 2.5, rtol=1e-14)
    out0 = oracle.paged_attention_decode(kp, vp, q, bt, [21], 0.0)
    np.testing.assert_allclose(out0[0, 0], DV[0][:, 0].mean(axis=0), rtol=1e-13)


def test_two_keys_sigmoid():
    rng = np.random.RandomState(13)
    kp, vp, bt, DK, DV = _paged_case(rng, [2], 1, 1, 5, 16)
    q = _rand(rng, 1, 1, 5)
    sc = 0.61
    s0 = sc * float(q[0, 0] @ DK[0][0, 0])
    s1 = sc * float(q[0, 0] @ DK[0][1, 0])
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    exp = w0 * DV[0][0, 0] + (1 - w0) * DV[0][1, 0]
    out = oracle.paged_attention_decode(kp, vp, q, bt, [2], sc)
    np.testing.assert_allclose(out[0, 0], exp, rtol=1e-12)


def test_gqa_head_mapping_is_contiguous_groups():
    """Query heads 2,3 read KV head 1 when G = 2 (hq // G, not hq % Hkv)."""
    rng = np.random.RandomState(14)
    kp, vp, bt, DK, DV = _paged_case(rng, [9], 4, 2, 4, 4)
    v2 = vp.copy()
    live = ~np.isnan(v2[:, :, 1])
    v2[:, :, 1][live] = -3.0
    q = _rand(rng, 1, 4, 4)
    out = oracle.paged_attention_decode(kp, v2, q, bt, [9], 0.5)
    np.testing.assert_allclose(out[0, 2], -3.0, rtol=1e-14)
    np.testing.assert_allclose(out[0, 3], -3.0, rtol=1e-14)
    assert np.all(np.abs(out[0, 0] + 3.0) > 1e-3)


def test_first_new_token_without_context_sees_only_itself():
    rng = np.random.RandomState(15)
    kp, vp, bt, DK, DV = _paged_case(rng, [5], 2, 2, 4, 4)
    q = _rand(rng, 5, 2, 4)
    out = oracle.paged_attention_prefill(kp, vp, q, [0, 5], bt, [5], 0.7)
    np.testing.assert_array_equal(out[0, 1], DV[0][0, 1])


def test_empty_sequence_and_overlong_query_give_zero():
    rng = np.random.RandomState(16)
    kp, vp, bt, _, _ = _paged_case(rng, [3], 2, 1, 4, 4)
    q = _rand(rng, 1, 2, 4)
    assert np.all(oracle.paged_attention_decode(kp, vp, q, bt, [0], 1.0) == 0)
    q5 = _rand(rng, 5, 2, 4)
    out = oracle.paged_attention_prefill(kp, vp, q5, [0, 5], bt, [3], 1.0)
    assert np.all(out[:2] == 0) and np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_page_permutation_invariance_bit_identical():
    rng = np.random.RandomState(17)
    lens = [5, 40, 17]
    kp, vp, bt, _, _ = _paged_case(rng, lens, 4, 2, 8, 4)
    q = _rand(rng, 3, 4, 8)
    ref = oracle.paged_attention_decode(kp, vp, q, bt, lens, 0.3)
    P = kp.shape[0]
    pi = rng.permutation(P)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[pi] = kp
    vp2[pi] = vp
    bt2 = np.where(bt >= 0, pi[np.clip(bt, 0, None)], -1)
    got = oracle.paged_attention_decode(kp2, vp2, q, bt2, lens, 0.3)
    assert np.array_equal(ref, got)


def test_shared_prefix_equals_duplicated_pages():
    rng = np.random.RandomState(18)
    ps, hkv, d, hq = 4, 2, 8, 4
    prefix_pages, own = 3, 2
    B = 3
    P = prefix_pages + B * own
    kp = _rand(rng, P, ps, hkv, d)
    vp = _rand(rng, P, ps, hkv, d)
    bt_shared = np.array([[0, 1, 2, 3 + 2 * b, 4 + 2 * b] for b in range(B)])
    # duplicated: every sequence gets private copies of the prefix pages
    P2 = B * (prefix_pages + own)
    kp2 = np.empty((P2, ps, hkv, d))
    vp2 = np.empty((P2, ps, hkv, d))
    bt_dup = np.zeros_like(bt_shared)
    for b in range(B):
        for m in range(prefix_pages + own):
            dst = b * (prefix_pages + own) + m
            kp2[dst] = kp[bt_shared[b, m]]
            vp2[dst] = vp[bt_shared[b, m]]
            bt_dup[b, m] = dst
    lens = [19, 20, 17]
    q = _rand(rng, B, hq, d)
    a = oracle.paged_attention_decode(kp, vp, q, bt_shared, lens, 0.4)
    c = oracle.paged_attention_decode(kp2, vp2, q, bt_dup, lens, 0.4)
    assert np.array_equal(a, c)


@pytest.mark.parametrize("poison", [np.nan, np.inf, -np.inf])
def test_dead_slots_do_not_leak(poison):
    rng = np.random.RandomState(19)
    lens = [6, 13]
    kp, vp, bt, _, _ = _paged_case(rng, lens, 2, 1, 4, 4, poison=poison)
    kz = np.where(np.isfinite(kp), kp, 0.0)
    vz = np.where(np.isfinite(vp), vp, 0.0)
    q = _rand(rng, 2, 2, 4)
    a = oracle.paged_attention_decode(kp, vp, q, bt, lens, 0.5)
    b = oracle.paged_attention_decode(kz, vz, q, bt, lens, 0.5)
    assert np.all(np.isfinite(a)) and np.array_equal(a, b)


def test_split_and_merge_equals_whole():
    rng = np.random.RandomState(20)
    lens = [50, 7]
    kp, vp, bt, _, _ = _paged_case(rng, lens, 4, 2, 8, 4)
    q = _rand(rng, 2, 4, 8) * 3.0
    whole = oracle.paged_attention_decode(kp, vp, q, bt, lens, 0.7)
    cuts = [(0, 13), (13, 31), (31, 64)]
    parts = [oracle.paged_attention_decode_partial(kp, vp, q, bt, lens, 0.7, [c, c])
             for c in cuts]
    merged = oracle.merge_partials(parts)
    np.testing.assert_allclose(merged, whole, rtol=1e-12, atol=1e-13)


def test_scale_argument_vs_prescaled_query():
    rng = np.random.RandomState(21)
    lens = [30]
    kp, vp, bt, _, _ = _paged_case(rng, lens, 2, 1, 8, 8)
    q = _rand(rng, 1, 2, 8)
    a = oracle.paged_attention_decode(kp, vp, q, bt, lens, 0.37)
    b = oracle.paged_attention_decode(kp, vp, q * 0.37, bt, lens, 1.0)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    c = oracle.paged_attention_decode(kp, vp, q, bt, lens, 1.0)
    assert np.max(np.abs(a - c)) > 1e-3    # scale is not silently ignored


# ---------------------------------------------------------------------------
# the workload generator feeds consistent inputs
# ---------------------------------------------------------------------------

def test_workload_plans_are_consistent():
    for plan in [wl.gqa_decode_plan(batch=6, lo=10, hi=70), wl.shared_prefix_plan(batch=3,
                 prefix_pages=4, unique_pages=2), wl.chunked_prefill_plan(new=(5, 9),
                 cached=(0, 33)), wl.long_context_plan(hkv=1, batch=4, lo=20, hi=90),
                 *wl.tiny_f32_plans()]:
        ps = plan.page_size
        assert np.all(plan.seq_lens == plan.cached + plan.new)
        live = plan.slot_mapping[plan.slot_mapping >= 0]
        assert np.unique(live).size == live.size
        assert np.all(live < plan.num_pages * ps)
        for b in range(plan.batch):
            n = (int(plan.seq_lens[b]) + ps - 1) // ps
            row = plan.block_table[b, :n]
            assert np.all((row >= 0) & (row < plan.num_pages))
            assert np.unique(row).size == n
        assert plan.query_start_loc[-1] == plan.total_new


def test_workload_materialize_poisons_dead_slots():
    plan = wl.gqa_decode_plan(batch=3, lo=5, hi=40)
    st = wl.materialize(plan)
    live = wl.live_slot_mask(plan)
    P, ps = plan.num_pages, plan.page_size
    flat = st.key_pool.float().view(P * ps, -1)
    assert torch.isnan(flat[torch.from_numpy(~live)]).all()
    assert torch.isfinite(flat[torch.from_numpy(live)]).all()


def test_tiny_config_decode_after_prefill_oracle_chain():
    """Config 1 through the oracle: append 100, prefill, append 1, decode."""
    pf, dc = wl.tiny_f32_plans()
    s1 = wl.materialize(pf)
    kp, vp = oracle.paged_kv_append(s1.key_pool.numpy(), s1.value_pool.numpy(),
                                    s1.key.numpy(), s1.value.numpy(), pf.slot_mapping)
    o1 = oracle.paged_attention_prefill(kp.astype(np.float64), vp.astype(np.float64),
                                        s1.q.numpy(), pf.query_start_loc, pf.block_table,
                                        pf.seq_lens, pf.scale)
    assert np.all(np.isfinite(o1))
    s2 = wl.materialize(dc, key_pool=torch.from_numpy(kp), value_pool=torch.from_numpy(vp))
    kp2, vp2 = oracle.paged_kv_append(kp, vp, s2.key.numpy(), s2.value.numpy(),
                                      dc.slot_mapping)
    o2 = oracle.paged_attention_decode(kp2.astype(np.float64), vp2.astype(np.float64),
                                       s2.q.numpy(), dc.block_table, dc.seq_lens, dc.scale)
    assert np.all(np.isfinite(o2))
    # the decode token at position 100 lands in page block_table[6], offset 4
    assert dc.slot_mapping[0] == dc.block_table[0, 6] * 16 + 4


# ---------------------------------------------------------------------------
# cascade decode: a prefix shared by every sequence, then each one's own pages
# ---------------------------------------------------------------------------

def _cascade_case(rng, prefix_len, lens, hq, hkv, d, ps):
    """A pool holding one shared prefix and per-sequence suffixes (NaN elsewhere)."""
    npre = (prefix_len + ps - 1) // ps
    need = [(L + ps - 1) // ps for L in lens]
    P = npre + sum(need) + 2
    perm = rng.permutation(P)
    kp = np.full((P, ps, hkv, d), np.nan)
    vp = np.full((P, ps, hkv, d), np.nan)
    pre_ids = perm[:npre].copy()
    for j in range(prefix_len):
        kp[pre_ids[j // ps], j % ps] = _rand(rng, hkv, d)
        vp[pre_ids[j // ps], j % ps] = _rand(rng, hkv, d)
    bt = np.full((len(lens), max(max(need), 1)), -1, dtype=np.int64)
    cur = npre
    for b, L in enumerate(lens):
        for m in range(need[b]):
            bt[b, m] = perm[cur]
            cur += 1
        for j in range(L):
            kp[bt[b, j // ps], j % ps] = _rand(rng, hkv, d)
            vp[bt[b, j // ps], j % ps] = _rand(rng, hkv, d)
    return kp, vp, pre_ids, bt


def _cascade_brute(kp, vp, q_row, pre_ids, prefix_len, bt_row, L, scale, hkv):
    """Pure-Python loops: key j < prefix_len at pool[pre_ids[j // ps], j % ps],
    key prefix_len + i at pool[bt_row[i // ps], i % ps]."""
    ps = len(kp[0])
    hq, d = len(q_row), len(q_row[0])
    G = hq // hkv
    locs = [(int(pre_ids[j // ps]), j % ps) for j in range(prefix_len)]
    locs += [(int(bt_row[i // ps]), i % ps) for i in range(L)]
    out = [[0.0] * d for _ in range(hq)]
    for h in range(hq):
        hk = h // G
        ss = []
        for page, off in locs:
            s = 0.0
            for e in range(d):
                s += float(q_row[h][e]) * float(kp[page][off][hk][e])
            ss.append(scale * s)
        if not ss:
            continue
        mx = max(ss)
        ws = [math.exp(x - mx) for x in ss]
        tot = sum(ws)
        for e in range(d):
            acc = 0.0
            for w, (page, off) in zip(ws, locs):
                acc += w * float(vp[page][off][hk][e])
            out[h][e] = acc / tot
    return np.array(out)


@pytest.mark.parametrize("prefix_len", [0, 5, 8, 13])
def test_cascade_bruteforce(prefix_len):
    rng = np.random.RandomState(30 + prefix_len)
    ps, hq, hkv, d = 4, 4, 2, 6
    lens = [0, 3, 9]
    kp, vp, pre_ids, bt = _cascade_case(rng, prefix_len, lens, hq, hkv, d, ps)
    q = _rand(rng, len(lens), hq, d)
    got = oracle.paged_attention_decode_cascade(kp, vp, q, pre_ids, prefix_len, bt, lens, 0.45)
    for b, L in enumerate(lens):
        exp = _cascade_brute(kp, vp, q[b], pre_ids, prefix_len, bt[b], L, 0.45, hkv)
        np.testing.assert_allclose(got[b], exp, rtol=1e-12, atol=1e-12)


def test_cascade_equals_decode_on_concatenated_tables():
    """Page-aligned prefix: identical to plain decode over prefix pages ++ own pages."""
    rng = np.random.RandomState(41)
    ps, hq, hkv, d = 4, 8, 2, 8
    prefix_len, lens = 12, [1, 6, 11, 0]
    kp, vp, pre_ids, bt = _cascade_case(rng, prefix_len, lens, hq, hkv, d, ps)
    q = _rand(rng, len(lens), hq, d)
    full = np.concatenate([np.tile(pre_ids, (len(lens), 1)), bt], axis=1)
    a = oracle.paged_attention_decode_cascade(kp, vp, q, pre_ids, prefix_len, bt, lens, 0.3)
    c = oracle.paged_attention_decode(kp, vp, q, full, [prefix_len + L for L in lens], 0.3)
    assert np.array_equal(a, c)


def test_cascade_is_merge_of_prefix_and_suffix_partials():
    """The prefix attended once for all queries, merged with each suffix."""
    rng = np.random.RandomState(42)
    ps, hq, hkv, d = 4, 4, 1, 8
    prefix_len, lens = 10, [7, 2, 0]
    kp, vp, pre_ids, bt = _cascade_case(rng, prefix_len, lens, hq, hkv, d, ps)
    q = _rand(rng, len(lens), hq, d) * 2.0
    Kp = oracle.gather_pages(kp, pre_ids, prefix_len)
    Vp = oracle.gather_pages(vp, pre_ids, prefix_len)
    pre = oracle.attend_partial(q, Kp, Vp, [prefix_len - 1] * len(lens), 0.6)
    suf = oracle.paged_attention_decode_partial(kp, vp, q, bt, lens, 0.6, [(0, L) for L in lens])
    merged = oracle.merge_partials([pre, suf])
    whole = oracle.paged_attention_decode_cascade(kp, vp, q, pre_ids, prefix_len, bt, lens, 0.6)
    np.testing.assert_allclose(merged, whole, rtol=1e-12, atol=1e-13)


def test_cascade_degenerate_cases():
    rng = np.random.RandomState(43)
    ps, hq, hkv, d = 4, 2, 1, 4
    kp, vp, pre_ids, bt = _cascade_case(rng, 0, [5, 0], hq, hkv, d, ps)
    q = _rand(rng, 2, hq, d)
    # no prefix: plain decode; no prefix and no own tokens: 0
    a = oracle.paged_attention_decode_cascade(kp, vp, q, pre_ids, 0, bt, [5, 0], 0.5)
    np.testing.assert_array_equal(a[0], oracle.paged_attention_decode(kp, vp, q, bt, [5, 0], 0.5)[0])
    assert np.all(a[1] == 0.0)
    # prefix only (every own length 0): the prefix attention for every query
    kp, vp, pre_ids, bt = _cascade_case(rng, 6, [0, 0], hq, hkv, d, ps)
    a = oracle.paged_attention_decode_cascade(kp, vp, q, pre_ids, 6, bt, [0, 0], 0.5)
    Kp = oracle.gather_pages(kp, pre_ids, 6)
    Vp = oracle.gather_pages(vp, pre_ids, 6)
    exp = oracle.attend(q, Kp, Vp, [5, 5], 0.5)
    np.testing.assert_allclose(a, exp, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# CSR page tables (kv_indptr / kv_indices / kv_last_page_len)
# ---------------------------------------------------------------------------

def _to_csr(bt, lens, ps):
    """Dense block-table rows -> (kv_indptr, kv_indices, kv_last_page_len), by hand."""
    indptr, indices, last = [0], [], []
    for b, L in enumerate(lens):
        n = (L + ps - 1) // ps
        indices.extend(int(x) for x in bt[b, :n])
        indptr.append(len(indices))
        last.append(L - (n - 1) * ps if n else 0)
    return np.array(indptr), np.array(indices, dtype=np.int64), np.array(last)


def test_csr_decode_bruteforce_and_dense_equivalence():
    rng = np.random.RandomState(50)
    ps, hq, hkv, d = 4, 4, 2, 6
    lens = [1, 4, 9, 0, 16]                 # full last pages, a partial one, an empty sequence
    kp, vp, bt, DK, DV = _paged_case(rng, lens, hq, hkv, d, ps)
    ip, ix, last = _to_csr(bt, lens, ps)
    q = _rand(rng, len(lens), hq, d)
    got = oracle.paged_attention_decode_csr(kp, vp, q, ip, ix, last, 0.41)
    for b, L in enumerate(lens):
        pages, LL = oracle.csr_pages(ip, ix, last, ps, b)
        assert LL == L                      # the key count the tokens laid down define
        exp = _attn_brute(kp, vp, q[b:b + 1], bt[b], L, 1, 0.41, hkv)[0] if L else np.zeros((hq, d))
        np.testing.assert_allclose(got[b], exp, rtol=1e-12, atol=1e-12)
    dense = oracle.paged_attention_decode(kp, vp, q, bt, lens, 0.41)
    assert np.array_equal(got, dense)


def test_csr_prefill_equals_dense_sdpa():
    rng = np.random.RandomState(51)
    ps, hq, hkv, d = 8, 8, 2, 16
    cached, new = [0, 17, 40], [9, 30, 1]
    lens = [c + n for c, n in zip(cached, new)]
    kp, vp, bt, DK, DV = _paged_case(rng, lens, hq, hkv, d, ps)
    ip, ix, last = _to_csr(bt, lens, ps)
    qsl = np.concatenate([[0], np.cumsum(new)])
    q = _rand(rng, int(qsl[-1]), hq, d)
    got = oracle.paged_attention_prefill_csr(kp, vp, q, qsl, ip, ix, last, 0.33)
    for b in range(len(lens)):
        exp = _sdpa_dense(q[qsl[b]:qsl[b + 1]], DK[b], DV[b], new[b], 0.33)
        np.testing.assert_allclose(got[qsl[b]:qsl[b + 1]], exp, rtol=1e-10, atol=1e-12)


def test_csr_shared_pages_between_sequences():
    """Two sequences whose CSR slices list the same physical pages read the same keys."""
    rng = np.random.RandomState(52)
    ps, hq, hkv, d = 4, 2, 1, 4
    kp = _rand(rng, 6, ps, hkv, d)
    vp = _rand(rng, 6, ps, hkv, d)
    ip = np.array([0, 3, 6])
    ix = np.array([2, 0, 5, 2, 0, 5])
    last = np.array([3, 3])
    q = np.repeat(_rand(rng, 1, hq, d), 2, axis=0)
    out = oracle.paged_attention_decode_csr(kp, vp, q, ip, ix, last, 0.5)
    assert np.array_equal(out[0], out[1])
