"""GPU parity: the C-ABI CUDA path against the fp64 oracle on the same
seeded inputs.

* append: the whole pool bit-exact (full-size pools: bit-exact on the
  written rows, untouched elsewhere, checked on the device);
* attention: max-abs <= 2e-2 and mean-abs <= 2e-3 for bf16, max-abs <= 1e-5
  for fp32, against the fp64 oracle;
* every pool slot that holds no live token is NaN (or +-Inf), so a read past
  seq_len or of a stale page shows up as a non-finite output.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import (assert_close, bits, compact_subset, gpu_step, oracle_step, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    build_mod.build()
    capi.lib()
    capi.device_error()  # clear


def _check_step(plan, device, where, seqs=None, rows=None, poison=float("nan")):
    st = wl.materialize(plan, device, poison=poison)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st, seqs=seqs, rows=rows)
    assert bits(kp).tobytes() == kb.tobytes(), f"{where}: key pool differs after append"
    assert bits(vp).tobytes() == vb.tobytes(), f"{where}: value pool differs after append"
    if plan.kind == "decode" and seqs is not None:
        r = list(seqs)
    else:
        r = None if rows is None else sorted(rows)
    res = assert_close(out, exp, plan.dtype, where, rows=r)
    assert capi.device_error() == (0, 0)
    return res


# ---------------------------------------------------------------------------
# configs at full size
# ---------------------------------------------------------------------------

def test_tiny_f32_prefill_then_decode(cuda_device):
    """Append 100, prefill, append 1, decode -- GPU chain vs oracle chain."""
    pf, dc = wl.tiny_f32_plans()
    s1 = wl.materialize(pf, cuda_device)
    kp, vp, out1 = gpu_step(s1)
    kb, vb, exp1 = oracle_step(s1)
    assert bits(kp).tobytes() == kb.tobytes()
    assert_close(out1, exp1, "f32", "tiny prefill")
    s2 = wl.materialize(dc, cuda_device, key_pool=kp, value_pool=vp)
    kp2, vp2, out2 = gpu_step(s2)
    kb2, vb2, exp2 = oracle_step(s2)
    assert bits(kp2).tobytes() == kb2.tobytes() and bits(vp2).tobytes() == vb2.tobytes()
    assert_close(out2, exp2, "f32", "tiny decode")


def test_gqa_decode_full(cuda_device):
    _check_step(wl.gqa_decode_plan(), cuda_device, "gqa_decode")


def test_shared_prefix_full(cuda_device):
    _check_step(wl.shared_prefix_plan(), cuda_device, "shared_prefix")


def test_chunked_prefill_full_every_row(cuda_device):
    """Config 4 at full size: the pools bit-exact after the append, and every
    one of the 10,496 rows (x 32 heads) against the oracle, which computes
    them sequence by sequence in chunks of 256 rows to bound its memory."""
    plan = wl.chunked_prefill_plan()
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value),
                                    plan.slot_mapping)
    assert bits(kp).tobytes() == kb.tobytes(), "chunked_prefill: key pool differs after append"
    assert bits(vp).tobytes() == vb.tobytes(), "chunked_prefill: value pool differs after append"
    K, V, q = to_f64(kb), to_f64(vb), to_f64(bits(st.q))
    exp = np.zeros(q.shape, dtype=np.float64)
    qsl = plan.query_start_loc
    for b in range(plan.batch):
        for r0 in range(int(qsl[b]), int(qsl[b + 1]), 256):
            rows = range(r0, min(r0 + 256, int(qsl[b + 1])))
            part = oracle.paged_attention_prefill(K, V, q, qsl, plan.block_table, plan.seq_lens, plan.scale,
                                                  rows=rows)
            exp[list(rows)] = part[list(rows)]
    assert_close(out, exp, "bf16", "chunked_prefill, every row")
    assert capi.device_error() == (0, 0)


def test_chunked_prefill_small_full_rows(cuda_device):
    plan = wl.chunked_prefill_plan(new=(64, 100, 1, 17, 250), cached=(0, 300, 47, 0, 33), seed=31)
    _check_step(plan, cuda_device, "chunked_prefill_small")


@pytest.mark.parametrize("hkv", [8, 1])
def test_long_context_full_every_sequence(cuda_device, hkv):
    """Config 5 at full size (256 sequences, contexts U[1024, 32768], the
    pool ~19 GB for 8 KV heads): the append checked on the device (written
    rows equal the new rows, every other slot untouched), then every
    sequence's output against the oracle.  The oracle runs on 16 sequences
    at a time, each batch on a host copy of only the pages it reads."""
    plan = wl.long_context_plan(hkv=hkv, seed=4 if hkv == 8 else 5)
    st = wl.materialize(plan, cuda_device)
    kp0 = st.key_pool
    kp, vp, out = gpu_step(st)
    P, ps = plan.num_pages, plan.page_size
    slots = st.slot_mapping
    assert torch.equal(kp.view(P * ps, -1)[slots].view(torch.int16),
                       st.key.view(len(slots), -1).view(torch.int16))
    assert torch.equal(vp.view(P * ps, -1)[slots].view(torch.int16),
                       st.value.view(len(slots), -1).view(torch.int16))
    mask = torch.ones(P * ps, dtype=torch.bool, device=cuda_device)
    mask[slots] = False
    assert torch.equal(kp.view(P * ps, -1)[mask].view(torch.int16),
                       kp0.view(P * ps, -1)[mask].view(torch.int16))
    del kp0, mask
    assert capi.device_error() == (0, 0)
    q_all = to_f64(bits(st.q))
    got_all = to_f64(bits(out))
    exp_all = np.zeros_like(q_all)
    for s0 in range(0, plan.batch, 16):
        seqs = list(range(s0, min(s0 + 16, plan.batch)))
        kpc, vpc, btc, slc, key_rows = compact_subset(st, seqs)
        kb, vb = oracle.paged_kv_append(kpc, vpc, bits(st.key)[key_rows], bits(st.value)[key_rows], slc)
        exp_all[seqs] = oracle.paged_attention_decode(to_f64(kb), to_f64(vb), q_all[seqs], btc,
                                                      plan.seq_lens[seqs], plan.scale)
        del kpc, vpc, kb, vb
    assert np.all(np.isfinite(got_all)), f"long hkv={hkv}: non-finite output"
    err = np.abs(got_all - exp_all)
    assert err.max() <= 2e-2, f"long hkv={hkv}: max abs {err.max():.3e}"
    assert err.mean() <= 2e-3, f"long hkv={hkv}: mean abs {err.mean():.3e}"
    # per sequence too: no sequence may hide behind the batch mean
    per_seq = err.reshape(plan.batch, -1).mean(axis=1)
    assert per_seq.max() <= 2e-3, f"long hkv={hkv}: sequence {int(per_seq.argmax())} mean abs {per_seq.max():.3e}"


# ---------------------------------------------------------------------------
# ragged, edge and degenerate cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (32, 8), (16, 1), (32, 1), (6, 3), (64, 2), (128, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_groups_and_head_dims(cuda_device, hq, hkv, d):
    lens = [1, 15, 16, 17, 31, 33, 100, 257, 1000]
    plan = wl.plan_from_lengths(f"dec_{hq}_{hkv}_{d}", "decode", "bf16", hq, hkv, d, 16,
                                np.array(lens) - 1, np.ones(len(lens)), seed=hq * 100 + hkv + d)
    _check_step(plan, cuda_device, plan.name)


def test_decode_32_row_groups_weighted_cut(cuda_device):
    """32 query heads per KV head with 4 KV heads (one box of 4): enough
    blocks per CTA that segment changes weigh in the cut of the units (the
    plain cut is used for the smaller shapes above)."""
    lens = np.full(32, 1000) + np.arange(32) * 37
    plan = wl.plan_from_lengths("dec_128_4_weighted", "decode", "bf16", 128, 4, 128, 16,
                                lens - 1, np.ones(32), seed=4141)
    _check_step(plan, cuda_device, plan.name)


def test_decode_16_row_groups_weighted_cut(cuda_device):
    """32/8 heads, d 128, 24 sequences (few enough that each spans several
    CTA ranges: segment changes weigh in the cut and a publisher warp counts
    the parts), with empty, one-key and one-page sequences between long ones."""
    rng = np.random.RandomState(77)
    lens = rng.randint(600, 5000, size=24)
    lens[[3, 11, 20]] = 0
    lens[[5, 17]] = 1
    lens[8] = 16
    plan = wl.plan_from_lengths("dec_16_rows_weighted", "decode", "bf16", 32, 8, 128, 16,
                                np.maximum(lens - 1, 0), (lens > 0).astype(int), seed=4242)
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert_close(out, exp, "bf16", plan.name)
    assert torch.all(out[3] == 0) and torch.all(out[11] == 0) and torch.all(out[20] == 0)


@pytest.mark.parametrize("ps", [8, 32, 64, 256])
def test_decode_page_sizes(cuda_device, ps):
    lens = [3, 64, 65, 190, 511]
    plan = wl.plan_from_lengths(f"dec_ps{ps}", "decode", "bf16", 32, 8, 128, ps,
                                np.array(lens) - 1, np.ones(len(lens)), seed=ps)
    _check_step(plan, cuda_device, plan.name)


def test_decode_with_empty_sequence(cuda_device):
    lens = np.array([0, 5, 0, 40])
    plan = wl.plan_from_lengths("dec_empty", "decode", "bf16", 8, 2, 128, 16,
                                np.maximum(lens - 1, 0), (lens > 0).astype(int), seed=3)
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert_close(out, exp, "bf16", "dec_empty")
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)


@pytest.mark.parametrize("poison", [float("inf"), float("-inf")])
def test_decode_inf_poison(cuda_device, poison):
    plan = wl.gqa_decode_plan(batch=7, lo=20, hi=300, seed=9)
    _check_step(plan, cuda_device, "inf poison", poison=poison)


def test_decode_large_batch_short_contexts(cuda_device):
    # many more (sequence, head) pairs than CTAs: most pairs complete in one CTA
    plan = wl.gqa_decode_plan(batch=600, lo=1, hi=40, seed=12)
    _check_step(plan, cuda_device, "dec_many_short")


def test_decode_scale_is_an_argument(cuda_device):
    plan = wl.gqa_decode_plan(batch=4, lo=30, hi=200, seed=5)
    plan.scale = 0.37
    st = wl.materialize(plan, cuda_device)
    _, _, a = gpu_step(st)
    st.q = (st.q.float() * 0.37).to(torch.bfloat16)
    plan.scale = 1.0
    kb, vb, exp = oracle_step(st)
    _, _, b = gpu_step(st)
    assert_close(b, exp, "bf16", "prescaled q, scale=1")
    # a (scale 0.37 on unscaled q) and b (pre-scaled q) agree within bf16 noise
    assert (a.float() - b.float()).abs().max().item() < 3e-2


def test_decode_max_seq_len_bound_is_only_a_bound(cuda_device):
    plan = wl.gqa_decode_plan(batch=9, lo=10, hi=500, seed=21)
    st = wl.materialize(plan, cuda_device)
    _, _, a = gpu_step(st, max_seq_len=plan.max_blocks * plan.page_size)
    _, _, b = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert_close(a, exp, "bf16", "loose bound")
    assert_close(b, exp, "bf16", "tight bound")


def test_decode_page_permutation_gives_identical_output(cuda_device):
    plan = wl.gqa_decode_plan(batch=8, lo=50, hi=700, seed=14)
    st = wl.materialize(plan, cuda_device)
    kp, vp, a = gpu_step(st)
    P = plan.num_pages
    pi = torch.randperm(P, generator=torch.Generator().manual_seed(3))
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[pi.to(cuda_device)] = kp
    vp2[pi.to(cuda_device)] = vp
    bt = st.block_table.long()
    bt2 = torch.where((bt >= 0) & (bt < P), pi.to(cuda_device)[bt.clamp(0, P - 1)], bt).int()
    b = capi.paged_attention_decode(kp2, vp2, st.q, bt2, st.seq_lens, plan.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_equals_duplicated_pages_on_gpu(cuda_device):
    shared = wl.shared_prefix_plan(batch=6, prefix_pages=20, unique_pages=3, seed=8)
    st = wl.materialize(shared, cuda_device)
    kp, vp, a = gpu_step(st)
    # duplicate the prefix pages per sequence
    ps = shared.page_size
    rows = []
    bt_dup = torch.full_like(st.block_table, -1)
    for b in range(shared.batch):
        n = (int(shared.seq_lens[b]) + ps - 1) // ps
        for m in range(n):
            bt_dup[b, m] = len(rows)
            rows.append(int(shared.block_table[b, m]))
    idx = torch.tensor(rows, device=cuda_device)
    kd, vd = kp[idx].contiguous(), vp[idx].contiguous()
    b_out = capi.paged_attention_decode(kd, vd, st.q, bt_dup, st.seq_lens, shared.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b_out.view(torch.int16))


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 1, 128), (4, 4, 64), (32, 1, 128)])
def test_prefill_ragged(cuda_device, hq, hkv, d):
    plan = wl.chunked_prefill_plan(new=(1, 7, 16, 65, 130, 3), cached=(0, 9, 100, 0, 31, 500),
                                   seed=hq + hkv + d, hq=hq, hkv=hkv, d=d)
    _check_step(plan, cuda_device, f"prefill {hq}/{hkv}/{d}")


@pytest.mark.parametrize("ps", [8, 32, 64, 256])
def test_prefill_page_sizes(cuda_device, ps):
    plan = wl.chunked_prefill_plan(new=(33, 90, 1), cached=(5, 64, 200), seed=ps, ps=ps)
    _check_step(plan, cuda_device, f"prefill ps={ps}")


def test_prefill_row_without_keys_is_zero(cuda_device):
    """n_b > L_b: the first n_b - L_b rows see no key (invalid input) -> 0."""
    plan = wl.chunked_prefill_plan(new=(6,), cached=(0,), seed=2)
    st = wl.materialize(plan, cuda_device)
    st.seq_lens = torch.tensor([4], dtype=torch.int32, device=cuda_device)
    plan_l = plan
    kp, vp, out = gpu_step(st)
    kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key),
                                    bits(st.value), plan.slot_mapping)
    exp = oracle.paged_attention_prefill(to_f64(kb), to_f64(vb), to_f64(bits(st.q)),
                                         plan_l.query_start_loc, plan_l.block_table, [4],
                                         plan_l.scale)
    assert_close(out, exp, "bf16", "rows without keys")
    assert torch.all(out[:2] == 0)


def test_append_padding_slots_and_determinism(cuda_device):
    plan = wl.chunked_prefill_plan(new=(40, 9), cached=(3, 0), seed=4)
    st = wl.materialize(plan, cuda_device)
    st.slot_mapping[5] = -1
    plan.slot_mapping = plan.slot_mapping.copy()
    plan.slot_mapping[5] = -1
    kp1, vp1 = st.key_pool.clone(), st.value_pool.clone()
    kp2, vp2 = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp1, vp1, st.key, st.value, st.slot_mapping)
    capi.paged_kv_append(kp2, vp2, st.key, st.value, st.slot_mapping)
    torch.cuda.synchronize()
    kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key),
                                    bits(st.value), plan.slot_mapping)
    assert bits(kp1).tobytes() == kb.tobytes() and bits(vp1).tobytes() == vb.tobytes()
    assert bits(kp1).tobytes() == bits(kp2).tobytes()


def test_append_f32_and_odd_row_bytes(cuda_device):
    """fp32 pool with head_dim 3 (12-byte rows: no 16-byte vectors)."""
    kp = torch.randn(10, 4, 1, 3, device=cuda_device)
    vp = torch.randn(10, 4, 1, 3, device=cuda_device)
    key = torch.randn(5, 1, 3, device=cuda_device)
    val = torch.randn(5, 1, 3, device=cuda_device)
    slots = torch.tensor([0, 39, 7, -1, 20], device=cuda_device)
    k2, v2 = kp.clone(), vp.clone()
    capi.paged_kv_append(k2, v2, key, val, slots)
    torch.cuda.synchronize()
    kb, vb = oracle.paged_kv_append(bits(kp), bits(vp), bits(key), bits(val), slots.cpu().numpy())
    assert bits(k2).tobytes() == kb.tobytes() and bits(v2).tobytes() == vb.tobytes()


def test_device_error_word_reports_bad_indices(cuda_device):
    plan = wl.gqa_decode_plan(batch=3, lo=20, hi=60, seed=2)
    st = wl.materialize(plan, cuda_device)
    capi.device_error()
    bad = st.slot_mapping.clone()
    bad[1] = plan.num_pages * plan.page_size + 5
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp, vp, st.key, st.value, bad)
    assert capi.device_error() == (2, plan.num_pages * plan.page_size + 5)
    bt = st.block_table.clone()
    bt[0, 0] = plan.num_pages + 100
    capi.paged_attention_decode(kp, vp, st.q, bt, st.seq_lens, plan.scale)
    code, detail = capi.device_error()
    assert code == 1 and detail == plan.num_pages + 100
    sl = st.seq_lens.clone()
    sl[2] = plan.max_blocks * plan.page_size + 1
    capi.paged_attention_decode(kp, vp, st.q, st.block_table, sl, plan.scale)
    assert capi.device_error()[0] == 3
