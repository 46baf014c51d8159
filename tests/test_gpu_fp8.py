"""GPU parity for e4m3 (fp8) KV pools: the quantising append bit-exact against
the oracle's quantiser, and decode against the oracle's attention over the
values the codes stand for.  The cached tokens' codes are written on the host
by the oracle; dead slots hold the NaN code, so any read of one shows up as a
non-finite output."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_fp8
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, to_f64

pytestmark = pytest.mark.gpu

KS, VS = 0.02, 0.03


def _fp8_step(plan, device, ks=KS, vs=VS):
    """(device e4m3 pools after the GPU append, host codes after the oracle append, state)."""
    st = wl.materialize(plan, device)
    kc0 = kv_fp8.quantize(to_f64(bits(st.key_pool)), ks)        # NaN (dead slots) -> 0x7F
    vc0 = kv_fp8.quantize(to_f64(bits(st.value_pool)), vs)
    kp = torch.from_numpy(kc0).to(device).view(torch.float8_e4m3fn)
    vp = torch.from_numpy(vc0).to(device).view(torch.float8_e4m3fn)
    if plan.total_new:
        capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping, k_scale=ks, v_scale=vs)
        kc, vc = kv_fp8.paged_kv_append_fp8(kc0, vc0, to_f64(bits(st.key)).astype(np.float32),
                                            to_f64(bits(st.value)).astype(np.float32), plan.slot_mapping, ks, vs)
    else:
        kc, vc = kc0, vc0
    torch.cuda.synchronize()
    return kp, vp, kc, vc, st


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


@pytest.mark.parametrize("name", ["gqa_decode", "long_small"])
def test_fp8_append_and_decode(cuda_device, name):
    plan = (wl.gqa_decode_plan() if name == "gqa_decode" else
            wl.long_context_plan(hkv=8, batch=12, lo=1000, hi=9000, seed=11))
    kp, vp, kc, vc, st = _fp8_step(plan, cuda_device)
    assert np.array_equal(_codes(kp), kc) and np.array_equal(_codes(vp), vc)   # append: every byte
    out = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                      max_seq_len=int(plan.seq_lens.max()), k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    exp = kv_fp8.paged_attention_decode_fp8(kc, vc, KS, VS, to_f64(bits(st.q)), plan.block_table, plan.seq_lens,
                                            plan.scale)
    assert_close(out, exp, "bf16", f"fp8 decode {name}")   # every sequence


@pytest.mark.parametrize("hq,hkv,d,ps", [(32, 1, 128, 16), (16, 4, 64, 8), (8, 8, 128, 64), (32, 8, 64, 16)])
def test_fp8_decode_ragged(cuda_device, hq, hkv, d, ps):
    lens = np.array([1, 15, 16, 17, 300, 2049, 64])
    plan = wl.plan_from_lengths(f"fp8_{hq}_{hkv}_{d}_{ps}", "decode", "bf16", hq, hkv, d, ps, lens - 1,
                                np.ones(len(lens)), seed=hq + d + ps, extra_free_pages=4)
    kp, vp, kc, vc, st = _fp8_step(plan, cuda_device, ks=0.05, vs=0.01)
    assert np.array_equal(_codes(kp), kc) and np.array_equal(_codes(vp), vc)
    out = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                      max_seq_len=int(lens.max()), k_scale=0.05, v_scale=0.01)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    exp = kv_fp8.paged_attention_decode_fp8(kc, vc, 0.05, 0.01, to_f64(bits(st.q)), plan.block_table,
                                            plan.seq_lens, plan.scale)
    assert_close(out, exp, "bf16", f"fp8 decode {hq}/{hkv}/{d} ps{ps}")


def test_fp8_decode_32_row_groups_weighted_cut(cuda_device):
    lens = np.full(32, 3000) + np.arange(32) * 7   # ~190 blocks a sequence on 1 KV head
    plan = wl.plan_from_lengths("fp8_mqa_weighted", "decode", "bf16", 32, 1, 128, 16, lens - 1,
                                np.ones(32), seed=49, extra_free_pages=4)
    kp, vp, kc, vc, st = _fp8_step(plan, cuda_device, ks=0.02, vs=0.03)
    out = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                      max_seq_len=int(lens.max()), k_scale=0.02, v_scale=0.03)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    exp = kv_fp8.paged_attention_decode_fp8(kc, vc, 0.02, 0.03, to_f64(bits(st.q)), plan.block_table,
                                            plan.seq_lens, plan.scale)
    assert_close(out, exp, "bf16", "fp8 decode 32-row groups")


def test_fp8_decode_csr_and_static_scratch_match(cuda_device):
    plan = wl.gqa_decode_plan(batch=9, lo=100, hi=2000, seed=21)
    kp, vp, kc, vc, st = _fp8_step(plan, cuda_device)
    msl = int(plan.seq_lens.max())
    a = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale, max_seq_len=msl,
                                    k_scale=KS, v_scale=VS)
    ip, ix, last = (torch.from_numpy(x).to(cuda_device) for x in wl.csr_tables(plan))
    b = capi.paged_attention_decode_csr(kp, vp, st.q, ip, ix, last, plan.scale, max_seq_len=msl,
                                        k_scale=KS, v_scale=VS)
    c = capi.paged_attention_decode_static_scratch(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                                   max_seq_len=msl, k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_fp8_quantiser_saturates_and_keeps_nan(cuda_device):
    """Rows past +-448*scale saturate; NaN rows stay NaN codes (the oracle's rule)."""
    P, ps, hkv, d = 4, 16, 2, 64
    kp = torch.zeros((P, ps, hkv, d), dtype=torch.float8_e4m3fn, device=cuda_device)
    vp = torch.zeros_like(kp)
    vals = torch.tensor([0.0, -0.0, 1e-9, 3.0, -9.0, 1e4, -1e4, float("nan")], dtype=torch.float32)
    key = vals.repeat(hkv * d // 8 * 3).reshape(3, hkv, d).to(torch.bfloat16).to(cuda_device)
    slots = torch.tensor([5, 17, 40], dtype=torch.int64, device=cuda_device)
    capi.paged_kv_append(kp, vp, key, key.clone(), slots, k_scale=0.5, v_scale=2.0)
    torch.cuda.synchronize()
    exp = kv_fp8.quantize(to_f64(bits(key)).astype(np.float32), 0.5)
    got = _codes(kp).reshape(P * ps, hkv, d)[[5, 17, 40]]
    assert np.array_equal(got, exp)
    assert (got == 0x7E).any() and (got == 0xFE).any() and (got == 0x7F).any()


# ---------------------------------------------------------------------------
# prefill over e4m3 pools
# ---------------------------------------------------------------------------

def _fp8_prefill(plan, device, ks=KS, vs=VS, rows=None):
    """Quantising append of the new rows, then prefill; (out, expected, codes ok)."""
    kp, vp, kc, vc, st = _fp8_step(plan, device, ks, vs)
    assert np.array_equal(_codes(kp), kc) and np.array_equal(_codes(vp), vc)   # append: every byte
    out = capi.paged_attention_prefill(kp, vp, st.q, st.query_start_loc, st.block_table, st.seq_lens,
                                       plan.scale, max_q_len=int(plan.new.max()),
                                       max_seq_len=int(plan.seq_lens.max()), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    q = to_f64(bits(st.q))
    exp = np.zeros(q.shape)
    qsl = plan.query_start_loc
    for b in range(plan.batch):   # 256 rows at a time bounds the oracle's memory
        for r0 in range(int(qsl[b]), int(qsl[b + 1]), 256):
            rr = list(range(r0, min(r0 + 256, int(qsl[b + 1]))))
            exp[rr] = kv_fp8.paged_attention_prefill_fp8(kc, vc, ks, vs, q, qsl, plan.block_table,
                                                         plan.seq_lens, plan.scale, rows=rr)[rr]
    return out, exp, (kp, vp, st)


def test_fp8_prefill_chunked_full_every_row(cuda_device):
    """The mixed chunked-prefill workload (8 sequences, 10,496 new rows after
    cached contexts up to 8192) on e4m3 pools: every row against the oracle."""
    plan = wl.chunked_prefill_plan()
    out, exp, _ = _fp8_prefill(plan, cuda_device)
    assert_close(out, exp, "bf16", "fp8 chunked prefill, every row")


def test_fp8_prefill_tiny_shape(cuda_device):
    """The tiny workload's shape (one sequence, 4 query / 2 KV heads, head_dim
    64, page 16, 7 of 64 pages) prefilled on an e4m3 pool."""
    rng = np.random.RandomState(0)
    pages = list(rng.choice(64, 7, replace=False))
    plan = wl._assemble("tiny_fp8_prefill", "prefill", "bf16", 4, 2, 64, 16, [0], [100], [pages], 64,
                        1.0 / 8.0, 0)
    out, exp, _ = _fp8_prefill(plan, cuda_device, ks=0.05, vs=0.01)
    assert_close(out, exp, "bf16", "fp8 tiny prefill")


@pytest.mark.parametrize("hq,hkv,d,ps", [(32, 8, 128, 16), (8, 1, 128, 8), (4, 4, 64, 32), (32, 1, 64, 64),
                                         (16, 4, 128, 256)])
def test_fp8_prefill_ragged(cuda_device, hq, hkv, d, ps):
    plan = wl.chunked_prefill_plan(new=(1, 7, 16, 65, 130, 3, 300), cached=(0, 9, 100, 0, 31, 500, 127),
                                   seed=hq + hkv + d + ps, hq=hq, hkv=hkv, d=d, ps=ps)
    out, exp, _ = _fp8_prefill(plan, cuda_device, ks=0.04, vs=0.02)
    assert_close(out, exp, "bf16", f"fp8 prefill {hq}/{hkv}/{d} ps{ps}")


def test_fp8_prefill_csr_matches_row_padded(cuda_device):
    plan = wl.chunked_prefill_plan(new=(40, 200, 3), cached=(17, 0, 900), seed=44)
    out, exp, (kp, vp, st) = _fp8_prefill(plan, cuda_device)
    assert_close(out, exp, "bf16", "fp8 prefill (row-padded)")
    ip, ix, last = (torch.from_numpy(x).to(cuda_device) for x in wl.csr_tables(plan))
    out2 = capi.paged_attention_prefill_csr(kp, vp, st.q, st.query_start_loc, ip, ix, last, plan.scale,
                                            max_q_len=int(plan.new.max()), max_seq_len=int(plan.seq_lens.max()),
                                            k_scale=KS, v_scale=VS)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_fp8_long_context_full_every_sequence(cuda_device):
    """The long-context GQA workload at full size (256 sequences, contexts
    U[1024, 32768]) on e4m3 pools.  The cached tokens' codes are made on the
    device by torch's own e4m3 conversion (x / scale, the oracle's rule for
    these in-range values); the appended rows go through the library's
    quantising append, checked byte for byte against the oracle's quantiser;
    then every sequence's decode output against the oracle on the codes, 16
    sequences at a time on host copies of only the pages they read."""
    from _parity import compact_subset
    plan = wl.long_context_plan(hkv=8, seed=4)
    st = wl.materialize(plan, cuda_device)
    for name in ("key_pool", "value_pool"):  # bf16 pool -> codes, in slices of pages
        src = getattr(st, name)
        dst = torch.empty(src.shape, dtype=torch.float8_e4m3fn, device=cuda_device)
        for i in range(0, src.shape[0], 4096):
            dst[i:i + 4096] = (src[i:i + 4096].float() / KS).to(torch.float8_e4m3fn)
        setattr(st, name, dst)
        del src
    torch.cuda.empty_cache()
    capi.paged_kv_append(st.key_pool, st.value_pool, st.key, st.value, st.slot_mapping, k_scale=KS, v_scale=KS)
    out = capi.paged_attention_decode(st.key_pool, st.value_pool, st.q, st.block_table, st.seq_lens, plan.scale,
                                      max_seq_len=int(plan.seq_lens.max()), k_scale=KS, v_scale=KS)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    P, ps = plan.num_pages, plan.page_size
    got_rows = st.key_pool.view(torch.uint8).view(P * ps, -1)[st.slot_mapping].cpu().numpy()
    exp_rows = kv_fp8.quantize(to_f64(bits(st.key)).astype(np.float32), KS).reshape(len(plan.slot_mapping), -1)
    assert np.array_equal(got_rows, exp_rows)              # the appended codes
    q_all = to_f64(bits(st.q))
    exp = np.zeros_like(q_all)
    for s0 in range(0, plan.batch, 16):
        seqs = list(range(s0, min(s0 + 16, plan.batch)))
        kc, vc, btc, _, _ = compact_subset(st, seqs)       # codes after the append, as uint8
        exp[seqs] = kv_fp8.paged_attention_decode_fp8(kc, vc, KS, KS, q_all[seqs], btc, plan.seq_lens[seqs],
                                                      plan.scale)
    assert_close(out, exp, "bf16", "fp8 long GQA, every sequence")
