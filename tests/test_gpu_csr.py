"""GPU parity of the CSR page-table calls (kv_indptr / kv_indices /
kv_last_page_len) against the oracle's CSR definitions, and bit-identity with
the row-padded calls on the same pages (the kernels are the same; only where
a sequence's page list and length come from differs)."""
import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, gpu_step, to_f64

pytestmark = pytest.mark.gpu


def _csr_dev(plan, device):
    ip, ix, last = wl.csr_tables(plan)
    return (torch.from_numpy(ip).to(device), torch.from_numpy(ix).to(device),
            torch.from_numpy(last).to(device)), (ip, ix, last)


def _oracle_pools(st):
    kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value),
                                    st.plan.slot_mapping)
    return to_f64(kb), to_f64(vb)


@pytest.mark.parametrize("name", ["gqa_decode", "shared_prefix"])
def test_decode_csr_full(cuda_device, name):
    plan = wl.named_plan(name)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    (ip, ix, last), host = _csr_dev(plan, cuda_device)
    msl = int(plan.seq_lens.max())
    out = capi.paged_attention_decode_csr(kp, vp, st.q, ip, ix, last, plan.scale, max_seq_len=msl)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    K, V = _oracle_pools(st)
    seqs = list(range(0, plan.batch, max(1, plan.batch // 16)))
    exp = oracle.paged_attention_decode_csr(K, V, to_f64(bits(st.q)), *host, plan.scale, seqs=seqs)
    assert_close(out, exp, plan.dtype, f"decode csr {name}", rows=seqs)


@pytest.mark.parametrize("hq,hkv,d,ps", [(32, 8, 128, 16), (32, 1, 128, 8), (4, 4, 64, 64)])
def test_decode_csr_ragged(cuda_device, hq, hkv, d, ps):
    lens = np.array([1, ps, ps + 1, 3 * ps, 7 * ps - 1, 200, 0, 1000])
    cached = np.maximum(lens - 1, 0)
    new = (lens > 0).astype(np.int64)
    plan = wl.plan_from_lengths(f"csr_{hq}_{hkv}_{ps}", "decode", "bf16", hq, hkv, d, ps, cached, new,
                                seed=ps + hkv, extra_free_pages=5)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    (ip, ix, last), host = _csr_dev(plan, cuda_device)
    out = capi.paged_attention_decode_csr(kp, vp, st.q, ip, ix, last, plan.scale,
                                          max_seq_len=int(lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    K, V = _oracle_pools(st)
    exp = oracle.paged_attention_decode_csr(K, V, to_f64(bits(st.q)), *host, plan.scale)
    assert_close(out, exp, plan.dtype, "decode csr ragged")


def test_decode_csr_32_row_groups(cuda_device):
    # 32 query heads on 1 KV head, ~190 blocks a sequence: the weighted cut
    lens = np.full(32, 3000) + np.arange(32) * 7
    plan = wl.plan_from_lengths("csr_mqa_weighted", "decode", "bf16", 32, 1, 128, 16, lens - 1,
                                np.ones(32), seed=48, extra_free_pages=5)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    (ip, ix, last), host = _csr_dev(plan, cuda_device)
    out = capi.paged_attention_decode_csr(kp, vp, st.q, ip, ix, last, plan.scale,
                                          max_seq_len=int(lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    K, V = _oracle_pools(st)
    seqs = list(range(0, plan.batch, 4))
    exp = oracle.paged_attention_decode_csr(K, V, to_f64(bits(st.q)), *host, plan.scale, seqs=seqs)
    assert_close(out, exp, plan.dtype, "decode csr 32-row groups", rows=seqs)


def test_decode_csr_16_row_groups_weighted(cuda_device):
    # 32/8 heads, 20 sequences of 800-4000 keys: each spans several CTA
    # ranges, so segment changes weigh in the cut (the weighted instantiation)
    lens = np.random.RandomState(49).randint(800, 4000, size=20)
    plan = wl.plan_from_lengths("csr_gqa_weighted", "decode", "bf16", 32, 8, 128, 16, lens - 1,
                                np.ones(20), seed=49, extra_free_pages=5)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    (ip, ix, last), host = _csr_dev(plan, cuda_device)
    out = capi.paged_attention_decode_csr(kp, vp, st.q, ip, ix, last, plan.scale,
                                          max_seq_len=int(lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    K, V = _oracle_pools(st)
    exp = oracle.paged_attention_decode_csr(K, V, to_f64(bits(st.q)), *host, plan.scale)
    assert_close(out, exp, plan.dtype, "decode csr 16-row groups, weighted cut")


@pytest.mark.parametrize("ps", [8, 16, 256])
def test_prefill_csr(cuda_device, ps):
    plan = wl.chunked_prefill_plan(new=(64, 100, 1, 17, 250), cached=(0, 300, 47, 0, 33), seed=ps, ps=ps)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    (ip, ix, last), host = _csr_dev(plan, cuda_device)
    out = capi.paged_attention_prefill_csr(kp, vp, st.q, st.query_start_loc, ip, ix, last, plan.scale,
                                           max_q_len=int(plan.new.max()),
                                           max_seq_len=int(plan.seq_lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(out.view(torch.int16), dense.view(torch.int16))
    K, V = _oracle_pools(st)
    exp = oracle.paged_attention_prefill_csr(K, V, to_f64(bits(st.q)), plan.query_start_loc, *host,
                                             plan.scale)
    assert_close(out, exp, plan.dtype, f"prefill csr ps{ps}")


def test_csr_tiny_f32_decode_after_prefill(cuda_device):
    """The fp32 configuration through the CSR calls: prefill 100 tokens, then decode 1."""
    pf, dc = wl.tiny_f32_plans()
    st = wl.materialize(pf, cuda_device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping)
    (ip, ix, last), host = _csr_dev(pf, cuda_device)
    out = capi.paged_attention_prefill_csr(kp, vp, st.q, st.query_start_loc, ip, ix, last, pf.scale,
                                           max_q_len=100, max_seq_len=100)
    torch.cuda.synchronize()
    K, V = _oracle_pools(st)
    exp = oracle.paged_attention_prefill_csr(K, V, bits(st.q).astype(np.float64), pf.query_start_loc, *host,
                                             pf.scale)
    assert_close(out, exp, "f32", "tiny f32 prefill csr")


def test_csr_bad_indptr_is_recorded_not_read(cuda_device):
    """A kv_indptr slice past the end of kv_indices counts as an empty sequence."""
    plan = wl.gqa_decode_plan(batch=4, lo=40, hi=90, seed=9)
    st = wl.materialize(plan, cuda_device)
    kp, vp, _ = gpu_step(st)
    (ip, ix, last), _ = _csr_dev(plan, cuda_device)
    ip_bad = ip.clone()
    ip_bad[3] = ix.numel() + 50                   # sequence 2 ends past kv_indices, 3 runs backwards
    capi.device_error()
    out = capi.paged_attention_decode_csr(kp, vp, st.q, ip_bad, ix, last, plan.scale, max_seq_len=200)
    torch.cuda.synchronize()
    code, _ = capi.device_error()
    assert code == 3
    assert torch.all(out[2:].float() == 0)
