"""GPU parity for bf16 pools whose page size the tensor-core kernels' TMA boxes
do not take (1, 2, 4 slots, or not a power of two): those calls run on the
CUDA-core path (fp32 arithmetic, one warp per query row and head).  Page size
1 is the token-granular layout of RadixAttention-style caches (mobius PR #395
summary).  Same bars as tests/test_gpu_parity.py: append bit-exact, bf16
outputs within max-abs 2e-2 / mean-abs 2e-3 of the fp64 oracle, NaN in every
slot that holds no live token."""
import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, gpu_step, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    build_mod.build()
    capi.lib()
    capi.device_error()  # clear


def _decode_plan(ps, seed):
    # ragged lengths with an empty sequence, one key, a page edge and a long one
    lens = np.array([0, 1, 3, 17, 64, 65, 190, 511])
    return wl.plan_from_lengths(f"dec_small_ps{ps}", "decode", "bf16", 32, 8, 128, ps,
                                np.maximum(lens - 1, 0), (lens > 0).astype(int), seed=seed)


@pytest.mark.parametrize("ps", [1, 2, 4, 12])
def test_decode_small_pages(cuda_device, ps):
    plan = _decode_plan(ps, 300 + ps)
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert bits(kp).tobytes() == kb.tobytes() and bits(vp).tobytes() == vb.tobytes()
    assert capi.device_error() == (0, 0)
    assert_close(out, exp, "bf16", plan.name)
    assert torch.all(out[0] == 0)  # the empty sequence


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 64), (16, 2, 96), (32, 1, 256)])
def test_decode_small_pages_shapes(cuda_device, hq, hkv, d):
    lens = np.array([5, 40, 300])
    plan = wl.plan_from_lengths(f"dec_small_{hq}_{hkv}_{d}", "decode", "bf16", hq, hkv, d, 4,
                                lens - 1, np.ones(3), seed=hq + d)
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert capi.device_error() == (0, 0)
    assert_close(out, exp, "bf16", plan.name)


@pytest.mark.parametrize("ps", [1, 4, 12])
def test_prefill_small_pages(cuda_device, ps):
    plan = wl.chunked_prefill_plan(new=(33, 90, 1, 17), cached=(5, 64, 200, 0), seed=ps, ps=ps)
    st = wl.materialize(plan, cuda_device)
    kp, vp, out = gpu_step(st)
    kb, vb, exp = oracle_step(st)
    assert bits(kp).tobytes() == kb.tobytes() and bits(vp).tobytes() == vb.tobytes()
    assert capi.device_error() == (0, 0)
    assert_close(out, exp, "bf16", f"prefill ps={ps}")


def test_fused_step_small_pages_is_append_then_decode(cuda_device):
    lens = np.array([1, 3, 17, 64, 65, 190, 511])  # every sequence takes a new token
    plan = wl.plan_from_lengths("fused_small_ps4", "decode", "bf16", 32, 8, 128, 4, lens - 1,
                                np.ones(len(lens)), seed=311)
    st = wl.materialize(plan, cuda_device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    out = capi.paged_attention_decode_append(kp, vp, st.key, st.value, st.slot_mapping, st.q, st.block_table,
                                             st.seq_lens, plan.scale, max_seq_len=int(plan.seq_lens.max()),
                                             out=torch.full_like(st.q, float("nan")))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    kb, vb, exp = oracle.paged_attention_decode_append(
        bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value), plan.slot_mapping,
        to_f64(bits(st.q)), plan.block_table, plan.seq_lens, plan.scale)
    assert bits(kp).tobytes() == kb.tobytes() and bits(vp).tobytes() == vb.tobytes()
    # the oracle attends over the appended pools (bits widened to fp64)
    exp = oracle.paged_attention_decode(to_f64(kb), to_f64(vb), to_f64(bits(st.q)), plan.block_table,
                                        plan.seq_lens, plan.scale)
    assert_close(out, exp, "bf16", "fused ps=4")
    kp2, vp2, out2 = gpu_step(st)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_csr_and_static_scratch_small_pages_match_dense(cuda_device):
    plan = _decode_plan(2, 312)
    st = wl.materialize(plan, cuda_device)
    kp, vp, dense = gpu_step(st)
    ip, ix, last = wl.csr_tables(plan)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    csr = capi.paged_attention_decode_csr(kp, vp, st.q, dev(ip), dev(ix), dev(last), plan.scale,
                                          max_seq_len=int(plan.seq_lens.max()))
    scratch = capi.paged_attention_decode_static_scratch(kp, vp, st.q, st.block_table, st.seq_lens,
                                                         plan.scale, max_seq_len=int(plan.seq_lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert torch.equal(csr.view(torch.int16), dense.view(torch.int16))
    assert torch.equal(scratch.view(torch.int16), dense.view(torch.int16))


def test_cascade_small_pages_is_unsupported(cuda_device):
    plan = _decode_plan(4, 313)
    st = wl.materialize(plan, cuda_device)
    pre = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    with pytest.raises(capi.PagedAttnError) as e:
        capi.paged_attention_decode_cascade(st.key_pool, st.value_pool, st.q, pre, 16, st.block_table,
                                            st.seq_lens, plan.scale, max_seq_len=int(plan.seq_lens.max()))
    assert e.value.status == capi.PA_ERR_UNSUPPORTED
