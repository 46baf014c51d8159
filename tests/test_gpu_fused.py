"""GPU parity of paged_attention_decode_append: one decode step (append of the
step's rows, then decode) in one launch, against the oracle's composition
(onnxruntime/mobius PR #395 "Add paged / block-table KV cache export", "How
it works (per attention layer)", steps 1 and 2).

* the pools after the call: bit-exact against the oracle's append;
* the outputs: within the bf16 tolerance of the oracle, and bit-identical to
  the two-launch path (paged_kv_append then paged_attention_decode), which
  reads the same values from the pool that the fused kernel takes from its
  input;
* the pool slots of the new tokens hold NaN before the call, so attending
  to a stale pool row instead of the input shows up as a non-finite output.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_fp8
from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    build_mod.build()
    capi.lib()
    capi.device_error()  # clear


def _fused(st, kp, vp, slots=None, seq_lens=None, ks=1.0, vs=1.0, out=None):
    p = st.plan
    return capi.paged_attention_decode_append(
        kp, vp, st.key, st.value, st.slot_mapping if slots is None else slots, st.q, st.block_table,
        st.seq_lens if seq_lens is None else seq_lens, p.scale, max_seq_len=int(p.seq_lens.max()),
        out=torch.full_like(st.q, float("nan")) if out is None else out, k_scale=ks, v_scale=vs)


def _check(plan, device, where):
    st = wl.materialize(plan, device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    out = _fused(st, kp, vp)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    kb, vb, exp = oracle.paged_attention_decode_append(
        bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value), plan.slot_mapping,
        to_f64(bits(st.q)), plan.block_table, plan.seq_lens, plan.scale)
    assert bits(kp).tobytes() == kb.tobytes(), f"{where}: key pool"
    assert bits(vp).tobytes() == vb.tobytes(), f"{where}: value pool"
    # the oracle attends over the appended pools (bits widened to fp64)
    exp = oracle.paged_attention_decode(to_f64(kb), to_f64(vb), to_f64(bits(st.q)), plan.block_table,
                                        plan.seq_lens, plan.scale)
    assert_close(out, exp, "bf16", where)
    # the two-launch path on the same inputs gives the same bits
    kp2, vp2 = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp2, vp2, st.key, st.value, st.slot_mapping)
    out2 = capi.paged_attention_decode(kp2, vp2, st.q, st.block_table, st.seq_lens, plan.scale,
                                       max_seq_len=int(plan.seq_lens.max()))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), f"{where}: fused != append + decode"


def test_fused_gqa_decode_full(cuda_device):
    _check(wl.gqa_decode_plan(), cuda_device, "fused gqa_decode")


@pytest.mark.parametrize("hq,hkv,d,ps", [(32, 1, 128, 16), (8, 8, 64, 8), (16, 4, 64, 64), (6, 3, 128, 32),
                                         (32, 8, 128, 256)])
def test_fused_ragged(cuda_device, hq, hkv, d, ps):
    lens = np.array([1, 2, 15, 16, 17, 33, 300, 1000])
    plan = wl.plan_from_lengths(f"fused_{hq}_{hkv}_{d}_{ps}", "decode", "bf16", hq, hkv, d, ps, lens - 1,
                                np.ones(len(lens)), seed=hq + hkv + d + ps, extra_free_pages=4)
    _check(plan, cuda_device, plan.name)


def test_fused_32_row_groups(cuda_device):
    # 32 query heads on 1 KV head, ~190 blocks a sequence: segment changes weigh
    # in the cut and a publisher warp counts the cut segments
    lens = np.full(32, 3000) + np.arange(32) * 7
    plan = wl.plan_from_lengths("fused_mqa_weighted", "decode", "bf16", 32, 1, 128, 16, lens - 1,
                                np.ones(32), seed=47, extra_free_pages=4)
    _check(plan, cuda_device, plan.name)


def test_fused_long_context(cuda_device):
    _check(wl.long_context_plan(hkv=8, batch=12, lo=1000, hi=9000, seed=41), cuda_device, "fused long")


def test_fused_some_sequences_without_new_token(cuda_device):
    plan = wl.gqa_decode_plan(batch=8, lo=40, hi=900, seed=43)
    st = wl.materialize(plan, cuda_device)
    none = [1, 4, 6]
    slots = plan.slot_mapping.copy()
    slots[none] = -1
    lens = plan.seq_lens.copy()
    lens[none] -= 1  # their keys are the cached ones only
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    out = _fused(st, kp, vp, slots=torch.from_numpy(slots).to(cuda_device),
                 seq_lens=torch.from_numpy(lens).to(cuda_device))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    kb, vb, exp = oracle.paged_attention_decode_append(
        bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value), slots,
        to_f64(bits(st.q)), plan.block_table, lens, plan.scale)
    assert bits(kp).tobytes() == kb.tobytes()
    exp = oracle.paged_attention_decode(to_f64(kb), to_f64(vb), to_f64(bits(st.q)), plan.block_table, lens,
                                        plan.scale)
    assert_close(out, exp, "bf16", "fused without new tokens")


def test_fused_slot_not_last_key_is_reported(cuda_device):
    plan = wl.gqa_decode_plan(batch=4, lo=40, hi=300, seed=44)
    st = wl.materialize(plan, cuda_device)
    slots = plan.slot_mapping.copy()
    ps = st.key_pool.shape[1]
    # a dead slot past the end of a sequence on its own last page: not its last key
    b = next(i for i, L in enumerate(plan.seq_lens) if (L - 1) % ps != ps - 1)
    L = int(plan.seq_lens[b])
    slots[b] = int(plan.block_table[b, (L - 1) // ps]) * ps + ps - 1
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    _fused(st, kp, vp, slots=torch.from_numpy(slots).to(cuda_device))
    torch.cuda.synchronize()
    assert capi.device_error() == (2, int(slots[b]))


def test_fused_e4m3_pools(cuda_device):
    plan = wl.long_context_plan(hkv=8, batch=8, lo=500, hi=5000, seed=45)
    st = wl.materialize(plan, cuda_device)
    ks, vs = 0.02, 0.03
    kc0 = kv_fp8.quantize(to_f64(bits(st.key_pool)), ks)  # NaN (dead and new slots) -> 0x7F
    vc0 = kv_fp8.quantize(to_f64(bits(st.value_pool)), vs)
    kp = torch.from_numpy(kc0).to(cuda_device).view(torch.float8_e4m3fn)
    vp = torch.from_numpy(vc0).to(cuda_device).view(torch.float8_e4m3fn)
    out = _fused(st, kp, vp, ks=ks, vs=vs)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    kc, vc, exp = kv_fp8.paged_attention_decode_append_fp8(
        kc0, vc0, to_f64(bits(st.key)).astype(np.float32), to_f64(bits(st.value)).astype(np.float32),
        plan.slot_mapping, ks, vs, to_f64(bits(st.q)), plan.block_table, plan.seq_lens, plan.scale)
    assert np.array_equal(kp.view(torch.uint8).cpu().numpy(), kc)
    assert np.array_equal(vp.view(torch.uint8).cpu().numpy(), vc)
    assert_close(out, exp, "bf16", "fused e4m3")


def test_fused_in_cuda_graph_replays(cuda_device):
    plan = wl.gqa_decode_plan(batch=16, seed=46)
    st = wl.materialize(plan, cuda_device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    out = torch.empty_like(st.q)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    s = torch.cuda.Stream()

    def call():
        capi.paged_attention_decode_append(kp, vp, st.key, st.value, st.slot_mapping, st.q, st.block_table,
                                           st.seq_lens, plan.scale, max_seq_len=int(plan.seq_lens.max()),
                                           out=out, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for rep in range(3):
        gen = torch.Generator().manual_seed(200 + rep)
        st.key.copy_(torch.randn(st.key.shape, generator=gen).to(st.key.dtype))
        st.value.copy_(torch.randn(st.value.shape, generator=gen).to(st.value.dtype))
        st.q.copy_(torch.randn(st.q.shape, generator=gen).to(st.q.dtype))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key), bits(st.value),
                                        plan.slot_mapping)
        assert bits(kp).tobytes() == kb.tobytes()
        exp = oracle.paged_attention_decode(to_f64(kb), to_f64(vb), to_f64(bits(st.q)), plan.block_table,
                                            plan.seq_lens, plan.scale)
        assert_close(out, exp, "bf16", f"fused graph replay {rep}")
