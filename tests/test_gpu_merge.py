"""GPU checks of the split-KV merge inside the decode kernel.

A segment (one sequence's keys for one box of KV heads) whose 16-key blocks
are cut across CTAs leaves one fp32 partial (m, l, o) per CTA.  Each CTA
counts its part on a per-segment word tagged with a per-launch epoch (kept at
the workspace's start), and after its own range every CTA that holds a part
waits -- bounded -- until all parts are counted and merges a slice of the
segment's rows with the combine identity (mobius PR #395 "Add paged /
block-table KV cache export": the decode output is softmax attention over all
seq_lens[b] keys, which the merge reassembles exactly up to rounding).  The
grid is launched cooperatively so that all its CTAs are resident; without
that launch the CTA that counts a segment's last part merges all of it.  So
the workspace needs no initialisation, and every launch -- eager or a CUDA
graph replay -- must merge afresh.  Each case below changes the inputs
between launches, so a launch that skipped its merge would leave a stale or
NaN output and fail against the oracle.  The last case makes the bounded
wait run out (through the library's test hook) and checks that the kernel
reports it and returns.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, gpu_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    build_mod.build()
    capi.lib()
    capi.device_error()  # clear


def _appended(plan, device):
    st = wl.materialize(plan, device)
    kp, vp, _ = gpu_step(st)
    return st, kp, vp


def _expect(st, kp, vp, q):
    p = st.plan
    return oracle.paged_attention_decode(to_f64(bits(kp)), to_f64(bits(vp)), to_f64(bits(q)),
                                         p.block_table, p.seq_lens, p.scale)


def _new_q(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(q.dtype).to(q.device)


def _decode(st, kp, vp, q, ws, out=None, stream=None):
    p = st.plan
    if out is None:  # NaN until written: a row the kernel skipped cannot pass
        out = torch.full_like(q, float("nan"))
    return capi.paged_attention_decode(kp, vp, q, st.block_table, st.seq_lens, p.scale,
                                       max_seq_len=int(p.seq_lens.max()), out=out, workspace=ws,
                                       stream=stream)


@pytest.mark.parametrize("fill", ["zeros", "ones", "pattern", "random"])
def test_merge_with_uninitialised_workspace(cuda_device, fill):
    plan = wl.gqa_decode_plan()  # 32 sequences of 512..4096 keys: most cut across CTAs
    st, kp, vp = _appended(plan, cuda_device)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    if fill == "zeros":
        ws.zero_()
    elif fill == "ones":
        ws.fill_(0xFF)
    elif fill == "pattern":
        ws.fill_(0x5A)
    else:
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, generator=torch.Generator().manual_seed(7)))
    out = _decode(st, kp, vp, st.q, ws)
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    assert_close(out, _expect(st, kp, vp, st.q), "bf16", f"merge, workspace {fill}")


def _mqa_plan(seed):
    # 32 query heads on 1 KV head (two 16-row tiles: the warps chain their
    # states, segment changes weigh in the cut and a publisher warp counts
    # the parts); ~190 blocks a sequence over 152 CTAs: every segment is cut
    return wl.plan_from_lengths(f"mqa_merge_{seed}", "decode", "bf16", 32, 1, 128, 16,
                                np.full(32, 3000) + np.arange(32) * 7, np.ones(32), seed=seed)


def test_merge_32_row_groups_uninitialised_workspace(cuda_device):
    plan = _mqa_plan(31)
    st, kp, vp = _appended(plan, cuda_device)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, generator=torch.Generator().manual_seed(8)))
    for rep in range(2):
        q = _new_q(st.q, 300 + rep)
        out = _decode(st, kp, vp, q, ws)
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        assert_close(out, _expect(st, kp, vp, q), "bf16", f"32-row merge rep {rep}")


def test_merge_repeated_calls_and_shapes_share_one_workspace(cuda_device):
    big = wl.gqa_decode_plan()
    small = wl.gqa_decode_plan(batch=5, lo=300, hi=6000, seed=9)
    mqa = wl.long_context_plan(hkv=1, batch=6, lo=1000, hi=9000, seed=13)  # 32 rows per KV head
    rigs = [_appended(p, cuda_device) for p in (big, small, mqa)]
    ws = capi.decode_workspace(big.batch, big.num_q_heads, rigs[0][1])
    for p, (st, kp, vp) in zip((big, small, mqa), rigs):
        need = capi.decode_workspace_size(p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim)
        assert need <= ws.numel()
    for rep in range(2):
        for i, (st, kp, vp) in enumerate(rigs):
            q = _new_q(st.q, 100 * rep + i)
            out = _decode(st, kp, vp, q, ws)
            torch.cuda.synchronize()
            assert capi.device_error() == (0, 0)
            assert_close(out, _expect(st, kp, vp, q), "bf16", f"merge rep {rep} plan {i}")


def _plan_of(shape, seed):
    # gqa: 16 or 32 long sequences, few enough that segment changes weigh in
    # the cut (the weighted instantiation); gqa_plain_cut: 64, cut plainly;
    # mqa: 32-row groups
    if shape == "gqa":
        return wl.gqa_decode_plan(batch=16 if seed == 5 else 32, seed=seed)
    if shape == "gqa_plain_cut":
        return wl.gqa_decode_plan(batch=64, seed=seed)
    return _mqa_plan(seed)


@pytest.mark.parametrize("shape", ["gqa", "gqa_plain_cut", "mqa"])
def test_merge_in_cuda_graph_replays(cuda_device, shape):
    plan = _plan_of(shape, 5)
    st, kp, vp = _appended(plan, cuda_device)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    q = st.q.clone()
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _decode(st, kp, vp, q, ws, out=out, stream=s)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _decode(st, kp, vp, q, ws, out=out, stream=s)
    for rep in range(4):
        qn = _new_q(q, 1000 + rep)
        q.copy_(qn)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        assert_close(out, _expect(st, kp, vp, qn), "bf16", f"graph replay {rep}")


def test_merge_e4m3_pools(cuda_device):
    plan = wl.long_context_plan(hkv=8, batch=8, lo=2000, hi=12000, seed=17)
    st, kp, vp = _appended(plan, cuda_device)
    ks, vs = 0.02, 0.03
    from oracle import kv_fp8
    kc = kv_fp8.quantize(to_f64(bits(kp)), ks)
    vc = kv_fp8.quantize(to_f64(bits(vp)), vs)
    kp8 = torch.from_numpy(kc).to(cuda_device).view(torch.float8_e4m3fn)
    vp8 = torch.from_numpy(vc).to(cuda_device).view(torch.float8_e4m3fn)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp8)
    ws.fill_(0xA5)
    for rep in range(2):
        q = _new_q(st.q, 50 + rep)
        out = torch.full_like(q, float("nan"))
        capi.paged_attention_decode(kp8, vp8, q, st.block_table, st.seq_lens, plan.scale,
                                    max_seq_len=int(plan.seq_lens.max()), out=out, workspace=ws,
                                    k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        exp = kv_fp8.paged_attention_decode_fp8(kc, vc, ks, vs, to_f64(bits(q)), plan.block_table,
                                                plan.seq_lens, plan.scale)
        assert_close(out, exp, "bf16", f"e4m3 merge rep {rep}")


_FALLBACK_SCRIPT = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import oracle
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl
from _parity import assert_close, bits, to_f64
dev = torch.device("cuda:0")
import numpy as np
plans = [wl.gqa_decode_plan(batch=16, seed=6), wl.gqa_decode_plan(batch=64, seed=6),
         wl.plan_from_lengths("mqa_fallback", "decode", "bf16", 32, 1, 128, 16,
                              np.full(32, 3000) + np.arange(32) * 7, np.ones(32), seed=6)]
for i, plan in enumerate(plans):
    st = wl.materialize(plan, dev)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping)  # eager: creates the device error word
    torch.cuda.synchronize()
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    out = torch.full_like(st.q, float("nan"))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):  # the process's first decode launch: inside a capture
        capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                    max_seq_len=int(plan.seq_lens.max()), out=out, workspace=ws, stream=s)
    for rep in range(2):
        st.q.copy_(torch.randn(st.q.shape, generator=torch.Generator().manual_seed(rep)).to(st.q.dtype))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        exp = oracle.paged_attention_decode(to_f64(bits(kp)), to_f64(bits(vp)), to_f64(bits(st.q)),
                                            plan.block_table, plan.seq_lens, plan.scale)
        assert_close(out, exp, "bf16", f"whole-segment merge, plan {i}, replay {rep}")
print("fallback merge ok")
"""


def test_merge_without_cooperative_launch():
    """The merge used when the grid is not launched cooperatively (the CTA
    counting a segment's last part merges all of it).  A process whose first
    decode launch happens inside a stream capture never tries the cooperative
    launch, so its graph replays take this path."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", _FALLBACK_SCRIPT, root], capture_output=True, text=True,
                         timeout=600, cwd=root)
    assert out.returncode == 0, (out.stdout[-1500:], out.stderr[-3000:])
    assert "fallback merge ok" in out.stdout


@pytest.mark.parametrize("shape", ["gqa", "gqa_plain_cut", "mqa"])
def test_bounded_part_wait_runs_out_and_is_reported(cuda_device, shape):
    """The decode kernel's one wait on other CTAs (a CTA holding part of a cut
    segment waits for the other parts before merging its slice) is bounded.
    Through the test hook every cut segment expects one part that never
    arrives and the limit is 1 ms: the call must return within a few ms
    instead of hanging, record code 5 (a bounded wait gave up, detail -2 =
    the part wait) in the device error word, and leave the context usable --
    a normal decode on the same workspace afterwards matches the oracle."""
    # ~145 (GQA) or ~190 (MQA) blocks a sequence over 152 CTAs: every segment is cut
    plan = _plan_of(shape, 23)
    st, kp, vp = _appended(plan, cuda_device)
    ws = capi.decode_workspace(plan.batch, plan.num_q_heads, kp)
    capi.device_error()
    pool = capi.make_pool(kp, vp)
    out = torch.full_like(st.q, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    status = capi.lib().pa_testing_decode_part_wait(
        ctypes.byref(pool), ctypes.c_void_p(st.q.data_ptr()), ctypes.c_void_p(out.data_ptr()), plan.batch,
        plan.num_q_heads, ctypes.c_void_p(st.block_table.data_ptr()), plan.max_blocks,
        ctypes.c_void_p(st.seq_lens.data_ptr()), int(plan.seq_lens.max()), plan.scale,
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), 1_000_000, 1, stream)
    assert status == capi.PA_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert capi.device_error() == (5, -2)
    assert elapsed < 1.0, f"the 1 ms part wait took {elapsed:.3f} s"
    # the same workspace, a normal call: unaffected
    for rep in range(2):
        q = _new_q(st.q, 90 + rep)
        got = _decode(st, kp, vp, q, ws)
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        assert_close(got, _expect(st, kp, vp, q), "bf16", f"decode after an expired wait, rep {rep}")
