"""paged_attention_decode_static_scratch: the decode entry point for callers
that cannot allocate device memory (a plugin whose host runtime owns all
device memory and gives it no allocator, or a serving loop that may not take
cudaMalloc's implicit synchronisation mid-step).  It keeps its split-KV
partials in the library's own static device array instead of a
caller-provided workspace.

Checked here through the C ABI: two calls in a row (different batch shapes,
so the shared array is reused with other contents) each match the regular
paged_attention_decode with a torch-allocated workspace, within the bf16
tolerance the parity tests use; a request too large for the array is
refused before any launch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def _stream_ptr():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call_static(lib, st, plan, out):
    pool = capi.make_pool(st.key_pool, st.value_pool)
    return lib.paged_attention_decode_static_scratch(
        ctypes.byref(pool), ctypes.c_void_p(st.q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        plan.batch, plan.num_q_heads, ctypes.c_void_p(st.block_table.data_ptr()), plan.max_blocks,
        ctypes.c_void_p(st.seq_lens.data_ptr()), int(plan.seq_lens.max()), plan.scale,
        _stream_ptr())


def _call_regular(lib, st, plan, out, ws):
    pool = capi.make_pool(st.key_pool, st.value_pool)
    return lib.paged_attention_decode(
        ctypes.byref(pool), ctypes.c_void_p(st.q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        plan.batch, plan.num_q_heads, ctypes.c_void_p(st.block_table.data_ptr()), plan.max_blocks,
        ctypes.c_void_p(st.seq_lens.data_ptr()), int(plan.seq_lens.max()), plan.scale,
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr())


def test_static_scratch_decode_matches_regular_decode_twice(cuda_device):
    build_mod.build()
    lib = capi.lib()
    plans = [wl.gqa_decode_plan(batch=32, seed=41),                       # GQA 4
             wl.long_context_plan(hkv=1, batch=24, lo=100, hi=3000, seed=42)]  # MQA
    for i, plan in enumerate(plans):
        st = wl.materialize(plan, cuda_device)
        capi.paged_kv_append(st.key_pool, st.value_pool, st.key, st.value, st.slot_mapping)
        ws = capi.decode_workspace(plan.batch, plan.num_q_heads, st.key_pool)
        ref = torch.full_like(st.q, float("nan"))
        got = torch.full_like(st.q, float("nan"))
        assert _call_regular(lib, st, plan, ref, ws) == capi.PA_OK
        assert _call_static(lib, st, plan, got) == capi.PA_OK
        torch.cuda.synchronize()
        err = (got.double() - ref.double()).abs()
        assert torch.isfinite(got).all(), f"call {i}: non-finite output"
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, f"call {i}"


def test_static_scratch_refuses_oversize_request(cuda_device):
    build_mod.build()
    lib = capi.lib()
    limit = 8 << 20
    # B * Hq * D * 4 bytes of partials alone exceed the array
    batch, hq, hkv, d = 4096, 32, 8, 128
    assert lib.paged_attention_decode_workspace_size(batch, hq, hkv, d, capi.PA_DTYPE_BF16) > limit
    kp = torch.zeros(4, 16, hkv, d, dtype=torch.bfloat16, device=cuda_device)
    pool = capi.make_pool(kp, kp.clone())
    q = torch.zeros(batch, hq, d, dtype=torch.bfloat16, device=cuda_device)
    out = torch.zeros_like(q)
    bt = torch.zeros(batch, 1, dtype=torch.int32, device=cuda_device)
    sl = torch.ones(batch, dtype=torch.int32, device=cuda_device)
    st = lib.paged_attention_decode_static_scratch(
        ctypes.byref(pool), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()), batch,
        hq, ctypes.c_void_p(bt.data_ptr()), 1, ctypes.c_void_p(sl.data_ptr()), 1, 0.1,
        _stream_ptr())
    assert st == capi.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0   # nothing was launched
