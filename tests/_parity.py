"""Helpers shared by the GPU parity tests: run one step through the C ABI and
through the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-5


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits (uint16 for bf16, uint8 codes for e4m3, float32 array
    for f32) on the host."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def to_f64(a: np.ndarray) -> np.ndarray:
    """Widen host bits/values to fp64 exactly."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def gpu_step(st: wl.StepTensors, clone_pools=True, max_seq_len=None, max_q_len=None):
    """append -> attend through the C ABI; returns (key_pool, value_pool, out)."""
    plan = st.plan
    kp = st.key_pool.clone() if clone_pools else st.key_pool
    vp = st.value_pool.clone() if clone_pools else st.value_pool
    capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping)
    msl = int(plan.seq_lens.max()) if max_seq_len is None else max_seq_len
    if plan.kind == "decode":
        out = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale,
                                          max_seq_len=msl)
    else:
        mql = int(plan.new.max()) if max_q_len is None else max_q_len
        out = capi.paged_attention_prefill(kp, vp, st.q, st.query_start_loc, st.block_table,
                                           st.seq_lens, plan.scale, max_q_len=mql,
                                           max_seq_len=msl)
    torch.cuda.synchronize()
    return kp, vp, out


def oracle_step(st: wl.StepTensors, seqs=None, rows=None):
    """The same step in the oracle: (key_bits, value_bits, out fp64)."""
    plan = st.plan
    kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key),
                                    bits(st.value), plan.slot_mapping)
    K, V = to_f64(kb), to_f64(vb)
    q = to_f64(bits(st.q))
    if plan.kind == "decode":
        out = oracle.paged_attention_decode(K, V, q, plan.block_table, plan.seq_lens, plan.scale,
                                            seqs=seqs)
    else:
        out = oracle.paged_attention_prefill(K, V, q, plan.query_start_loc, plan.block_table,
                                             plan.seq_lens, plan.scale, rows=rows)
    return kb, vb, out


def assert_close(got: torch.Tensor, exp: np.ndarray, dtype: str, where: str = "", rows=None):
    g = to_f64(bits(got))
    if rows is not None:
        g = g[rows]
        exp = exp[rows]
    assert np.all(np.isfinite(g)), f"{where}: non-finite output"
    err = np.abs(g - exp)
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{where}: max abs {err.max():.3e} > {F32_MAX_ABS}"
    else:
        assert err.max() <= BF16_MAX_ABS, f"{where}: max abs {err.max():.3e} > {BF16_MAX_ABS}"
        assert err.mean() <= BF16_MEAN_ABS, f"{where}: mean abs {err.mean():.3e} > {BF16_MEAN_ABS}"
    return float(err.max()), float(err.mean())


def compact_subset(st: wl.StepTensors, seqs):
    """Host copy of only the pages the given sequences use, with remapped tables.

    For full-size pools too large to bring to the host: the oracle then runs
    on exactly the values those sequences read.
    """
    plan = st.plan
    ps = plan.page_size
    pages = []
    for b in seqs:
        n = (int(plan.seq_lens[b]) + ps - 1) // ps
        pages.extend(int(x) for x in plan.block_table[b, :n])
    uniq = sorted(set(pages))
    remap = {p: i for i, p in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=st.key_pool.device)
    raw = lambda t: t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t  # e4m3: select the code bytes
    kp = bits(raw(st.key_pool).index_select(0, idx))
    vp = bits(raw(st.value_pool).index_select(0, idx))
    mb = plan.block_table.shape[1]
    bt = np.full((len(seqs), mb), -1, dtype=np.int64)
    slots = []
    key_rows = []
    for i, b in enumerate(seqs):
        n = (int(plan.seq_lens[b]) + ps - 1) // ps
        bt[i, :n] = [remap[int(x)] for x in plan.block_table[b, :n]]
        t0, t1 = int(plan.query_start_loc[b]), int(plan.query_start_loc[b + 1])
        for t in range(t0, t1):
            s = int(plan.slot_mapping[t])
            slots.append(remap[s // ps] * ps + s % ps)
            key_rows.append(t)
    return kp, vp, bt, np.asarray(slots, dtype=np.int64), key_rows
