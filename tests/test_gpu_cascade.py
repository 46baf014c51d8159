"""GPU parity of cascade decode (a prefix shared by the whole batch, then each
sequence's own pages) against the fp64 oracle's cascade definition, on the
same seeded inputs.  Dead pool slots are NaN-poisoned, so a read of a slot
outside the prefix or past a sequence's own tokens shows up as non-finite."""
import numpy as np
import pytest
import torch

import oracle
from serving_slot_mapping_gb300 import capi
from serving_slot_mapping_gb300 import workloads as wl

from _parity import assert_close, bits, to_f64

pytestmark = pytest.mark.gpu


def _plan(name, hq, hkv, d, ps, prefix_pages, own, seed):
    """Sequences listing the same first ``prefix_pages`` pages, then ``own[b]``
    tokens of their own (the last one appended this step when own[b] > 0)."""
    total = np.asarray([prefix_pages * ps + o for o in own], dtype=np.int64)
    new = np.asarray([1 if o > 0 else 0 for o in own], dtype=np.int64)
    return wl.plan_from_lengths(name, "decode", "bf16", hq, hkv, d, ps, total - new, new, seed,
                                extra_free_pages=3, shared_prefix_pages=prefix_pages)


def _run(plan, device, prefix_pages, prefix_len, where):
    st = wl.materialize(plan, device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    if plan.total_new:
        capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping)
    pre, plen, own_bt, own_lens = wl.cascade_tables(plan, prefix_pages, prefix_len)
    dev = lambda a: torch.from_numpy(a).to(device)
    out = capi.paged_attention_decode_cascade(kp, vp, st.q, dev(pre), plen, dev(own_bt), dev(own_lens),
                                              plan.scale, max_seq_len=int(own_lens.max()))
    torch.cuda.synchronize()
    assert capi.device_error() == (0, 0)
    if plan.total_new:
        kb, vb = oracle.paged_kv_append(bits(st.key_pool), bits(st.value_pool), bits(st.key),
                                        bits(st.value), plan.slot_mapping)
    else:
        kb, vb = bits(st.key_pool), bits(st.value_pool)
    exp = oracle.paged_attention_decode_cascade(to_f64(kb), to_f64(vb), to_f64(bits(st.q)), pre, plen,
                                                own_bt, own_lens, plan.scale)
    assert_close(out, exp, "bf16", where)
    return kp, vp, st, out


def test_cascade_shared_prefix_full(cuda_device):
    """The shared-prefix decode workload at full size: 64 sequences, 128 shared
    pages (2048 tokens), 16 own pages each."""
    plan = wl.shared_prefix_plan()
    _run(plan, cuda_device, 128, 128 * plan.page_size, "cascade shared_prefix")


@pytest.mark.parametrize("hq,hkv,d,ps,batch,prefix_pages,cut", [
    (32, 8, 128, 16, 70, 12, 5),    # 280 query rows: two row tiles; prefix ends mid-page
    (32, 1, 128, 16, 9, 40, 3),     # MQA, 288 rows; 5 key tiles over several chunks
    (4, 4, 64, 8, 33, 30, 0),       # G 1, head_dim 64, page 8
    (8, 2, 128, 64, 5, 3, 50),      # page 64, prefix of 142 tokens
])
def test_cascade_ragged(cuda_device, hq, hkv, d, ps, batch, prefix_pages, cut):
    rng = np.random.RandomState(batch + prefix_pages)
    own = rng.randint(1, 3 * ps, size=batch).tolist()
    own[0] = 0                       # prefix only
    own[-1] = 1                      # the appended token alone
    plan = _plan(f"casc_{hq}_{hkv}_{d}_{ps}", hq, hkv, d, ps, prefix_pages, own, seed=batch)
    _run(plan, cuda_device, prefix_pages, prefix_pages * ps - cut, f"cascade {hq}/{hkv}/{d} ps{ps}")


def test_cascade_long_prefix_many_chunks(cuda_device):
    """A 6000-token prefix: 47 key tiles cut into chunks across the whole GPU."""
    plan = _plan("casc_long", 32, 8, 128, 16, 375, [16, 200, 1, 33], seed=3)
    _run(plan, cuda_device, 375, 375 * 16, "cascade long prefix")


def test_cascade_zero_prefix_is_plain_decode(cuda_device):
    plan = _plan("casc_zero", 32, 8, 128, 16, 0, [40, 1, 300], seed=5)
    kp, vp, st, out = _run(plan, cuda_device, 0, 0, "cascade no prefix")
    ref = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_cascade_close_to_plain_decode_over_full_tables(cuda_device):
    """Page-aligned prefix: cascade and plain decode over prefix ++ own pages
    attend to the same keys (different reduction order, same tolerance)."""
    plan = _plan("casc_vs_plain", 32, 8, 128, 16, 20, [5, 100, 37, 250, 1], seed=6)
    kp, vp, st, out = _run(plan, cuda_device, 20, 320, "cascade vs plain")
    ref = capi.paged_attention_decode(kp, vp, st.q, st.block_table, st.seq_lens, plan.scale)
    torch.cuda.synchronize()
    diff = (out.float() - ref.float()).abs()
    assert diff.max().item() <= 2e-2 and diff.mean().item() <= 2e-3


def test_cascade_large_batch(cuda_device):
    """640 sequences (10 tiles of 256 query rows per KV head in the prefix
    pass); own parts are ragged, some sequences have none."""
    rng = np.random.RandomState(7)
    own = rng.randint(0, 40, size=640).tolist()
    plan = _plan("casc_large", 32, 8, 128, 16, 9, own, seed=12)
    _run(plan, cuda_device, 9, 9 * 16 - 3, "cascade, large batch")


def test_cascade_many_short_and_empty_own_parts(cuda_device):
    """Many segments of a few blocks each; a third of the sequences have no
    key of their own (their rows come from the prefix alone)."""
    rng = np.random.RandomState(8)
    own = rng.randint(1, 20, size=150).tolist()
    for b in range(0, 150, 3):
        own[b] = 0
    plan = _plan("casc_short", 16, 4, 128, 16, 30, own, seed=13)
    _run(plan, cuda_device, 30, 30 * 16, "cascade, short own parts")


def test_cascade_graph_replays_on_a_garbage_workspace(cuda_device):
    """A workspace filled with random bytes, then CUDA graph replays with new
    queries: every replay must recompute and merge all partials."""
    plan = wl.shared_prefix_plan(batch=24, prefix_pages=40, unique_pages=6, seed=15)
    st = wl.materialize(plan, cuda_device)
    kp, vp = st.key_pool.clone(), st.value_pool.clone()
    capi.paged_kv_append(kp, vp, st.key, st.value, st.slot_mapping)
    pre, plen, own_bt, own_lens = wl.cascade_tables(plan, 40, 40 * plan.page_size)
    dev = lambda a: torch.from_numpy(a).to(cuda_device)
    pre_t, bt_t, sl_t = dev(pre), dev(own_bt), dev(own_lens)
    ws = capi.cascade_workspace(plan.batch, plan.num_q_heads, kp)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, generator=torch.Generator().manual_seed(2)))
    q = st.q.clone()
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()

    def call():
        capi.paged_attention_decode_cascade(kp, vp, q, pre_t, plen, bt_t, sl_t, plan.scale,
                                            max_seq_len=int(own_lens.max()), out=out, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        call()                        # eager first: the first cascade call on a thread precedes any capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    kb, vb = bits(kp), bits(vp)
    for rep in range(3):
        q.copy_(torch.randn(q.shape, generator=torch.Generator().manual_seed(30 + rep)).to(q.dtype))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert capi.device_error() == (0, 0)
        exp = oracle.paged_attention_decode_cascade(to_f64(kb), to_f64(vb), to_f64(bits(q)), pre, plen, own_bt,
                                                    own_lens, plan.scale)
        assert_close(out, exp, "bf16", f"cascade graph replay {rep}")
