"""The workload builders' alternative page-table forms name the same keys.

The CSR form (``kv_indptr`` / ``kv_indices`` / ``kv_last_page_len``,
NVIDIA/recsys-examples PR #400, KVCacheMetadata) and the cascade form (shared
prefix pages + each sequence's own pages) are inputs to both the CUDA path and
the oracle in the GPU tests, so they are checked here against the dense
block table directly: slot by slot, every sequence must list the same pool
slots in the same order.
"""
import numpy as np
import pytest

from serving_slot_mapping_gb300 import workloads as wl


def _dense_slots(plan, b):
    ps, L = plan.page_size, int(plan.seq_lens[b])
    return [int(plan.block_table[b, j // ps]) * ps + j % ps for j in range(L)]


@pytest.mark.parametrize("plan", [
    wl.gqa_decode_plan(batch=7, lo=1, hi=200, seed=3),
    wl.plan_from_lengths("ragged", "decode", "bf16", 8, 2, 64, 8, np.array([0, 7, 8, 9, 63]),
                         np.ones(5), seed=4),
    wl.chunked_prefill_plan(new=(5, 40, 17), cached=(0, 33, 90), seed=7),
])
def test_csr_tables_list_the_dense_slots(plan):
    ip, ix, last = wl.csr_tables(plan)
    ps = plan.page_size
    assert ip[0] == 0 and (np.diff(ip) >= 0).all() and ip.dtype == np.int32 and ix.dtype == np.int32
    for b in range(plan.batch):
        pages = ix[ip[b]:ip[b + 1]]
        n = len(pages)
        L = (n - 1) * ps + int(last[b]) if n else 0
        assert L == int(plan.seq_lens[b])
        assert n == 0 or 1 <= last[b] <= ps
        slots = [int(pages[j // ps]) * ps + j % ps for j in range(L)]
        assert slots == _dense_slots(plan, b)


@pytest.mark.parametrize("prefix_pages,cut", [(4, 0), (4, 5), (1, 3)])
def test_cascade_tables_split_the_dense_slots(prefix_pages, cut):
    plan = wl.shared_prefix_plan(batch=5, prefix_pages=prefix_pages, unique_pages=3, seed=8, hq=8, hkv=2, d=64)
    ps = plan.page_size
    assert wl.shared_prefix_pages(plan) >= prefix_pages
    prefix_len = prefix_pages * ps - cut  # the prefix may end inside its last page
    pre, plen, own_bt, own_lens = wl.cascade_tables(plan, prefix_pages, prefix_len)
    assert plen == prefix_len and len(pre) == prefix_pages
    for b in range(plan.batch):
        dense = _dense_slots(plan, b)
        prefix = [int(pre[j // ps]) * ps + j % ps for j in range(plen)]
        own = [int(own_bt[b, j // ps]) * ps + j % ps for j in range(int(own_lens[b]))]
        # the cascade keys are the dense row's first prefix_len slots, then the
        # slots on the sequence's own pages (after the shared ones); slots of
        # the last shared page at or past prefix_len belong to neither list
        assert prefix == dense[:plen]
        assert own == dense[prefix_pages * ps:]
        if cut == 0:
            assert prefix + own == dense
