"""Seeded synthetic workloads for paged KV-cache append + attention.

This module only *builds inputs*: sequence lengths, a page allocation
(block_table), the slot each new token is written to (slot_mapping), and
N(0,1) tensor values rounded to the pool dtype.  It contains none of the
attention or scatter arithmetic; both the CUDA path and the CPU oracle
receive exactly the arrays produced here.

Workload shapes follow the five cases the pages' method is exercised on
(tiny fp32 case, GQA decode batch, shared-prefix decode batch, mixed
chunked prefill, long-context decode with GQA and MQA).  Layout conventions
come from the I/O contract of onnxruntime/mobius PR #395 "Add paged /
block-table KV cache export" (section "ONNX I/O contract"):

* pools ``[num_pages, page_size, num_kv_heads, head_dim]`` in the model dtype;
* ``slot_mapping`` int64, one entry ``page_id * page_size + offset`` per new
  token;
* ``seq_lens`` (``nonpad_kv_seqlen``) counts the tokens already written plus
  the ones appended this step.

Pool slots that hold no live token are filled with NaN ("poisoned"), the way
recycled pages keep stale data until overwritten (ROCm/maxtext PR #93
"[Draft] kv paged kernels", allocator section on dirty pages).  Block-table
entries past a sequence's last page hold garbage (-1 or num_pages + 7).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass
class StepPlan:
    """Host-side (small) description of one append + attend step."""

    name: str
    kind: str                  # "decode" (one new token per sequence) or "prefill"
    dtype: str                 # "f32" | "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    scale: float
    seed: int
    cached: np.ndarray         # int64 [B] tokens already in the pool
    new: np.ndarray            # int64 [B] tokens appended this step
    block_table: np.ndarray    # int32 [B, max_blocks] (row padded with garbage)
    slot_mapping: np.ndarray   # int64 [T]
    query_start_loc: np.ndarray  # int32 [B+1]

    @property
    def batch(self) -> int:
        return int(self.cached.shape[0])

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.cached + self.new).astype(np.int32)

    @property
    def total_new(self) -> int:
        return int(self.new.sum())

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _pages_for(n_tokens: int, page_size: int) -> int:
    return (int(n_tokens) + page_size - 1) // page_size


def _assemble(name, kind, dtype, hq, hkv, d, ps, cached, new, page_lists, num_pages,
              scale, seed) -> StepPlan:
    """Row-pad the block tables and derive slot_mapping for the new tokens."""
    cached = np.asarray(cached, dtype=np.int64)
    new = np.asarray(new, dtype=np.int64)
    B = cached.shape[0]
    mb = max(1, max(len(p) for p in page_lists))
    bt = np.empty((B, mb), dtype=np.int64)
    for b in range(B):
        pad = -1 if b % 2 == 0 else num_pages + 7
        bt[b, :] = pad
        bt[b, : len(page_lists[b])] = page_lists[b]
    slots = []
    for b in range(B):
        for pos in range(int(cached[b]), int(cached[b] + new[b])):
            page = page_lists[b][pos // ps]
            slots.append(page * ps + pos % ps)
    qsl = np.zeros(B + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(new)
    return StepPlan(name=name, kind=kind, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=d, page_size=ps, num_pages=int(num_pages), scale=float(scale),
                    seed=seed, cached=cached, new=new, block_table=bt.astype(np.int32),
                    slot_mapping=np.asarray(slots, dtype=np.int64),
                    query_start_loc=qsl.astype(np.int32))


def plan_from_lengths(name, kind, dtype, hq, hkv, d, ps, cached, new, seed,
                      free_frac=0.0, extra_free_pages=0, shared_prefix_pages=0,
                      scale=None) -> StepPlan:
    """Allocate pages for sequences of the given lengths.

    Every sequence owns ``ceil((cached+new)/ps)`` pages, drawn without
    replacement from a randomly permuted pool.  With ``shared_prefix_pages``
    all sequences list the same first physical pages (RadixAttention-style
    sharing, mobius PR #395 "What this adds").
    """
    rng = np.random.RandomState(seed)
    cached = np.asarray(cached, dtype=np.int64)
    new = np.asarray(new, dtype=np.int64)
    B = len(cached)
    total = cached + new
    need = [_pages_for(t, ps) for t in total]
    shared = shared_prefix_pages
    own = [n - shared for n in need]
    assert all(o >= 0 for o in own)
    used = shared + sum(own)
    num_pages = used + extra_free_pages + int(math.ceil(free_frac * used))
    perm = rng.permutation(num_pages)
    shared_ids = list(perm[:shared])
    cursor = shared
    lists = []
    for b in range(B):
        lists.append(shared_ids + list(perm[cursor: cursor + own[b]]))
        cursor += own[b]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return _assemble(name, kind, dtype, hq, hkv, d, ps, cached, new, lists, num_pages,
                     scale, seed)


# ---------------------------------------------------------------------------
# The five workload families.
# ---------------------------------------------------------------------------

def tiny_f32_plans():
    """One fp32 sequence: append+prefill 100 tokens, then append+decode 1.

    GQA 2 (4 query / 2 KV heads), head_dim 64, page_size 16, a pool of 64
    pages of which 7 distinct ones (random order) hold the sequence.
    Returns (prefill_plan, decode_plan); the decode step runs on the pool the
    prefill step's append produced.
    """
    rng = np.random.RandomState(0)
    pages = list(rng.choice(64, 7, replace=False))
    pf = _assemble("tiny_f32_prefill", "prefill", "f32", 4, 2, 64, 16, [0], [100], [pages],
                   64, 1.0 / 8.0, 0)
    dc = _assemble("tiny_f32_decode", "decode", "f32", 4, 2, 64, 16, [100], [1], [pages],
                   64, 1.0 / 8.0, 0)
    return pf, dc


def gqa_decode_plan(batch=32, lo=512, hi=4096, seed=1, hq=32, hkv=8, d=128, ps=16,
                    name="gqa_decode"):
    """Llama-3-8B-like decode batch: L ~ U[lo, hi], one appended token each."""
    rng = np.random.RandomState(seed + 1000)
    L = rng.randint(lo, hi + 1, size=batch)
    return plan_from_lengths(name, "decode", "bf16", hq, hkv, d, ps, L - 1, np.ones(batch),
                             seed)


def shared_prefix_plan(batch=64, prefix_pages=128, unique_pages=16, seed=2, hq=32, hkv=8,
                       d=128, ps=16, name="shared_prefix"):
    """All sequences share ``prefix_pages`` physical pages, then own ``unique_pages``."""
    L = np.full(batch, (prefix_pages + unique_pages) * ps, dtype=np.int64)
    return plan_from_lengths(name, "decode", "bf16", hq, hkv, d, ps, L - 1, np.ones(batch),
                             seed, shared_prefix_pages=prefix_pages)


CHUNKED_NEW = (512, 768, 1024, 1024, 1536, 1536, 2048, 2048)
CHUNKED_CACHED = (0, 1024, 2048, 4096, 0, 8192, 512, 6144)


def chunked_prefill_plan(new=CHUNKED_NEW, cached=CHUNKED_CACHED, seed=3, hq=32, hkv=8, d=128,
                         ps=16, name="chunked_prefill"):
    """Varlen causal prefill of ``new`` tokens after ``cached`` context tokens."""
    return plan_from_lengths(name, "prefill", "bf16", hq, hkv, d, ps, cached, new, seed)


def long_context_plan(hkv=8, batch=256, lo=1024, hi=32768, seed=4, hq=32, d=128, ps=16,
                      name=None):
    """Long-context decode; pool = used pages + 10% free (poisoned) pages."""
    rng = np.random.RandomState(seed + 1000)
    L = rng.randint(lo, hi + 1, size=batch)
    name = name or ("long_gqa" if hkv > 1 else "long_mqa")
    return plan_from_lengths(name, "decode", "bf16", hq, hkv, d, ps, L - 1, np.ones(batch),
                             seed, free_frac=0.10)


def shared_prefix_pages(plan: StepPlan) -> int:
    """Number of leading block-table columns that every sequence shares."""
    bt = plan.block_table
    n = 0
    while n < bt.shape[1] and (bt[:, n] == bt[0, n]).all():
        n += 1
    return n


def cascade_tables(plan: StepPlan, prefix_pages: int, prefix_len: int):
    """Describe a plan whose sequences all list the same first ``prefix_pages``
    pages as a cascade decode call: (prefix page ids int32 [prefix_pages],
    prefix_len, own block table int32 [B, MB - prefix_pages], own token counts
    int32 [B]).  A sequence's own tokens are those on its pages after the
    shared ones; slots of the last shared page at or past ``prefix_len`` are
    not part of the prefix.
    """
    bt = plan.block_table
    B = bt.shape[0]
    pre = np.ascontiguousarray(bt[0, :prefix_pages]).astype(np.int32)
    assert prefix_pages == 0 or (bt[:, :prefix_pages] == pre[None, :]).all()
    assert 0 <= prefix_len <= prefix_pages * plan.page_size
    own_bt = np.ascontiguousarray(bt[:, prefix_pages:]).astype(np.int32)
    if own_bt.shape[1] == 0:
        own_bt = np.full((B, 1), -1, dtype=np.int32)
    own_lens = (plan.seq_lens.astype(np.int64) - prefix_pages * plan.page_size).astype(np.int32)
    assert (own_lens >= 0).all()
    return pre, int(prefix_len), own_bt, own_lens


def csr_tables(plan: StepPlan):
    """The plan's page table in CSR form: (kv_indptr int32 [B+1], kv_indices
    int32 [nnz], kv_last_page_len int32 [B]); each sequence lists its
    ceil(L/ps) pages, the last one holding L - (n-1)*ps tokens."""
    ps = plan.page_size
    indptr, indices, last = [0], [], []
    for b, L in enumerate(plan.seq_lens.tolist()):
        n = (L + ps - 1) // ps
        indices.extend(plan.block_table[b, :n].tolist())
        indptr.append(len(indices))
        last.append(L - (n - 1) * ps if n else 0)
    return (np.asarray(indptr, dtype=np.int32), np.asarray(indices or [0], dtype=np.int32),
            np.asarray(last, dtype=np.int32))


def named_plan(name: str) -> StepPlan:
    table = {
        "gqa_decode": lambda: gqa_decode_plan(),
        "shared_prefix": lambda: shared_prefix_plan(),
        "chunked_prefill": lambda: chunked_prefill_plan(),
        "long_gqa": lambda: long_context_plan(hkv=8, seed=4),
        "long_mqa": lambda: long_context_plan(hkv=1, seed=5),
    }
    return table[name]()


# ---------------------------------------------------------------------------
# Materialisation: tensors on a device.
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class StepTensors:
    plan: StepPlan
    key_pool: torch.Tensor        # [P, ps, Hkv, D]  (state before this step's append)
    value_pool: torch.Tensor
    key: torch.Tensor             # [T, Hkv, D] new rows
    value: torch.Tensor
    q: torch.Tensor               # [B, Hq, D] (decode) or [T, Hq, D] (prefill)
    slot_mapping: torch.Tensor    # int64 [T]
    block_table: torch.Tensor     # int32 [B, MB]
    seq_lens: torch.Tensor        # int32 [B]
    query_start_loc: torch.Tensor  # int32 [B+1]


def _randn(shape, gen, device, dtype, chunk_elems=1 << 28):
    """N(0,1) fp32 draws rounded (RNE) to ``dtype``, generated in chunks."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def live_slot_mask(plan: StepPlan, include_new: bool = False) -> np.ndarray:
    """Boolean [P*ps]: slots holding a cached token (optionally also new ones)."""
    P, ps = plan.num_pages, plan.page_size
    mask = np.zeros(P * ps, dtype=bool)
    for b in range(plan.batch):
        n_live = int(plan.cached[b] + (plan.new[b] if include_new else 0))
        row = plan.block_table[b]
        full, rem = divmod(n_live, ps)
        for m in range(full):
            mask[int(row[m]) * ps: int(row[m]) * ps + ps] = True
        if rem:
            mask[int(row[full]) * ps: int(row[full]) * ps + rem] = True
    return mask


def materialize(plan: StepPlan, device="cpu", poison=float("nan"),
                key_pool: Optional[torch.Tensor] = None,
                value_pool: Optional[torch.Tensor] = None) -> StepTensors:
    """Draw the step's tensors with a torch generator seeded by ``plan.seed``.

    Cached-context slots get N(0,1) values, every other slot ``poison``.  If
    pools are passed in (a later step of the same sequences), they are used
    as they are.
    """
    device = torch.device(device)
    dt = DTYPES[plan.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(int(plan.seed) * 7919 + 17)
    P, ps, hkv, d = plan.num_pages, plan.page_size, plan.num_kv_heads, plan.head_dim
    if key_pool is None:
        key_pool = _randn((P, ps, hkv, d), gen, device, dt)
        value_pool = _randn((P, ps, hkv, d), gen, device, dt)
        dead = torch.from_numpy(~live_slot_mask(plan)).to(device)
        key_pool.view(P * ps, hkv, d)[dead] = poison
        value_pool.view(P * ps, hkv, d)[dead] = poison
    T = plan.total_new
    key = _randn((T, hkv, d), gen, device, dt)
    value = _randn((T, hkv, d), gen, device, dt)
    rows = plan.batch if plan.kind == "decode" else T
    q = _randn((rows, plan.num_q_heads, d), gen, device, dt)
    return StepTensors(
        plan=plan, key_pool=key_pool, value_pool=value_pool, key=key, value=value, q=q,
        slot_mapping=torch.from_numpy(plan.slot_mapping).to(device),
        block_table=torch.from_numpy(plan.block_table).to(device),
        seq_lens=torch.from_numpy(plan.seq_lens).to(device),
        query_start_loc=torch.from_numpy(plan.query_start_loc).to(device))


def subset_plan(plan: StepPlan, seqs: Sequence[int]) -> StepPlan:
    """The same step restricted to some sequences (for sampled oracle checks).

    Block tables, slots and the pool geometry are unchanged, so the subset
    reads the very pages the full batch reads.
    """
    seqs = list(seqs)
    lists = []
    for b in seqs:
        n = _pages_for(plan.cached[b] + plan.new[b], plan.page_size)
        lists.append(list(plan.block_table[b, :n]))
    return _assemble(plan.name + "_subset", plan.kind, plan.dtype, plan.num_q_heads,
                     plan.num_kv_heads, plan.head_dim, plan.page_size, plan.cached[seqs],
                     plan.new[seqs], lists, plan.num_pages, plan.scale, plan.seed)


# ---------------------------------------------------------------------------
# Algorithmic work (for throughput accounting, not for computing results).
# ---------------------------------------------------------------------------

def elem_bytes(plan: StepPlan) -> int:
    return 4 if plan.dtype == "f32" else 2


def decode_kv_bytes(plan: StepPlan) -> int:
    """K and V bytes a decode step must read once: sum_b L_b * Hkv * D * 2 * elem."""
    return int(plan.seq_lens.astype(np.int64).sum()) * plan.num_kv_heads * plan.head_dim * 2 \
        * elem_bytes(plan)


def decode_unique_kv_bytes(plan: StepPlan) -> int:
    """Bytes of distinct live slots (shared prefix pages counted once)."""
    pages = set()
    slots = 0
    for b in range(plan.batch):
        L = int(plan.seq_lens[b])
        for m in range(_pages_for(L, plan.page_size)):
            pid = int(plan.block_table[b, m])
            if pid not in pages:
                pages.add(pid)
                slots += min(plan.page_size, L - m * plan.page_size)
    return slots * plan.num_kv_heads * plan.head_dim * 2 * elem_bytes(plan)


def decode_io_bytes(plan: StepPlan) -> int:
    """q in + out + block table rows + seq_lens."""
    e = elem_bytes(plan)
    qo = 2 * plan.batch * plan.num_q_heads * plan.head_dim * e
    bt = int(sum(_pages_for(l, plan.page_size) for l in plan.seq_lens)) * 4 + plan.batch * 4
    return qo + bt


def append_bytes(plan: StepPlan) -> int:
    """Rows read + written once, plus the slot ids."""
    T = plan.total_new
    return 2 * 2 * T * plan.num_kv_heads * plan.head_dim * elem_bytes(plan) + 8 * T


def prefill_visible_pairs(plan: StepPlan) -> int:
    """Number of (query token, key) pairs the causal mask lets through."""
    n = plan.new.astype(np.int64)
    c = plan.cached.astype(np.int64)
    return int((n * c + n * (n + 1) // 2).sum())


def prefill_flops(plan: StepPlan) -> int:
    """QK^T and PV over visible pairs: 2 matmuls x 2 flop/MAC x D, per query head."""
    return prefill_visible_pairs(plan) * 4 * plan.head_dim * plan.num_q_heads
