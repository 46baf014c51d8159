"""Plain fp64 statement of paged KV append + paged attention (test oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Imports: numpy.

Notation: B sequences, Hq query heads, Hkv KV heads, G = Hq // Hkv,
D head_dim, ps page_size, P num_pages.  Pools are ``[P, ps, Hkv, D]``.
Sequence b has ``L_b = seq_lens[b]`` valid KV tokens (``nonpad_kv_seqlen``)
of which the last ``n_b`` were appended this step.

Readings of points the pages leave open (each is the plainest reading that
the rest of the pages support):

1. Causal alignment.  The new tokens are the last ``n_b`` of the sequence:
   new token i sits at absolute position ``p = L_b - n_b + i`` (the write
   start plus i, because ``nonpad_kv_seqlen = write_start +
   valid_token_count``, mobius PR #395 "ONNX I/O contract") and sees keys
   ``0..p``.  Decode is the case ``n_b = 1``: the query sees all L_b keys.
2. A query row with no visible key (p < 0, i.e. n_b > L_b) has output 0;
   a decode row with L_b = 0 has output 0.
3. ``slot_mapping`` entries < 0 are padding tokens and are skipped; an entry
   >= P*ps is an error; duplicate slots in one call are an error (ScatterND
   leaves them undefined).
4. block_table entries past ``ceil(L_b/ps)`` are never read.
5. Query head hq reads KV head ``hq // G`` (contiguous groups).
6. ``scale`` multiplies q.k; it is an argument with no default.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Append: ScatterND on the flattened pool.
# ---------------------------------------------------------------------------

def paged_kv_append(key_pool, value_pool, key, value, slot_mapping):
    """Return copies of the pools with ``key[t]``/``value[t]`` written at slot t.

    ScatterND with ``indices = slot_mapping[:, None]`` on the pools viewed as
    ``[P*ps, Hkv, D]`` (mobius PR #395, "How it works (per attention layer)",
    step 1).  Works on any dtype, including raw bf16 bit patterns (uint16),
    so the comparison with a GPU pool can be bit-exact.
    """
    key_pool = np.asarray(key_pool)
    value_pool = np.asarray(value_pool)
    P, ps, hkv, d = key_pool.shape
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    key = np.asarray(key).reshape(slots.shape[0], hkv, d)
    value = np.asarray(value).reshape(slots.shape[0], hkv, d)
    live = slots[slots >= 0]
    if np.any(live >= P * ps):
        raise ValueError("slot_mapping entry out of range")
    if np.unique(live).shape[0] != live.shape[0]:
        raise ValueError("duplicate slot in one append")
    kp = key_pool.copy()
    vp = value_pool.copy()
    kflat = kp.reshape(P * ps, hkv, d)
    vflat = vp.reshape(P * ps, hkv, d)
    for t in range(slots.shape[0]):
        s = slots[t]
        if s < 0:
            continue
        kflat[s] = key[t]
        vflat[s] = value[t]
    return kp, vp


# ---------------------------------------------------------------------------
# Gather: the sequence's pages, contiguous.
# ---------------------------------------------------------------------------

def gather_pages(pool, block_table_row, seq_len):
    """``Gather(pool, block_table)`` truncated to the sequence's L tokens.

    Returns ``[L, Hkv, D]``: the first ``ceil(L/ps)`` listed pages, in order,
    concatenated (mobius PR #395, "How it works", step 2).
    """
    pool = np.asarray(pool)
    ps = pool.shape[1]
    L = int(seq_len)
    if L <= 0:
        return pool[:0, 0]
    n_pages = (L + ps - 1) // ps
    pages = [pool[int(block_table_row[m])] for m in range(n_pages)]
    return np.concatenate(pages, axis=0)[:L]


# ---------------------------------------------------------------------------
# Dense masked attention over one sequence.
# ---------------------------------------------------------------------------

def _scores(q, keys, scale, G):
    """scale * q.k for every (query row, query head, key): [n, Hq, L]."""
    n, hq, d = q.shape
    L = keys.shape[0]
    s = np.empty((n, hq, L), dtype=np.float64)
    for h in range(hq):
        s[:, h, :] = scale * (q[:, h, :] @ keys[:, h // G, :].T)
    return s


def attend_partial(q, keys, values, positions, scale):
    """Unnormalised softmax pieces over the given keys.

    For each query row i and head h, over keys j <= positions[i]:
    ``m = max_j s_j``, ``l = sum_j exp(s_j - m)``,
    ``o = sum_j exp(s_j - m) v_j``.  Rows with no visible key get
    ``m = -inf, l = 0, o = 0``.
    Returns (m [n,Hq], l [n,Hq], o [n,Hq,D]).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    n, hq, d = q.shape
    L, hkv, _ = keys.shape
    G = hq // hkv
    positions = np.asarray(positions, dtype=np.int64).reshape(n)
    m = np.full((n, hq), -np.inf)
    l = np.zeros((n, hq))
    o = np.zeros((n, hq, d))
    if L == 0:
        return m, l, o
    s = _scores(q, keys, scale, G)
    visible = np.arange(L)[None, :] <= positions[:, None]          # [n, L]
    for h in range(hq):
        sh = np.where(visible, s[:, h, :], -np.inf)
        mh = sh.max(axis=1)
        has = visible.any(axis=1)
        safe_m = np.where(has, mh, 0.0)
        w = np.where(visible, np.exp(sh - safe_m[:, None]), 0.0)
        m[:, h] = np.where(has, mh, -np.inf)
        l[:, h] = w.sum(axis=1)
        o[:, h, :] = w @ values[:, h // G, :]
    return m, l, o


def attend(q, keys, values, positions, scale):
    """softmax(scale * q K^T, masked to keys <= position) V for one sequence.

    ``q [n, Hq, D]``, ``keys/values [L, Hkv, D]``; query head h reads KV head
    ``h // G``.  Rows with no visible key give 0.
    """
    m, l, o = attend_partial(q, keys, values, positions, scale)
    out = np.zeros_like(o)
    ok = l > 0
    out[ok] = o[ok] / l[ok][:, None]
    return out


def merge_partials(parts):
    """Combine (m, l, o) partials over disjoint key sets into the output.

    ``M = max_i m_i``;  ``o = sum_i e^{m_i - M} o_i / sum_i e^{m_i - M} l_i``.
    This is the identity a split-KV (flash-decoding) combine relies on; it
    is exact up to rounding.  Entries whose l sums to 0 give 0.
    """
    ms = np.stack([p[0] for p in parts])            # [k, ...]
    ls = np.stack([p[1] for p in parts])
    os_ = np.stack([p[2] for p in parts])           # [k, ..., D]
    M = ms.max(axis=0)
    safe = np.where(np.isfinite(M), M, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - safe[None]), 0.0)
    num = (w[..., None] * os_).sum(axis=0)
    den = (w * ls).sum(axis=0)
    out = np.zeros_like(num)
    ok = den > 0
    out[ok] = num[ok] / den[ok][..., None]
    return out


# ---------------------------------------------------------------------------
# Paged entry points (the GPU path's three calls, stated plainly).
# ---------------------------------------------------------------------------

def paged_attention_decode(key_pool, value_pool, q, block_table, seq_lens, scale, seqs=None):
    """One query token per sequence, attending to all ``L_b`` keys.

    ``q [B, Hq, D]`` -> ``[B, Hq, D]`` (only rows in ``seqs`` are computed if
    given; the others stay 0).
    """
    q = np.asarray(q, dtype=np.float64)
    B = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    for b in (range(B) if seqs is None else seqs):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        K = gather_pages(key_pool, block_table[b], L)
        V = gather_pages(value_pool, block_table[b], L)
        out[b] = attend(q[b:b + 1], K, V, [L - 1], scale)[0]
    return out


def paged_attention_decode_append(key_pool, value_pool, key, value, slot_mapping, q, block_table,
                                  seq_lens, scale, seqs=None):
    """One decode step as one call: this step's K/V rows ``key/value [B, Hkv, D]``
    are appended at ``slot_mapping [B]`` (step 1 of mobius PR #395, "How it
    works (per attention layer)"), then every sequence attends over the
    updated pools with ``seq_lens`` that count the new token (step 2).
    Returns ``(key_pool', value_pool', out)``."""
    kp, vp = paged_kv_append(key_pool, value_pool, key, value, slot_mapping)
    return kp, vp, paged_attention_decode(kp, vp, q, block_table, seq_lens, scale, seqs=seqs)


def paged_attention_decode_partial(key_pool, value_pool, q, block_table, seq_lens, scale,
                                   key_ranges):
    """Decode partials over key ranges ``key_ranges[b] = (lo, hi)`` (fp64).

    Returns (m [B,Hq], l [B,Hq], o [B,Hq,D]) for keys ``lo <= j < hi`` of each
    sequence (the pieces a split-KV or cascade combine merges).
    """
    q = np.asarray(q, dtype=np.float64)
    B, hq, d = q.shape
    m = np.full((B, hq), -np.inf)
    l = np.zeros((B, hq))
    o = np.zeros((B, hq, d))
    for b in range(B):
        L = int(seq_lens[b])
        lo, hi = key_ranges[b]
        hi = min(hi, L)
        if hi <= lo:
            continue
        K = gather_pages(key_pool, block_table[b], L)[lo:hi]
        V = gather_pages(value_pool, block_table[b], L)[lo:hi]
        mb, lb, ob = attend_partial(q[b:b + 1], K, V, [hi - lo - 1], scale)
        m[b], l[b], o[b] = mb[0], lb[0], ob[0]
    return m, l, o


def paged_attention_prefill(key_pool, value_pool, q, query_start_loc, block_table, seq_lens,
                            scale, rows=None):
    """Varlen causal prefill: rows ``query_start_loc[b]..[b+1]`` of ``q [T, Hq, D]``
    are sequence b's ``n_b`` newest tokens.

    Token i of sequence b is at position ``L_b - n_b + i`` and sees keys up to
    it.  If ``rows`` (a set of packed row indices) is given, only those rows
    are computed.
    """
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.float64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    B = qsl.shape[0] - 1
    want = None if rows is None else set(int(r) for r in rows)
    for b in range(B):
        s0, s1 = int(qsl[b]), int(qsl[b + 1])
        n = s1 - s0
        if n <= 0:
            continue
        idx = list(range(s0, s1)) if want is None else [r for r in range(s0, s1) if r in want]
        if not idx:
            continue
        L = int(seq_lens[b])
        if L <= 0:
            continue
        K = gather_pages(key_pool, block_table[b], L)
        V = gather_pages(value_pool, block_table[b], L)
        pos = [L - n + (r - s0) for r in idx]
        out[idx] = attend(q[idx], K, V, pos, scale)
    return out


def paged_attention_decode_cascade(key_pool, value_pool, q, prefix_block_ids, prefix_len,
                                   block_table, seq_lens, scale, seqs=None):
    """Decode where every sequence's keys begin with one shared prefix.

    Sequence b attends to the ``prefix_len`` tokens held on the pages
    ``prefix_block_ids`` -- the same physical pages for every sequence of the
    batch, as when block tables alias the pages of a shared prompt prefix
    (the RadixAttention case of mobius PR #395, summary; the page-granular
    prefix index of ROCm/maxtext PR #93, the prefix cache (M5) commit) --
    followed by its own ``seq_lens[b]`` tokens on ``block_table[b]``.  The
    plain definition: gather both page lists, concatenate the keys (and the
    values), attend with the one decode query.  ``seq_lens`` counts only the
    sequence's own tokens; a sequence with ``prefix_len + seq_lens[b] = 0``
    gives 0.
    """
    q = np.asarray(q, dtype=np.float64)
    B = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    Kp = gather_pages(key_pool, prefix_block_ids, prefix_len)
    Vp = gather_pages(value_pool, prefix_block_ids, prefix_len)
    for b in (range(B) if seqs is None else seqs):
        L = int(seq_lens[b])
        K = np.concatenate([Kp, gather_pages(key_pool, block_table[b], L)], axis=0)
        V = np.concatenate([Vp, gather_pages(value_pool, block_table[b], L)], axis=0)
        if K.shape[0] == 0:
            continue
        out[b] = attend(q[b:b + 1], K, V, [K.shape[0] - 1], scale)[0]
    return out


def csr_pages(kv_indptr, kv_indices, kv_last_page_len, page_size, b):
    """Sequence b of a CSR page table: (its page ids, its key count).

    The compressed page-table metadata of NVIDIA/recsys-examples PR #400
    (KVCacheMetadata: kv_indices, kv_indptr, kv_last_page_len), read plainly:
    the pages are ``kv_indices[kv_indptr[b]:kv_indptr[b+1]]`` in order and the
    last one holds ``kv_last_page_len[b]`` tokens, so the sequence has
    ``(n_pages - 1) * page_size + kv_last_page_len[b]`` keys (0 without pages).
    """
    lo, hi = int(kv_indptr[b]), int(kv_indptr[b + 1])
    pages = [int(x) for x in kv_indices[lo:hi]]
    if not pages:
        return pages, 0
    return pages, (len(pages) - 1) * page_size + int(kv_last_page_len[b])


def paged_attention_decode_csr(key_pool, value_pool, q, kv_indptr, kv_indices, kv_last_page_len,
                               scale, seqs=None):
    """Decode with the page table in CSR form (see :func:`csr_pages`)."""
    q = np.asarray(q, dtype=np.float64)
    ps = np.asarray(key_pool).shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    for b in (range(q.shape[0]) if seqs is None else seqs):
        pages, L = csr_pages(kv_indptr, kv_indices, kv_last_page_len, ps, b)
        if L <= 0:
            continue
        K = gather_pages(key_pool, pages, L)
        V = gather_pages(value_pool, pages, L)
        out[b] = attend(q[b:b + 1], K, V, [L - 1], scale)[0]
    return out


def paged_attention_prefill_csr(key_pool, value_pool, q, query_start_loc, kv_indptr, kv_indices,
                                kv_last_page_len, scale, rows=None):
    """Varlen causal prefill with the page table in CSR form (see
    :func:`csr_pages` and :func:`paged_attention_prefill`)."""
    q = np.asarray(q, dtype=np.float64)
    ps = np.asarray(key_pool).shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    want = None if rows is None else set(int(r) for r in rows)
    for b in range(qsl.shape[0] - 1):
        s0, s1 = int(qsl[b]), int(qsl[b + 1])
        n = s1 - s0
        idx = list(range(s0, s1)) if want is None else [r for r in range(s0, s1) if r in want]
        if n <= 0 or not idx:
            continue
        pages, L = csr_pages(kv_indptr, kv_indices, kv_last_page_len, ps, b)
        if L <= 0:
            continue
        K = gather_pages(key_pool, pages, L)
        V = gather_pages(value_pool, pages, L)
        out[idx] = attend(q[idx], K, V, [L - n + (r - s0) for r in idx], scale)
    return out
