"""fp64 CPU oracle for paged KV-cache append and paged attention.

TEST INFRASTRUCTURE.  This package is the slow, plain statement of what the
GPU path computes.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import it; the library under
``serving_slot_mapping_gb300`` never does, and it shares no code with it.
It imports nothing but the Python standard library and numpy.

What it follows:

* append: the ScatterND write of new K/V rows into the per-layer page pool at
  ``slot_mapping`` (onnxruntime/mobius PR #395 "Add paged / block-table KV
  cache export", sections "How it works (per attention layer)" and "ONNX I/O
  contract");
* gather: ``Gather(pool, block_table)`` assembling a sequence's physical
  pages contiguously (same page, same sections);
* attention: softmax attention with causal + padding masking derived from
  ``is_causal=1`` and ``nonpad_kv_seqlen`` (same page, "ONNX I/O contract"),
  grouped-query heads where query head ``i`` reads KV head ``i // G``
  (ROCm/maxtext PR #93 "[Draft] kv paged kernels", the KV-pool sharding
  commit), and an explicit softmax scale (same page, the ``gpu_paged``
  commit and the double-scaling fix);
* the split-softmax merge identity used to combine partial results;
* decode over a prefix shared by the whole batch (block tables aliasing the
  pages of a common prompt prefix: the RadixAttention case of the mobius
  page, summary, and the prefix index of the maxtext page, M5 commit),
  defined plainly as attention over the prefix keys followed by the
  sequence's own keys;
* fp8 (e4m3) pools with one scale per tensor (:mod:`oracle.kv_fp8`): the
  quantising append and decode over the values the codes stand for;
* the compressed (CSR) page-table form ``kv_indptr`` / ``kv_indices`` /
  ``kv_last_page_len`` named by NVIDIA/recsys-examples PR #400
  (KVCacheMetadata);
* one decode step as one call: the append of the step's rows followed by
  the decode that attends to them (mobius page, "How it works (per
  attention layer)", steps 1 and 2).

Readings where the pages are silent are listed in the module docstring of
:mod:`oracle.paged_attention`.

Every function is pinned by the ``-m "not gpu"`` tests in ``tests/``
(brute force, closed forms, a library attention routine on dense data,
page-permutation and shared-prefix invariants); none is "parity unpinned".
"""
from .paged_attention import (  # noqa: F401
    paged_kv_append,
    gather_pages,
    attend,
    attend_partial,
    merge_partials,
    paged_attention_decode,
    paged_attention_prefill,
    paged_attention_decode_partial,
    paged_attention_decode_cascade,
    paged_attention_decode_append,
    csr_pages,
    paged_attention_decode_csr,
    paged_attention_prefill_csr,
)
from . import kv_fp8  # noqa: F401,E402
