"""Paged (block-table) KV-cache append and attention for one GB300 (sm_103a).

The computation lives in ``libpagedattn.so`` (C ABI: ``include/paged_attn.h``);
:mod:`serving_slot_mapping_gb300.capi` is its thin Python binding and
:mod:`serving_slot_mapping_gb300.build` compiles it.
"""
from .capi import (  # noqa: F401
    paged_kv_append,
    paged_attention_decode,
    paged_attention_prefill,
    decode_workspace,
    decode_workspace_size,
    device_error,
    PagedAttnError,
    make_pool,
)
