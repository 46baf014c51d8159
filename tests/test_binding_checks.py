"""The ctypes binding's tensor checks (no GPU: every call below is refused in
Python before the library is called).  The C ABI takes untyped pointers, so
the binding is where a query, output or new-row tensor of the wrong dtype or
head size is caught."""
import pytest
import torch

from serving_slot_mapping_gb300 import capi


def _pools(dtype=torch.bfloat16, P=4, ps=16, hkv=2, d=64):
    return torch.zeros(P, ps, hkv, d, dtype=dtype), torch.zeros(P, ps, hkv, d, dtype=dtype)


def _tables(B=3, mb=2):
    return torch.zeros(B, mb, dtype=torch.int32), torch.ones(B, dtype=torch.int32)


@pytest.mark.parametrize("pool_dtype,q", [
    (torch.bfloat16, torch.zeros(3, 4, 64)),                          # f32 q on a bf16 pool
    (torch.bfloat16, torch.zeros(3, 4, 32, dtype=torch.bfloat16)),   # head_dim mismatch
    (torch.float8_e4m3fn, torch.zeros(3, 4, 64, dtype=torch.float8_e4m3fn)),  # e4m3 pools take bf16 q
    (torch.float32, torch.zeros(3, 4, 64, dtype=torch.bfloat16)),    # f32 pools take f32 q
])
def test_decode_rejects_query_of_wrong_dtype_or_head_dim(pool_dtype, q):
    kp, vp = _pools(pool_dtype)
    bt, sl = _tables()
    with pytest.raises(ValueError, match="q must be"):
        capi.paged_attention_decode(kp, vp, q, bt, sl, 0.1)


def test_decode_rejects_mismatched_out():
    kp, vp = _pools()
    bt, sl = _tables()
    q = torch.zeros(3, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must match"):
        capi.paged_attention_decode(kp, vp, q, bt, sl, 0.1, out=torch.zeros(3, 4, 64))


def test_prefill_and_csr_wrappers_check_the_query_too():
    kp, vp = _pools()
    bt, sl = _tables()
    qsl = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    bad = torch.zeros(3, 4, 64)
    with pytest.raises(ValueError, match="q must be"):
        capi.paged_attention_prefill(kp, vp, bad, qsl, bt, sl, 0.1, max_q_len=1)
    ip = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    with pytest.raises(ValueError, match="q must be"):
        capi.paged_attention_decode_csr(kp, vp, bad, ip, ip[:3], sl, 0.1, max_seq_len=16)


def test_fused_wrapper_checks_its_new_rows():
    kp, vp = _pools()
    bt, sl = _tables()
    q = torch.zeros(3, 4, 64, dtype=torch.bfloat16)
    slots = torch.zeros(3, dtype=torch.int64)
    good = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="key must be"):
        capi.paged_attention_decode_append(kp, vp, torch.zeros(3, 2, 64), good, slots, q, bt, sl, 0.1)
    with pytest.raises(ValueError, match="value must be"):
        capi.paged_attention_decode_append(kp, vp, good, torch.zeros(3, 2, 32, dtype=torch.bfloat16), slots,
                                           q, bt, sl, 0.1)
    with pytest.raises(ValueError, match="slot_mapping"):
        capi.paged_attention_decode_append(kp, vp, good, good, slots[:2], q, bt, sl, 0.1)
    with pytest.raises(TypeError, match="int64"):
        capi.paged_attention_decode_append(kp, vp, good, good, slots.int(), q, bt, sl, 0.1)
