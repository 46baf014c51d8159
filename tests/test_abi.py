"""The C ABI: the library builds, loads, and exports every declared symbol;
host-side argument checks return the documented status codes.  No kernel
is launched here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from serving_slot_mapping_gb300 import build as build_mod
from serving_slot_mapping_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return capi.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("paged_kv_append", "paged_attention_decode", "paged_attention_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(L, n), f"missing export {n}"
        assert n in capi.SIGNATURES, f"binding does not declare {n}"


def test_abi_version(L):
    assert L.pa_abi_version() == 2
    assert b"PA_ERR_SHAPE" in L.pa_status_string(2)


def _pool(dtype=capi.PA_DTYPE_BF16, hkv=8, d=128, ps=16, P=64, k=0x10000, v=0x20000, ks=1.0, vs=1.0):
    return capi.PaKvPool(k, v, P, ps, hkv, d, dtype, ks, vs)


FAKE = ctypes.c_void_p(0x40000)  # never dereferenced: every call below fails validation


def test_append_validation(L):
    assert L.paged_kv_append(None, FAKE, FAKE, FAKE, 4, None) == capi.PA_ERR_NULL
    p = _pool(dtype=7)
    assert L.paged_kv_append(ctypes.byref(p), FAKE, FAKE, FAKE, 4, None) == capi.PA_ERR_DTYPE
    p = _pool(P=0)
    assert L.paged_kv_append(ctypes.byref(p), FAKE, FAKE, FAKE, 4, None) == capi.PA_ERR_SHAPE
    p = _pool()
    assert L.paged_kv_append(ctypes.byref(p), FAKE, FAKE, FAKE, -1, None) == capi.PA_ERR_SHAPE
    assert L.paged_kv_append(ctypes.byref(p), None, FAKE, FAKE, 4, None) == capi.PA_ERR_NULL
    assert L.paged_kv_append(ctypes.byref(p), FAKE, FAKE, ctypes.c_void_p(0x40004), 4,
                             None) == capi.PA_ERR_ALIGN
    # zero tokens: nothing to do, no launch
    assert L.paged_kv_append(ctypes.byref(p), None, None, None, 0, None) == capi.PA_OK


def _decode(L, pool, hq=32, batch=2, mb=4, msl=64, scale=0.1, ws=None, wsb=0, q=FAKE, out=None):
    return L.paged_attention_decode(ctypes.byref(pool), q, out or ctypes.c_void_p(0x50000), batch, hq,
                                    FAKE, mb, FAKE, msl, scale, ws, wsb, None)


def test_decode_validation(L):
    assert _decode(L, _pool(), hq=12) == capi.PA_ERR_SHAPE          # 12 % 8 != 0
    assert _decode(L, _pool(d=96)) == capi.PA_ERR_UNSUPPORTED       # bf16 head_dim
    # e4m3 pools: page sizes of whole 8-slot blocks only (no CUDA-core path)
    assert _decode(L, _pool(dtype=capi.PA_DTYPE_FP8_E4M3, ps=12), msl=40) == capi.PA_ERR_UNSUPPORTED
    assert _decode(L, _pool(dtype=capi.PA_DTYPE_FP8_E4M3, ps=4), msl=16) == capi.PA_ERR_UNSUPPORTED
    # bf16 pools of other page sizes take the CUDA-core path: its limits
    assert _decode(L, _pool(ps=4, d=320), msl=16) == capi.PA_ERR_UNSUPPORTED  # head_dim <= 256
    assert _decode(L, _pool(ps=4), msl=16, q=None) == capi.PA_ERR_NULL
    assert _decode(L, _pool(ps=4), msl=17) == capi.PA_ERR_SHAPE      # > max_blocks * page_size
    assert _decode(L, _pool(hkv=1), hq=64) == capi.PA_ERR_UNSUPPORTED  # group 64
    assert _decode(L, _pool(), scale=float("nan")) == capi.PA_ERR_RANGE
    assert _decode(L, _pool(), msl=65) == capi.PA_ERR_SHAPE          # > max_blocks * page_size
    assert _decode(L, _pool(), q=None) == capi.PA_ERR_NULL
    assert _decode(L, _pool(), out=FAKE) == capi.PA_ERR_SHAPE        # out aliases q
    assert _decode(L, _pool(), batch=0) == capi.PA_OK
    assert _decode(L, _pool(k=0x10008)) == capi.PA_ERR_ALIGN         # bf16 pool needs 16 B
    assert _decode(L, _pool(), ws=None, wsb=0) == capi.PA_ERR_WORKSPACE
    assert _decode(L, _pool(P=1 << 27)) == capi.PA_ERR_RANGE         # 2^31 slots: past the 32-bit row
    assert _decode(L, _pool(), batch=40000, mb=1 << 20, msl=1 << 24) == capi.PA_ERR_RANGE  # 2^30+ blocks


def test_prefill_validation(L):
    p = _pool()
    f = L.paged_attention_prefill
    assert f(ctypes.byref(p), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 10, 0, FAKE, 4, FAKE, 64,
             0.1, None) == capi.PA_ERR_SHAPE                      # max_q_len 0 with tokens
    assert f(ctypes.byref(p), FAKE, ctypes.c_void_p(0x50000), 2, 32, None, 10, 5, FAKE, 4, FAKE, 64,
             0.1, None) == capi.PA_ERR_NULL
    assert f(ctypes.byref(p), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 0, 5, FAKE, 4, FAKE, 64,
             0.1, None) == capi.PA_OK                             # nothing to do
    assert f(ctypes.byref(p), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 10, 5, FAKE, 4, FAKE, 64,
             float("inf"), None) == capi.PA_ERR_RANGE
    assert f(ctypes.byref(p), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 10, 1 << 29, FAKE, 4, FAKE, 64,
             0.1, None) == capi.PA_ERR_RANGE                      # 2^29 tokens x G 4 packed rows
    p4 = _pool(dtype=capi.PA_DTYPE_FP8_E4M3, ps=4)                 # e4m3: page_size >= 8
    assert f(ctypes.byref(p4), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 10, 5, FAKE, 4, FAKE, 16,
             0.1, None) == capi.PA_ERR_UNSUPPORTED


def test_workspace_size_is_zero_for_f32_and_positive_for_bf16(L):
    assert L.paged_attention_decode_workspace_size(4, 32, 8, 128, capi.PA_DTYPE_F32) == 0
    assert L.paged_attention_decode_workspace_size(4, 32, 8, 128, capi.PA_DTYPE_BF16) > 0


def test_cascade_validation(L):
    f = L.paged_attention_decode_cascade
    p = _pool()
    args = lambda **k: dict(dict(q=FAKE, out=ctypes.c_void_p(0x50000), batch=2, hq=32, pre=FAKE, plen=64,
                                 bt=FAKE, mb=4, sl=FAKE, msl=64, scale=0.1, ws=FAKE, wsb=1 << 30), **k)
    call = lambda pool, a: f(ctypes.byref(pool), a["q"], a["out"], a["batch"], a["hq"], a["pre"], a["plen"],
                             a["bt"], a["mb"], a["sl"], a["msl"], a["scale"], a["ws"], a["wsb"], None)
    assert call(_pool(dtype=capi.PA_DTYPE_F32), args()) == capi.PA_ERR_UNSUPPORTED   # bf16 only
    assert call(p, args(plen=-1)) == capi.PA_ERR_SHAPE
    assert call(p, args(pre=None)) == capi.PA_ERR_NULL
    assert call(p, args(wsb=16)) == capi.PA_ERR_WORKSPACE
    assert call(p, args(batch=0)) == capi.PA_OK
    # the prefix pass is the tensor-core kernel: bf16 pages of whole 8-slot blocks
    assert call(_pool(ps=4), args(msl=16)) == capi.PA_ERR_UNSUPPORTED
    assert L.paged_attention_decode_cascade_workspace_size(4, 32, 8, 128, capi.PA_DTYPE_F32) == 0


def test_e4m3_pool_validation(L):
    f8 = capi.PA_DTYPE_FP8_E4M3
    assert _decode(L, _pool(dtype=f8, ks=0.0)) == capi.PA_ERR_RANGE              # scale must be > 0
    assert _decode(L, _pool(dtype=f8, vs=float("inf"))) == capi.PA_ERR_RANGE
    assert _decode(L, _pool(dtype=f8), ws=None, wsb=0) == capi.PA_ERR_WORKSPACE  # same workspace as bf16
    assert L.paged_attention_decode_workspace_size(4, 32, 8, 128, f8) == \
        L.paged_attention_decode_workspace_size(4, 32, 8, 128, capi.PA_DTYPE_BF16)
    p = _pool(dtype=f8)
    # prefill on an e4m3 pool reads q rows 16 bytes at a time
    assert L.paged_attention_prefill(ctypes.byref(p), ctypes.c_void_p(0x40008), ctypes.c_void_p(0x50000), 2, 32,
                                     FAKE, 10, 5, FAKE, 4, FAKE, 64, 0.1, None) == capi.PA_ERR_ALIGN
    assert L.paged_attention_prefill(ctypes.byref(_pool(dtype=f8, ks=-1.0)), FAKE, ctypes.c_void_p(0x50000), 2,
                                     32, FAKE, 10, 5, FAKE, 4, FAKE, 64, 0.1, None) == capi.PA_ERR_RANGE
    assert _decode(L, _pool(dtype=3)) == capi.PA_ERR_DTYPE


def test_decode_append_validation(L):
    f = L.paged_attention_decode_append
    p = _pool()

    def call(pool=p, key=FAKE, value=FAKE, slots=FAKE, q=FAKE, out=ctypes.c_void_p(0x50000), batch=2, hq=32,
             msl=64, scale=0.1, ws=None, wsb=0):
        return f(ctypes.byref(pool), key, value, slots, q, out, batch, hq, FAKE, 4, FAKE, msl, scale, ws, wsb,
                 None)
    assert call(batch=0) == capi.PA_OK                                   # nothing to do
    assert call(key=None) == capi.PA_ERR_NULL
    assert call(slots=None) == capi.PA_ERR_NULL
    assert call(slots=ctypes.c_void_p(0x40004)) == capi.PA_ERR_ALIGN     # int64 slots: 8 B
    assert call(key=ctypes.c_void_p(0x40008)) == capi.PA_ERR_ALIGN       # 8 bf16 per access: 16 B
    assert call(out=FAKE) == capi.PA_ERR_SHAPE                           # out aliases q
    assert call(hq=12) == capi.PA_ERR_SHAPE
    assert call(scale=float("nan")) == capi.PA_ERR_RANGE
    assert call() == capi.PA_ERR_WORKSPACE                               # bf16 needs the decode workspace


def test_part_wait_hook_validation(L):
    """The wait-expiry test hook can only shorten a wait: limits outside
    1 us .. 2 s, negative or huge part counts, f32 pools and bf16 pages the
    tensor-core kernel does not take are refused before any launch."""
    f = L.pa_testing_decode_part_wait
    p = _pool()

    def call(pool=p, wait_ns=1_000_000, extra=1, ws=FAKE, wsb=1 << 30):
        return f(ctypes.byref(pool), FAKE, ctypes.c_void_p(0x50000), 2, 32, FAKE, 4, FAKE, 64, 0.1, ws, wsb,
                 wait_ns, extra, None)
    assert call(wait_ns=999) == capi.PA_ERR_RANGE
    assert call(wait_ns=2_000_000_001) == capi.PA_ERR_RANGE
    assert call(extra=-1) == capi.PA_ERR_RANGE
    assert call(extra=1025) == capi.PA_ERR_RANGE
    assert call(pool=_pool(dtype=capi.PA_DTYPE_F32)) == capi.PA_ERR_UNSUPPORTED
    assert call(pool=_pool(ps=4)) == capi.PA_ERR_UNSUPPORTED   # the CUDA-core path has no wait
    assert call(ws=None, wsb=0) == capi.PA_ERR_WORKSPACE
    assert f(None, FAKE, FAKE, 2, 32, FAKE, 4, FAKE, 64, 0.1, FAKE, 1, 1_000_000, 1, None) == capi.PA_ERR_NULL
