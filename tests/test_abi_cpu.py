"""CPU-only checks of the C ABI: the library loads, exports every declared
symbol, reports cache layout sizes, and rejects bad arguments before any
device work (no GPU needed: validation returns before a launch)."""
import ctypes
import os
import re

import numpy as np
import pytest

from attention_group_quantized_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(kvq.LIB_PATH):
        from attention_group_quantized_gb300 import build
        build.build()
    return kvq.lib()


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert set(declared) == set(kvq.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for s in range(8):
        assert L.kvq_status_str(s)
    assert L.kvq_status_str(99) == b"unknown status"


def test_cache_layout_sizes(L):
    hb = np.array([8, 4, 4, 8], np.int8)
    B, Tcap, D = 3, 128, 128
    nc, ns = kvq.cache_nbytes(hb, B, Tcap, D)
    assert nc == B * Tcap * (2 * 128 + 2 * 64)
    assert ns == 4 * B * Tcap * 4 * 4
    cs = kvq.CCache(None, None, hb.ctypes.data, B, 4, Tcap, D)
    offs = [L.kvq_cache_head_offset(ctypes.byref(cs), h) for h in range(4)]
    plane8, plane4 = B * Tcap * 128, B * Tcap * 64
    # 8-bit planes first in head order, then 4-bit planes in head order
    assert offs == [0, 2 * plane8, 2 * plane8 + plane4, plane8]
    assert L.kvq_cache_head_offset(ctypes.byref(cs), 4) == -1


def test_cache_layout_rejects_bad_shapes(L):
    hb = np.array([8, 5], np.int8)
    cs = kvq.CCache(None, None, hb.ctypes.data, 1, 2, 64, 128)
    assert L.kvq_cache_codes_bytes(ctypes.byref(cs)) == -1
    hb = np.array([8], np.int8)
    for B, Tcap, D in [(0, 64, 128), (1, 100, 128), (1, 64, 96)]:
        cs = kvq.CCache(None, None, hb.ctypes.data, B, 1, Tcap, D)
        assert L.kvq_cache_codes_bytes(ctypes.byref(cs)) == -1


def _cache(hb, B=1, Tcap=64, D=128, codes=0x1000, sz=0x2000):
    hb = np.asarray(hb, np.int8)
    return kvq.CCache(codes, sz, hb.ctypes.data, B, len(hb), Tcap, D), hb


def test_quantize_validation_without_launch(L):
    c, hb = _cache([8])
    P = ctypes.byref
    assert L.kvq_quantize(None, 0, 0, 128, 0, 1, P(c), None, None) == 1
    assert L.kvq_quantize(0x3000, 0, 0, 128, 0, 65, P(c), None, None) == 1        # past capacity
    assert L.kvq_quantize(0x3000, 0, 0, 128, -1, 1, P(c), None, None) == 1
    assert L.kvq_quantize(0x3002, 0, 0, 128, 0, 1, P(c), None, None) == 1        # misaligned rows
    assert L.kvq_quantize(0x3000, 0, 0, 100, 0, 1, P(c), None, None) == 1        # row stride not 16 B
    c2, hb2 = _cache([8], D=96)
    assert L.kvq_quantize(0x3000, 0, 0, 96, 0, 1, P(c2), None, None) == 2
    assert L.kvq_quantize(0x3000, 0, 0, 128, 0, 0, P(c), None, None) == 0        # nothing to do


def test_decode_validation_without_launch(L):
    k, hk = _cache([8, 8])
    v, hv = _cache([8, 8])
    P = ctypes.byref
    q, lens, out, ws = 0x4000, 0x5000, 0x6000, 0x7000
    assert L.kvq_decode_attention(None, P(k), P(v), lens, 8, 0.0, out, 0, ws, 1 << 20, None, None) == 1
    assert L.kvq_decode_attention(q, P(k), P(v), lens, 7, 0.0, out, 0, ws, 1 << 20, None, None) == 1   # Hq % Hkv
    assert L.kvq_decode_attention(q, P(k), P(v), lens, 32, 0.0, out, 0, ws, 1 << 20, None, None) == 2  # 16 per KV
    assert L.kvq_decode_attention(q, P(k), P(v), lens, 8, 0.0, out, 5, ws, 1 << 20, None, None) == 1   # dtype
    v2, hv2 = _cache([8, 4])
    assert L.kvq_decode_attention(q, P(k), P(v2), lens, 8, 0.0, out, 0, ws, 1 << 20, None, None) == 1  # bits differ
    assert L.kvq_decode_attention(q + 8, P(k), P(v), lens, 8, 0.0, out, 0, ws, 1 << 20, None, None) == 1


def test_prefill_validation_without_launch(L):
    k, hk = _cache([8, 8], Tcap=256)
    v, hv = _cache([8, 8], Tcap=256)
    P = ctypes.byref
    a = 0x8000
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, 256, 128, 2, 0.0, None, 128, P(k), P(v), a, 0, None, None) == 2
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, 256, 128, 1, 0.0, None, 64, P(k), P(v), a, 0, None, None) == 2
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, 200, 128, 1, 0.0, None, 128, P(k), P(v), a, 0, None, None) == 2
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, 512, 128, 1, 0.0, None, 128, P(k), P(v), a, 0, None, None) == 1
    assert L.kvq_prefill_attention(a, a, a, 1, 3, 2, 256, 128, 1, 0.0, None, 128, P(k), P(v), a, 0, None, None) == 1
    # head dims other than 64 and 128 are refused (4-bit and mixed per-head caches are accepted)
    k96, _ = _cache([8, 4], Tcap=256, D=96)
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, 256, 96, 1, 0.0, None, 128, P(k96), P(k96), a, 0, None,
                                   None) == 2


def test_prefill_varlen_validation_without_launch(L):
    """The varlen entry point checks what the plain one checks, plus its lengths pointer, before any launch."""
    k, hk = _cache([8, 8], Tcap=256)
    v, hv = _cache([8, 8], Tcap=256)
    P = ctypes.byref
    a, lens = 0x8000, 0x9000
    call = lambda **o: L.kvq_prefill_attention_varlen(
        a, a, a, 1, o.get("Hq", 4), 2, o.get("S", 256), 128, o.get("lens", lens), o.get("causal", 1), 0.0, None,
        o.get("tile", 128), P(k), P(v), a, 0, None, None)
    assert call(lens=None) == 1
    assert call(causal=2) == 2
    assert call(tile=64) == 2
    assert call(S=200) == 2
    assert call(S=512) == 1          # longer than the caches
    assert call(Hq=3) == 1


def test_prefill_rejects_a_mask_too_large_to_index(L):
    """nT * nT >= 2^31 with a mask: unsupported before any other check needs the caches."""
    k, hk = _cache([8, 8], Tcap=128)
    v, hv = _cache([8, 8], Tcap=128)
    P = ctypes.byref
    a = 0x8000
    S = 46341 * 128                    # nT = 46341, nT^2 > 2^31
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, S, 128, 1, 0.0, a, 128, P(k), P(v), a, 0, None, None) == 2
    # the same length without a mask gets as far as the cache-shape check
    assert L.kvq_prefill_attention(a, a, a, 1, 4, 2, S, 128, 1, 0.0, None, 128, P(k), P(v), a, 0, None, None) == 1


def test_decode_step_validation_without_launch(L):
    k, hk = _cache([8, 8])
    v, hv = _cache([8, 8])
    P = ctypes.byref
    q, kn, vn, lens, out, ws = 0x4000, 0x9000, 0xA000, 0x5000, 0x6000, 0x7000
    args = lambda **o: [o.get("q", q), o.get("kn", kn), o.get("vn", vn), P(k), P(o.get("v", v)), lens,
                        o.get("Hq", 8), 0.0, out, o.get("dt", 0), ws, 1 << 20, None, None]
    assert L.kvq_decode_step(*args(kn=None)) == 1
    assert L.kvq_decode_step(*args(vn=vn + 4)) == 1          # misaligned new row
    assert L.kvq_decode_step(*args(q=None)) == 1
    assert L.kvq_decode_step(*args(Hq=7)) == 1
    assert L.kvq_decode_step(*args(Hq=32)) == 2              # 16 query heads per KV head
    assert L.kvq_decode_step(*args(dt=5)) == 1
    v2, hv2 = _cache([8, 4])
    assert L.kvq_decode_step(*args(v=v2)) == 1               # bit-widths differ


def test_decode_step_staging_bytes(L):
    r = lambda x: (x + 255) // 256 * 256
    for B, Hq, Hkv, D, dt in [(8, 32, 8, 128, 0), (8, 32, 8, 128, 1), (3, 4, 4, 64, 0), (1, 1, 1, 64, 1)]:
        q, kv = B * Hq * D * 2, B * Hkv * D * 2
        o = B * Hq * D * (4 if dt == 0 else 2)
        assert L.kvq_decode_step_staging_bytes(B, Hq, Hkv, D, dt) == r(q) + 2 * r(kv) + r(o)
    assert L.kvq_decode_step_staging_bytes(1, 3, 2, 128, 0) == 0
    assert L.kvq_decode_step_staging_bytes(1, 4, 2, 96, 0) == 0
    assert L.kvq_decode_step_staging_bytes(1, 4, 2, 128, 7) == 0


def test_decode_step_host_validation_without_launch(L):
    k, hk = _cache([8, 8])
    v, hv = _cache([8, 8])
    P = ctypes.byref
    h, lens, st, ws = 0x10000, 0x5000, 0x20000, 0x7000
    need = L.kvq_decode_step_staging_bytes(1, 8, 2, 128, 0)
    call = lambda stg, n, qh=h, dt=0: L.kvq_decode_step_host(qh, h, h, P(k), P(v), lens, 8, 0.0, h, dt, stg, n,
                                                             ws, 1 << 20, None, None)
    assert call(st, need, qh=None) == 1
    assert call(None, need) == 1
    assert call(st, need - 1) == 1                            # staging too small
    assert call(st + 16, need) == 1                           # staging not 256-byte aligned
    assert call(st, need, dt=3) == 1


def test_policy_defaults_and_validation_without_launch(L):
    """kvq_policy_default fills the values the plain calls use; an
    out-of-range field is refused before any device work."""
    p = kvq.CPolicy()
    L.kvq_policy_default(ctypes.byref(p))
    assert (p.decode_ring_tiles, p.decode_l2_warm_tiles, p.wait_limit_us, p.test_issue_limit) == (4, 5, 2_000_000, -1)
    c, hb = _cache([8], B=1, Tcap=64)
    c128, hb128 = _cache([8], B=1, Tcap=128)
    P = ctypes.byref
    bad = [("decode_ring_tiles", 1), ("decode_ring_tiles", 3), ("decode_ring_tiles", 5), ("decode_l2_warm_tiles", -1),
           ("decode_l2_warm_tiles", 17), ("wait_limit_us", 0),
           ("wait_limit_us", 60_000_001)]
    for field, val in bad:
        q = kvq.CPolicy()
        L.kvq_policy_default(ctypes.byref(q))
        setattr(q, field, val)
        st = L.kvq_decode_attention_ex(0x3000, P(c), P(c), 0x4000, 4, 0.0, 0x5000, 0, 0x6000, 1 << 20, P(q),
                                       None, None)
        assert st == 1, (field, val)
        st = L.kvq_prefill_attention_ex(0x3000, 0x3000, 0x3000, 1, 4, 1, 128, 128, None, 1, 0.0, None, 128,
                                        P(c128), P(c128), 0x5000, 0, P(q), None, None)
        assert st == 1, (field, val)


class _FakeBuf:
    """Stands in for a tensor: an address and a size, never dereferenced (the call fails first)."""

    def __init__(self, ptr, n=0, shape=()):
        self.ptr, self.n, self.shape = ptr, n, shape

    def data_ptr(self):
        return self.ptr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


class _FakeStream:
    cuda_stream = None


def test_prepared_decode_step_host_marshals_its_arguments(L):
    """DecodeStepHost converts every argument once and calls through a handle
    without ctypes conversion: a staging buffer one byte short must come back
    as INVALID_ARG, one of the exact size must pass that check and fail only
    at the first CUDA call (no GPU here), and a second run reuses the caches'
    C views."""
    B, Hq, Hkv, D = 1, 8, 2, 128
    need = L.kvq_decode_step_staging_bytes(B, Hq, Hkv, D, 0)
    mk = lambda: kvq.QuantCache(_FakeBuf(0x100000), _FakeBuf(0x200000), np.array([8, 8], np.int8), B, Hkv, 128, D)
    k, v = mk(), mk()
    q, kn = _FakeBuf(0x10000, shape=(B, Hq, D)), _FakeBuf(0x11000, shape=(B, Hkv, D))
    args = (q, kn, _FakeBuf(0x12000), _FakeBuf(0x5000), _FakeBuf(0x13000))
    short = kvq.DecodeStepHost(*args, 0.1, staging=_FakeBuf(0x20000, need - 1), workspace=_FakeBuf(0x7000, 1 << 20),
                               stream=_FakeStream())
    with pytest.raises(kvq.KvqError) as e:
        short.run(k, v)
    assert e.value.status == 1
    exact = kvq.DecodeStepHost(*args, 0.1, staging=_FakeBuf(0x20000, need), workspace=_FakeBuf(0x7000, 1 << 20),
                               stream=_FakeStream())
    for _ in range(2):
        with pytest.raises(kvq.KvqError) as e:
            exact.run(k, v)
        assert e.value.status not in (0, 1)
    assert len(exact._views) == 2


def test_debug_library_exports_every_declared_symbol(L):
    """libkvq_debug.so (the kernels with index checks) is a drop-in: same exports,
    and the status it adds has its own string."""
    if not os.path.exists(kvq.DEBUG_LIB_PATH):
        from attention_group_quantized_gb300 import build
        build.build(debug=True)
    D = ctypes.CDLL(kvq.DEBUG_LIB_PATH)
    for name in _declared_functions():
        assert hasattr(D, name), name
    D.kvq_status_str.restype = ctypes.c_char_p
    assert D.kvq_status_str(7) == b"device index check failed (debug build)"
    assert L.kvq_status_str(7) == D.kvq_status_str(7)


def test_decode_refuses_more_sequences_than_its_length_table(L):
    """4097 sequences: KVQ_ERR_UNSUPPORTED before any launch (the decode kernel's
    shared-memory length table holds 4096)."""
    k, hk = _cache([8], B=4097, Tcap=64)
    v, hv = _cache([8], B=4097, Tcap=64)
    P = ctypes.byref
    st = L.kvq_decode_attention(0x10000, P(k), P(v), 0x5000, 8, 0.0, 0x20000, 0, 0x30000, 1 << 30, None, None)
    assert st == 2
