"""Thin Python binding of libkvq (the C ABI declared in include/kvq.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  If the
library has not been built, :func:`lib` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")
# the same kernels built with KVQ_DEBUG=1 (device index checks; see build.py)
DEBUG_LIB_PATH = os.path.join(HERE, "libkvq_debug.so")

KVQ_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
                4: "workspace", 5: "timeout", 6: "non-finite", 7: "index check (debug build)"}
OUT_F32 = 0
OUT_BF16 = 1
GROUP = 32
TILE_TOKENS = 64

# every symbol include/kvq.h declares
EXPORTS = ("kvq_cache_codes_bytes", "kvq_cache_sz_bytes", "kvq_cache_head_offset", "kvq_quantize",
           "kvq_decode_workspace_bytes", "kvq_decode_attention", "kvq_prefill_attention",
           "kvq_decode_attention_noalloc", "kvq_decode_step", "kvq_decode_step_staging_bytes",
           "kvq_decode_step_host", "kvq_quantize_paged", "kvq_decode_attention_paged", "kvq_decode_step_paged",
           "kvq_build_tile_mask", "kvq_prefill_attention_varlen", "kvq_head_error_stats_workspace_bytes", "kvq_head_error_stats",
           "kvq_allocate_head_bits", "kvq_status_str", "kvq_policy_default", "kvq_decode_attention_ex",
           "kvq_prefill_attention_ex")


class CBlockTable(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("B", ctypes.c_int32), ("max_pages", ctypes.c_int32)]


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status})")
        self.status = status


class CPolicy(ctypes.Structure):
    _fields_ = [("decode_ring_tiles", ctypes.c_int32), ("decode_l2_warm_tiles", ctypes.c_int32),
                ("wait_limit_us", ctypes.c_uint32), ("test_issue_limit", ctypes.c_int32)]


class CCache(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sz", ctypes.c_void_p), ("head_bits", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("Tcap", ctypes.c_int32),
                ("D", ctypes.c_int32)]


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libkvq.so (once).  Raises if it is missing: there is no CPU path."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so not found at {LIB_PATH}; build it with "
                               "attention_group_quantized_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        CP = ctypes.POINTER(CCache)
        L.kvq_cache_codes_bytes.argtypes = [CP]; L.kvq_cache_codes_bytes.restype = I64
        L.kvq_cache_sz_bytes.argtypes = [CP]; L.kvq_cache_sz_bytes.restype = I64
        L.kvq_cache_head_offset.argtypes = [CP, I32]; L.kvq_cache_head_offset.restype = I64
        L.kvq_quantize.argtypes = [P, I64, I64, I64, I32, I32, CP, P, P]; L.kvq_quantize.restype = I32
        L.kvq_decode_workspace_bytes.argtypes = [I32, I32, I32, I32]; L.kvq_decode_workspace_bytes.restype = SZ
        L.kvq_decode_attention.argtypes = [P, CP, CP, P, I32, F32, P, I32, P, SZ, P, P]
        L.kvq_decode_attention.restype = I32
        L.kvq_prefill_attention.argtypes = [P, P, P, I32, I32, I32, I32, I32, I32, F32, P, I32, CP, CP, P, I32,
                                            P, P]
        L.kvq_prefill_attention.restype = I32
        L.kvq_prefill_attention_varlen.argtypes = [P, P, P, I32, I32, I32, I32, I32, P, I32, F32, P, I32, CP, CP,
                                                   P, I32, P, P]
        L.kvq_prefill_attention_varlen.restype = I32
        L.kvq_decode_attention_noalloc.argtypes = [P, CP, CP, P, I32, F32, P, I32, P, P]
        L.kvq_decode_attention_noalloc.restype = I32
        L.kvq_decode_step.argtypes = [P, P, P, CP, CP, P, I32, F32, P, I32, P, SZ, P, P]
        L.kvq_decode_step.restype = I32
        L.kvq_decode_step_staging_bytes.argtypes = [I32, I32, I32, I32, I32]
        L.kvq_decode_step_staging_bytes.restype = SZ
        L.kvq_decode_step_host.argtypes = [P, P, P, CP, CP, P, I32, F32, P, I32, P, SZ, P, SZ, P, P]
        L.kvq_decode_step_host.restype = I32
        BT = ctypes.POINTER(CBlockTable)
        L.kvq_quantize_paged.argtypes = [P, I64, I64, I64, I32, I32, CP, BT, P, P]
        L.kvq_quantize_paged.restype = I32
        L.kvq_decode_attention_paged.argtypes = [P, CP, CP, BT, P, I32, F32, P, I32, P, SZ, P, P]
        L.kvq_decode_attention_paged.restype = I32
        L.kvq_decode_step_paged.argtypes = [P, P, P, CP, CP, BT, P, I32, F32, P, I32, P, SZ, P, P]
        L.kvq_decode_step_paged.restype = I32
        L.kvq_build_tile_mask.argtypes = [P, I32, I32, I32, ctypes.c_uint64, P]
        L.kvq_build_tile_mask.restype = I32
        L.kvq_head_error_stats_workspace_bytes.argtypes = [I32]
        L.kvq_head_error_stats_workspace_bytes.restype = SZ
        L.kvq_head_error_stats.argtypes = [P, I32, I32, I32, I32, P, P, I32, P, P, SZ, P, P]
        L.kvq_head_error_stats.restype = I32
        L.kvq_allocate_head_bits.argtypes = [P, P, I32, I32, I32, P, P]
        L.kvq_allocate_head_bits.restype = I32
        L.kvq_status_str.argtypes = [I32]; L.kvq_status_str.restype = ctypes.c_char_p
        PP = ctypes.POINTER(CPolicy)
        L.kvq_policy_default.argtypes = [PP]; L.kvq_policy_default.restype = None
        L.kvq_decode_attention_ex.argtypes = [P, CP, CP, P, I32, F32, P, I32, P, SZ, PP, P, P]
        L.kvq_decode_attention_ex.restype = I32
        L.kvq_prefill_attention_ex.argtypes = [P, P, P, I32, I32, I32, I32, I32, P, I32, F32, P, I32, CP, CP, P,
                                               I32, PP, P, P]
        L.kvq_prefill_attention_ex.restype = I32
        _LIB = L
    return _LIB


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KvqError(status, what)


def _stream_ptr(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class QuantCache:
    """A quantised K or V cache in libkvq's layout, backed by torch tensors."""
    codes: "object"           # torch.uint8 [codes_bytes]
    sz: "object"              # torch.int32 [Hkv*B*Tcap*D/32] (fp16 scale | fp16 zero << 16)
    head_bits: np.ndarray     # int8 [Hkv] (host)
    B: int
    Hkv: int
    Tcap: int
    D: int

    def c_struct(self) -> CCache:
        """The C view of the cache, rebuilt only when a backing buffer changed."""
        key = (self.codes.data_ptr(), self.sz.data_ptr(), id(self.head_bits), self.B, self.Hkv, self.Tcap, self.D)
        cached = self.__dict__.get("_c_view")
        if cached is not None and cached[0] == key:
            return cached[1]
        hb = np.ascontiguousarray(self.head_bits, dtype=np.int8)
        self.head_bits = hb
        cs = CCache(self.codes.data_ptr(), self.sz.data_ptr(), hb.ctypes.data, self.B, self.Hkv, self.Tcap, self.D)
        key = (self.codes.data_ptr(), self.sz.data_ptr(), id(hb), self.B, self.Hkv, self.Tcap, self.D)
        self.__dict__["_c_view"] = (key, cs, hb)
        return cs

    def head_offset(self, h: int) -> int:
        cs = self.c_struct()
        return int(lib().kvq_cache_head_offset(ctypes.byref(cs), h))


def cache_nbytes(head_bits: Sequence[int], B: int, Tcap: int, D: int):
    """(codes bytes, sz bytes) of a cache with this shape."""
    hb = np.ascontiguousarray(head_bits, dtype=np.int8)
    cs = CCache(None, None, hb.ctypes.data, B, len(hb), Tcap, D)
    nc = int(lib().kvq_cache_codes_bytes(ctypes.byref(cs)))
    ns = int(lib().kvq_cache_sz_bytes(ctypes.byref(cs)))
    if nc < 0 or ns < 0:
        raise KvqError(1, "cache shape")
    return nc, ns


def empty_cache(head_bits: Sequence[int], B: int, Tcap: int, D: int, device="cuda") -> QuantCache:
    import torch
    nc, ns = cache_nbytes(head_bits, B, Tcap, D)
    codes = torch.empty(nc, dtype=torch.uint8, device=device)
    sz = torch.empty(ns // 4, dtype=torch.int32, device=device)
    return QuantCache(codes, sz, np.asarray(head_bits, np.int8), B, len(head_bits), Tcap, D)


def quantize(x, cache: QuantCache, t0: int = 0, status=None, stream=None):
    """Quantise bf16 x[B][Hkv][T][D] (strided, channels contiguous) into cache positions t0.."""
    assert x.dtype.itemsize == 2 and x.stride(-1) == 1
    cs = cache.c_struct()
    st = lib().kvq_quantize(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2), t0, x.shape[2],
                            ctypes.byref(cs), status.data_ptr() if status is not None else None,
                            _stream_ptr(stream))
    _check(st, "kvq_quantize")


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, D: int) -> int:
    return int(lib().kvq_decode_workspace_bytes(B, Hq, Hkv, D))


def decode_workspace(B: int, Hq: int, Hkv: int, D: int, device="cuda"):
    """A zero-filled decode workspace (the library keeps it zeroed between calls)."""
    import torch
    n = decode_workspace_bytes(B, Hq, Hkv, D)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def policy(**fields) -> CPolicy:
    """A kvq_policy: the library's defaults with the given fields replaced
    (decode_ring_tiles, decode_l2_warm_tiles, wait_limit_us, test_issue_limit)."""
    p = CPolicy()
    lib().kvq_policy_default(ctypes.byref(p))
    for k, val in fields.items():
        if not hasattr(p, k):
            raise TypeError(f"kvq_policy has no field {k}")
        setattr(p, k, int(val))
    return p


def decode_attention(q, k: QuantCache, v: QuantCache, seq_lens, softmax_scale: float = 0.0,
                     out=None, out_dtype: int = OUT_F32, workspace=None, status=None, stream=None,
                     policy: Optional[CPolicy] = None):
    """Decode attention: q bf16 [B][Hq][D] over the caches; returns out [B][Hq][D].
    With a policy (see :func:`policy`) the call goes through kvq_decode_attention_ex."""
    import torch
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, k.Hkv, D, q.device)
    kc, vc = k.c_struct(), v.c_struct()
    status_p = status.data_ptr() if status is not None else None
    ws_n = workspace.numel() * workspace.element_size()
    if policy is None:
        st = lib().kvq_decode_attention(q.data_ptr(), ctypes.byref(kc), ctypes.byref(vc), seq_lens.data_ptr(),
                                        Hq, float(softmax_scale), out.data_ptr(), out_dtype,
                                        workspace.data_ptr(), ws_n, status_p, _stream_ptr(stream))
        _check(st, "kvq_decode_attention")
    else:
        st = lib().kvq_decode_attention_ex(q.data_ptr(), ctypes.byref(kc), ctypes.byref(vc), seq_lens.data_ptr(),
                                           Hq, float(softmax_scale), out.data_ptr(), out_dtype,
                                           workspace.data_ptr(), ws_n, ctypes.byref(policy), status_p,
                                           _stream_ptr(stream))
        _check(st, "kvq_decode_attention_ex")
    return out


def decode_attention_noalloc(q, k: QuantCache, v: QuantCache, seq_lens, softmax_scale: float = 0.0,
                             out=None, out_dtype: int = OUT_F32, status=None, stream=None):
    """Decode attention with the library's built-in scratch (no workspace argument).

    For callers that cannot allocate device memory; the output buffer must be
    given by the caller in that case (``out``).  Calls on one device share the
    scratch, so they must be ordered on the GPU.
    """
    import torch
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    kc, vc = k.c_struct(), v.c_struct()
    st = lib().kvq_decode_attention_noalloc(q.data_ptr(), ctypes.byref(kc), ctypes.byref(vc), seq_lens.data_ptr(),
                                            Hq, float(softmax_scale), out.data_ptr(), out_dtype,
                                            status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_decode_attention_noalloc")
    return out


def decode_step(q, k_new, v_new, k: QuantCache, v: QuantCache, seq_lens, softmax_scale: float = 0.0,
                out=None, out_dtype: int = OUT_F32, workspace=None, status=None, stream=None):
    """One decode step: append k_new/v_new bf16 [B][Hkv][D] at position seq_lens[b] - 1 of the
    caches, then attend q bf16 [B][Hq][D] over seq_lens[b] tokens; returns out [B][Hq][D]."""
    import torch
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, k.Hkv, D, q.device)
    kc, vc = k.c_struct(), v.c_struct()
    st = lib().kvq_decode_step(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), ctypes.byref(kc), ctypes.byref(vc),
                               seq_lens.data_ptr(), Hq, float(softmax_scale), out.data_ptr(), out_dtype,
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_decode_step")
    return out


def decode_step_staging(B: int, Hq: int, Hkv: int, D: int, out_dtype: int = OUT_F32, device="cuda"):
    """Device staging buffer for decode_step_host (256-byte aligned)."""
    import torch
    n = int(lib().kvq_decode_step_staging_bytes(B, Hq, Hkv, D, out_dtype))
    if n == 0:
        raise KvqError(1, "kvq_decode_step_staging_bytes: invalid shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode_step_host(q_host, k_new_host, v_new_host, k: QuantCache, v: QuantCache, seq_lens, out_host,
                     softmax_scale: float = 0.0, out_dtype: int = OUT_F32, staging=None, workspace=None,
                     status=None, stream=None):
    """decode_step with the inputs (q_host, k_new_host, v_new_host, bf16 CPU tensors) and the
    output (out_host, CPU tensor of out_dtype) in host memory.  With pinned tensors the launches
    read and write them in place; otherwise they are copied through `staging`.  Everything is
    enqueued on `stream`; out_host is valid after a synchronisation."""
    B, Hq, D = q_host.shape
    dev = k.codes.device
    if staging is None:
        staging = decode_step_staging(B, Hq, k.Hkv, D, out_dtype, dev)
    if workspace is None:
        workspace = decode_workspace(B, Hq, k.Hkv, D, dev)
    kc, vc = k.c_struct(), v.c_struct()
    st = lib().kvq_decode_step_host(q_host.data_ptr(), k_new_host.data_ptr(), v_new_host.data_ptr(),
                                    ctypes.byref(kc), ctypes.byref(vc), seq_lens.data_ptr(), Hq,
                                    float(softmax_scale), out_host.data_ptr(), out_dtype,
                                    staging.data_ptr(), staging.numel(),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_decode_step_host")
    return out_host


class DecodeStepHost:
    """A decode_step_host call with its host buffers, staging, workspace and stream bound once,
    for serving loops that run it every token: ``run(k, v)`` enqueues one step on the caches
    given with little Python work per call.

    Every argument but the two caches is converted to its C type once; the call goes through a
    second handle on the same library function without ctypes argument conversion (the
    converted values are passed as they are), and each cache's C view is reused while the cache
    object and its buffers are unchanged."""

    def __init__(self, q_host, k_new_host, v_new_host, seq_lens, out_host, softmax_scale: float = 0.0,
                 out_dtype: int = OUT_F32, staging=None, workspace=None, status=None, stream=None,
                 Hkv: Optional[int] = None, device="cuda"):
        B, Hq, D = q_host.shape
        Hkv = int(k_new_host.shape[1]) if Hkv is None else Hkv
        self.staging = staging if staging is not None else decode_step_staging(B, Hq, Hkv, D, out_dtype, device)
        self.workspace = workspace if workspace is not None else decode_workspace(B, Hq, Hkv, D, device)
        self._keep = (q_host, k_new_host, v_new_host, seq_lens, out_host, status, stream)
        P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        self._head = (P(q_host.data_ptr()), P(k_new_host.data_ptr()), P(v_new_host.data_ptr()))
        self._tail = (P(seq_lens.data_ptr()), I32(Hq), F32(float(softmax_scale)), P(out_host.data_ptr()),
                      I32(out_dtype), P(self.staging.data_ptr()), SZ(self.staging.numel()),
                      P(self.workspace.data_ptr()), SZ(self.workspace.numel() * self.workspace.element_size()),
                      P(status.data_ptr() if status is not None else None), P(_stream_ptr(stream)))
        lib()   # loads the library and checks its exports
        raw = ctypes.CDLL(LIB_PATH).kvq_decode_step_host
        raw.restype = ctypes.c_int32
        self._fn = raw
        self._views = {}

    def _view(self, c: QuantCache):
        """byref of the cache's C view, reused while the cache object, the buffer objects it holds
        and its shape fields are the same (a buffer resized in place needs a new call object)."""
        hit = self._views.get(id(c))
        if (hit is not None and hit[0] is c and hit[1] is c.codes and hit[2] is c.sz and hit[3] is c.head_bits
                and hit[4] == (c.B, c.Hkv, c.Tcap, c.D)):
            return hit[5]
        ref = ctypes.byref(c.c_struct())
        if len(self._views) > 64:
            self._views.clear()
        self._views[id(c)] = (c, c.codes, c.sz, c.head_bits, (c.B, c.Hkv, c.Tcap, c.D), ref)
        return ref

    def run(self, k: QuantCache, v: QuantCache):
        st = self._fn(*self._head, self._view(k), self._view(v), *self._tail)
        if st != KVQ_OK:
            raise KvqError(st, "kvq_decode_step_host")


PAGE_TOKENS = 64


def empty_page_pool(head_bits: Sequence[int], n_pages: int, D: int, device="cuda") -> QuantCache:
    """A page pool: a cache of n_pages pages of 64 tokens (B = n_pages, Tcap = 64)."""
    return empty_cache(head_bits, n_pages, PAGE_TOKENS, D, device=device)


def _table(block_table) -> CBlockTable:
    """block_table: device int32 [B][max_pages] of page ids."""
    assert block_table.dtype.itemsize == 4 and block_table.dim() == 2 and block_table.is_contiguous()
    return CBlockTable(block_table.data_ptr(), int(block_table.shape[0]), int(block_table.shape[1]))


def quantize_paged(x, pool: QuantCache, block_table, t0: int = 0, status=None, stream=None):
    """Quantise bf16 x[B][Hkv][T][D] (strided, channels contiguous) into positions t0.. of the
    sequences of block_table, stored in the page pool."""
    assert x.dtype.itemsize == 2 and x.stride(-1) == 1
    cs, bt = pool.c_struct(), _table(block_table)
    st = lib().kvq_quantize_paged(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2), t0, x.shape[2],
                                  ctypes.byref(cs), ctypes.byref(bt),
                                  status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_quantize_paged")


def decode_attention_paged(q, k_pool: QuantCache, v_pool: QuantCache, block_table, seq_lens,
                           softmax_scale: float = 0.0, out=None, out_dtype: int = OUT_F32, workspace=None,
                           status=None, stream=None):
    """Decode attention over page pools through a block table; returns out [B][Hq][D]."""
    import torch
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, k_pool.Hkv, D, q.device)
    kc, vc, bt = k_pool.c_struct(), v_pool.c_struct(), _table(block_table)
    st = lib().kvq_decode_attention_paged(q.data_ptr(), ctypes.byref(kc), ctypes.byref(vc), ctypes.byref(bt),
                                          seq_lens.data_ptr(), Hq, float(softmax_scale), out.data_ptr(), out_dtype,
                                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                          status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_decode_attention_paged")
    return out


def decode_step_paged(q, k_new, v_new, k_pool: QuantCache, v_pool: QuantCache, block_table, seq_lens,
                      softmax_scale: float = 0.0, out=None, out_dtype: int = OUT_F32, workspace=None, status=None,
                      stream=None):
    """decode_step over page pools: append at position seq_lens[b] - 1 through the block table, then attend."""
    import torch
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, k_pool.Hkv, D, q.device)
    kc, vc, bt = k_pool.c_struct(), v_pool.c_struct(), _table(block_table)
    st = lib().kvq_decode_step_paged(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), ctypes.byref(kc),
                                     ctypes.byref(vc), ctypes.byref(bt), seq_lens.data_ptr(), Hq,
                                     float(softmax_scale), out.data_ptr(), out_dtype,
                                     workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                     status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_decode_step_paged")
    return out


def build_tile_mask(nT: int, skip_num: int, skip_den: int, seed: int, device="cuda", out=None, stream=None):
    """A prefill tile mask uint8 [nT][nT] built on the GPU: per query tile, floor((qt-1)*num/den) of the
    key tiles in [1, qt) skipped (smallest SplitMix64 keys); tile 0 and the diagonal kept."""
    import torch
    if out is None:
        out = torch.empty((nT, nT), dtype=torch.uint8, device=device)
    st = lib().kvq_build_tile_mask(out.data_ptr(), nT, skip_num, skip_den, int(seed) & 0xFFFFFFFFFFFFFFFF,
                                   _stream_ptr(stream))
    _check(st, "kvq_build_tile_mask")
    return out


def head_error_stats_workspace(H: int, device="cuda"):
    import torch
    n = lib().kvq_head_error_stats_workspace_bytes(H)
    return torch.empty(n, dtype=torch.uint8, device=device)


def head_error_stats(x, bits: int = 4, seq_lens=None, weights=None, workspace=None, out=None, status=None,
                     stream=None):
    """Per-head (weighted squared quantisation error, weighted squared norm) of bf16 x [B][H][T][D] at `bits`
    bits: a device float64 tensor [H][2].  seq_lens: device int32 [B]; weights: device float32 [B][H][T]."""
    import torch
    B, H, T, D = x.shape
    if workspace is None:
        workspace = head_error_stats_workspace(H, x.device)
    if out is None:
        out = torch.empty((H, 2), dtype=torch.float64, device=x.device)
    st = lib().kvq_head_error_stats(x.data_ptr(), B, H, T, D,
                                    seq_lens.data_ptr() if seq_lens is not None else None,
                                    weights.data_ptr() if weights is not None else None, bits,
                                    out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                    status.data_ptr() if status is not None else None, _stream_ptr(stream))
    _check(st, "kvq_head_error_stats")
    return out


def allocate_head_bits(k_stats, v_stats, n_high: int, low_bits: int = 4):
    """(head_bits int8 [H], score float64 [H]) from K and V statistics (kvq_head_error_stats results, on the
    device or the host): 8 bits for the n_high most sensitive heads, low_bits for the others."""
    import numpy as np
    ks = np.ascontiguousarray(k_stats.cpu().numpy() if hasattr(k_stats, "cpu") else k_stats, dtype=np.float64)
    vs = np.ascontiguousarray(v_stats.cpu().numpy() if hasattr(v_stats, "cpu") else v_stats, dtype=np.float64)
    H = ks.shape[0]
    bits = np.empty(H, dtype=np.int8)
    score = np.empty(H, dtype=np.float64)
    st = lib().kvq_allocate_head_bits(ks.ctypes.data, vs.ctypes.data, H, n_high, low_bits, bits.ctypes.data,
                                      score.ctypes.data)
    _check(st, "kvq_allocate_head_bits")
    return bits, score


def prefill_attention(q, k, v, k_cache: QuantCache, v_cache: QuantCache, softmax_scale: float = 0.0,
                      tile_mask=None, out=None, out_dtype: int = OUT_F32, status=None, stream=None,
                      causal: bool = True, seq_lens=None, policy: Optional[CPolicy] = None):
    """Prefill (causal by default): q bf16 [B][Hq][S][D], k/v bf16 [B][Hkv][S][D]; fills the caches, returns out.
    seq_lens (device int32 [B]): per-sequence lengths within the padded S (kvq_prefill_attention_varlen).
    With a policy (see :func:`policy`) the call goes through kvq_prefill_attention_ex."""
    import torch
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty((B, Hq, S, D), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
                          device=q.device)
    kc, vc = k_cache.c_struct(), v_cache.c_struct()
    mask_p = tile_mask.data_ptr() if tile_mask is not None else None
    status_p = status.data_ptr() if status is not None else None
    if policy is not None:
        st = lib().kvq_prefill_attention_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Hq, Hkv, S, D,
                                            seq_lens.data_ptr() if seq_lens is not None else None,
                                            1 if causal else 0, float(softmax_scale), mask_p, 128,
                                            ctypes.byref(kc), ctypes.byref(vc), out.data_ptr(), out_dtype,
                                            ctypes.byref(policy), status_p, _stream_ptr(stream))
        _check(st, "kvq_prefill_attention_ex")
    elif seq_lens is None:
        st = lib().kvq_prefill_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Hq, Hkv, S, D,
                                         1 if causal else 0, float(softmax_scale), mask_p, 128,
                                         ctypes.byref(kc), ctypes.byref(vc), out.data_ptr(), out_dtype,
                                         status_p, _stream_ptr(stream))
        _check(st, "kvq_prefill_attention")
    else:
        st = lib().kvq_prefill_attention_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Hq, Hkv, S, D,
                                                seq_lens.data_ptr(), 1 if causal else 0, float(softmax_scale),
                                                mask_p, 128, ctypes.byref(kc), ctypes.byref(vc), out.data_ptr(),
                                                out_dtype, status_p, _stream_ptr(stream))
        _check(st, "kvq_prefill_attention_varlen")
    return out
