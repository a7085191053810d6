"""The same kernels built with index checks (libkvq_debug.so, KVQ_DEBUG=1).

In that build every global-memory index the kernels compute is checked before
use -- the decode's code-copy coordinates, its scale/zero-word and query copies,
block-table reads, workspace slots and output rows; the prefill's code and word
loads and output rows; the quantiser's and the append's code and word stores --
and a failed check reports KVQ_ERR_BOUNDS (7) in the status word instead of
touching memory.  Representative calls run on both libraries: the debug build's
status must stay 0 and its results must be byte-identical to the shipped
library's (the checks change no arithmetic).  It stands in for a memory
checker, with checks that record a status rather than stop the kernel.
"""
import contextlib

import numpy as np
import pytest

import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from attention_group_quantized_gb300 import kvq as K
    if not os.path.exists(K.DEBUG_LIB_PATH):
        from attention_group_quantized_gb300 import build
        build.build(debug=True)
    K.lib()
    return K


@contextlib.contextmanager
def _library(K, path):
    """Route the binding's calls to the library at `path` for the duration."""
    old_path, old_lib = K.LIB_PATH, K._LIB
    K.LIB_PATH, K._LIB = path, None
    try:
        K.lib()
        yield
    finally:
        K.LIB_PATH, K._LIB = old_path, old_lib


def _both(K, fn):
    """fn() -> (list of result tensors, status tensor), run on each library; the
    debug run must report no failed check and give the same bytes."""
    results = []
    for path in (K.LIB_PATH, K.DEBUG_LIB_PATH):
        with _library(K, path):
            outs, status = fn()
            torch.cuda.synchronize()
            results.append(([o.detach().cpu().clone() for o in outs], int(status.item())))
    (plain, st_plain), (dbg, st_dbg) = results
    assert st_plain == 0
    assert st_dbg == 0, f"debug build reported status {st_dbg}"
    for a, b in zip(plain, dbg):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


DECODE_CASES = [
    # name, seed, B, Hq, Hkv, D, Tcap, lens, bits
    ("gqa4_int8_ragged", 301, 3, 8, 2, 128, 512, [512, 77, 300], "8"),
    ("gqa3_int4_ragged", 302, 2, 6, 2, 64, 384, [1, 383], "4"),
    ("mixed_d128", 303, 2, 16, 4, 128, 256, [256, 129], "mixed"),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_debug_build_quantize_and_decode(kvq, case):
    name, seed, B, Hq, Hkv, D, Tcap, lens, bits = case
    inp = W.make_decode(name, seed, B, Hq, Hkv, D, Tcap, lens=lens, bits=bits)

    def run():
        st = _status()
        kc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
        vc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
        for c in (kc, vc):
            c.codes.zero_()
            c.sz.zero_()
        kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
        kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
        sl = torch.from_numpy(inp.seq_lens.astype(np.int32)).cuda()
        out = kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, sl, inp.softmax_scale, status=st)
        return [kc.codes, kc.sz, vc.codes, vc.sz, out], st

    _both(kvq, run)


def test_debug_build_paged_quantize_and_decode(kvq):
    inp = W.make_decode("paged_dbg", 304, 3, 8, 2, 128, 256, lens=[256, 65, 190], bits="mixed")
    max_pages = inp.Tcap // 64
    n_pages = inp.B * max_pages + 5
    table = np.random.default_rng(305).permutation(n_pages)[:inp.B * max_pages].reshape(inp.B, max_pages)

    def run():
        st = _status()
        bt = torch.from_numpy(table.astype(np.int32)).cuda()
        kp = kvq.empty_page_pool(inp.head_bits, n_pages, inp.D)
        vp = kvq.empty_page_pool(inp.head_bits, n_pages, inp.D)
        for c in (kp, vp):
            c.codes.zero_()
            c.sz.zero_()
        kvq.quantize_paged(U.to_dev_bf16(inp.k), kp, bt, 0, st)
        kvq.quantize_paged(U.to_dev_bf16(inp.v), vp, bt, 0, st)
        sl = torch.from_numpy(inp.seq_lens.astype(np.int32)).cuda()
        out = kvq.decode_attention_paged(U.to_dev_bf16(inp.q), kp, vp, bt, sl, inp.softmax_scale, status=st)
        return [kp.codes, kp.sz, vp.codes, vp.sz, out], st

    _both(kvq, run)


def test_debug_build_decode_step(kvq):
    """Append (quantise-on-write of the new token) then decode, from device buffers."""
    inp = W.make_decode("step_dbg", 306, 2, 8, 2, 128, 256, lens=[200, 37], bits="mixed")
    rng = np.random.default_rng(307)
    k_new = W._draw_bf16(rng, (inp.B, inp.Hkv, inp.D))
    v_new = W._draw_bf16(rng, (inp.B, inp.Hkv, inp.D))

    def run():
        st = _status()
        kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
        vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
        for c in (kc, vc):
            c.codes.zero_()
            c.sz.zero_()
        kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
        kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
        sl = torch.from_numpy(inp.seq_lens.astype(np.int32)).cuda()
        out = kvq.decode_step(U.to_dev_bf16(inp.q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc, sl,
                              inp.softmax_scale, status=st)
        return [kc.codes, kc.sz, vc.codes, vc.sz, out], st

    _both(kvq, run)


PREFILL_CASES = [
    # name, seed, B, Hq, Hkv, D, S, head bits, causal, lens
    ("causal_int8_masked", 311, 1, 8, 2, 128, 384, [8, 8], True, None),
    ("noncausal_mixed_d64", 312, 2, 4, 2, 64, 256, [4, 8], False, None),
    ("varlen_int4_d128", 313, 3, 4, 2, 128, 384, [4, 4], True, [384, 200, 1]),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_debug_build_prefill(kvq, case):
    name, seed, B, Hq, Hkv, D, S, hb, causal, lens = case
    inp = W.make_prefill(name, seed, B, Hq, Hkv, D, S, mask_seed=seed if causal else None)

    def run():
        st = _status()
        kc = kvq.empty_cache(np.asarray(hb, np.int8), B, S, D)
        vc = kvq.empty_cache(np.asarray(hb, np.int8), B, S, D)
        for c in (kc, vc):   # rows past a short sequence are not written
            c.codes.zero_()
            c.sz.zero_()
        mask = torch.from_numpy(inp.tile_mask).cuda() if inp.tile_mask is not None else None
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
        out = kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                                    inp.softmax_scale, mask, status=st, causal=causal, seq_lens=sl)
        return [out, kc.codes, vc.codes, kc.sz, vc.sz], st

    _both(kvq, run)
