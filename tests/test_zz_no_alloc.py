"""The decode entry point for callers that cannot allocate device memory.

kvq_decode_attention_noalloc uses a fixed scratch array inside the library
instead of a caller workspace.  Through the C ABI, two calls in a row must
give the same outputs as kvq_decode_attention (within the parity tolerance of
the other tests) and match the oracle directly, and a shape too large for the
built-in scratch must be refused without a launch.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import kvq_workloads as W
from oracle import kvq_oracle as O
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq as K
    K.lib()
    return K


def _caches(kvq, inp):
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    kvq.quantize(U.to_dev_bf16(inp.k), kc)
    kvq.quantize(U.to_dev_bf16(inp.v), vc)
    return kc, vc


def _noalloc(kvq, q, kc, vc, sl, scale, out, status):
    """The raw C-ABI call (plain pointers, the current stream)."""
    k_s, v_s = kc.c_struct(), vc.c_struct()
    return kvq.lib().kvq_decode_attention_noalloc(
        q.data_ptr(), ctypes.byref(k_s), ctypes.byref(v_s), sl.data_ptr(), q.shape[1], float(scale),
        out.data_ptr(), kvq.OUT_F32, status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls(kvq):
    inputs = [W.make_decode("noalloc_a", 61, 3, 8, 2, 128, 2048, lens=[2048, 777, 64], bits="mixed",
                            outliers_per_head=2, outlier_head_mult=8.0),
              W.make_decode("noalloc_b", 62, 4, 16, 4, 128, 1024, lens=[1, 1024, 500, 0], bits="8")]
    for inp in inputs:
        kc, vc = _caches(kvq, inp)
        q = U.to_dev_bf16(inp.q)
        sl = torch.from_numpy(inp.seq_lens).cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=status)
        # the oracle over its own dequantised cache, for a direct check as well
        _, _, _, kd = U.oracle_quantize(inp.k, inp.head_bits)
        _, _, _, vd = U.oracle_quantize(inp.v, inp.head_bits)
        oracle = O.decode_attention(inp.q, kd, vd, inp.seq_lens, inp.softmax_scale)
        for call in range(2):
            out = torch.full((inp.B, inp.Hq, inp.D), float("nan"), dtype=torch.float32, device="cuda")
            assert _noalloc(kvq, q, kc, vc, sl, inp.softmax_scale, out, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            got = out.cpu().numpy()
            U.assert_close(got, ref.cpu().numpy().astype(np.float64), f"{inp.name} call {call}")
            U.assert_close(got, oracle, f"{inp.name} call {call} vs oracle")


def test_noalloc_refuses_shapes_beyond_its_scratch(kvq):
    # B=4096 sequences x 8 KV heads needs far more than the built-in scratch
    hb = np.full(8, 8, np.int8)
    k_s = kvq.CCache(0x1000, 0x2000, hb.ctypes.data, 4096, 8, 64, 128)
    st = kvq.lib().kvq_decode_attention_noalloc(0x3000, ctypes.byref(k_s), ctypes.byref(k_s), 0x4000, 32, 0.0,
                                                0x5000, 0, None, None)
    assert st == 4   # KVQ_ERR_WORKSPACE, nothing launched
