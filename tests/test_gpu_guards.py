"""Guard bytes around every buffer the kernels write (compute-sanitizer is not available, so writes outside
a buffer are caught this way): caches, outputs, statistics, workspaces and masks are views into larger
buffers whose leading and trailing 256 bytes hold a sentinel that must survive each call."""
import numpy as np
import pytest

import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GUARD = 256   # bytes on each side (keeps the views 16-byte aligned)
SENT = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq
    kvq.lib()


def _kvq():
    from attention_group_quantized_gb300 import kvq
    return kvq


class Guarded:
    """A byte buffer of n bytes between two sentinel regions; view(dtype, shape) is the usable part."""

    def __init__(self, n: int):
        self.n = n
        self.buf = torch.full((n + 2 * GUARD,), SENT, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool(torch.all(self.buf[:GUARD] == SENT)) and bool(torch.all(self.buf[GUARD + self.n:] == SENT))


def _guarded_cache(bits, B, Tcap, D):
    kvq = _kvq()
    nc, ns = kvq.cache_nbytes(bits, B, Tcap, D)
    gc, gs = Guarded(nc), Guarded(ns)
    cache = kvq.QuantCache(gc.view(torch.uint8, (nc,)), gs.view(torch.int32, (ns // 4,)), np.asarray(bits, np.int8),
                           B, len(bits), Tcap, D)
    return cache, gc, gs


def test_quantize_and_decode_step_stay_inside_the_caches():
    kvq = _kvq()
    inp = W.make_decode("guard_q", 81, 3, 8, 2, 128, 192, lens=[192, 5, 100], bits="mixed")
    kc, gkc, gks = _guarded_cache(inp.head_bits, 3, 192, 128)
    vc, gvc, gvs = _guarded_cache(inp.head_bits, 3, 192, 128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, status)
    kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, status)
    # one decode step at the last position of each sequence (append + decode), output guarded too
    gout = Guarded(3 * 8 * 128 * 4)
    out = gout.view(torch.float32, (3, 8, 128))
    k_new = U.to_dev_bf16(np.stack([inp.k[b, :, inp.seq_lens[b] - 1] for b in range(3)]))
    v_new = U.to_dev_bf16(np.stack([inp.v[b, :, inp.seq_lens[b] - 1] for b in range(3)]))
    kvq.decode_step(U.to_dev_bf16(inp.q), k_new, v_new, kc, vc, torch.from_numpy(inp.seq_lens).cuda(),
                    inp.softmax_scale, out=out, status=status)
    assert int(status.item()) == 0
    for g in (gkc, gks, gvc, gvs, gout):
        assert g.intact()


def test_prefill_stays_inside_its_buffers():
    kvq = _kvq()
    inp = W.make_prefill("guard_p", 82, 2, 4, 2, 128, 384, mask_seed=3)
    bits = np.full(2, 8, np.int8)
    for lens in (None, [384, 130]):
        kc, gkc, gks = _guarded_cache(bits, 2, 384, 128)
        vc, gvc, gvs = _guarded_cache(bits, 2, 384, 128)
        gout = Guarded(2 * 4 * 384 * 128 * 2)
        out = gout.view(torch.bfloat16, (2, 4, 384, 128))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
        kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                              inp.softmax_scale, torch.from_numpy(inp.tile_mask).cuda(), out=out,
                              out_dtype=kvq.OUT_BF16, status=status, seq_lens=sl)
        assert int(status.item()) == 0
        for g in (gkc, gks, gvc, gvs, gout):
            assert g.intact(), lens


def test_statistics_and_mask_stay_inside_their_buffers():
    kvq = _kvq()
    inp = W.make_sensitivity("guard_s", 83, 2, 4, 128, 200, [1])
    H = 4
    gst = Guarded(H * 2 * 8)
    stats = gst.view(torch.float64, (H, 2))
    nws = int(kvq.lib().kvq_head_error_stats_workspace_bytes(H))
    gws = Guarded(nws)
    ws = gws.view(torch.uint8, (nws,))
    kvq.head_error_stats(U.to_dev_bf16(inp.k), 4, weights=torch.from_numpy(inp.weights).cuda(), workspace=ws,
                         out=stats)
    assert gst.intact() and gws.intact()
    for nT in (1, 3, 129):
        gm = Guarded(nT * nT)
        mask = gm.view(torch.uint8, (nT, nT))
        kvq.build_tile_mask(nT, 1, 3, 9, out=mask)
        assert gm.intact(), nT
