"""GPU parity of the paged-cache calls (page pools + block tables) against the oracle.

Every live token row read back through the block table must equal the
oracle's quantisation bit for bit; decode outputs must satisfy
|o - ref| <= 2e-3 + 2e-3 |ref| against the fp64 oracle, and a paged decode
must give exactly the bytes of the same data decoded from contiguous caches.
"""
import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq
    kvq.lib()


def _kvq():
    from attention_group_quantized_gb300 import kvq
    return kvq


def _block_table(B: int, max_pages: int, n_pages: int, seed: int) -> np.ndarray:
    """Each sequence's pages drawn without replacement from a shuffled pool."""
    perm = np.random.default_rng(seed).permutation(n_pages)
    return perm[:B * max_pages].reshape(B, max_pages).astype(np.int32)


def _paged(inp: W.DecodeInputs, seed: int, spare_pages: int = 7):
    kvq = _kvq()
    max_pages = inp.Tcap // 64
    n_pages = inp.B * max_pages + spare_pages
    table = _block_table(inp.B, max_pages, n_pages, seed)
    kp = kvq.empty_page_pool(inp.head_bits, n_pages, inp.D)
    vp = kvq.empty_page_pool(inp.head_bits, n_pages, inp.D)
    for c in (kp, vp):
        c.codes.fill_(0xA5)
        c.sz.fill_(-1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(table).cuda()
    kvq.quantize_paged(U.to_dev_bf16(inp.k), kp, bt, 0, status)
    kvq.quantize_paged(U.to_dev_bf16(inp.v), vp, bt, 0, status)
    return kp, vp, bt, table, status


def _check_pool_exact(pool, x, head_bits, lens, table):
    planes, scale, zero = U.read_cache(pool, 64)          # per page: [n_pages][64][R], [n_pages][Hkv][64][G]
    o_planes, o_scale, o_zero, deq = U.oracle_quantize(x, head_bits)
    for b, L in enumerate(lens):
        for t in range(0, int(L), 64):
            n = min(64, int(L) - t)
            page = table[b, t // 64]
            for h in range(len(head_bits)):
                assert np.array_equal(planes[h][page, :n], o_planes[h][b, t:t + n]), (b, t, h)
            assert np.array_equal(scale[page, :, :n].view(np.uint16), o_scale[b, :, t:t + n].view(np.uint16)), (b, t)
            assert np.array_equal(zero[page, :, :n].view(np.uint16), o_zero[b, :, t:t + n].view(np.uint16)), (b, t)
    return deq


PAGED = [
    # name, seed, B, Hq, Hkv, D, Tcap, lens, bits
    ("paged_int8_ragged", 41, 3, 8, 2, 128, 512, [512, 77, 1], "8"),
    ("paged_mixed", 42, 2, 16, 4, 128, 640, [640, 333], "mixed"),
    ("paged_d64_int4", 43, 4, 8, 4, 64, 256, [2, 64, 129, 256], "4"),
    ("paged_many_sequences", 44, 20, 4, 1, 128, 192, list(np.random.default_rng(1).integers(0, 193, 20)), "mixed"),
]


@pytest.mark.parametrize("case", PAGED, ids=[c[0] for c in PAGED])
def test_paged_quantize_and_decode_parity(case):
    name, seed, B, Hq, Hkv, D, Tcap, lens, bits = case
    kvq = _kvq()
    inp = W.make_decode(name, seed, B, Hq, Hkv, D, Tcap, lens=list(lens), bits=bits,
                        outliers_per_head=2, outlier_head_mult=8.0)
    kp, vp, bt, table, status = _paged(inp, seed)
    deq_k = _check_pool_exact(kp, inp.k, inp.head_bits, inp.seq_lens, table)
    deq_v = _check_pool_exact(vp, inp.v, inp.head_bits, inp.seq_lens, table)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    out = kvq.decode_attention_paged(U.to_dev_bf16(inp.q), kp, vp, bt, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.decode_attention(inp.q, deq_k, deq_v, inp.seq_lens, inp.softmax_scale)
    U.assert_close(out.cpu().numpy(), ref, name)


def test_paged_decode_gives_the_contiguous_bytes():
    """Same data in page pools and in contiguous caches: identical outputs."""
    kvq = _kvq()
    inp = W.make_decode("paged_vs_contiguous", 45, 4, 32, 8, 128, 1024, lens=[1024, 700, 64, 513], bits="mixed",
                        outliers_per_head=2, outlier_head_mult=8.0)
    kp, vp, bt, table, status = _paged(inp, 45)
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, status)
    kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, status)
    q = U.to_dev_bf16(inp.q)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    a = kvq.decode_attention_paged(q, kp, vp, bt, sl, inp.softmax_scale, status=status)
    b = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a, b)


def test_paged_decode_steps_append_through_the_table():
    kvq = _kvq()
    T_final = [130, 64, 7]
    inp = W.make_decode("paged_steps", 46, 3, 8, 2, 128, 192, lens=T_final, bits="8",
                        outliers_per_head=2, outlier_head_mult=8.0)
    B, Hq, Hkv, D = inp.B, inp.Hq, inp.Hkv, inp.D
    n_steps = 3
    start = [L - n_steps for L in T_final]
    pre_k, pre_v = inp.k.copy(), inp.v.copy()
    for b, L0 in enumerate(start):
        pre_k[b, :, L0:] = 0
        pre_v[b, :, L0:] = 0
    pre = W.DecodeInputs(inp.name, inp.q, pre_k, pre_v, np.array(start, np.int32), inp.head_bits,
                         inp.softmax_scale, Hq, Hkv, D, inp.Tcap)
    kp, vp, bt, table, status = _paged(pre, 46)
    ws = kvq.decode_workspace(B, Hq, Hkv, D, "cuda")
    deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
    rng = np.random.default_rng(47)
    for s in range(n_steps):
        lens = np.array([L0 + s + 1 for L0 in start], dtype=np.int32)
        k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(B)])
        v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(B)])
        q = W._draw_bf16(rng, (B, Hq, D))
        out = kvq.decode_step_paged(U.to_dev_bf16(q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kp, vp, bt,
                                    torch.from_numpy(lens).cuda(), inp.softmax_scale, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        U.assert_close(out.cpu().numpy(), O.decode_attention(q, deq_k, deq_v, lens, inp.softmax_scale), f"step {s}")
    _check_pool_exact(kp, inp.k, inp.head_bits, np.array(T_final), table)


def test_paged_page_id_outside_the_pool_is_reported():
    kvq = _kvq()
    inp = W.make_decode("paged_bad_page", 48, 2, 4, 1, 128, 128, lens=[128, 100], bits="8")
    kp, vp, bt, table, status = _paged(inp, 48)
    before = kp.codes.clone()
    bad = bt.clone()
    bad[1, 1] = kp.B + 5                         # sequence 1, tokens 64..127
    status.zero_()
    kvq.quantize_paged(U.to_dev_bf16(inp.k), kp, bad, 0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    # only the rows of the bad page were skipped; everything else was rewritten identically
    assert torch.equal(kp.codes, before)
    status.zero_()
    sl = torch.from_numpy(inp.seq_lens).cuda()
    out = kvq.decode_attention_paged(U.to_dev_bf16(inp.q), kp, vp, bad, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.isfinite(out).all()
    # sequence 0 never touches the bad entry: its output is the oracle's
    deq_k = U.oracle_quantize(inp.k[:1], inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v[:1], inp.head_bits)[3]
    ref = O.decode_attention(inp.q[:1], deq_k, deq_v, inp.seq_lens[:1], inp.softmax_scale)
    U.assert_close(out[:1].cpu().numpy(), ref, "sequence 0")
