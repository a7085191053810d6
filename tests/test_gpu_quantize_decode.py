"""GPU parity of kvq_quantize and kvq_decode_attention against the oracle.

Codes, scales and zero points must be bit-exact; attention outputs must
satisfy |o - ref| <= 2e-3 + 2e-3 |ref| against the fp64 oracle fed the same
dequantised cache.  Small cases are compared element by element (several
64-token tiles and ragged tails); the full-size workloads are compared on
every cache row and every output row, segment by segment.
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


def _quantized_caches(inp: W.DecodeInputs, fill_garbage=True):
    kvq = _kvq()
    B, Hkv, Tcap, D = inp.B, inp.Hkv, inp.Tcap, inp.D
    kc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    vc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    if fill_garbage:   # stale cache contents past each sequence must never matter
        for c in (kc, vc):
            c.codes.fill_(0xA5)
            c.sz.fill_(-1)       # fp16 NaN scale and zero
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd, vd = U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v)
    kvq.quantize(kd, kc, 0, status)
    kvq.quantize(vd, vc, 0, status)
    return kc, vc, status


def _check_cache_exact(cache, bits_in: np.ndarray, head_bits, lens):
    """Bit-exact comparison of the cache rows that hold live tokens."""
    planes, scale, zero = U.read_cache(cache, bits_in.shape[2])
    o_planes, o_scale, o_zero, deq = U.oracle_quantize(bits_in, head_bits)
    for b, L in enumerate(lens):
        for h in range(len(head_bits)):
            assert np.array_equal(planes[h][b, :L], o_planes[h][b, :L]), (b, h)
        assert np.array_equal(scale[b, :, :L].view(np.uint16), o_scale[b, :, :L].view(np.uint16)), b
        assert np.array_equal(zero[b, :, :L].view(np.uint16), o_zero[b, :, :L].view(np.uint16)), b
    return deq


def _run_decode_case(inp: W.DecodeInputs, out_dtype=0):
    kvq = _kvq()
    kc, vc, status = _quantized_caches(inp)
    lens = inp.seq_lens
    deq_k = _check_cache_exact(kc, inp.k, inp.head_bits, lens)
    deq_v = _check_cache_exact(vc, inp.v, inp.head_bits, lens)
    q = U.to_dev_bf16(inp.q)
    sl = torch.from_numpy(lens.astype(np.int32)).cuda()
    out = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.float().cpu().numpy()
    ref = O.decode_attention(inp.q, deq_k, deq_v, lens, inp.softmax_scale)
    m = U.Margin(inp.name)
    m.add(U.assert_close(got, ref, inp.name, out_bf16=out_dtype == 1), inp.B * inp.Hq)
    m.report()
    return m.worst


SMALL = [
    # name, seed, B, Hq, Hkv, D, Tcap, lens, bits
    ("gqa_int8_ragged", 11, 2, 8, 2, 128, 1024, [1000, 77], "8"),
    ("int4_ragged", 12, 3, 8, 2, 128, 2048, [1, 1500, 2048], "4"),
    ("mixed_heads", 13, 2, 16, 4, 128, 640, [640, 333], "mixed"),
    ("d64_int8_mha", 14, 2, 4, 4, 64, 512, [512, 129], "8"),
    ("d64_int4_gqa2", 15, 2, 8, 4, 64, 256, [31, 255], "4"),
    ("edge_lengths", 16, 9, 8, 1, 128, 192, [0, 1, 31, 33, 63, 64, 65, 127, 192], "8"),
    ("many_sequences", 17, 40, 4, 1, 128, 256, list(np.random.default_rng(0).integers(0, 257, 40)), "mixed"),
    # at the limits: 4096 sequences (the most the decode's length table holds),
    # 8 query heads per KV head; and 64 KV heads (the most a cache may have)
    ("max_4096_sequences", 18, 4096, 8, 1, 64, 64, list(np.random.default_rng(1).integers(0, 65, 4096)), "8"),
    ("max_64_kv_heads", 19, 2, 64, 64, 128, 128, [128, 70], "mixed"),
]
# GQA ratios 3, 5, 6 and 7 (the MMA's 8 head columns partly unused), both head
# dims and both bit-widths, with a ragged tail in every case
SMALL += [(f"gqa{r}_d{D}_int{bits}", 100 + 10 * r + D // 64 + (bits == 4), 2, 2 * r, 2, D, 512,
           [512, 64 * r + 13], str(bits))
          for r in (3, 5, 6, 7) for D in (64, 128) for bits in (8, 4)]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_decode_small_parity(case):
    name, seed, B, Hq, Hkv, D, Tcap, lens, bits = case
    inp = W.make_decode(name, seed, B, Hq, Hkv, D, Tcap, lens=list(lens), bits=bits,
                        outliers_per_head=2, outlier_head_mult=8.0)
    _run_decode_case(inp)


def test_decode_bf16_output():
    inp = W.make_decode("bf16_out", 21, 2, 8, 2, 128, 512, lens=[512, 300], bits="8")
    _run_decode_case(inp, out_dtype=1)


def test_decode_tiny_workload_includes_quantize():
    inp = W.decode_tiny()
    _run_decode_case(inp)


def test_quantize_strided_input_and_offset_positions():
    """Quantise a strided view into cache positions t0.. ; bit-exact against the oracle."""
    kvq = _kvq()
    rng = np.random.default_rng(5)
    B, Hkv, T, D, Tcap, t0 = 2, 3, 100, 128, 256, 64
    x = W.bf16_bits(rng.standard_normal((B, T, Hkv, D)).astype(np.float32) * 3)
    xd = U.to_dev_bf16(x).permute(0, 2, 1, 3)          # [B][Hkv][T][D] view, strides (T*Hkv*D, D, Hkv*D, 1)
    for hb in ([8, 8, 8], [4, 8, 4]):
        c = kvq.empty_cache(np.array(hb, np.int8), B, Tcap, D)
        kvq.quantize(xd, c, t0)
        torch.cuda.synchronize()
        planes, scale, zero = U.read_cache(c, Tcap)
        o_planes, o_scale, o_zero, _ = U.oracle_quantize(np.ascontiguousarray(x.transpose(0, 2, 1, 3)), hb)
        for h in range(Hkv):
            assert np.array_equal(planes[h][:, t0:t0 + T], o_planes[h])
        assert np.array_equal(scale[:, :, t0:t0 + T].view(np.uint16), o_scale.view(np.uint16))
        assert np.array_equal(zero[:, :, t0:t0 + T].view(np.uint16), o_zero.view(np.uint16))


def test_quantize_special_groups_bit_exact():
    """All-zero, constant, one-sided, tiny, huge and tie-producing groups."""
    kvq = _kvq()
    rng = np.random.default_rng(8)
    rows = [np.zeros(128), np.full(128, 3.25), -np.abs(rng.standard_normal(128)) - 1,
            np.abs(rng.standard_normal(128)) * 1e-6, rng.standard_normal(128) * 3e4,
            np.repeat([-1.0, 3.0, 0.0, 0.5], 32), (np.arange(128) % 16 - 7.5) * 0.125]
    x = W.bf16_bits(np.stack(rows).astype(np.float32))[None, None]   # [1][1][7][128]
    for bits in (8, 4):
        c = kvq.empty_cache(np.array([bits], np.int8), 1, 64, 128)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.quantize(U.to_dev_bf16(x), c, 0, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        planes, scale, zero = U.read_cache(c, 7)
        o_planes, o_scale, o_zero, _ = U.oracle_quantize(x, [bits])
        assert np.array_equal(planes[0], o_planes[0])
        assert np.array_equal(scale.view(np.uint16), o_scale.view(np.uint16))
        assert np.array_equal(zero.view(np.uint16), o_zero.view(np.uint16))


def _near_tie_rows(bits: int, n_rows: int = 64, seed: int = 9):
    """bf16 rows [n][128] whose groups hold quotients x / s exactly on a
    half-integer (scale 1/16 from a range of 15.9375 (8-bit) or 0.9375
    (4-bit)) and, from a seeded search, within 2^-13 of one: the cases where
    a reciprocal-based quotient could round differently from the IEEE
    division."""
    qmax = 2 ** bits - 1
    hi, lo = (8.0, -7.9375) if bits == 8 else (0.5, -0.4375)
    rows = []
    ties = np.array([(2 * k + 1) / 32.0 for k in range(-16, 16)], np.float32)
    ties = ties[(ties <= hi) & (ties >= lo)]
    g = np.concatenate([[hi, lo], ties, np.zeros(32)])[:32].astype(np.float32)
    rows.append(np.tile(g, 4))
    rng = np.random.default_rng(seed)
    found = []
    while len(found) < 8 * (n_rows - 1):
        cand = W.bf16_bits((rng.standard_normal((256, 32)) * rng.uniform(0.1, 50.0)).astype(np.float32))
        xf = O.bf16_to_f32(cand)
        _, sc, _ = O.quantize_groups(cand, bits)
        q = xf / sc.astype(np.float32)                  # IEEE fp32 quotients
        d = np.abs(q - np.floor(q) - np.float32(0.5))
        hit = (d <= np.float32(2.0 ** -13)).any(axis=-1)
        found.extend(xf[hit])
    rows.extend(np.stack(found[: 4 * (n_rows - 1)]).reshape(n_rows - 1, 128))
    return W.bf16_bits(np.stack(rows).astype(np.float32))


@pytest.mark.parametrize("bits", [8, 4])
def test_quantize_near_tie_quotients_bit_exact(bits):
    """Quotients on or next to a half-integer take the kernel's exact-division
    path; codes must still equal the oracle's bit for bit."""
    kvq = _kvq()
    x = _near_tie_rows(bits)[None, None]            # [1][1][n][128]
    n = x.shape[2]
    c = kvq.empty_cache(np.array([bits], np.int8), 1, ((n + 63) // 64) * 64, 128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize(U.to_dev_bf16(x), c, 0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    planes, scale, zero = U.read_cache(c, n)
    o_planes, o_scale, o_zero, _ = U.oracle_quantize(x, [bits])
    assert np.array_equal(planes[0], o_planes[0])
    assert np.array_equal(scale.view(np.uint16), o_scale.view(np.uint16))
    assert np.array_equal(zero.view(np.uint16), o_zero.view(np.uint16))


@pytest.mark.parametrize("bad,where", [(np.inf, "inf"), (-np.inf, "-inf"), (np.nan, "nan in a live group"),
                                       (np.nan, "nan in an all-zero group")],
                         ids=["inf", "neg_inf", "nan_live", "nan_zero_group"])
def test_quantize_reports_nonfinite(bad, where):
    kvq = _kvq()
    rng = np.random.default_rng(5)
    x = np.zeros((1, 1, 2, 128), np.float32)
    if where != "nan in an all-zero group":
        x[0, 0, :] = rng.standard_normal((2, 128))
    x[0, 0, 1, 37] = bad
    for bits in (8, 4):
        c = kvq.empty_cache(np.array([bits], np.int8), 1, 64, 128)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.quantize(U.to_dev_bf16(W.bf16_bits(x)), c, 0, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 6, (where, bits)


def test_decode_reports_length_beyond_capacity():
    kvq = _kvq()
    inp = W.make_decode("too_long", 3, 1, 4, 1, 128, 128, lens=[128], bits="8")
    kc, vc, status = _quantized_caches(inp)
    sl = torch.tensor([129], dtype=torch.int32, device="cuda")
    kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, sl, 0.0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


def test_decode_workspace_too_small_is_rejected():
    kvq = _kvq()
    inp = W.make_decode("ws", 3, 1, 4, 1, 128, 128, lens=[128], bits="8")
    kc, vc, _ = _quantized_caches(inp)
    sl = torch.tensor([128], dtype=torch.int32, device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, sl, 0.0, workspace=ws)
    assert e.value.status == 4


def test_decode_output_guard_bytes_untouched():
    kvq = _kvq()
    inp = W.make_decode("guard", 4, 3, 8, 2, 128, 256, lens=[256, 10, 200], bits="mixed")
    kc, vc, status = _quantized_caches(inp)
    n = 3 * 8 * 128
    buf = torch.full((n + 64,), 12345.0, dtype=torch.float32, device="cuda")
    out = buf[:n].view(3, 8, 128)
    kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, torch.from_numpy(inp.seq_lens).cuda(), 0.0, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 12345.0)


# ---------------------------------------------------------------------------
# full-size workloads: every token row of the caches and every output row
# ---------------------------------------------------------------------------

def _full_size_check(inp: W.DecodeInputs):
    """The full workload, segment by segment (sequence, KV head): the codes,
    scales and zero points of every live token bit-exact, and every query
    head's output against the oracle attention over the oracle's own
    dequantised cache.  Reports the worst err / bound ratio."""
    kvq = _kvq()
    kc, vc, status = _quantized_caches(inp, fill_garbage=False)
    q = U.to_dev_bf16(inp.q)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    out = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    B, Hq, Hkv, D = inp.B, inp.Hq, inp.Hkv, inp.D
    rep = Hq // Hkv
    kp, ks, kz = U.read_cache(kc, inp.Tcap)
    vp, vs, vz = U.read_cache(vc, inp.Tcap)
    margin = U.Margin(inp.name)
    for b in range(B):
        L = int(inp.seq_lens[b])
        qf = O.bf16_to_f32(inp.q[b]).astype(np.float64)
        for kv in range(Hkv):
            bits = int(inp.head_bits[kv])
            deq = []
            for src, planes, sc, zz in ((inp.k, kp, ks, kz), (inp.v, vp, vs, vz)):
                c, s, z = O.quantize_groups(src[b, kv, :L], bits)
                packed = c if bits == 8 else O.pack_int4(c)
                assert np.array_equal(planes[kv][b, :L], packed), (inp.name, b, kv)
                assert np.array_equal(sc[b, kv, :L].view(np.uint16), s.view(np.uint16)), (inp.name, b, kv)
                assert np.array_equal(zz[b, kv, :L].view(np.uint16), z.view(np.uint16)), (inp.name, b, kv)
                deq.append(O.dequantize(c, s, z))
            hs = slice(kv * rep, (kv + 1) * rep)
            ref = O.attention(qf[hs], deq[0], deq[1], inp.softmax_scale) if L > 0 else np.zeros((rep, D))
            margin.add(U.assert_close(got[b, hs], ref, f"{inp.name} b={b} kv={kv}"), rep)
    margin.report()


def test_full_decode_gqa():
    _full_size_check(W.decode_gqa())


def test_full_decode_long_ragged():
    _full_size_check(W.decode_long_ragged())


def test_full_decode_mixed():
    _full_size_check(W.decode_mixed())


def test_decode_workspace_reused_across_calls():
    """The arrival counters in the workspace are back at zero after every call."""
    kvq = _kvq()
    ws = kvq.decode_workspace(6, 8, 2, 128)
    for i, lens in enumerate(([1000, 77, 512, 0, 3, 640], [64, 65, 1024, 1, 900, 333], [1024] * 6)):
        inp = W.make_decode(f"reuse{i}", 40 + i, 6, 8, 2, 128, 1024, lens=lens, bits="8")
        kc, vc, status = _quantized_caches(inp)
        out = kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, torch.from_numpy(inp.seq_lens).cuda(),
                                   inp.softmax_scale, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _, _, _, kd = U.oracle_quantize(inp.k, inp.head_bits)
        _, _, _, vd = U.oracle_quantize(inp.v, inp.head_bits)
        ref = O.decode_attention(inp.q, kd, vd, inp.seq_lens, inp.softmax_scale)
        U.assert_close(out.cpu().numpy(), ref, f"reuse call {i}")
    n_cnt = 6 * 2 * 4
    assert int(ws[:n_cnt].sum().item()) == 0
