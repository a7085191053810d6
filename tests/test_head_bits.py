"""Sensitivity-driven per-head bit allocation.

CPU: the oracle's error statistics pinned to closed forms (values on the code
grid give no error, a half-way value rounds to even and costs exactly
(s/2)^2, power-of-two scaling, the s/2 bound, weights and lengths), the
allocation's order and ties, and the host allocator of the C ABI against the
oracle.  GPU: kvq_head_error_stats against the oracle (relative 1e-5: fp32
within a group, fp64 beyond), the same bit-widths chosen, and a decode over a
cache laid out with those bit-widths.
"""
import ctypes

import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W


def _bf16(x):
    """float -> bf16 bits (the values used here are exact in bf16)."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "test values must be exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _one_group(values):
    """x [1][1][1][32] holding one group: the given values, then zeros."""
    g = np.zeros(32, dtype=np.float32)
    g[:len(values)] = values
    return _bf16(g).reshape(1, 1, 1, 32)


# ---------------------------------------------------------------- oracle pins

def test_values_on_the_code_grid_have_no_error():
    # 0..15 with INT4: range 15, s = 15/15 = 1 exactly, z = 0, every value a code
    x = _one_group(np.arange(16))
    st = O.head_error_stats(x, 4)
    assert st[0, 0] == 0.0
    assert st[0, 1] == float(np.sum(np.arange(16) ** 2))      # 1240
    # 0, 0.5, ..., 127.5 with INT8: s = 127.5 / 255 = 0.5 exactly
    x8 = _bf16(np.concatenate([np.arange(0, 16) * 0.5, np.arange(240, 256) * 0.5])).reshape(1, 1, 1, 32)
    assert O.head_error_stats(x8, 8)[0, 0] == 0.0


def test_half_way_value_rounds_to_even():
    # range [0, 15], s = 1: 7.5 -> rne(7.5) = 8, error 0.5^2
    st = O.head_error_stats(_one_group([15.0, 7.5]), 4)
    assert st[0, 0] == 0.25
    # range [-15, 0], s = 1, z = 15: -7.5 -> rne(-7.5) = -8, code 7, x_hat = -8
    st = O.head_error_stats(_one_group([-15.0, -7.5]), 4)
    assert st[0, 0] == 0.25
    # 6.5 -> 6 (even), error 0.25 again; two such values add
    st = O.head_error_stats(_one_group([15.0, 6.5, 9.5]), 4)
    assert st[0, 0] == 0.5


def test_error_bound_and_power_of_two_scaling():
    rng = np.random.default_rng(3)
    f = rng.standard_normal((2, 3, 5, 64)).astype(np.float32)
    x = (f.view(np.uint32) >> 16).astype(np.uint16)           # truncated to bf16: exact values
    xf = O.bf16_to_f32(x).astype(np.float64)
    for bits in (4, 8):
        st = O.head_error_stats(x, bits)
        # every value lies inside the widened range, so each error is at most s/2 (up to the fp32
        # quotient's rounding), with s the fp16 round-up of range / qmax
        g = xf.reshape(2, 3, 5, 2, 32)
        rng_g = np.maximum(g.max(-1), 0) - np.minimum(g.min(-1), 0)
        s_max = rng_g / (2 ** bits - 1) * (1 + 2 ** -10)
        bound = np.sum(32 * (s_max / 2) ** 2, axis=(0, 2, 3)) * 1.0001
        assert np.all(st[:, 0] <= bound)
        assert np.all(st[:, 0] > 0)
        # x * 4 is exact in bf16; scales, codes and zero points scale along, so both sums scale by 16
        x4 = ((O.bf16_to_f32(x) * np.float32(4)).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(O.bf16_to_f32(x4), O.bf16_to_f32(x) * 4)
        st4 = O.head_error_stats(x4, bits)
        assert np.array_equal(st4, st * 16)


def test_weights_and_lengths():
    rng = np.random.default_rng(4)
    B, H, T, D = 3, 2, 7, 32
    x = (rng.standard_normal((B, H, T, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    base = O.head_error_stats(x, 4)
    assert np.allclose(O.head_error_stats(x, 4, weights=np.full((B, H, T), 2.5, np.float32)), 2.5 * base,
                       rtol=1e-15)
    # a length cut equals dropping those tokens; weight 0 on a token equals dropping it too
    lens = np.array([7, 0, 3])
    cut = O.head_error_stats(x, 4, seq_lens=lens)
    manual = O.head_error_stats(x[0:1], 4) + O.head_error_stats(x[2:3, :, :3], 4)
    assert np.allclose(cut, manual, rtol=1e-14)
    w = np.ones((B, H, T), np.float32)
    w[1] = 0
    w[2, :, 3:] = 0
    assert np.allclose(O.head_error_stats(x, 4, weights=w), cut, rtol=1e-14)
    # per-token weights pick out single tokens
    w = np.zeros((B, H, T), np.float32)
    w[2, 1, 5] = 1
    one = O.head_error_stats(x[2:3, 1:2, 5:6], 4)
    assert np.array_equal(O.head_error_stats(x, 4, weights=w)[1], one[0])


def test_sensitivity_and_allocation_rules():
    k = np.array([[1.0, 10.0], [0.0, 0.0], [3.0, 10.0], [1.0, 10.0]])
    v = np.array([[1.0, 4.0], [2.0, 4.0], [0.0, 4.0], [1.0, 4.0]])
    sc = O.head_sensitivity(k, v)
    assert np.allclose(sc, [0.35, 0.5, 0.3, 0.35])          # 0 / 0 counts 0
    assert list(O.allocate_head_bits(sc, 1)) == [4, 8, 4, 4]
    assert list(O.allocate_head_bits(sc, 2)) == [8, 8, 4, 4]  # tie between heads 0 and 3: the smaller index
    assert list(O.allocate_head_bits(sc, 3)) == [8, 8, 4, 8]
    assert list(O.allocate_head_bits(sc, 0)) == [4, 4, 4, 4]
    assert list(O.allocate_head_bits(sc, 4)) == [8, 8, 8, 8]


def test_outlier_heads_are_the_sensitive_ones():
    inp = W.make_sensitivity("pin", 1, 2, 8, 128, 256, [1, 4, 6])
    sc = O.head_sensitivity(O.head_error_stats(inp.k, 4, inp.seq_lens, inp.weights),
                            O.head_error_stats(inp.v, 4, inp.seq_lens, inp.weights))
    assert list(np.flatnonzero(O.allocate_head_bits(sc, 3) == 8)) == [1, 4, 6]


# ------------------------------------------------------ host ABI (no launch)

@pytest.fixture(scope="module")
def L():
    from attention_group_quantized_gb300 import kvq
    return kvq.lib()


def _alloc(L, ks, vs, n_high, low=4):
    ks = np.ascontiguousarray(ks, np.float64)
    vs = np.ascontiguousarray(vs, np.float64)
    H = ks.shape[0]
    bits = np.zeros(H, np.int8)
    score = np.zeros(H)
    st = L.kvq_allocate_head_bits(ks.ctypes.data, vs.ctypes.data, H, n_high, low, bits.ctypes.data,
                                  score.ctypes.data)
    return st, bits, score


def test_host_allocator_matches_the_oracle(L):
    rng = np.random.default_rng(5)
    for H in (1, 3, 8, 32, 64):
        ks = np.stack([rng.random(H), rng.random(H) + 0.5], 1)
        vs = np.stack([rng.random(H), rng.random(H) + 0.5], 1)
        ks[rng.integers(0, H)] = 0                  # a zero-norm head
        if H > 3:
            ks[2], vs[2] = ks[1], vs[1]             # an exact tie
        for n_high in sorted({0, 1, H // 2, H}):
            st, bits, score = _alloc(L, ks, vs, n_high)
            assert st == 0
            want = O.head_sensitivity(ks, vs)
            assert np.array_equal(score, want)
            assert np.array_equal(bits, O.allocate_head_bits(want, n_high))
    st, bits, _ = _alloc(L, ks, vs, 3, low=8)
    assert st == 0 and np.all(bits == 8)


def test_host_allocator_rejects(L):
    ks = np.ones((4, 2))
    assert _alloc(L, ks, ks, 5)[0] == 1
    assert _alloc(L, ks, ks, -1)[0] == 1
    assert _alloc(L, ks, ks, 2, low=5)[0] == 1
    bad = ks.copy()
    bad[1, 0] = np.nan
    st, bits, _ = _alloc(L, bad, ks, 2)
    assert st == 6 and np.all(bits == 0)             # nothing written
    assert L.kvq_allocate_head_bits(None, ks.ctypes.data, 4, 1, 4, None, None) == 1


def test_stats_validation_without_launch(L):
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 255) & ~255
    need = L.kvq_head_error_stats_workspace_bytes(8)
    assert need >= 8 * 2 * 8
    assert L.kvq_head_error_stats_workspace_bytes(0) == 0
    call = lambda **kw: L.kvq_head_error_stats(kw.get("x", a), kw.get("B", 1), kw.get("H", 8), kw.get("T", 64),
                                               kw.get("D", 128), None, None, kw.get("bits", 4), kw.get("st", a),
                                               kw.get("ws", a), kw.get("wsb", need), None, None)
    assert call(x=None) == 1
    assert call(st=None) == 1
    assert call(B=0) == 1
    assert call(T=0) == 1
    assert call(bits=5) == 1
    assert call(D=96) == 2
    assert call(x=a + 8) == 1
    assert call(st=a + 4) == 1
    assert call(ws=None) == 4
    assert call(wsb=need - 1) == 4
    assert call(B=1 << 16, T=1 << 15) == 1


# ---------------------------------------------------------------------- GPU

torch = pytest.importorskip("torch")


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq
    kvq.lib()
    return kvq


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


STATS = [
    # name, seed, B, H, T, D, outlier heads, lens, weights, bits
    ("full_d128_int4", 61, 2, 8, 300, 128, [1, 4, 6], "full", True, 4),
    ("ragged_d64_int8", 62, 3, 4, 257, 64, [0], [257, 0, 31], True, 8),
    ("unweighted_one_head", 63, 1, 1, 5, 128, [], "full", False, 4),
    ("many_heads", 64, 2, 32, 70, 128, [3, 17, 30], [70, 9], False, 4),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", STATS, ids=[c[0] for c in STATS])
def test_stats_parity(case):
    kvq = _gpu()
    name, seed, B, H, T, D, oh, lens, weighted, bits = case
    inp = W.make_sensitivity(name, seed, B, H, D, T, oh, lens=lens, weights=weighted)
    sl = torch.from_numpy(inp.seq_lens).cuda() if not isinstance(lens, str) else None
    w = torch.from_numpy(inp.weights).cuda() if weighted else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for x in (inp.k, inp.v):
        got = kvq.head_error_stats(_dev_bf16(x), bits, seq_lens=sl, weights=w, status=status).cpu().numpy()
        want = O.head_error_stats(x, bits, inp.seq_lens if sl is not None else None, inp.weights)
        assert np.allclose(got, want, rtol=1e-5, atol=1e-30), (name, got, want)
        again = kvq.head_error_stats(_dev_bf16(x), bits, seq_lens=sl, weights=w, status=status).cpu().numpy()
        assert np.array_equal(got, again)          # a fixed summation order
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_stats_report_nonfinite():
    kvq = _gpu()
    inp = W.make_sensitivity("nan", 65, 1, 2, 128, 64, [], weights=False)
    x = inp.k.copy()
    x[0, 1, 10, 7] = 0x7FC0                         # NaN
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.head_error_stats(_dev_bf16(x), 4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6


@pytest.mark.gpu
def test_allocation_then_decode_over_the_chosen_bits():
    """Statistics on the GPU, allocation on the host, a cache laid out with the chosen bit-widths,
    quantise and decode: the bits are the oracle's and the decode matches the oracle."""
    kvq = _gpu()
    from tests import kvq_testutil as U
    B, Hq, H, D, T = 2, 16, 8, 128, 512
    inp = W.make_sensitivity("alloc", 66, B, H, D, T, [1, 4, 6], lens=[512, 300])
    sl = torch.from_numpy(inp.seq_lens).cuda()
    w = torch.from_numpy(inp.weights).cuda()
    ks = kvq.head_error_stats(_dev_bf16(inp.k), 4, seq_lens=sl, weights=w)
    vs = kvq.head_error_stats(_dev_bf16(inp.v), 4, seq_lens=sl, weights=w)
    bits, score = kvq.allocate_head_bits(ks, vs, 3)
    o_sc = O.head_sensitivity(O.head_error_stats(inp.k, 4, inp.seq_lens, inp.weights),
                              O.head_error_stats(inp.v, 4, inp.seq_lens, inp.weights))
    o_bits = O.allocate_head_bits(o_sc, 3)
    srt = np.sort(o_sc)[::-1]
    assert srt[2] - srt[3] > 1e-3 * srt[2]            # the cut is far from a tie at this tolerance
    assert np.allclose(score, o_sc, rtol=1e-5)
    assert np.array_equal(bits, o_bits)
    assert list(np.flatnonzero(bits == 8)) == [1, 4, 6]
    kc = kvq.empty_cache(bits, B, T, D)
    vc = kvq.empty_cache(bits, B, T, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize(_dev_bf16(inp.k), kc, 0, status)
    kvq.quantize(_dev_bf16(inp.v), vc, 0, status)
    rng = np.random.default_rng(67)
    q = W._draw_bf16(rng, (B, Hq, D))
    out = kvq.decode_attention(_dev_bf16(q), kc, vc, sl, 1.0 / np.sqrt(D), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    deq_k = U.oracle_quantize(inp.k, bits)[3]
    deq_v = U.oracle_quantize(inp.v, bits)[3]
    ref = O.decode_attention(q, deq_k, deq_v, inp.seq_lens, 1.0 / np.sqrt(D))
    U.assert_close(out.cpu().numpy(), ref, "decode over allocated bits")


@pytest.mark.gpu
def test_stats_full_size_workload():
    """The bench's workload (B8, 8 heads, D128, 8192 tokens, weighted): statistics of K and V against the
    oracle, and the outlier heads chosen."""
    kvq = _gpu()
    inp = W.head_bits_kv()
    w = torch.from_numpy(inp.weights).cuda()
    ks = kvq.head_error_stats(_dev_bf16(inp.k), 4, weights=w).cpu().numpy()
    vs = kvq.head_error_stats(_dev_bf16(inp.v), 4, weights=w).cpu().numpy()
    o_ks = O.head_error_stats(inp.k, 4, None, inp.weights)
    o_vs = O.head_error_stats(inp.v, 4, None, inp.weights)
    assert np.allclose(ks, o_ks, rtol=1e-5)
    assert np.allclose(vs, o_vs, rtol=1e-5)
    bits, _ = kvq.allocate_head_bits(ks, vs, len(inp.outlier_heads))
    assert list(np.flatnonzero(bits == 8)) == list(inp.outlier_heads)


# ------------------------------------------------------------ properties (CPU)

def test_allocation_is_equivariant_and_nested():
    """Permuting the heads permutes the bit-widths (distinct scores); raising n_high only adds 8-bit heads."""
    rng = np.random.default_rng(21)
    for H in (2, 5, 16, 64):
        sc = rng.random(H)
        perm = rng.permutation(H)
        for n_high in range(H + 1):
            bits = O.allocate_head_bits(sc, n_high)
            assert np.array_equal(O.allocate_head_bits(sc[perm], n_high), bits[perm])
            assert int(np.sum(bits == 8)) == n_high
            if n_high > 0:
                prev = O.allocate_head_bits(sc, n_high - 1)
                assert np.all((prev == 8) <= (bits == 8))          # nested: the set only grows
        # the chosen heads are exactly the n_high largest scores
        n = H // 2
        chosen = set(np.flatnonzero(O.allocate_head_bits(sc, n) == 8))
        assert chosen == set(np.argsort(-sc)[:n])


def test_statistics_add_over_sequences_and_ignore_token_order():
    rng = np.random.default_rng(22)
    B, H, T, D = 3, 2, 9, 64
    x = (rng.standard_normal((B, H, T, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = rng.exponential(1.0, (B, H, T)).astype(np.float32)
    whole = O.head_error_stats(x, 4, weights=w)
    parts = sum(O.head_error_stats(x[b:b + 1], 4, weights=w[b:b + 1]) for b in range(B))
    assert np.allclose(whole, parts, rtol=1e-14)
    perm = rng.permutation(T)
    assert np.allclose(O.head_error_stats(x[:, :, perm], 4, weights=w[:, :, perm]), whole, rtol=1e-14)


def test_host_allocator_is_equivariant(L):
    rng = np.random.default_rng(23)
    H = 24
    ks = np.stack([rng.random(H), rng.random(H) + 0.5], 1)
    vs = np.stack([rng.random(H), rng.random(H) + 0.5], 1)
    perm = rng.permutation(H)
    for n_high in (0, 5, 12, 24):
        st, bits, score = _alloc(L, ks, vs, n_high)
        st2, bits2, score2 = _alloc(L, ks[perm], vs[perm], n_high)
        assert st == st2 == 0
        assert np.array_equal(bits2, bits[perm]) and np.array_equal(score2, score[perm])
