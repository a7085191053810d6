"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each test ties one oracle function to something independent of it: an
exhaustive table, a hand-worked fixture, a closed form, an invariant, or a
brute force written in plain Python scalar arithmetic.  The planted-mistake
tests at the end show that plausible slips in the oracle fail these pins.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_of(x):
    return W.bf16_bits(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

_ALL_F16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
_FINITE_F16 = np.unique(_ALL_F16[np.isfinite(_ALL_F16)].astype(np.float64))


def test_f16_round_up_matches_exhaustive_table():
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        rng.uniform(-70000, 70000, 20000),
        rng.standard_normal(20000) * 1e-3,
        rng.standard_normal(20000) * 1e-6,           # subnormal fp16 range
        _FINITE_F16[::97],                            # exact fp16 values
        (_FINITE_F16[1:] + _FINITE_F16[:-1])[::89] / 2,  # midpoints
        [0.0, -0.0, 65504.0, -65504.0, 6.1035156e-05, 5.96e-08],
    ]).astype(np.float32)
    xs = xs[np.abs(xs) <= 65504]
    got = O.f16_round_up(xs).astype(np.float64)
    idx = np.searchsorted(_FINITE_F16, xs.astype(np.float64), side="left")
    want = _FINITE_F16[idx]
    assert np.array_equal(got, want)


def test_rne_matches_python_bankers_rounding():
    vals = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.49999, 3.5, 254.5, 255.5, -127.5,
                     0.49999997, 1e-8, -7.000001], dtype=np.float32)
    got = O.rne_int(vals)
    want = [round(float(v)) for v in vals]          # Python rounds half to even
    assert list(got) == want


def test_bf16_decode_and_generator_rounding():
    import torch
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(10000) * rng.choice([1e-30, 1e-3, 1, 1e3, 1e30], 10000)).astype(np.float32)
    bits = W.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = O.bf16_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------------------
# quantisation
# ---------------------------------------------------------------------------

def _load_golden():
    cases = []
    with open(os.path.join(HERE, "golden", "quant_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, xs, fill, scale, zero, codes, fillcode = [p.strip() for p in line.split("|")]
            num, den = scale.split("/")
            cases.append(dict(bits=int(bits), xs=[float(v) for v in xs.split()], fill=float(fill),
                              scale=Fraction(int(num), int(den)), zero=int(zero),
                              codes=[int(c) for c in codes.split()], fillcode=int(fillcode)))
    return cases


@pytest.mark.parametrize("case", _load_golden())
def test_quantize_hand_worked_cases(case):
    x = np.full(32, case["fill"], dtype=np.float32)
    x[:len(case["xs"])] = case["xs"]
    codes, scale, zero = O.quantize_groups(_bf16_of(x)[None, :], case["bits"])
    assert Fraction(float(scale[0, 0])) == case["scale"]
    assert int(zero[0, 0]) == case["zero"]
    want = np.full(32, case["fillcode"])
    want[:len(case["codes"])] = case["codes"]
    assert np.array_equal(codes[0], want)


def test_int4_packing_hand_worked():
    # case B of the golden file: codes 4 7 15 2 then 4s -> bytes 0x74 0x2F 0x44...
    codes = np.array([4, 7, 15, 2] + [4] * 28, dtype=np.uint8)
    packed = O.pack_int4(codes)
    assert packed[0] == 0x74 and packed[1] == 0x2F and np.all(packed[2:] == 0x44)
    assert np.array_equal(O.unpack_int4(packed), codes)


def _random_groups(rng, n):
    """Rows of 32 channels with assorted shapes: normal, outliers, one-sided, constant, zero, tiny."""
    rows = []
    rows.append(rng.standard_normal((n, 32)))
    o = rng.standard_normal((n, 32)); o[:, rng.integers(0, 32, n)] *= 50; rows.append(o)
    rows.append(np.abs(rng.standard_normal((n, 32))) + 0.1)
    rows.append(-np.abs(rng.standard_normal((n, 32))) - 3.0)
    rows.append(np.repeat(rng.standard_normal((n, 1)), 32, axis=1))
    rows.append(np.zeros((4, 32)))
    rows.append(rng.standard_normal((n, 32)) * 1e-6)
    rows.append(rng.standard_normal((n, 32)) * 1e4)
    z = rng.standard_normal((n, 32)); z[:, :31] = 0; rows.append(z)
    return np.concatenate(rows).astype(np.float32)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantize_invariants(bits):
    rng = np.random.default_rng(bits)
    x = _random_groups(rng, 300)
    xb = _bf16_of(x)
    xf = O.bf16_to_f32(xb).astype(np.float64)
    codes, scale, zero = O.quantize_groups(xb, bits)
    qmax = 2 ** bits - 1
    s = scale.astype(np.float64)[:, 0]
    z = zero.astype(np.float64)[:, 0]
    assert codes.max() <= qmax and zero.min() >= 0 and zero.max() <= qmax
    # reconstruction error <= scale * (1/2 + 2^-16) for every element
    xh = O.dequantize(codes, scale, zero)
    err = np.abs(xh - xf)
    assert np.all(err <= s[:, None] * (0.5 + 2.0 ** -16))
    # scale is the smallest fp16 >= (hi - lo) / qmax, on the range widened to contain 0
    lo = np.minimum(0, xf.min(axis=1)); hi = np.maximum(0, xf.max(axis=1))
    r = (hi - lo).astype(np.float32)
    nz = r > 0
    step = (r / np.float32(qmax)).astype(np.float64)
    idx = np.searchsorted(_FINITE_F16, step[nz], side="left")
    assert np.array_equal(s[nz], _FINITE_F16[idx])
    assert np.all(s[~nz] == 1.0) and np.all(z[~nz] == 0) and np.all(codes[~nz] == 0)
    # zero maps back to exactly 0: the zero point is an integer code
    assert np.all(z == np.round(z))
    # the group's extremes use the ends of the code space (within one step)
    cmin = codes.min(axis=1).astype(int); cmax = codes.max(axis=1).astype(int)
    # (only where the scale is a normal fp16: below 2^-14 its grid is too coarse)
    normal = (r / np.float32(qmax)) >= 2.0 ** -14
    has_neg = (xf.min(axis=1) < 0) & normal
    has_pos = (xf.max(axis=1) > 0) & normal
    assert np.all(cmin[has_neg] <= 1)
    assert np.all(cmax[has_pos] >= qmax - 1)
    # one-sided groups: zero point sits at an end of the code space
    assert np.all(z[nz & (xf.min(axis=1) >= 0)] == 0)
    assert np.all(z[nz & normal & (xf.max(axis=1) <= 0)] == qmax)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantize_codes_are_nearest_brute_force(bits):
    """Each code is a nearest point of the grid {(c - zero) * scale, c = 0..qmax}."""
    rng = np.random.default_rng(100 + bits)
    x = _random_groups(rng, 20)
    xb = _bf16_of(x)
    xf = O.bf16_to_f32(xb).astype(np.float64)
    codes, scale, zero = O.quantize_groups(xb, bits)
    qmax = 2 ** bits - 1
    for r in range(x.shape[0]):
        s = float(scale[r, 0]); zz = float(zero[r, 0])
        grid = (np.arange(qmax + 1) - zz) * s
        d = np.abs(xf[r][:, None] - grid[None, :])
        best = d.min(axis=1)
        chosen = d[np.arange(32), codes[r].astype(int)]
        # equal up to the float32 rounding of the quotient x / scale
        assert np.all(chosen <= best + s * 2.0 ** -15)


def test_quantize_exact_grid_reconstructs_exactly():
    rng = np.random.default_rng(5)
    for bits in (8, 4):
        qmax = 2 ** bits - 1
        for _ in range(50):
            e = int(rng.integers(-8, 3))
            s0 = 2.0 ** e
            z0 = int(rng.integers(0, qmax + 1))
            k = rng.integers(0, qmax + 1, 32)
            k[0], k[1] = 0, qmax
            x = ((k - z0) * s0).astype(np.float32)
            codes, scale, zero = O.quantize_groups(_bf16_of(x)[None, :], bits)
            assert float(scale[0, 0]) == s0
            assert int(zero[0, 0]) == z0
            assert np.array_equal(codes[0], k)
            assert np.array_equal(O.dequantize(codes, scale, zero)[0], x.astype(np.float64))


def test_dequantize_hand_worked():
    codes = np.array([[0, 255] + [64] * 30], dtype=np.uint8)
    scale = np.array([[1029 / 65536]], dtype=np.float16)
    zero = np.array([[64]], dtype=np.float16)
    xh = O.dequantize(codes, scale, zero)
    assert xh[0, 0] == -64 * 1029 / 65536 and xh[0, 1] == 191 * 1029 / 65536 and xh[0, 5] == 0.0


# ---------------------------------------------------------------------------
# attention: closed forms, invariants and a scalar brute force
# ---------------------------------------------------------------------------

def _brute_attention(q, k, v, scale, allowed=None):
    """Scalar Python: softmax via log-sum-exp with math.fsum, then a weighted sum."""
    nq, nk, d = len(q), len(k), len(v[0])
    out = []
    for i in range(nq):
        keys = [j for j in range(nk) if allowed is None or allowed[i][j]]
        s = {j: scale * math.fsum(q[i][c] * k[j][c] for c in range(d)) for j in keys}
        mx = max(s.values())
        lse = mx + math.log(math.fsum(math.exp(s[j] - mx) for j in keys))
        out.append([math.fsum(math.exp(s[j] - lse) * v[j][c] for j in keys) for c in range(d)])
    return np.array(out)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(0)
    s = rng.standard_normal((50, 300)) * rng.uniform(0.1, 30, (50, 1))
    s[:, ::7] = -np.inf
    p = O.softmax_rows(s)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(p[:, ::7] == 0)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(1)
    for nq, nk, d in [(1, 1, 4), (2, 5, 4), (3, 8, 4), (1, 8, 3)]:
        q = rng.standard_normal((nq, d)); k = rng.standard_normal((nk, d)); v = rng.standard_normal((nk, d))
        allowed = rng.random((nq, nk)) < 0.7
        allowed[:, 0] = True
        for al in (None, allowed):
            got = O.attention(q, k, v, 0.7, al)
            want = _brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.7, None if al is None else al.tolist())
            assert np.allclose(got, want, rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    d = 8
    v = rng.standard_normal((6, d)); k = rng.standard_normal((6, d))
    # a single key returns its value
    assert np.allclose(O.attention(rng.standard_normal((1, d)), k[:1], v[:1], 1.0), v[:1], rtol=0, atol=1e-15)
    # a zero query weights every key equally: the mean of V
    assert np.allclose(O.attention(np.zeros((1, d)), k, v, 1.0)[0], v.mean(axis=0), atol=1e-14)
    # two keys with scores a, b: logistic weights
    q = np.zeros((1, d)); q[0, 0] = 1.0
    kk = np.zeros((2, d)); kk[0, 0] = 0.3; kk[1, 0] = -1.1
    w0 = 1.0 / (1.0 + math.exp(-(0.3 - -1.1) * 2.0))
    assert np.allclose(O.attention(q, kk, v[:2], 2.0)[0], w0 * v[0] + (1 - w0) * v[1], atol=1e-14)
    # permuting the keys (with their values) changes nothing
    p = rng.permutation(6)
    qq = rng.standard_normal((3, d))
    assert np.allclose(O.attention(qq, k, v, 0.5), O.attention(qq, k[p], v[p], 0.5), atol=1e-14)
    # an overwhelming score selects its key
    kk = np.zeros((3, d)); kk[1, 0] = 1.0
    assert np.allclose(O.attention(q, kk, v[:3], 1e4)[0], v[1], atol=1e-12)


def test_decode_attention_gqa_mapping_and_empty_sequence():
    """Query head h must read KV head h // (Hq/Hkv): plant constant V per KV head, Q = 0."""
    B, Hq, Hkv, T, D = 2, 8, 2, 5, 4
    q = _bf16_of(np.zeros((B, Hq, D)))
    k = np.random.default_rng(0).standard_normal((B, Hkv, T, D))
    v = np.zeros((B, Hkv, T, D))
    for h in range(Hkv):
        v[:, h] = 10.0 * (h + 1)
    out = O.decode_attention(q, k, v, np.array([5, 0]), 1.0)
    for h in range(Hq):
        assert np.allclose(out[0, h], 10.0 * (h // (Hq // Hkv) + 1))
    assert np.all(out[1] == 0)


def test_decode_attention_brute_force():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, T, D = 2, 4, 2, 7, 4
    q = _bf16_of(rng.standard_normal((B, Hq, D)))
    k = rng.standard_normal((B, Hkv, T, D)); v = rng.standard_normal((B, Hkv, T, D))
    lens = np.array([7, 3])
    out = O.decode_attention(q, k, v, lens, 0.9)
    qf = O.bf16_to_f32(q).astype(np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // 2
            want = _brute_attention([qf[b, h].tolist()], k[b, kv, :lens[b]].tolist(),
                                    v[b, kv, :lens[b]].tolist(), 0.9)
            assert np.allclose(out[b, h], want[0], rtol=1e-12, atol=1e-13)


def test_prefill_mask_semantics_brute_force():
    """Causal + tile mask with tile 2 on 7 tokens, against key deletion in scalar Python."""
    rng = np.random.default_rng(6)
    S, D, tile = 7, 4, 2
    q = _bf16_of(rng.standard_normal((1, 2, S, D)))
    k = rng.standard_normal((1, 1, S, D)); v = rng.standard_normal((1, 1, S, D))
    n_t = 4
    mask = np.tril(np.ones((n_t, n_t), np.uint8)); mask[2, 1] = 0; mask[3, 1] = 0; mask[3, 2] = 0
    rows = np.arange(S)
    qf = O.bf16_to_f32(q).astype(np.float64)
    for h in range(2):
        got = O.prefill_rows(q, k, v, 0, h, rows, mask, 0.8, tile)
        for i in range(S):
            keys = [j for j in range(i + 1) if j // tile == i // tile or mask[i // tile, j // tile]]
            want = _brute_attention([qf[0, h, i].tolist()], k[0, 0, keys].tolist(), v[0, 0, keys].tolist(), 0.8)
            assert np.allclose(got[i], want[0], rtol=1e-12, atol=1e-13)
    # row 0 sees only key 0
    assert np.allclose(O.prefill_rows(q, k, v, 0, 0, np.array([0]), mask, 0.8, tile)[0], v[0, 0, 0])


def test_prefill_non_causal_mask_semantics_brute_force():
    """Non-causal + tile mask (entries above and below the diagonal) with tile 2
    on 7 tokens, against key deletion in scalar Python."""
    rng = np.random.default_rng(16)
    S, D, tile = 7, 4, 2
    q = _bf16_of(rng.standard_normal((1, 3, S, D)))
    k = rng.standard_normal((1, 1, S, D)); v = rng.standard_normal((1, 1, S, D))
    mask = np.ones((4, 4), np.uint8); mask[0, 3] = 0; mask[1, 0] = 0; mask[1, 2] = 0; mask[3, 1] = 0
    mask[2, 2] = 0                                   # a diagonal entry is ignored: the tile is always kept
    rows = np.arange(S)
    qf = O.bf16_to_f32(q).astype(np.float64)
    for h in range(3):
        got = O.prefill_rows(q, k, v, 0, h, rows, mask, 0.8, tile, causal=False)
        for i in range(S):
            keys = [j for j in range(S) if j // tile == i // tile or mask[i // tile, j // tile]]
            want = _brute_attention([qf[0, h, i].tolist()], k[0, 0, keys].tolist(), v[0, 0, keys].tolist(), 0.8)
            assert np.allclose(got[i], want[0], rtol=1e-12, atol=1e-13)
    # the last row, non-causal with no mask, is plain attention over all keys; row 0 too
    for r in (0, S - 1):
        want = _brute_attention([qf[0, 0, r].tolist()], k[0, 0].tolist(), v[0, 0].tolist(), 0.8)
        got = O.prefill_rows(q, k, v, 0, 0, np.array([r]), None, 0.8, tile, causal=False)
        assert np.allclose(got[0], want[0], rtol=1e-12, atol=1e-13)
    # causal and non-causal agree on the last row when the mask keeps every tile
    a = O.prefill_rows(q, k, v, 0, 1, np.array([S - 1]), None, 0.8, tile, causal=True)
    b = O.prefill_rows(q, k, v, 0, 1, np.array([S - 1]), None, 0.8, tile, causal=False)
    assert np.array_equal(a, b)


def test_prefill_seq_len_equals_truncated_inputs():
    """A sequence of length L inside a padded S: the same as the oracle on inputs cut to L (both modes, with a
    mask), and padding keys never matter (they are overwritten with large values here)."""
    rng = np.random.default_rng(17)
    S, L, D, tile = 12, 7, 4, 4
    q = _bf16_of(rng.standard_normal((1, 2, S, D)))
    k = rng.standard_normal((1, 1, S, D)); v = rng.standard_normal((1, 1, S, D))
    k[:, :, L:] = 1e6; v[:, :, L:] = -1e6
    mask = np.ones((3, 3), np.uint8); mask[1, 0] = 0; mask[0, 1] = 0
    rows = np.arange(L)
    for causal in (True, False):
        for h in range(2):
            a = O.prefill_rows(q, k, v, 0, h, rows, mask, 0.5, tile, causal=causal, seq_len=L)
            b = O.prefill_rows(q[:, :, :L], k[:, :, :L], v[:, :, :L], 0, h, rows, mask, 0.5, tile, causal=causal)
            assert np.array_equal(a, b)
    with pytest.raises(AssertionError):
        O.prefill_rows(q, k, v, 0, 0, np.array([L]), None, 0.5, tile, seq_len=L)


def test_prefill_all_ones_mask_equals_dense_causal():
    rng = np.random.default_rng(7)
    S, D = 300, 16
    q = _bf16_of(rng.standard_normal((1, 4, S, D)))
    k = rng.standard_normal((1, 2, S, D)); v = rng.standard_normal((1, 2, S, D))
    ones = np.ones((3, 3), np.uint8)
    rows = np.array([0, 1, 127, 128, 129, 255, 256, 299])
    for h in range(4):
        a = O.prefill_rows(q, k, v, 0, h, rows, ones, 0.25)
        b = O.prefill_rows(q, k, v, 0, h, rows, None, 0.25)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("tile", [1, 7, 32, 128])
def test_online_softmax_equals_one_shot(tile):
    rng = np.random.default_rng(tile)
    T, D = 1000, 16
    q = rng.standard_normal(D) * 2; k = rng.standard_normal((T, D)); v = rng.standard_normal((T, D))
    ref = O.attention(q[None], k, v, 0.6)[0]
    bounds = list(range(0, T, tile)) + [T]
    got = O.online_softmax_attention(q, k, v, 0.6, bounds)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)
    cut = sorted(set([0, T] + list(rng.integers(0, T, 9))))
    assert np.allclose(O.online_softmax_attention(q, k, v, 0.6, cut), ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(O.lse_merge(O.split_partials(q, k, v, 0.6, cut)), ref, rtol=1e-12, atol=1e-13)


def test_lse_merge_with_empty_split():
    rng = np.random.default_rng(9)
    T, D = 50, 8
    q = rng.standard_normal(D); k = rng.standard_normal((T, D)); v = rng.standard_normal((T, D))
    parts = O.split_partials(q, k, v, 1.0, [0, 20, 20, 50])
    assert parts[1][1] == -np.inf
    assert np.allclose(O.lse_merge(parts), O.attention(q[None], k, v, 1.0)[0], atol=1e-13)


# ---------------------------------------------------------------------------
# planted mistakes: each plausible slip in the oracle must break a pin above
# ---------------------------------------------------------------------------

def _run_pins(fns):
    failed = 0
    for fn in fns:
        try:
            fn()
        except AssertionError:
            failed += 1
    return failed


def test_planted_quantize_mistakes_are_caught(monkeypatch):
    orig = O.quantize_groups
    golden = _load_golden()

    def pins():
        for c in golden:
            test_quantize_hand_worked_cases(c)
        test_quantize_invariants(8)
        test_quantize_exact_grid_reconstructs_exactly()

    # (a) zero point added with the wrong sign
    def bad_sign(x, bits):
        c, s, z = orig(x, bits)
        qmax = 2 ** bits - 1
        xf = O.bf16_to_f32(x)
        g = xf.reshape(xf.shape[:-1] + (-1, 32))
        cc = np.clip(O.rne_int(g / s.astype(np.float32)[..., None]) - z.astype(np.int64)[..., None], 0, qmax)
        return cc.reshape(xf.shape).astype(np.uint8), s, z
    # (b) scale rounded to nearest instead of up
    def bad_round(x, bits):
        c, s, z = orig(x, bits)
        xf = O.bf16_to_f32(x).reshape(x.shape[:-1] + (-1, 32))
        lo = np.minimum(0, xf.min(-1)); hi = np.maximum(0, xf.max(-1))
        s2 = ((hi - lo) / np.float32(2 ** bits - 1)).astype(np.float16)
        s2 = np.where(hi - lo == 0, np.float16(1), s2)
        return c, s2.astype(np.float16), z
    # (c) range not widened to contain zero (min/max of the data only)
    def bad_range(x, bits):
        qmax = 2 ** bits - 1
        xf = O.bf16_to_f32(x)
        g = xf.reshape(xf.shape[:-1] + (-1, 32))
        lo = g.min(-1); hi = g.max(-1); r = (hi - lo).astype(np.float32)
        s = O.f16_round_up(r / np.float32(qmax)); s = np.where(r == 0, np.float16(1), s).astype(np.float16)
        z = np.clip(O.rne_int(-lo / s.astype(np.float32)), 0, qmax)
        cc = np.clip(O.rne_int(g / s.astype(np.float32)[..., None]) + z[..., None], 0, qmax)
        return cc.reshape(xf.shape).astype(np.uint8), s, z.astype(np.float16)
    for bad in (bad_sign, bad_round, bad_range):
        monkeypatch.setattr(O, "quantize_groups", bad)
        assert _run_pins([pins]) == 1, bad.__name__
    monkeypatch.setattr(O, "quantize_groups", orig)
    assert _run_pins([pins]) == 0


def test_planted_attention_mistakes_are_caught(monkeypatch):
    orig = O.attention

    def pins():
        test_attention_brute_force_tiny()
        test_attention_closed_forms()

    def no_scale(q, k, v, scale, allowed=None):
        return orig(q, k, v, 1.0, allowed)
    def transposed_v(q, k, v, scale, allowed=None):
        qq = np.asarray(q, np.float64)
        s = scale * (qq @ np.asarray(k, np.float64).T)
        if allowed is not None:
            s = np.where(allowed, s, -np.inf)
        p = O.softmax_rows(s)
        vv = np.asarray(v, np.float64)
        return p @ vv[::-1]
    def ignores_mask(q, k, v, scale, allowed=None):
        return orig(q, k, v, scale, None)
    for bad in (no_scale, transposed_v, ignores_mask):
        monkeypatch.setattr(O, "attention", bad)
        assert _run_pins([pins]) == 1, bad.__name__
    monkeypatch.setattr(O, "attention", orig)
    assert _run_pins([pins]) == 0
