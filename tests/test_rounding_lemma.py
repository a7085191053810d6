"""The rounding fact the quantiser's fast path rests on, checked on the CPU.

The specification rounds the IEEE fp32 quotient: code = rne(fl(x / s)) + z.
For a bf16 value x and an fp16 scale s (|x / s| <= 256) that equals the
exact rne(x / s): fl(x / s) lands on a half-integer h only when x / s is h
exactly, and otherwise stays on the same side of every half-integer.  The
kernels therefore decide each code from an exact fp32 remainder x - u * s
instead of a division.  Here every finite bf16 x is tried against a spread of
fp16 scales (normal and subnormal), with the exact quotient decided in
float64 (x and (k + 1/2) * s are exact there).
"""
import numpy as np


def _all_bf16():
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    return x[np.isfinite(x)]


def _exact_rne(x: np.ndarray, s: np.float32) -> np.ndarray:
    """rne(x / s) from exact comparisons: k = floor(x / s), then compare x with (k + 1/2) s."""
    xd = x.astype(np.float64)
    sd = np.float64(s)
    k = np.floor(xd / sd)
    # float64 division may be off by one ulp near integers; settle k exactly
    k = np.where(k * sd > xd, k - 1, k)
    k = np.where((k + 1) * sd <= xd, k + 1, k)
    mid = (k + 0.5) * sd                      # exact: k + 1/2 has at most 10 significant bits here
    up = (xd > mid) | ((xd == mid) & (np.mod(k, 2) == 1))
    return k + up


def test_rne_of_fp32_quotient_equals_exact_rne():
    rng = np.random.default_rng(11)
    x = _all_bf16()
    scales = np.concatenate([rng.uniform(2.0 ** -24, 2.0 ** -14, 40), rng.uniform(2.0 ** -14, 2.0 ** 8, 160),
                             2.0 ** np.arange(-24, 9), [1.0341796875, 3.0, 6.5, 0.1]])
    scales = np.unique(scales.astype(np.float16).astype(np.float32))
    scales = scales[scales > 0]
    ties = 0
    for s in scales:
        s = np.float32(s)
        sel = np.abs(x.astype(np.float64) / np.float64(s)) <= 256
        xs = x[sel]
        spec = np.rint((xs / s).astype(np.float32)).astype(np.float64)    # rne of the IEEE fp32 quotient
        exact = _exact_rne(xs, s)
        assert np.array_equal(spec, exact), f"scale {s}"
        mid = (np.floor(xs.astype(np.float64) / np.float64(s)) + 0.5) * np.float64(s)
        ties += int(np.sum(xs.astype(np.float64) == mid))
    assert ties > 1000                        # exact ties do occur, so the tie rule is exercised


def test_the_fp32_quotient_can_round_onto_a_half_integer_only_from_it():
    """A constructed near-tie: x / s just off a half-integer never rounds onto it in fp32 (bf16 x, fp16 s)."""
    allx = _all_bf16()
    for s in (np.float32(3.0), np.float32(1.0341796875), np.float32(0.0999755859375)):
        x = allx[np.abs(allx.astype(np.float64) / np.float64(s)) <= 256]
        q32 = (x / s).astype(np.float32)
        frac = q32.astype(np.float64) - np.floor(q32.astype(np.float64))
        on_half = frac == 0.5
        xd = x.astype(np.float64)
        assert np.all(xd[on_half] == (np.floor(q32[on_half].astype(np.float64)) + 0.5) * np.float64(s))
