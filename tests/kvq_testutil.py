"""Test glue: move seeded inputs to the GPU, read caches back, compare with the oracle."""
from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O

TOL_ABS = 2e-3
TOL_REL = 2e-3


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def read_cache(cache, T: int):
    """GPU cache -> (packed code rows per head, scale f16 [B][Hkv][T][G], zero f16).

    codes is a list over heads of uint8 arrays [B][T][D*bits/8] as stored.
    """
    codes = cache.codes.cpu().numpy()
    sz = cache.sz.cpu().numpy().view(np.uint32)
    B, Hkv, Tcap, D = cache.B, cache.Hkv, cache.Tcap, cache.D
    G = D // 32
    planes = []
    for h in range(Hkv):
        bits = int(cache.head_bits[h])
        R = D * bits // 8
        off = cache.head_offset(h)
        planes.append(codes[off:off + B * Tcap * R].reshape(B, Tcap, R)[:, :T])
    szv = sz.reshape(Hkv, B, Tcap, G)[:, :, :T].transpose(1, 0, 2, 3)
    scale = (szv & 0xFFFF).astype(np.uint16).view(np.float16)
    zero = (szv >> 16).astype(np.uint16).view(np.float16)
    return planes, scale, zero


def oracle_quantize(kbits: np.ndarray, head_bits) -> tuple:
    """Oracle quantisation of bf16 [B][Hkv][T][D] with per-head bits.

    Returns (packed planes list per head [B][T][R], scale, zero, dequantised f64).
    """
    B, Hkv, T, D = kbits.shape
    planes, scales, zeros = [], [], []
    deq = np.empty((B, Hkv, T, D), dtype=np.float64)
    for h in range(Hkv):
        bits = int(head_bits[h])
        c, s, z = O.quantize_groups(kbits[:, h], bits)
        planes.append(c if bits == 8 else O.pack_int4(c))
        scales.append(s)
        zeros.append(z)
        deq[:, h] = O.dequantize(c, s, z)
    return planes, np.stack(scales, 1), np.stack(zeros, 1), deq


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "", out_bf16: bool = False):
    """|got - ref| <= 2e-3 + 2e-3 |ref|; a bf16 output may also differ by its own
    rounding, at most half a bf16 ulp = 2^-8 |ref| (8 significant bits).

    Returns the largest err / bound over the elements (1.0 = at the tolerance)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = TOL_ABS + (TOL_REL + (2.0 ** -8 if out_bf16 else 0.0)) * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    return float((err / bound).max()) if err.size else 0.0


class Margin:
    """Worst err / bound ratio over several assert_close calls of one case.

    ``report()`` prints it and, when the environment names a file in
    KVQ_MARGIN_LOG, appends one JSON line there, so a test run can record how
    far each workload stays inside the tolerance."""

    def __init__(self, name: str):
        self.name = name
        self.worst = 0.0
        self.n = 0

    def add(self, ratio: float, count: int = 1):
        self.worst = max(self.worst, ratio)
        self.n += count

    def report(self):
        import json
        import os
        line = {"case": self.name, "worst_err_over_bound": self.worst, "rows": self.n}
        print(f"parity margin {self.name}: worst err/bound {self.worst:.4f} over {self.n} rows")
        path = os.environ.get("KVQ_MARGIN_LOG")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps(line) + "\n")
