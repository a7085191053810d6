"""Seeded synthetic inputs for the quantised-KV attention path.

This module draws random numbers and shapes them; it holds none of the
method's arithmetic (no quantisation, no attention).  Both the CUDA path
(through the tests and the benchmark) and the CPU oracle consume what it
returns, so the two sides always see identical inputs.

Recipe (every workload):
  * ``numpy.random.Generator(PCG64(seed))``;
  * draw order: per-workload structure first (sequence lengths, per-head
    bit-widths, outlier channels), then Q, K, V in that order, each drawn in
    C order ``[B][H][T][D]`` as float32 ``standard_normal`` and rounded to
    bf16 with round-half-to-even;
  * outlier channels multiply the float32 draw before the bf16 rounding.

bf16 tensors are returned as ``uint16`` bit patterns (numpy has no bf16).
The shapes follow the long-context GQA serving setting of the source pages
(7B-class models, 32 query / 8 KV heads of width 128, 8K-128K contexts); the
pages' own datasets and models are not available, so these draws stand in
for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

GROUP = 32


def bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round half to even); returns uint16 bits."""
    u = np.ascontiguousarray(x_f32, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _draw_bf16(rng: np.random.Generator, shape, scale_cols: Optional[np.ndarray] = None,
               chunk: int = 1 << 24) -> np.ndarray:
    """Draw N(0,1) float32 in C order, optionally scale columns, round to bf16.

    ``scale_cols`` has the shape of the trailing two axes ``[H, D]`` (or
    broadcasts to it) and multiplies the draw before rounding.  Drawing is done
    in chunks of whole rows; the stream is identical to one single draw.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1, shape[-1])
    D = shape[-1]
    rows = flat.shape[0]
    rows_per_chunk = max(1, chunk // D)
    # row index -> head index, for outlier scaling
    T = shape[-2] if len(shape) >= 2 else 1
    H = shape[-3] if len(shape) >= 3 else 1
    for r0 in range(0, rows, rows_per_chunk):
        r1 = min(rows, r0 + rows_per_chunk)
        x = rng.standard_normal((r1 - r0, D), dtype=np.float32)
        if scale_cols is not None:
            heads = (np.arange(r0, r1) // T) % H
            x *= np.asarray(scale_cols, dtype=np.float32)[heads]
        flat[r0:r1] = bf16_bits(x)
    return out


@dataclass
class DecodeInputs:
    """One decode batch: q[B][Hq][D], k/v[B][Hkv][Tcap][D] (bf16 bits), lengths."""
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    seq_lens: np.ndarray          # int32 [B]
    head_bits: np.ndarray         # int8 [Hkv], 4 or 8
    softmax_scale: float
    Hq: int
    Hkv: int
    D: int
    Tcap: int
    include_quantize: bool = False

    @property
    def B(self) -> int:
        return int(self.q.shape[0])


@dataclass
class PrefillInputs:
    """One causal prefill: q[B][Hq][S][D], k/v[B][Hkv][S][D] (bf16 bits), tile mask."""
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    tile_mask: Optional[np.ndarray]   # uint8 [S/128][S/128], 1 = keep, or None (dense)
    softmax_scale: float
    Hq: int
    Hkv: int
    D: int
    S: int
    head_bits: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int8))

    @property
    def B(self) -> int:
        return int(self.q.shape[0])


# ----------------------------------------------------------------------------
# decode workloads
# ----------------------------------------------------------------------------

def make_decode(name: str, seed: int, B: int, Hq: int, Hkv: int, D: int, Tcap: int,
                lens: str = "full", len_range=None, bits: str = "8",
                outliers_shared: int = 0, outlier_shared_mult: float = 1.0,
                outliers_per_head: int = 0, outlier_head_mult: float = 1.0,
                softmax_scale: Optional[float] = None,
                include_quantize: bool = False) -> DecodeInputs:
    """Generic decode workload.

    lens: "full" (every sequence Tcap long), "uniform" (integers in
    ``len_range`` inclusive, one per sequence), or an explicit list.
    bits: "8", "4" or "mixed" (per KV head 8 if a uniform draw < 0.5 else 4).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    # 1. structure: lengths, per-head bit-widths, outlier channels
    if isinstance(lens, (list, tuple, np.ndarray)):
        seq_lens = np.asarray(lens, dtype=np.int32)
    elif lens == "full":
        seq_lens = np.full(B, Tcap, dtype=np.int32)
    elif lens == "uniform":
        lo, hi = len_range
        seq_lens = rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    else:
        raise ValueError(lens)
    if bits == "mixed":
        head_bits = np.array([8 if rng.random() < 0.5 else 4 for _ in range(Hkv)], dtype=np.int8)
    else:
        head_bits = np.full(Hkv, int(bits), dtype=np.int8)
    kscale = np.ones((Hkv, D), dtype=np.float32)
    if outliers_shared:
        ch = rng.choice(D, outliers_shared, replace=False)
        kscale[:, ch] *= np.float32(outlier_shared_mult)
    if outliers_per_head:
        for h in range(Hkv):
            ch = rng.choice(D, outliers_per_head, replace=False)
            kscale[h, ch] *= np.float32(outlier_head_mult)
    # 2. Q, K, V (K and V only for the live tokens of each sequence)
    q = _draw_bf16(rng, (B, Hq, D))
    k = np.zeros((B, Hkv, Tcap, D), dtype=np.uint16)
    v = np.zeros((B, Hkv, Tcap, D), dtype=np.uint16)
    if np.all(seq_lens == Tcap):
        k[:] = _draw_bf16(rng, (B, Hkv, Tcap, D), kscale)
        v[:] = _draw_bf16(rng, (B, Hkv, Tcap, D))
    else:
        for b in range(B):
            L = int(seq_lens[b])
            k[b, :, :L] = _draw_bf16(rng, (Hkv, L, D), kscale)
        for b in range(B):
            L = int(seq_lens[b])
            v[b, :, :L] = _draw_bf16(rng, (Hkv, L, D))
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    return DecodeInputs(name, q, k, v, seq_lens, head_bits, float(softmax_scale),
                        Hq, Hkv, D, Tcap, include_quantize)


def make_tile_mask(seed: int, n_tiles: int, skip_fraction: float = 0.25) -> np.ndarray:
    """Block-sparse causal tile mask (1 = keep).

    Of the strictly-below-diagonal tiles, ``round(skip_fraction * count)`` are
    skipped, drawn uniformly without replacement from those with key tile >= 1,
    so diagonal tiles and key tile 0 are always kept (no query row is starved
    of its first block).  Entries above the diagonal are 0 and unused.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    mask = np.tril(np.ones((n_tiles, n_tiles), dtype=np.uint8))
    below = n_tiles * (n_tiles - 1) // 2
    n_skip = int(round(skip_fraction * below))
    cand = [(qt, kt) for qt in range(n_tiles) for kt in range(1, qt)]
    pick = rng.choice(len(cand), n_skip, replace=False) if n_skip else []
    for i in pick:
        qt, kt = cand[int(i)]
        mask[qt, kt] = 0
    return mask


def make_prefill(name: str, seed: int, B: int, Hq: int, Hkv: int, D: int, S: int,
                 mask_seed: Optional[int] = None, skip_fraction: float = 0.25,
                 tile: int = 128, softmax_scale: Optional[float] = None) -> PrefillInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _draw_bf16(rng, (B, Hq, S, D))
    k = _draw_bf16(rng, (B, Hkv, S, D))
    v = _draw_bf16(rng, (B, Hkv, S, D))
    n_t = (S + tile - 1) // tile
    mask = make_tile_mask(mask_seed, n_t, skip_fraction) if mask_seed is not None else None
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    return PrefillInputs(name, q, k, v, mask, float(softmax_scale), Hq, Hkv, D, S,
                         np.full(Hkv, 8, dtype=np.int8))


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

def decode_tiny() -> DecodeInputs:
    """Decode, tiny: B1, 4/4 heads, D64, 512 tokens, INT8, seed 0; includes quantize."""
    return make_decode("decode_tiny_b1_h4_d64_t512_int8", 0, 1, 4, 4, 64, 512,
                       include_quantize=True)


def decode_gqa() -> DecodeInputs:
    """Decode GQA: B8, 32/8 heads, D128, 8192 tokens, INT8, 4 shared K outlier channels x10."""
    return make_decode("decode_gqa_b8_h32kv8_d128_t8192_int8", 1, 8, 32, 8, 128, 8192,
                       outliers_shared=4, outlier_shared_mult=10.0)


def decode_long_ragged() -> DecodeInputs:
    """Decode long ragged: B4, 32/8 heads, D128, lengths U[32768,131072], INT4."""
    return make_decode("decode_ragged_b4_h32kv8_d128_t32k-128k_int4", 2, 4, 32, 8, 128, 131072,
                       lens="uniform", len_range=(32768, 131072), bits="4")


def prefill_noncausal() -> PrefillInputs:
    """Prefill non-causal: the causal workload's shapes (B1, 32/8 heads, D128, S32768, INT8 KV), no tile mask."""
    return make_prefill("prefill_noncausal_b1_h32kv8_d128_s32768_dense", 3, 1, 32, 8, 128, 32768,
                        mask_seed=None)


def prefill_varlen():
    """Prefill varlen: B4 sequences padded to S8192, 32/8 heads, D128, INT8 KV, causal, no mask; lengths
    U[2048, 8192] from their own generator (seed 7), so the padded draws match make_prefill's recipe.
    Returns (inputs, lengths int32 [B])."""
    inp = make_prefill("prefill_varlen_b4_h32kv8_d128_s8192_len2k-8k", 6, 4, 32, 8, 128, 8192, mask_seed=None)
    lens = np.random.Generator(np.random.PCG64(7)).integers(2048, 8192, size=4, endpoint=True).astype(np.int32)
    return inp, lens


def prefill_causal() -> PrefillInputs:
    """Prefill causal: B1, 32/8 heads, D128, S32768, INT8 KV, 25% of below-diagonal tiles skipped."""
    return make_prefill("prefill_causal_b1_h32kv8_d128_s32768_skip25", 3, 1, 32, 8, 128, 32768,
                        mask_seed=4)


def decode_mixed() -> DecodeInputs:
    """Decode mixed: B16, 32/8 heads, D128, 32768 tokens, INT8/INT4 per KV head, 2 outliers x8 per head."""
    return make_decode("decode_mixed_b16_h32kv8_d128_t32768_int8int4", 5, 16, 32, 8, 128, 32768,
                       bits="mixed", outliers_per_head=2, outlier_head_mult=8.0)


@dataclass
class SensitivityInputs:
    """K and V rows [B][H][T][D] (bf16 bits) whose per-head statistics choose the bit-widths."""
    name: str
    k: np.ndarray
    v: np.ndarray
    seq_lens: np.ndarray                  # int32 [B]
    weights: Optional[np.ndarray]         # float32 [B][H][T] attention mass per token, or None
    outlier_heads: np.ndarray             # heads whose K carries outlier channels
    H: int
    D: int
    T: int


def make_sensitivity(name: str, seed: int, B: int, H: int, D: int, T: int, outlier_heads,
                     n_outlier_ch: int = 4, outlier_mult: float = 10.0, lens="full",
                     weights: bool = True) -> SensitivityInputs:
    """Heads listed in ``outlier_heads`` get ``n_outlier_ch`` K channels scaled by
    ``outlier_mult`` (channels drawn per head); the other heads are plain N(0,1).
    Draw order: outlier channels, K, V (each [B][H][T][D] in C order), then the
    weights, float32 exponential(1) per token ([B][H][T]); lengths "full" or an
    explicit list (tokens past a sequence's length are zero)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = (np.full(B, T, dtype=np.int32) if isinstance(lens, str)
                else np.asarray(lens, dtype=np.int32))
    kscale = np.ones((H, D), dtype=np.float32)
    for h in outlier_heads:
        ch = rng.choice(D, n_outlier_ch, replace=False)
        kscale[h, ch] *= np.float32(outlier_mult)
    k = _draw_bf16(rng, (B, H, T, D), kscale)
    v = _draw_bf16(rng, (B, H, T, D))
    w = rng.exponential(1.0, size=(B, H, T)).astype(np.float32) if weights else None
    for b in range(B):
        k[b, :, seq_lens[b]:] = 0
        v[b, :, seq_lens[b]:] = 0
    return SensitivityInputs(name, k, v, seq_lens, w, np.asarray(sorted(outlier_heads), dtype=np.int32),
                             H, D, T)


def head_bits_kv() -> SensitivityInputs:
    """Per-head bit allocation input: decode_gqa's K/V shape (B8, 8 KV heads, D128, 8192 tokens);
    heads 1, 4, 6 carry 4 K outlier channels x10; exponential(1) attention-mass weights."""
    return make_sensitivity("head_bits_b8_h8_d128_t8192_outliers3", 5, 8, 8, 128, 8192, [1, 4, 6])


NAMED = {
    "decode_tiny": decode_tiny,
    "decode_gqa": decode_gqa,
    "decode_long_ragged": decode_long_ragged,
    "prefill_causal": prefill_causal,
    "decode_mixed": decode_mixed,
}
