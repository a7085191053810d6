"""CPU oracle for group-quantised KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy.  Only the test suite, the package's
``smoke()`` check and the benchmark's CPU-baseline leg may import this
module; the library never calls it and shares no code with it.

What it follows (the source pages are four web articles; citations give each
page's title and the section on it):

* [P4] 《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》 (xdnf.cn)
    - §2.4 "KV Cache分组量化": the KV cache is quantised in groups of adjacent
      values along the channel (head_dim) axis, each group with its own scale
      factor and zero point; sensitive heads may keep a higher bit-width.
    - §3.2: the integration hook fixes the group size at 32
      (``kv_quant_group_size=32``).
    - §2.2: attention is computed tile by tile, each tile's local softmax
      statistics (maximum and normaliser) carried forward and merged, and a
      final correction makes the tiled result equal the global softmax.
    - §1.3 / §2.3: a block-sparse mask skips whole tiles of the score matrix.
* [P1] 《一只"兔子"如何搅动大模型推理赛道的底层逻辑》 (m.xxqk.cn) §3.1:
  Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V.

* [P4] §2.3 also caps the skipped share so that no block is starved: the
  tile-mask builder below skips, per query tile, a fixed fraction of its
  candidate key tiles and always keeps key tile 0 and the diagonal.

Readings taken where the pages are silent (each listed in the design notes):

* Quantiser form (P4 §2.4 says only "scale factor and zero point per group"):
  the textbook asymmetric scheme with an integer zero point.  The group range
  is widened to contain 0, the fp16 scale is rounded UP from (hi-lo)/qmax so
  the range never overflows the code space, the zero point is
  rne(-lo/scale), and code = clamp(rne(x/scale) + zero, 0, qmax).
  Every division is an IEEE float32 division and rne is round-half-to-even.
  An all-zero group stores scale 1, zero 0 and codes 0.
* INT4 packing: two codes per byte, even channel in the low nibble.
* Dequantisation: x_hat = (code - zero) * scale, evaluated exactly in float64.
* Decode: the single query of sequence b attends keys 0 .. len_b-1.
* Prefill: causal (key j visible to query i iff j <= i) or non-causal (every
  key of the sequence visible); a tile-mask entry 0 at an off-diagonal
  (query tile, key tile) removes those keys from the softmax entirely, as if
  their scores were -inf; diagonal tiles are always computed (with the
  element-wise causal rule when causal).
* GQA: query head h reads KV head h // (Hq / Hkv).

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

GROUP = 32  # P4 §3.2: kv_quant_group_size=32


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_round_up(x: np.ndarray) -> np.ndarray:
    """Smallest fp16 value >= x, for finite float32 x (IEEE round toward +inf).

    numpy's float32 -> float16 cast rounds to nearest even; if that lands
    below x, step one fp16 ulp toward +inf.
    """
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
        below = h.astype(np.float32) < x
        h = np.where(below, np.nextafter(h, np.float16(np.inf)), h)
    return h.astype(np.float16)


def rne_int(x: np.ndarray) -> np.ndarray:
    """Round-half-to-even of float32 values to integers (as int64)."""
    return np.rint(np.asarray(x, dtype=np.float32)).astype(np.int64)


# ----------------------------------------------------------------------------
# quantise / dequantise (P4 §2.4, group of 32 from P4 §3.2)
# ----------------------------------------------------------------------------

def quantize_groups(x_bits: np.ndarray, bits: int):
    """Quantise bf16 rows group by group.

    x_bits: uint16 bf16 patterns, shape [..., D] with D a multiple of 32.
    Returns (codes uint8 [..., D] unpacked, scale float16 [..., D/32],
    zero float16 [..., D/32]).

    Steps, per group of 32 adjacent channels, qmax = 2**bits - 1:
      1. xf = float32(x)                          (exact)
      2. lo = min(0, min xf), hi = max(0, max xf)
      3. r = hi - lo in float32; r == 0 -> scale 1, zero 0, codes 0
      4. scale = fp16 round-up of r / qmax        (IEEE fp32 division)
      5. zero = clamp(rne(-lo / scale), 0, qmax)
      6. code = clamp(rne(xf / scale) + zero, 0, qmax)
    """
    assert bits in (4, 8)
    qmax = np.float32(2 ** bits - 1)
    xf = bf16_to_f32(x_bits)
    assert np.all(np.isfinite(xf)), "oracle inputs must be finite"
    D = xf.shape[-1]
    assert D % GROUP == 0
    g = xf.reshape(xf.shape[:-1] + (D // GROUP, GROUP))
    lo = np.minimum(np.float32(0), g.min(axis=-1))
    hi = np.maximum(np.float32(0), g.max(axis=-1))
    r = (hi - lo).astype(np.float32)
    zero_range = r == np.float32(0)
    step = (r / qmax).astype(np.float32)
    scale_h = f16_round_up(step)
    assert np.all(np.isfinite(scale_h.astype(np.float32))), "fp16 scale overflow"
    scale_h = np.where(zero_range, np.float16(1.0), scale_h).astype(np.float16)
    sf = scale_h.astype(np.float32)
    z = rne_int((-lo).astype(np.float32) / sf)
    z = np.clip(z, 0, int(qmax))
    z = np.where(zero_range, 0, z)
    q = rne_int(g / sf[..., None]) + z[..., None]
    codes = np.clip(q, 0, int(qmax))
    codes = np.where(zero_range[..., None], 0, codes).astype(np.uint8)
    return (codes.reshape(xf.shape), scale_h, z.astype(np.float16))


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes two per byte: channel 2i in the low nibble, 2i+1 in the high."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0 and np.all(c < 16)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequantize(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """x_hat = (code - zero) * scale per group, exactly, in float64."""
    c = np.asarray(codes, dtype=np.float64)
    D = c.shape[-1]
    s = np.repeat(np.asarray(scale, dtype=np.float64), GROUP, axis=-1)
    z = np.repeat(np.asarray(zero, dtype=np.float64), GROUP, axis=-1)
    assert s.shape[-1] == D
    return (c - z) * s


# ----------------------------------------------------------------------------
# attention (P1 §3.1 definition; P4 §2.2-2.3 tiling and tile skipping)
# ----------------------------------------------------------------------------

def softmax_rows(scores: np.ndarray) -> np.ndarray:
    """Row softmax in float64; -inf entries get weight 0 (stable: max subtracted)."""
    s = np.asarray(scores, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, softmax_scale: float,
              allowed: np.ndarray | None = None) -> np.ndarray:
    """O = softmax(scale * Q K^T, restricted to allowed keys) V, in float64.

    q: [Nq, D]; k_hat, v_hat: [Nk, D]; allowed: bool [Nq, Nk] or None (all).
    Every row must allow at least one key.
    """
    q = np.asarray(q, dtype=np.float64)
    s = softmax_scale * (q @ np.asarray(k_hat, dtype=np.float64).T)
    if allowed is not None:
        assert np.all(allowed.any(axis=-1)), "a query row with no visible key"
        s = np.where(allowed, s, -np.inf)
    return softmax_rows(s) @ np.asarray(v_hat, dtype=np.float64)


def decode_attention(q_bits: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray,
                     seq_lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    """One query token per (sequence, query head) over that sequence's cached keys.

    q_bits: bf16 [B][Hq][D]; k_hat, v_hat: float64 [B][Hkv][T][D] (dequantised);
    seq_lens: [B].  Returns float64 [B][Hq][D]; a sequence of length 0 gives 0.
    """
    B, Hq, D = q_bits.shape
    Hkv = k_hat.shape[1]
    assert Hq % Hkv == 0
    rep = Hq // Hkv
    q = bf16_to_f32(q_bits).astype(np.float64)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            kv = h // rep
            out[b, h] = attention(q[b, h][None, :], k_hat[b, kv, :L], v_hat[b, kv, :L],
                                  softmax_scale)[0]
    return out


def prefill_allowed(rows: np.ndarray, n_keys: int, tile_mask: np.ndarray | None,
                    tile: int = 128, causal: bool = True) -> np.ndarray:
    """Visibility of keys 0..n_keys-1 to the given query rows.

    Key j is visible to query i iff (j <= i, when causal) and, for key tiles
    other than the query's own tile, tile_mask[i // tile][j // tile] == 1.
    """
    i = np.asarray(rows)[:, None]
    j = np.arange(n_keys)[None, :]
    ok = j <= i if causal else np.ones((i.shape[0], n_keys), dtype=bool)
    if tile_mask is not None:
        qt = i // tile
        kt = j // tile
        keep = np.asarray(tile_mask)[np.minimum(qt, tile_mask.shape[0] - 1),
                                     np.minimum(kt, tile_mask.shape[1] - 1)] != 0
        ok &= (kt == qt) | keep
    return ok


def prefill_rows(q_bits: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, b: int, h: int,
                 rows: np.ndarray, tile_mask: np.ndarray | None, softmax_scale: float,
                 tile: int = 128, causal: bool = True, seq_len: int | None = None) -> np.ndarray:
    """(Tile-masked) attention output for selected query rows of one head.

    q_bits: bf16 [B][Hq][S][D]; k_hat, v_hat: float64 [B][Hkv][S][D].  The
    sequence is seq_len long (S when None; the rows must lie inside it).
    Causal rows see keys up to their own position, non-causal rows all
    seq_len keys.  Returns float64 [len(rows)][D].
    """
    Hq = q_bits.shape[1]
    Hkv = k_hat.shape[1]
    kv = h // (Hq // Hkv)
    rows = np.asarray(rows)
    L = q_bits.shape[2] if seq_len is None else int(seq_len)
    assert rows.max() < L, "query rows must lie inside the sequence"
    n_keys = int(rows.max()) + 1 if causal else L
    q = bf16_to_f32(q_bits[b, h, rows]).astype(np.float64)
    allowed = prefill_allowed(rows, n_keys, tile_mask, tile, causal)
    return attention(q, k_hat[b, kv, :n_keys], v_hat[b, kv, :n_keys], softmax_scale, allowed)


# ----------------------------------------------------------------------------
# online softmax over tiles and the split merge (P4 §2.2)
# ----------------------------------------------------------------------------

def online_softmax_attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray,
                             softmax_scale: float, bounds) -> np.ndarray:
    """Tile-by-tile attention for one query vector, carrying (max, normaliser, acc).

    ``bounds`` lists the tile edges [0, b1, ..., Nk].  For each tile:
        m' = max(m, max s);  l' = l e^(m-m') + sum e^(s-m');
        acc' = acc e^(m-m') + sum e^(s-m') v;
    and the result is acc / l after the last tile (the final correction).
    Used only to show that the tiled form equals the one-shot softmax.
    """
    q = np.asarray(q, dtype=np.float64)
    m = -np.inf
    l = 0.0
    acc = np.zeros(v_hat.shape[-1], dtype=np.float64)
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        if t1 <= t0:
            continue
        s = softmax_scale * (np.asarray(k_hat[t0:t1], np.float64) @ q)
        m_new = max(m, float(np.max(s)))
        corr = np.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.exp(s - m_new)
        l = l * corr + float(np.sum(p))
        acc = acc * corr + p @ np.asarray(v_hat[t0:t1], np.float64)
        m = m_new
    return acc / l


def split_partials(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, softmax_scale: float,
                   bounds):
    """Per split [t0, t1): normalised partial output o_s and natural-log LSE."""
    q = np.asarray(q, dtype=np.float64)
    parts = []
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        if t1 <= t0:
            parts.append((np.zeros(v_hat.shape[-1]), -np.inf))
            continue
        s = softmax_scale * (np.asarray(k_hat[t0:t1], np.float64) @ q)
        m = float(np.max(s))
        p = np.exp(s - m)
        l = float(np.sum(p))
        parts.append((p @ np.asarray(v_hat[t0:t1], np.float64) / l, m + np.log(l)))
    return parts


def lse_merge(parts) -> np.ndarray:
    """Merge split partials: O = sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M)."""
    lses = np.array([p[1] for p in parts], dtype=np.float64)
    M = np.max(lses)
    w = np.exp(lses - M)
    o = sum(wi * p[0] for wi, p in zip(w, parts))
    return o / np.sum(w)


# ---------------------------------------------------------------------------
# Tile-mask builder (P4 §2.3: whole tiles are skipped, the skipped share is
# capped so no block is starved).  Reading: per query tile qt, of the key
# tiles kt in [1, qt) skip floor(n * num / den) (n = max(qt - 1, 0)), those
# with the smallest SplitMix64 keys, ties to the smaller kt; keep tile 0 and
# the diagonal; zero above the diagonal.
# ---------------------------------------------------------------------------

_SM64_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_SM64_M1 = np.uint64(0xBF58476D1CE4E5B9)
_SM64_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: np.ndarray) -> np.ndarray:
    """Output number n (1-based) of SplitMix64 seeded with `seed` (Steele, Lea
    and Flood, "Fast splittable pseudorandom number generators", 2014): the
    state after n steps is seed + n * gamma (mod 2^64), mixed by the
    generator's finaliser."""
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + n * _SM64_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _SM64_M1
        z = (z ^ (z >> np.uint64(27))) * _SM64_M2
    return z ^ (z >> np.uint64(31))


def build_tile_mask(nT: int, skip_num: int, skip_den: int, seed: int) -> np.ndarray:
    """uint8 [nT][nT]: 1 = key tile kept for that query tile."""
    mask = np.zeros((nT, nT), dtype=np.uint8)
    for qt in range(nT):
        mask[qt, :qt + 1] = 1
        cand = np.arange(1, qt, dtype=np.int64)
        k = (len(cand) * skip_num) // skip_den
        if k == 0:
            continue
        keys = splitmix64(seed, qt * nT + cand + 1)
        order = np.argsort(keys, kind="stable")     # equal keys keep the smaller kt first
        mask[qt, cand[order[:k]]] = 0
    return mask


# ---------------------------------------------------------------------------
# Per-head sensitivity and bit allocation (P4 §2.4: every attention head gets
# a sensitivity score, sensitive heads are stored at the higher bit-width and
# the rest at the lower one; P4 §3.4: keeping more heads at high precision
# lowers the compression from about 4x to 2.5x).  The pages give no formula.
# Reading: a head's sensitivity is the relative error its cached K and V
# would carry at the low bit-width, each token weighted by a caller-given
# attention mass w (1 when absent):
#   e_h = sum_{b, t < len_b} w[b,h,t] * sum_d (x - x_hat)^2,
#   n_h = sum_{b, t < len_b} w[b,h,t] * sum_d x^2,
#   score_h = e_h(K) / n_h(K) + e_h(V) / n_h(V)   (a 0 / 0 term counts 0);
# the n_high heads with the largest scores (ties to the smaller head index)
# get 8 bits, the others the low bit-width.
# ---------------------------------------------------------------------------

def head_error_stats(x_bits: np.ndarray, bits: int, seq_lens=None, weights=None) -> np.ndarray:
    """float64 [H][2]: (weighted squared quantisation error, weighted squared norm) per head.

    x_bits: bf16 patterns [B][H][T][D]; seq_lens: [B] (tokens t >= len_b are
    left out; None = all T); weights: [B][H][T] float32 (None = 1).
    x_hat is the dequantised value the cache would hold at `bits` bits.
    """
    x_bits = np.asarray(x_bits)
    B, H, T, D = x_bits.shape
    c, sc, z = quantize_groups(x_bits, bits)
    x_hat = dequantize(c, sc, z)                       # float64, exact
    xf = bf16_to_f32(x_bits).astype(np.float64)
    err_tok = np.sum((xf - x_hat) ** 2, axis=-1)       # [B][H][T]
    nrm_tok = np.sum(xf * xf, axis=-1)
    w = np.ones((B, H, T)) if weights is None else np.asarray(weights, dtype=np.float32).astype(np.float64)
    live = np.ones((B, T), dtype=bool)
    if seq_lens is not None:
        live = np.arange(T)[None, :] < np.asarray(seq_lens)[:, None]
    w = np.where(live[:, None, :], w, 0.0)
    out = np.zeros((H, 2))
    out[:, 0] = np.sum(w * err_tok, axis=(0, 2))
    out[:, 1] = np.sum(w * nrm_tok, axis=(0, 2))
    return out


def head_sensitivity(k_stats: np.ndarray, v_stats: np.ndarray) -> np.ndarray:
    """score_h = relative low-bit error of K plus that of V (0 / 0 counts 0)."""
    def rel(st):
        st = np.asarray(st, dtype=np.float64)
        return np.divide(st[:, 0], st[:, 1], out=np.zeros(st.shape[0]), where=st[:, 1] != 0)
    return rel(k_stats) + rel(v_stats)


def allocate_head_bits(score: np.ndarray, n_high: int, low_bits: int = 4) -> np.ndarray:
    """int8 [H]: 8 bits for the n_high largest scores (ties to the smaller index), low_bits elsewhere."""
    score = np.asarray(score, dtype=np.float64)
    order = sorted(range(len(score)), key=lambda h: (-score[h], h))
    bits = np.full(len(score), low_bits, dtype=np.int8)
    bits[order[:n_high]] = 8
    return bits

