"""Planted mistakes in the oracle: each plausible slip in one of its functions
(a dropped term, a wrong sign, index or operand order, an off-by-one) must
break at least one of the pins that check that function, and the oracle as it
stands must pass them all.  The pins are the tests of test_oracle_pins.py,
test_tile_mask.py and test_head_bits.py, called directly; each mistake is
planted in the oracle module on the CPU and removed again.
"""
import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests import test_head_bits as HB
from tests import test_oracle_pins as P
from tests import test_tile_mask as TM

GROUP = 32


def _failures(pins):
    n = 0
    for fn in pins:
        try:
            fn()
        except AssertionError:
            n += 1
    return n


def _check(monkeypatch, name, variants, pins):
    orig = getattr(O, name)
    for bad in variants:
        monkeypatch.setattr(O, name, bad)
        assert _failures(pins) >= 1, f"{name}: {bad.__name__} passes every pin"
    monkeypatch.setattr(O, name, orig)
    assert _failures(pins) == 0


# ---------------------------------------------------------------- dequantise

def test_planted_dequantize_mistakes(monkeypatch):
    def zero_added(codes, scale, zero):
        c = np.asarray(codes, np.float64)
        s = np.repeat(np.asarray(scale, np.float64), GROUP, axis=-1)
        z = np.repeat(np.asarray(zero, np.float64), GROUP, axis=-1)
        return (c + z) * s

    def groups_interleaved(codes, scale, zero):   # channel c takes group c % G instead of c // 32
        c = np.asarray(codes, np.float64)
        G = c.shape[-1] // GROUP
        s = np.tile(np.asarray(scale, np.float64), GROUP)
        z = np.tile(np.asarray(zero, np.float64), GROUP)
        assert s.shape[-1] == G * GROUP
        return (c - z) * s

    def scale_before_zero(codes, scale, zero):     # c * s - z: the zero point not scaled
        c = np.asarray(codes, np.float64)
        s = np.repeat(np.asarray(scale, np.float64), GROUP, axis=-1)
        z = np.repeat(np.asarray(zero, np.float64), GROUP, axis=-1)
        return c * s - z

    _check(monkeypatch, "dequantize", (zero_added, groups_interleaved, scale_before_zero),
           [P.test_dequantize_hand_worked, P.test_quantize_exact_grid_reconstructs_exactly,
            HB.test_values_on_the_code_grid_have_no_error, HB.test_error_bound_and_power_of_two_scaling])


# ----------------------------------------------------------------- 4-bit packing

def test_planted_int4_packing_mistakes(monkeypatch):
    def nibbles_swapped(codes):
        c = np.asarray(codes, dtype=np.uint8)
        return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)

    def halves_not_interleaved(codes):   # channel i and i + D/2 share a byte
        c = np.asarray(codes, dtype=np.uint8)
        h = c.shape[-1] // 2
        return (c[..., :h] | (c[..., h:] << 4)).astype(np.uint8)

    _check(monkeypatch, "pack_int4", (nibbles_swapped, halves_not_interleaved), [P.test_int4_packing_hand_worked])


# ---------------------------------------------------------------- decode

def test_planted_decode_mistakes(monkeypatch):
    orig = O.decode_attention

    def heads_modulo(q_bits, k_hat, v_hat, seq_lens, softmax_scale):   # query head h reads KV head h % Hkv
        B, Hq, D = q_bits.shape
        Hkv = k_hat.shape[1]
        q = O.bf16_to_f32(q_bits).astype(np.float64)
        out = np.zeros((B, Hq, D))
        for b in range(B):
            L = int(seq_lens[b])
            if L == 0:
                continue
            for h in range(Hq):
                out[b, h] = O.attention(q[b, h][None, :], k_hat[b, h % Hkv, :L], v_hat[b, h % Hkv, :L],
                                        softmax_scale)[0]
        return out

    def last_token_dropped(q_bits, k_hat, v_hat, seq_lens, softmax_scale):
        lens = np.maximum(np.asarray(seq_lens) - 1, 0)
        return orig(q_bits, k_hat, v_hat, lens, softmax_scale)

    _check(monkeypatch, "decode_attention", (heads_modulo, last_token_dropped),
           [P.test_decode_attention_gqa_mapping_and_empty_sequence, P.test_decode_attention_brute_force])


# ---------------------------------------------------------------- prefill visibility

def test_planted_prefill_mask_mistakes(monkeypatch):
    orig = O.prefill_allowed

    def causal_strict(rows, n_keys, tile_mask, tile=128, causal=True):   # a query does not see itself
        ok = orig(rows, n_keys, tile_mask, tile, causal)
        if causal:
            ok &= np.arange(n_keys)[None, :] != np.asarray(rows)[:, None]
        return ok

    def mask_transposed(rows, n_keys, tile_mask, tile=128, causal=True):
        return orig(rows, n_keys, None if tile_mask is None else np.asarray(tile_mask).T, tile, causal)

    def diagonal_not_exempt(rows, n_keys, tile_mask, tile=128, causal=True):
        i = np.asarray(rows)[:, None]
        j = np.arange(n_keys)[None, :]
        ok = j <= i if causal else np.ones((i.shape[0], n_keys), dtype=bool)
        if tile_mask is not None:
            m = np.asarray(tile_mask)
            ok &= m[np.minimum(i // tile, m.shape[0] - 1), np.minimum(j // tile, m.shape[1] - 1)] != 0
        return ok

    def causal_ignored(rows, n_keys, tile_mask, tile=128, causal=True):
        return orig(rows, n_keys, tile_mask, tile, False)

    _check(monkeypatch, "prefill_allowed", (causal_strict, mask_transposed, diagonal_not_exempt, causal_ignored),
           [P.test_prefill_mask_semantics_brute_force, P.test_prefill_non_causal_mask_semantics_brute_force,
            P.test_prefill_all_ones_mask_equals_dense_causal, P.test_prefill_seq_len_equals_truncated_inputs])


# ---------------------------------------------------------------- online softmax and the split merge

def test_planted_merge_mistakes(monkeypatch):
    def unnormalised(parts):
        lses = np.array([p[1] for p in parts], dtype=np.float64)
        w = np.exp(lses - np.max(lses))
        return sum(wi * p[0] for wi, p in zip(w, parts))

    def weights_inverted(parts):
        lses = np.array([p[1] for p in parts], dtype=np.float64)
        fin = np.isfinite(lses)
        w = np.where(fin, np.exp(np.max(lses) - np.where(fin, lses, 0.0)), 0.0)
        return sum(wi * p[0] for wi, p in zip(w, parts)) / np.sum(w)

    def plain_average(parts):
        live = [p[0] for p in parts if np.isfinite(p[1])]
        return sum(live) / len(live)

    pins = [lambda: P.test_online_softmax_equals_one_shot(7), P.test_lse_merge_with_empty_split]
    _check(monkeypatch, "lse_merge", (unnormalised, weights_inverted, plain_average), pins)

    orig_split = O.split_partials

    def partial_lse_without_log(q, k_hat, v_hat, softmax_scale, bounds):   # e^lse passed on instead of lse
        return [(o, lse if not np.isfinite(lse) else float(np.exp(lse)))
                for o, lse in orig_split(q, k_hat, v_hat, softmax_scale, bounds)]

    _check(monkeypatch, "split_partials", (partial_lse_without_log,), pins)

    def correction_inverted(q, k_hat, v_hat, softmax_scale, bounds):
        q = np.asarray(q, dtype=np.float64)
        m, l = -np.inf, 0.0
        acc = np.zeros(v_hat.shape[-1])
        for t0, t1 in zip(bounds[:-1], bounds[1:]):
            if t1 <= t0:
                continue
            s = softmax_scale * (np.asarray(k_hat[t0:t1], np.float64) @ q)
            m_new = max(m, float(np.max(s)))
            corr = np.exp(m_new - m) if np.isfinite(m) else 0.0
            p = np.exp(s - m_new)
            l = l * corr + float(np.sum(p))
            acc = acc * corr + p @ np.asarray(v_hat[t0:t1], np.float64)
            m = m_new
        return acc / l

    _check(monkeypatch, "online_softmax_attention", (correction_inverted,), pins)


# ---------------------------------------------------------------- tile-mask builder

def test_planted_tile_mask_mistakes(monkeypatch):
    orig = O.build_tile_mask

    def diagonal_dropped(nT, num, den, seed):
        m = orig(nT, num, den, seed)
        for qt in range(1, nT):
            m[qt, qt] = 0
        return m

    def tile0_skippable(nT, num, den, seed):
        mask = np.zeros((nT, nT), dtype=np.uint8)
        for qt in range(nT):
            mask[qt, :qt + 1] = 1
            cand = np.arange(0, qt, dtype=np.int64)
            k = (len(cand) * num) // den
            if k:
                keys = O.splitmix64(seed, qt * nT + cand + 1)
                mask[qt, cand[np.argsort(keys, kind="stable")[:k]]] = 0
        return mask

    def count_rounded_up(nT, num, den, seed):
        mask = np.zeros((nT, nT), dtype=np.uint8)
        for qt in range(nT):
            mask[qt, :qt + 1] = 1
            cand = np.arange(1, qt, dtype=np.int64)
            k = -((-len(cand) * num) // den)
            if k:
                keys = O.splitmix64(seed, qt * nT + cand + 1)
                mask[qt, cand[np.argsort(keys, kind="stable")[:k]]] = 0
        return mask

    def largest_keys_skipped(nT, num, den, seed):
        mask = np.zeros((nT, nT), dtype=np.uint8)
        for qt in range(nT):
            mask[qt, :qt + 1] = 1
            cand = np.arange(1, qt, dtype=np.int64)
            k = (len(cand) * num) // den
            if k:
                keys = O.splitmix64(seed, qt * nT + cand + 1)
                mask[qt, cand[np.argsort(keys, kind="stable")[::-1][:k]]] = 0
        return mask

    params = [(1, 1, 4, 0), (2, 1, 4, 3), (9, 1, 4, 7), (33, 7, 20, 11), (64, 1, 2, 5), (40, 0, 1, 9), (40, 1, 1, 9)]
    pins = [lambda a=a: TM.test_tile_mask_invariants(*a) for a in params]
    pins.append(TM.test_tile_mask_skips_the_smallest_keys_by_brute_force)
    _check(monkeypatch, "build_tile_mask", (diagonal_dropped, tile0_skippable, count_rounded_up, largest_keys_skipped),
           pins)


# ---------------------------------------------------------------- per-head statistics and allocation

_HB_PINS = [HB.test_values_on_the_code_grid_have_no_error, HB.test_half_way_value_rounds_to_even,
            HB.test_error_bound_and_power_of_two_scaling, HB.test_weights_and_lengths,
            HB.test_outlier_heads_are_the_sensitive_ones, HB.test_statistics_add_over_sequences_and_ignore_token_order]


def test_planted_head_stats_mistakes(monkeypatch):
    orig = O.head_error_stats

    def weights_ignored(x_bits, bits, seq_lens=None, weights=None):
        return orig(x_bits, bits, seq_lens, None)

    def lengths_ignored(x_bits, bits, seq_lens=None, weights=None):
        return orig(x_bits, bits, None, weights)

    def columns_swapped(x_bits, bits, seq_lens=None, weights=None):
        return orig(x_bits, bits, seq_lens, weights)[:, ::-1].copy()

    def absolute_error(x_bits, bits, seq_lens=None, weights=None):
        x_bits = np.asarray(x_bits)
        B, H, T, D = x_bits.shape
        c, sc, z = O.quantize_groups(x_bits, bits)
        xf = O.bf16_to_f32(x_bits).astype(np.float64)
        err = np.sum(np.abs(xf - O.dequantize(c, sc, z)), axis=-1)
        nrm = np.sum(xf * xf, axis=-1)
        w = np.ones((B, H, T)) if weights is None else np.asarray(weights, np.float32).astype(np.float64)
        if seq_lens is not None:
            w = np.where((np.arange(T)[None, :] < np.asarray(seq_lens)[:, None])[:, None, :], w, 0.0)
        return np.stack([np.sum(w * err, axis=(0, 2)), np.sum(w * nrm, axis=(0, 2))], axis=1)

    _check(monkeypatch, "head_error_stats", (weights_ignored, lengths_ignored, columns_swapped, absolute_error),
           _HB_PINS)


def test_planted_sensitivity_and_allocation_mistakes(monkeypatch):
    def keys_only(k_stats, v_stats):
        st = np.asarray(k_stats, dtype=np.float64)
        return np.divide(st[:, 0], st[:, 1], out=np.zeros(st.shape[0]), where=st[:, 1] != 0)

    def ratio_inverted(k_stats, v_stats):
        def rel(st):
            st = np.asarray(st, dtype=np.float64)
            return np.divide(st[:, 1], st[:, 0], out=np.zeros(st.shape[0]), where=st[:, 0] != 0)
        return rel(k_stats) + rel(v_stats)

    pins = [HB.test_sensitivity_and_allocation_rules, HB.test_outlier_heads_are_the_sensitive_ones]
    _check(monkeypatch, "head_sensitivity", (keys_only, ratio_inverted), pins)

    def smallest_get_8(score, n_high, low_bits=4):
        score = np.asarray(score, dtype=np.float64)
        order = sorted(range(len(score)), key=lambda h: (score[h], h))
        bits = np.full(len(score), low_bits, dtype=np.int8)
        bits[order[:n_high]] = 8
        return bits

    def ties_to_larger_index(score, n_high, low_bits=4):
        score = np.asarray(score, dtype=np.float64)
        order = sorted(range(len(score)), key=lambda h: (-score[h], -h))
        bits = np.full(len(score), low_bits, dtype=np.int8)
        bits[order[:n_high]] = 8
        return bits

    _check(monkeypatch, "allocate_head_bits", (smallest_get_8, ties_to_larger_index),
           pins + [HB.test_allocation_is_equivariant_and_nested])


@pytest.mark.parametrize("name", ["quantize_groups", "dequantize", "attention", "build_tile_mask", "head_error_stats"])
def test_planting_restores_the_oracle(name):
    """No planted function leaks out of its test (the module attributes are the oracle's own)."""
    fn = getattr(O, name)
    assert fn.__module__ == O.__name__ and fn.__qualname__ == name
