"""The tile-mask builder: oracle pins on CPU, and the GPU builder bit for bit
against the oracle (GPU tests marked)."""
import numpy as np
import pytest

from oracle import kvq_oracle as O


# SplitMix64 seeded with 0: its first outputs as printed by the generator's
# reference C implementation (Vigna's splitmix64.c, after Steele, Lea and
# Flood 2014) and quoted widely as the test vector of the generator.
SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_published_first_outputs():
    got = [int(x) for x in O.splitmix64(0, np.arange(1, 4))]
    assert got == SPLITMIX64_SEED0


def test_splitmix64_seed_shifts_the_sequence():
    # seeding with s is the sequence of seed 0 started at the state s: output
    # n of seed (m * gamma) is output n + m of seed 0
    gamma = 0x9E3779B97F4A7C15
    for m in (1, 5, 1000):
        a = O.splitmix64((m * gamma) % (1 << 64), np.arange(1, 20))
        b = O.splitmix64(0, np.arange(1 + m, 20 + m))
        assert np.array_equal(a, b)


@pytest.mark.parametrize("nT,num,den,seed", [(1, 1, 4, 0), (2, 1, 4, 3), (9, 1, 4, 7), (33, 7, 20, 11),
                                             (64, 1, 2, 5), (40, 0, 1, 9), (40, 1, 1, 9)])
def test_tile_mask_invariants(nT, num, den, seed):
    m = O.build_tile_mask(nT, num, den, seed)
    assert m.shape == (nT, nT) and m.dtype == np.uint8
    for qt in range(nT):
        assert m[qt, 0] == 1 and m[qt, qt] == 1
        assert np.all(m[qt, qt + 1:] == 0)
        n = max(qt - 1, 0)
        skipped = int(n - m[qt, 1:qt].sum()) if qt > 1 else 0
        assert skipped == (n * num) // den
    if num == 0:
        assert np.array_equal(m, np.tril(np.ones((nT, nT), np.uint8)))
    if num == den:
        expect = np.zeros((nT, nT), np.uint8)
        expect[:, 0] = 1
        np.fill_diagonal(expect, 1)
        assert np.array_equal(m, expect)


def test_tile_mask_skips_the_smallest_keys_by_brute_force():
    nT, num, den, seed = 12, 1, 3, 21
    m = O.build_tile_mask(nT, num, den, seed)
    for qt in range(2, nT):
        cand = list(range(1, qt))
        keys = {kt: int(O.splitmix64(seed, np.array([qt * nT + kt + 1]))[0]) for kt in cand}
        k = (len(cand) * num) // den
        # rank by pairwise comparison (key, kt), no sorting routine
        rank = {kt: sum(1 for o in cand if (keys[o], o) < (keys[kt], kt)) for kt in cand}
        for kt in cand:
            assert m[qt, kt] == (0 if rank[kt] < k else 1), (qt, kt)


# ---------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("nT,num,den,seed", [(1, 1, 4, 0), (2, 1, 4, 1), (7, 1, 4, 2), (256, 1, 4, 4),
                                             (256, 7, 20, 5), (300, 1, 2, 6), (1000, 1, 4, 7), (4096, 1, 4, 8),
                                             (64, 0, 1, 9), (64, 1, 1, 10)])
def test_gpu_tile_mask_bit_exact(nT, num, den, seed):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq
    got = kvq.build_tile_mask(nT, num, den, seed + (1 << 63)).cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(got, O.build_tile_mask(nT, num, den, seed + (1 << 63)))


@pytest.mark.gpu
def test_gpu_prefill_with_a_device_built_mask():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq
    import kvq_workloads as W
    from tests import kvq_testutil as U
    S, Hq, Hkv, D = 1024, 4, 2, 128
    nT = S // 128
    rng = np.random.default_rng(77)
    q = W._draw_bf16(rng, (1, Hq, S, D))
    k = W._draw_bf16(rng, (1, Hkv, S, D))
    v = W._draw_bf16(rng, (1, Hkv, S, D))
    mask = kvq.build_tile_mask(nT, 1, 2, 99)
    kc = kvq.empty_cache([8] * Hkv, 1, S, D)
    vc = kvq.empty_cache([8] * Hkv, 1, S, D)
    out = kvq.prefill_attention(U.to_dev_bf16(q), U.to_dev_bf16(k), U.to_dev_bf16(v), kc, vc, 0.0, tile_mask=mask)
    torch.cuda.synchronize()
    m = O.build_tile_mask(nT, 1, 2, 99)
    assert np.array_equal(mask.cpu().numpy(), m)
    deq_k = U.oracle_quantize(k, [8] * Hkv)[3]
    deq_v = U.oracle_quantize(v, [8] * Hkv)[3]
    rows = np.arange(0, S, 37)
    for h in range(Hq):
        ref = O.prefill_rows(q, deq_k, deq_v, 0, h, rows, m, 1.0 / np.sqrt(D))
        U.assert_close(out[0, h].cpu().numpy()[rows], ref, f"head {h}")
