"""GPU parity of the prefill over 4-bit, mixed per-head and head-dim-64 caches.

The page stores sensitive heads at the higher bit-width and the rest at the
lower one; a cache laid out that way is filled by the prefill call itself
(quantise-on-write, bit-exact against the oracle) and its dequantised codes
are attended.  Outputs must satisfy |o - ref| <= 2e-3 + 2e-3 |ref| against
the fp64 oracle fed the same dequantised cache, on every row.  The last test
runs the whole chain: statistics, allocation, prefill into the allocated
cache, then decode over it.
"""
import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq as K
    K.lib()
    return K


def _full_mask(n_t: int, seed: int, keep: float = 0.7) -> np.ndarray:
    return (np.random.default_rng(seed).random((n_t, n_t)) < keep).astype(np.uint8)


def _run(kvq, inp, head_bits, causal=True, out_dtype=0, lens=None):
    B, Hkv, S, D = inp.B, inp.Hkv, inp.S, inp.D
    hb = np.asarray(head_bits, np.int8)
    kc = kvq.empty_cache(hb, B, S, D)
    vc = kvq.empty_cache(hb, B, S, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.from_numpy(inp.tile_mask).cuda() if inp.tile_mask is not None else None
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    out = kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                                inp.softmax_scale, mask, out_dtype=out_dtype, status=status, causal=causal,
                                seq_lens=sl)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.float().cpu().numpy(), kc, vc


def _check(inp, head_bits, got, kc, vc, causal=True, out_bf16=False, lens=None):
    margin = U.Margin(inp.name)
    lens = lens if lens is not None else [inp.S] * inp.B
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0)
            continue
        planes_o, sc_o, z_o, kd = U.oracle_quantize(inp.k[b:b + 1, :, :L], head_bits)
        vplanes_o, vsc_o, vz_o, vd = U.oracle_quantize(inp.v[b:b + 1, :, :L], head_bits)
        # the caches this call wrote: bit-exact codes, scales and zero points
        for cache, (pl, sc, z) in ((kc, (planes_o, sc_o, z_o)), (vc, (vplanes_o, vsc_o, vz_o))):
            planes, scale, zero = U.read_cache(cache, L)
            for h in range(inp.Hkv):
                assert np.array_equal(planes[h][b], pl[h][0]), (inp.name, b, h)
            assert np.array_equal(scale[b].view(np.uint16), sc[0].view(np.uint16))
            assert np.array_equal(zero[b].view(np.uint16), z[0].view(np.uint16))
        for h in range(inp.Hq):
            ref = O.prefill_rows(inp.q[b:b + 1, :, :L], kd, vd, 0, h, np.arange(L), inp.tile_mask,
                                 inp.softmax_scale, causal=causal)
            margin.add(U.assert_close(got[b, h, :L], ref, f"{inp.name} b={b} h={h}", out_bf16), L)
        assert np.all(got[b, :, L:] == 0)
    margin.report()


CASES = [
    # name, seed, B, Hq, Hkv, D, S, head bits, causal, mask ("causal" seed / "full" seed / None)
    ("int4_rep2_d128", 81, 1, 4, 2, 128, 384, [4, 4], True, ("causal", 3)),
    ("mixed_rep4_d128", 82, 1, 16, 4, 128, 512, [8, 4, 4, 8], True, ("causal", 4)),
    ("mixed_rep3_d128", 88, 1, 6, 2, 128, 256, [4, 8], True, None),
    ("d64_int8_rep2", 83, 1, 4, 2, 64, 384, [8, 8], True, None),
    ("d64_int4_rep3", 84, 1, 6, 2, 64, 256, [4, 4], True, ("causal", 5)),
    ("d64_mixed_batch2", 89, 2, 4, 2, 64, 384, [8, 4], True, ("causal", 6)),
    ("d64_mixed_noncausal", 85, 2, 4, 2, 64, 384, [4, 8], False, ("full", 7)),
    ("mixed_noncausal_d128", 86, 1, 8, 2, 128, 384, [8, 4], False, None),
    ("int4_mha_d128", 90, 1, 2, 2, 128, 256, [4, 4], True, None),
    ("max_64_kv_heads_d64", 97, 1, 64, 64, 64, 256, [8, 4] * 32, True, ("causal", 11)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_bits_parity(kvq, case):
    name, seed, B, Hq, Hkv, D, S, hb, causal, mk = case
    inp = W.make_prefill(name, seed, B, Hq, Hkv, D, S, mask_seed=None)
    if mk is not None:
        kind, mseed = mk
        inp.tile_mask = W.make_tile_mask(mseed, S // 128) if kind == "causal" else _full_mask(S // 128, mseed)
    got, kc, vc = _run(kvq, inp, hb, causal=causal)
    _check(inp, hb, got, kc, vc, causal=causal)


def test_prefill_bits_bf16_output_d64(kvq):
    inp = W.make_prefill("d64_bf16", 91, 1, 4, 2, 64, 256, mask_seed=8)
    got, kc, vc = _run(kvq, inp, [4, 8], out_dtype=1)
    _check(inp, [4, 8], got, kc, vc, out_bf16=True)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_prefill_bits_varlen(kvq, causal):
    inp = W.make_prefill("vl_mixed", 87, 3, 4, 2, 128, 512, mask_seed=None)
    lens = [512, 300, 1]
    got, kc, vc = _run(kvq, inp, [4, 8], causal=causal, lens=lens)
    _check(inp, [4, 8], got, kc, vc, causal=causal, lens=lens)


def test_prefill_int8_heads_unchanged_by_a_4bit_neighbour(kvq):
    """The 8-bit heads of a mixed cache give the same output bytes as an all-8-bit cache."""
    inp = W.make_prefill("neighbour", 92, 1, 8, 2, 128, 384, mask_seed=9)
    mixed, _, _ = _run(kvq, inp, [8, 4])
    plain, _, _ = _run(kvq, inp, [8, 8])
    assert np.array_equal(mixed[:, :4], plain[:, :4])


def test_allocation_prefill_then_decode(kvq):
    """Per-head statistics on the GPU, allocation on the host, a prefill that
    quantises into the allocated cache and attends it, and a decode of a new
    query over the same cache: each against the oracle."""
    B, Hq, H, D, S = 2, 16, 8, 128, 512
    # outlier channels x4: the allocation still singles out heads 2 and 5, and
    # the prefill's fp16 K_hat operand (one rounding of (c - z) s) keeps the
    # score error well inside the tolerance (it grows with |q| |k|)
    sens = W.make_sensitivity("alloc_prefill", 93, B, H, D, S, [2, 5], outlier_mult=4.0, lens=[S, S])
    ks = kvq.head_error_stats(U.to_dev_bf16(sens.k), 4)
    vs = kvq.head_error_stats(U.to_dev_bf16(sens.v), 4)
    bits, _ = kvq.allocate_head_bits(ks, vs, 2)
    assert list(np.flatnonzero(bits == 8)) == [2, 5]
    rng = np.random.default_rng(94)
    q = W._draw_bf16(rng, (B, Hq, S, D))
    inp = W.PrefillInputs("alloc_prefill", q, sens.k, sens.v, W.make_tile_mask(10, S // 128), 1.0 / np.sqrt(D),
                          Hq, H, D, S, bits)
    got, kc, vc = _run(kvq, inp, bits)
    _check(inp, bits, got, kc, vc)
    # decode of a new query over the cache the prefill wrote
    qd = W._draw_bf16(rng, (B, Hq, D))
    sl = torch.full((B,), S, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.decode_attention(U.to_dev_bf16(qd), kc, vc, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kd = U.oracle_quantize(sens.k, bits)[3]
    vd = U.oracle_quantize(sens.v, bits)[3]
    ref = O.decode_attention(qd, kd, vd, np.full(B, S), inp.softmax_scale)
    U.assert_close(out.cpu().numpy(), ref, "decode after prefill over allocated bits")


JUMPS = [(128 + 70, "tile1_chunk2"), (256 + 5, "tile2_chunk0"), (256 + 100, "tile2_chunk3")]


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("tok", [t for t, _ in JUMPS], ids=[n for _, n in JUMPS])
def test_prefill_running_max_jumps(kvq, causal, tok):
    """One key token of large values in the middle of a later key tile: in
    the rows whose score against it is large the tile's max exceeds the running
    max by far more than the rescale threshold, so the running max moves in
    the middle of the sequence and the O accumulated so far is rescaled (after
    the previous P.V product has finished); in those rows that key then
    dominates, so an unrescaled O would show at full weight.  Every row
    against the oracle, over an 8-bit and a 4-bit KV head.  (The key's values
    are chosen so that the fp16 K operand holds them exactly: with ordinary
    bf16 values of that size the operand's rounding alone moves such scores by
    percents, and the check would measure that instead of the rescale.)"""
    inp = W.make_prefill("max_jump", 95, 1, 4, 2, 128, 512, mask_seed=None)
    kf = (inp.k.astype(np.uint32) << 16).view(np.float32).copy()
    # The large key: per 32-channel group, integers n spanning exactly the code
    # range ([-128, 127] at 8 bits, [-8, 7] at 4) times a power of two, so the
    # group's scale is that power of two and its dequantised values are exact
    # in fp16 -- the scores against it then carry no operand rounding.
    rng = np.random.default_rng(96)
    for h, (lo, hi, step) in enumerate(((-128, 127, 0.5), (-8, 7, 8.0))):
        n = rng.integers(lo, hi + 1, size=(128,)).astype(np.float64)
        n[0::32], n[1::32] = lo, hi
        kf[0, h, tok] = (n * step).astype(np.float32)
    inp.k = (kf.view(np.uint32) >> 16).astype(np.uint16)
    got, kc, vc = _run(kvq, inp, [8, 4], causal=causal)
    _check(inp, [8, 4], got, kc, vc, causal=causal)
