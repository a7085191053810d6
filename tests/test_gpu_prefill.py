"""GPU parity of kvq_prefill_attention (tcgen05 prefill) against the oracle.

The call quantises K and V into the caches (bit-exact against the oracle)
and computes causal or non-causal, tile-masked attention over the
dequantised cache;
outputs must satisfy |o - ref| <= 2e-3 + 2e-3 |ref| against the fp64 oracle.
Small cases are compared on every row; the full-size workload on sampled
rows of every query head.
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


def _run(inp: W.PrefillInputs, out_dtype=0, Tcap=None, causal=True):
    from attention_group_quantized_gb300 import kvq
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.S, inp.D
    Tcap = Tcap or S
    kc = kvq.empty_cache(np.full(Hkv, 8, np.int8), B, Tcap, D)
    vc = kvq.empty_cache(np.full(Hkv, 8, np.int8), B, Tcap, D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.from_numpy(inp.tile_mask).cuda() if inp.tile_mask is not None else None
    out = kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                                inp.softmax_scale, mask, out_dtype=out_dtype, status=status, causal=causal)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.float().cpu().numpy(), kc, vc


def _oracle_deq(x):
    c, s, z = O.quantize_groups(x, 8)
    return O.dequantize(c, s, z)


def _check_all_rows(inp, got, out_bf16=False, causal=True):
    kd, vd = _oracle_deq(inp.k), _oracle_deq(inp.v)
    rows = np.arange(inp.S)
    for b in range(inp.B):
        for h in range(inp.Hq):
            ref = O.prefill_rows(inp.q, kd, vd, b, h, rows, inp.tile_mask, inp.softmax_scale, causal=causal)
            U.assert_close(got[b, h], ref, f"{inp.name} b={b} h={h}", out_bf16)


CASES = [
    # name, seed, B, Hq, Hkv, S, mask seed (None = dense causal)
    ("dense_rep2", 31, 1, 4, 2, 256, None),
    ("masked_rep4", 32, 1, 8, 2, 640, 7),
    ("mha_rep1", 33, 1, 2, 2, 384, 8),
    ("odd_rep3", 34, 1, 6, 2, 256, None),
    ("batch2", 35, 2, 4, 1, 512, 9),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_small_parity(case):
    name, seed, B, Hq, Hkv, S, mseed = case
    inp = W.make_prefill(name, seed, B, Hq, Hkv, 128, S, mask_seed=mseed)
    got, kc, vc = _run(inp)
    _check_all_rows(inp, got)
    # the caches written by the same call are bit-exact
    planes, scale, zero = U.read_cache(kc, S)
    o_planes, o_scale, o_zero, _ = U.oracle_quantize(inp.k, [8] * Hkv)
    for h in range(Hkv):
        assert np.array_equal(planes[h], o_planes[h])
    assert np.array_equal(scale.view(np.uint16), o_scale.view(np.uint16))
    assert np.array_equal(zero.view(np.uint16), o_zero.view(np.uint16))


def test_prefill_all_ones_mask_equals_dense():
    inp = W.make_prefill("ones", 36, 1, 4, 2, 128, 384, mask_seed=None)
    dense, _, _ = _run(inp)
    inp.tile_mask = np.ones((3, 3), np.uint8)
    ones, _, _ = _run(inp)
    assert np.array_equal(dense, ones)


def test_prefill_bf16_output_and_larger_capacity():
    inp = W.make_prefill("bf16", 37, 1, 4, 1, 128, 256, mask_seed=3)
    got, _, _ = _run(inp, out_dtype=1, Tcap=512)
    _check_all_rows(inp, got, out_bf16=True)


def test_prefill_full_size_sampled_rows():
    inp = W.prefill_causal()
    got, _, _ = _run(inp)
    rng = np.random.default_rng(0)
    rep = inp.Hq // inp.Hkv
    for kv in range(inp.Hkv):
        kd = _oracle_deq(inp.k[:, kv:kv + 1])
        vd = _oracle_deq(inp.v[:, kv:kv + 1])
        for h in range(kv * rep, (kv + 1) * rep):
            rows = np.sort(np.concatenate([rng.integers(0, inp.S, 6), [0, 127, 128, inp.S - 1]]))
            sub_q = inp.q[:, h:h + 1]
            ref = O.prefill_rows(sub_q, kd, vd, 0, 0, rows, inp.tile_mask, inp.softmax_scale)
            U.assert_close(got[0, h, rows], ref, f"full prefill h={h}")


def _full_mask(n_t: int, seed: int, keep: float = 0.7) -> np.ndarray:
    """A tile mask with random entries above and below the diagonal."""
    return (np.random.default_rng(seed).random((n_t, n_t)) < keep).astype(np.uint8)


NON_CAUSAL = [
    # name, seed, B, Hq, Hkv, S, mask seed (None = every tile)
    ("nc_dense_rep2", 51, 1, 4, 2, 256, None),
    ("nc_masked_rep4", 52, 1, 8, 2, 640, 17),
    ("nc_mha_rep1", 53, 1, 2, 2, 384, 18),
    ("nc_odd_rep3", 54, 1, 6, 2, 256, 19),
    ("nc_batch2", 55, 2, 4, 1, 512, None),
]


@pytest.mark.parametrize("case", NON_CAUSAL, ids=[c[0] for c in NON_CAUSAL])
def test_prefill_non_causal_small_parity(case):
    name, seed, B, Hq, Hkv, S, mseed = case
    inp = W.make_prefill(name, seed, B, Hq, Hkv, 128, S, mask_seed=None)
    if mseed is not None:
        inp.tile_mask = _full_mask(S // 128, mseed)
    got, _, _ = _run(inp, causal=False)
    _check_all_rows(inp, got, causal=False)


def test_prefill_non_causal_row_with_every_tile_skipped_but_its_own():
    """Every off-diagonal tile masked out: each query tile sees only its own 128 keys."""
    inp = W.make_prefill("nc_diag_only", 56, 1, 4, 1, 128, 384, mask_seed=None)
    inp.tile_mask = np.zeros((3, 3), np.uint8)
    got, _, _ = _run(inp, causal=False)
    _check_all_rows(inp, got, causal=False)


def test_prefill_non_causal_all_ones_mask_equals_no_mask():
    inp = W.make_prefill("nc_ones", 57, 1, 4, 2, 128, 384, mask_seed=None)
    dense, _, _ = _run(inp, causal=False)
    inp.tile_mask = np.ones((3, 3), np.uint8)
    ones, _, _ = _run(inp, causal=False)
    assert np.array_equal(dense, ones)


def test_prefill_non_causal_medium_sampled_rows():
    """B1, 32/8 heads, S 4096, random off-diagonal mask: sampled rows of every head."""
    inp = W.make_prefill("nc_medium", 58, 1, 32, 8, 128, 4096, mask_seed=None)
    inp.tile_mask = _full_mask(32, 20, keep=0.75)
    got, _, _ = _run(inp, causal=False)
    rng = np.random.default_rng(1)
    rep = inp.Hq // inp.Hkv
    for kv in range(inp.Hkv):
        kd = _oracle_deq(inp.k[:, kv:kv + 1])
        vd = _oracle_deq(inp.v[:, kv:kv + 1])
        for h in range(kv * rep, (kv + 1) * rep):
            rows = np.sort(np.concatenate([rng.integers(0, inp.S, 6), [0, 127, 128, inp.S - 1]]))
            ref = O.prefill_rows(inp.q[:, h:h + 1], kd, vd, 0, 0, rows, inp.tile_mask, inp.softmax_scale,
                                 causal=False)
            U.assert_close(got[0, h, rows], ref, f"non-causal prefill h={h}")
