"""GPU parity of kvq_prefill_attention (tcgen05 prefill) against the oracle.

The call quantises K and V into the caches (bit-exact against the oracle)
and computes causal or non-causal, tile-masked attention over the
dequantised cache;
outputs must satisfy |o - ref| <= 2e-3 + 2e-3 |ref| against the fp64 oracle.
Small cases are compared on every row; the full-size workload on two rows
of every query tile of every query head.
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
    margin = U.Margin(inp.name + ("" if causal else " non-causal"))
    for b in range(inp.B):
        for h in range(inp.Hq):
            ref = O.prefill_rows(inp.q, kd, vd, b, h, rows, inp.tile_mask, inp.softmax_scale, causal=causal)
            margin.add(U.assert_close(got[b, h], ref, f"{inp.name} b={b} h={h}", out_bf16), len(rows))
    margin.report()


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


def test_prefill_full_size_rows_of_every_query_tile():
    """prefill_causal at full size: per query head, two rows of every one of
    the 256 query tiles -- a tile edge (first row of even tiles, last row of
    odd ones, so rows 128k - 1 and 128k both occur) and a seeded random row --
    plus the sequence's last row, against the oracle."""
    inp = W.prefill_causal()
    got, _, _ = _run(inp)
    rng = np.random.default_rng(0)
    rep = inp.Hq // inp.Hkv
    n_t = inp.S // 128
    margin = U.Margin(inp.name)
    for kv in range(inp.Hkv):
        kd = _oracle_deq(inp.k[:, kv:kv + 1])
        vd = _oracle_deq(inp.v[:, kv:kv + 1])
        for h in range(kv * rep, (kv + 1) * rep):
            qt = np.arange(n_t)
            edge = 128 * qt + np.where(qt % 2 == 0, 0, 127)
            rows = np.unique(np.concatenate([edge, 128 * qt + rng.integers(0, 128, n_t), [inp.S - 1]]))
            sub_q = inp.q[:, h:h + 1]
            for part in np.array_split(rows, 4):
                ref = O.prefill_rows(sub_q, kd, vd, 0, 0, part, inp.tile_mask, inp.softmax_scale)
                margin.add(U.assert_close(got[0, h, part], ref, f"full prefill h={h}"), len(part))
    margin.report()


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


# ---------------------------------------------------------------- varlen

NAN_BF16 = 0x7FC0


def _run_varlen(inp, lens, causal, out_dtype=0):
    """Padding rows of q, k, v hold NaN and the caches hold a NaN-scale sentinel, so any padding value that
    reached a valid row, or any cache slot that was written past a sequence's end, shows."""
    from attention_group_quantized_gb300 import kvq
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.S, inp.D
    q, k, v = inp.q.copy(), inp.k.copy(), inp.v.copy()
    for b, L in enumerate(lens):
        q[b, :, L:] = NAN_BF16
        k[b, :, L:] = NAN_BF16
        v[b, :, L:] = NAN_BF16
    kc = kvq.empty_cache(np.full(Hkv, 8, np.int8), B, S, D)
    vc = kvq.empty_cache(np.full(Hkv, 8, np.int8), B, S, D)
    for c in (kc, vc):
        c.codes.fill_(0xA5)
        c.sz.fill_(-1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.from_numpy(inp.tile_mask).cuda() if inp.tile_mask is not None else None
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = kvq.prefill_attention(U.to_dev_bf16(q), U.to_dev_bf16(k), U.to_dev_bf16(v), kc, vc, inp.softmax_scale,
                                mask, out_dtype=out_dtype, status=status, causal=causal, seq_lens=sl)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), kc, vc, int(status.item())


def _check_varlen(inp, lens, causal, got, kc, out_bf16=False):
    S, Hkv = inp.S, inp.Hkv
    planes, scale, zero = U.read_cache(kc, S)
    for b, L in enumerate(lens):
        L = min(max(L, 0), S)
        assert np.all(got[b, :, L:] == 0), f"padding rows of sequence {b} are not zero"
        if L > 0:
            kd = _oracle_deq(inp.k[b:b + 1, :, :L])
            vd = _oracle_deq(inp.v[b:b + 1, :, :L])
            for h in range(inp.Hq):
                ref = O.prefill_rows(inp.q[b:b + 1, :, :L], kd, vd, 0, h, np.arange(L), inp.tile_mask,
                                     inp.softmax_scale, causal=causal)
                U.assert_close(got[b, h, :L], ref, f"{inp.name} b={b} h={h}", out_bf16)
            o_planes, o_scale, o_zero, _ = U.oracle_quantize(inp.k[b:b + 1, :, :L], [8] * Hkv)
            for h in range(Hkv):
                assert np.array_equal(planes[h][b, :L], o_planes[h][0]), (b, h)
            assert np.array_equal(scale[b, :, :L].view(np.uint16), o_scale[0].view(np.uint16))
            assert np.array_equal(zero[b, :, :L].view(np.uint16), o_zero[0].view(np.uint16))
        # cache positions past the sequence: cleared to the end of its 128-token tile, untouched after
        E = (L + 127) // 128 * 128
        for h in range(Hkv):
            assert np.all(planes[h][b, L:E] == 0), (b, h)
            assert np.all(planes[h][b, E:] == 0xA5), (b, h)
        assert np.all(scale[b, :, L:E].view(np.uint16) == 0) and np.all(zero[b, :, L:E].view(np.uint16) == 0)
        assert np.all(scale[b, :, E:].view(np.uint16) == 0xFFFF)


VARLEN = [
    # name, seed, B, Hq, Hkv, S, lens, causal, mask ("causal" seed / "full" seed / None)
    ("vl_causal", 71, 3, 4, 2, 512, [512, 300, 1], True, None),
    ("vl_causal_masked", 72, 2, 8, 2, 640, [640, 129], True, ("causal", 5)),
    ("vl_noncausal", 73, 3, 4, 1, 384, [384, 200, 127], False, None),
    ("vl_noncausal_masked", 74, 2, 6, 2, 512, [511, 256], False, ("full", 6)),
    ("vl_empty_and_one_tile", 75, 2, 2, 1, 256, [0, 128], True, None),
    ("vl_tile_edges_causal", 79, 5, 4, 2, 1024, [1024, 1023, 897, 128, 0], True, ("causal", 8)),
    ("vl_tile_edges_noncausal", 80, 5, 4, 2, 1024, [1, 1023, 897, 129, 1024], False, ("full", 9)),
]


@pytest.mark.parametrize("case", VARLEN, ids=[c[0] for c in VARLEN])
def test_prefill_varlen_parity(case):
    name, seed, B, Hq, Hkv, S, lens, causal, mk = case
    inp = W.make_prefill(name, seed, B, Hq, Hkv, 128, S, mask_seed=None)
    if mk is not None:
        kind, mseed = mk
        inp.tile_mask = (W.make_tile_mask(mseed, S // 128) if kind == "causal" else _full_mask(S // 128, mseed))
    got, kc, vc, status = _run_varlen(inp, lens, causal)
    assert status == 0
    _check_varlen(inp, lens, causal, got, kc)


def test_prefill_varlen_bf16_out():
    inp = W.make_prefill("vl_bf16", 76, 2, 4, 2, 128, 384, mask_seed=None)
    got, kc, vc, status = _run_varlen(inp, [383, 130], True, out_dtype=1)
    assert status == 0
    _check_varlen(inp, [383, 130], True, got, kc, out_bf16=True)


def test_prefill_varlen_full_lengths_equal_the_plain_call():
    inp = W.make_prefill("vl_same", 77, 2, 4, 2, 128, 256, mask_seed=3)
    plain, _, _ = _run(inp)
    got, _, _, status = _run_varlen(inp, [256, 256], True)
    assert status == 0
    assert np.array_equal(plain, got)


def test_prefill_varlen_length_out_of_range_is_reported_and_clamped():
    inp = W.make_prefill("vl_bad", 78, 2, 2, 1, 128, 256, mask_seed=None)
    from attention_group_quantized_gb300 import kvq
    kc = kvq.empty_cache(np.full(1, 8, np.int8), 2, 256, 128)
    vc = kvq.empty_cache(np.full(1, 8, np.int8), 2, 256, 128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.tensor([300, -5], dtype=torch.int32, device="cuda")
    out = kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                                inp.softmax_scale, None, status=status, seq_lens=sl)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    got = out.cpu().numpy()
    assert np.all(got[1] == 0)                      # -5 -> 0: nothing
    kd, vd = _oracle_deq(inp.k[:1]), _oracle_deq(inp.v[:1])
    for h in range(2):                              # 300 -> 256: the whole sequence
        ref = O.prefill_rows(inp.q[:1], kd, vd, 0, h, np.arange(256), None, inp.softmax_scale)
        U.assert_close(got[0, h], ref, f"clamped h={h}")
