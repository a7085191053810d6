"""Seeded random configurations of quantise + decode and of prefill against
the oracle: batch, query/KV head counts (every GQA ratio the calls accept),
head dim, capacity, ragged lengths (0, 1, tile edges), per-head bit widths,
masks, causal and non-causal, varlen and output dtype all drawn from the
case's seed, at sizes where the oracle checks every output row.

Codes, scales and zero points must equal the oracle's bit for bit;
outputs must satisfy |o - ref| <= 2e-3 + 2e-3 |ref| (plus half a bf16 ulp
of the result for bf16 output).
"""
import os

import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# cases per test (more with KVQ_SWEEP_CASES for a longer search)
N_CASES = int(os.environ.get("KVQ_SWEEP_CASES", "24"))


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq as K
    K.lib()
    return K


def _lens(rng, B, cap, tile):
    """Ragged lengths with the edge cases mixed in: 0, 1, a tile edge, the capacity."""
    special = [min(x, cap) for x in (0, 1, tile - 1, tile, tile + 1, cap)]
    return [int(rng.choice(special)) if rng.random() < 0.5 else int(rng.integers(1, cap + 1)) for _ in range(B)]


def _check_caches(kc, vc, inp, head_bits, lens):
    for cache, x in ((kc, inp.k), (vc, inp.v)):
        planes, scale, zero = U.read_cache(cache, inp.Tcap if hasattr(inp, "Tcap") else inp.S)
        o_planes, o_scale, o_zero, deq = U.oracle_quantize(x, head_bits)
        for b, L in enumerate(lens):
            for h in range(len(head_bits)):
                assert np.array_equal(planes[h][b, :L], o_planes[h][b, :L]), (b, h)
            assert np.array_equal(scale[b, :, :L].view(np.uint16), o_scale[b, :, :L].view(np.uint16)), b
            assert np.array_equal(zero[b, :, :L].view(np.uint16), o_zero[b, :, :L].view(np.uint16)), b


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_quantize_and_decode(kvq, seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 5))
    Hkv = int(rng.choice([1, 2, 3, 4]))
    rep = int(rng.choice([1, 2, 3, 4, 5, 8]))
    D = int(rng.choice([64, 128]))
    Tcap = 64 * int(rng.integers(1, 9))
    lens = _lens(rng, B, Tcap, 64)
    bits = str(rng.choice(["8", "4", "mixed"]))
    out_dtype = int(rng.integers(0, 2))
    inp = W.make_decode(f"sweep_decode_{seed}", 2000 + seed, B, Hkv * rep, Hkv, D, Tcap, lens=lens, bits=bits,
                        outliers_per_head=int(rng.integers(0, 3)), outlier_head_mult=8.0)
    kc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    vc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
    kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
    out = kvq.decode_attention(U.to_dev_bf16(inp.q), kc, vc, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                               inp.softmax_scale, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_caches(kc, vc, inp, inp.head_bits, [Tcap] * B)
    deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
    ref = O.decode_attention(inp.q, deq_k, deq_v, np.asarray(lens, np.int32), inp.softmax_scale)
    U.assert_close(out.float().cpu().numpy(), ref, f"sweep decode {seed} B{B} Hkv{Hkv} rep{rep} D{D} "
                   f"T{Tcap} lens{lens} bits {list(inp.head_bits)}", out_bf16=out_dtype == 1)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_prefill(kvq, seed):
    rng = np.random.default_rng(3000 + seed)
    B = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2, 3]))
    rep = int(rng.choice([1, 2, 3, 4, 5]))
    D = int(rng.choice([64, 128]))
    n_t = int(rng.integers(1, 5))
    S = 128 * n_t
    causal = bool(rng.random() < 0.6)
    head_bits = np.asarray([8 if rng.random() < 0.5 else 4 for _ in range(Hkv)], np.int8)
    varlen = bool(rng.random() < 0.5)
    lens = _lens(rng, B, S, 128) if varlen else [S] * B
    mask_kind = str(rng.choice(["none", "random"]))
    out_dtype = int(rng.integers(0, 2))
    inp = W.make_prefill(f"sweep_prefill_{seed}", 4000 + seed, B, Hkv * rep, Hkv, D, S, mask_seed=None)
    if mask_kind == "random":
        inp.tile_mask = (rng.random((n_t, n_t)) < 0.6).astype(np.uint8)
    kc = kvq.empty_cache(head_bits, B, S, D)
    vc = kvq.empty_cache(head_bits, B, S, D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.from_numpy(inp.tile_mask).cuda() if inp.tile_mask is not None else None
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda") if varlen else None
    out = kvq.prefill_attention(U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v), kc, vc,
                                inp.softmax_scale, mask, out_dtype=out_dtype, status=st, causal=causal, seq_lens=sl)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.float().cpu().numpy()
    what = (f"sweep prefill {seed} B{B} Hkv{Hkv} rep{rep} D{D} S{S} causal={causal} lens{lens} "
            f"mask={mask_kind} bits {list(head_bits)}")
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0), what
            continue
        o_planes, o_scale, o_zero, kd = U.oracle_quantize(inp.k[b:b + 1, :, :L], head_bits)
        vd = U.oracle_quantize(inp.v[b:b + 1, :, :L], head_bits)[3]
        planes, scale, zero = U.read_cache(kc, L)
        for h in range(Hkv):
            assert np.array_equal(planes[h][b], o_planes[h][0]), (what, b, h)
        assert np.array_equal(scale[b].view(np.uint16), o_scale[0].view(np.uint16)), (what, b)
        assert np.array_equal(zero[b].view(np.uint16), o_zero[0].view(np.uint16)), (what, b)
        for h in range(inp.Hq):
            ref = O.prefill_rows(inp.q[b:b + 1, :, :L], kd, vd, 0, h, np.arange(L), inp.tile_mask,
                                 inp.softmax_scale, causal=causal)
            U.assert_close(got[b, h, :L], ref, f"{what} b={b} h={h}", out_bf16=out_dtype == 1)
        assert np.all(got[b, :, L:] == 0), what


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_paged_decode_and_step(kvq, seed):
    """Paged decode through a random block table (byte-equal to the contiguous
    decode of the same data), then one decode step on contiguous caches whose
    new-token rows held other values."""
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 6))
    Hkv = int(rng.choice([1, 2, 4]))
    rep = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 128]))
    max_pages = int(rng.integers(1, 6))
    Tcap = 64 * max_pages
    lens = [max(L, 1) for L in _lens(rng, B, Tcap, 64)]   # a step appends at len - 1
    bits = str(rng.choice(["8", "4", "mixed"]))
    inp = W.make_decode(f"sweep_paged_{seed}", 6000 + seed, B, Hkv * rep, Hkv, D, Tcap, lens=lens, bits=bits,
                        outliers_per_head=int(rng.integers(0, 3)), outlier_head_mult=8.0)
    what = f"sweep paged/step {seed} B{B} Hkv{Hkv} rep{rep} D{D} T{Tcap} lens{lens} bits {list(inp.head_bits)}"
    n_pages = B * max_pages + int(rng.integers(0, 8))
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    bt = torch.from_numpy(table).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp = kvq.empty_page_pool(inp.head_bits, n_pages, D)
    vp = kvq.empty_page_pool(inp.head_bits, n_pages, D)
    kvq.quantize_paged(U.to_dev_bf16(inp.k), kp, bt, 0, st)
    kvq.quantize_paged(U.to_dev_bf16(inp.v), vp, bt, 0, st)
    kc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    vc = kvq.empty_cache(inp.head_bits, B, Tcap, D)
    kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
    kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = U.to_dev_bf16(inp.q)
    paged = kvq.decode_attention_paged(q, kp, vp, bt, sl, inp.softmax_scale, status=st)
    contiguous = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, what
    assert torch.equal(paged, contiguous), what
    deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
    ref = O.decode_attention(inp.q, deq_k, deq_v, np.asarray(lens, np.int32), inp.softmax_scale)
    U.assert_close(paged.cpu().numpy(), ref, what)
    # the step: caches quantised from inputs whose row len - 1 held other values
    stale_k, stale_v = inp.k.copy(), inp.v.copy()
    for b, L in enumerate(lens):
        for x in (stale_k, stale_v):
            f = (rng.standard_normal((Hkv, D)) * 3.0).astype(np.float32)
            x[b, :, L - 1] = (f.view(np.uint32) >> 16).astype(np.uint16)
    kvq.quantize(U.to_dev_bf16(stale_k), kc, 0, st)
    kvq.quantize(U.to_dev_bf16(stale_v), vc, 0, st)
    k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(B)])
    v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(B)])
    out = kvq.decode_step(q, U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc, sl, inp.softmax_scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, what
    assert torch.equal(out, contiguous), what   # the same cache contents as the contiguous decode above
    _check_caches(kc, vc, inp, inp.head_bits, lens)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_head_error_stats_and_allocation(kvq, seed):
    """Per-head error statistics (fixed summation order: the same bytes twice)
    against the oracle, and the host allocator's choice from those statistics
    against the oracle's allocation rule applied to the same statistics (near
    ties between heads could order differently from the oracle's own
    statistics within the 1e-5 tolerance)."""
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 9))
    D = int(rng.choice([64, 128]))
    T = 64 * int(rng.integers(1, 9))
    bits = int(rng.choice([4, 8]))
    outliers = sorted(int(h) for h in rng.choice(H, int(rng.integers(0, H + 1)), replace=False))
    ragged = bool(rng.random() < 0.5)
    lens = _lens(rng, B, T, 64) if ragged else "full"
    weighted = bool(rng.random() < 0.5)
    inp = W.make_sensitivity(f"sweep_stats_{seed}", 8000 + seed, B, H, D, T, outliers, lens=lens, weights=weighted)
    what = f"sweep stats {seed} B{B} H{H} D{D} T{T} bits{bits} outliers{outliers} lens{lens} weighted={weighted}"
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    sl = torch.from_numpy(inp.seq_lens).cuda() if ragged else None
    w = torch.from_numpy(inp.weights).cuda() if weighted else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = []
    for x in (inp.k, inp.v):
        a = kvq.head_error_stats(dev(x), bits, seq_lens=sl, weights=w, status=st).cpu().numpy()
        b = kvq.head_error_stats(dev(x), bits, seq_lens=sl, weights=w, status=st).cpu().numpy()
        want = O.head_error_stats(x, bits, inp.seq_lens if ragged else None, inp.weights)
        assert np.array_equal(a, b), what
        assert np.allclose(a, want, rtol=1e-5, atol=1e-30), (what, a, want)
        got.append((a, want))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, what
    n_high = int(rng.integers(0, H + 1))
    hb, _ = kvq.allocate_head_bits(torch.from_numpy(got[0][0]), torch.from_numpy(got[1][0]), n_high=n_high,
                                   low_bits=4)
    o_bits = O.allocate_head_bits(O.head_sensitivity(got[0][0], got[1][0]), n_high, 4)
    assert np.array_equal(np.asarray(hb), np.asarray(o_bits)), (what, hb, o_bits)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_tile_mask(kvq, seed):
    """The device mask builder against the oracle, bit for bit, over random grid
    sizes (a single tile up to 700 tiles a side), skip ratios (none to all of the
    candidates) and 64-bit seeds."""
    rng = np.random.default_rng(9000 + seed)
    nT = int(rng.choice([1, 2, 3, int(rng.integers(4, 129)), int(rng.integers(129, 701))]))
    den = int(rng.integers(1, 21))
    num = int(rng.integers(0, den + 1))
    mseed = int(rng.integers(0, 1 << 62)) * 4 + int(rng.integers(0, 4))
    got = kvq.build_tile_mask(nT, num, den, mseed).cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(got, O.build_tile_mask(nT, num, den, mseed)), (nT, num, den, mseed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_strided_quantize_into_a_window(kvq, seed):
    """Quantise-on-write of a strided view (sequence, head or token strides
    padded, or the head and token axes swapped in memory) into positions
    [t0, t0 + nt) of a cache: those rows bit-exact against the oracle, every
    other row of the cache untouched."""
    rng = np.random.default_rng(11000 + seed)
    B = int(rng.integers(1, 4))
    Hkv = int(rng.integers(1, 5))
    D = int(rng.choice([64, 128]))
    Tcap = 64 * int(rng.integers(1, 5))
    t0 = int(rng.integers(0, Tcap))
    nt = int(rng.integers(1, Tcap - t0 + 1))
    head_bits = np.asarray([8 if rng.random() < 0.5 else 4 for _ in range(Hkv)], np.int8)
    full = W.make_decode(f"sweep_quant_{seed}", 12000 + seed, B, Hkv, Hkv, D, nt, lens="full",
                         outliers_per_head=int(rng.integers(0, 3)), outlier_head_mult=8.0).k   # [B][Hkv][nt][D]
    layout = str(rng.choice(["contiguous", "padded", "heads_inner"]))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    if layout == "contiguous":
        xv = dev(full)
    elif layout == "padded":   # every stride padded by a multiple of 8 elements
        pad = dev(np.zeros((B, Hkv + 1, nt + 3, D + 8 * int(rng.integers(1, 3))), np.uint16))
        pad[:, :Hkv, :nt, :D] = dev(full)
        xv = pad[:, :Hkv, :nt, :D]
    else:                      # memory order [B][T][Hkv][D]
        xv = dev(np.ascontiguousarray(full.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    kc = kvq.empty_cache(head_bits, B, Tcap, D)
    kc.codes.fill_(0x5A)
    kc.sz.fill_(0x1234567)
    codes0, sz0 = kc.codes.clone(), kc.sz.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.quantize(xv, kc, t0, st)
    torch.cuda.synchronize()
    what = f"sweep quantize {seed} B{B} Hkv{Hkv} D{D} Tcap{Tcap} t0={t0} nt={nt} {layout} bits {list(head_bits)}"
    assert int(st.item()) == 0, what
    planes, scale, zero = U.read_cache(kc, Tcap)
    p0, s0, z0 = U.read_cache(kvq.QuantCache(codes0, sz0, head_bits, B, Hkv, Tcap, D), Tcap)
    o_planes, o_scale, o_zero, _ = U.oracle_quantize(full, head_bits)
    for h in range(Hkv):
        assert np.array_equal(planes[h][:, t0:t0 + nt], o_planes[h]), (what, h)
        assert np.array_equal(planes[h][:, :t0], p0[h][:, :t0]), (what, h)
        assert np.array_equal(planes[h][:, t0 + nt:], p0[h][:, t0 + nt:]), (what, h)
    assert np.array_equal(scale[:, :, t0:t0 + nt].view(np.uint16), o_scale.view(np.uint16)), what
    assert np.array_equal(zero[:, :, t0:t0 + nt].view(np.uint16), o_zero.view(np.uint16)), what
    for a, b in ((scale, s0), (zero, z0)):
        assert np.array_equal(a[:, :, :t0].view(np.uint16), b[:, :, :t0].view(np.uint16)), what
        assert np.array_equal(a[:, :, t0 + nt:].view(np.uint16), b[:, :, t0 + nt:].view(np.uint16)), what
