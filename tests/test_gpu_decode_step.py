"""GPU parity of kvq_decode_step / kvq_decode_step_host (append the new token's
K/V, then attend) against the oracle.

The cache is first filled from a copy of the inputs whose new-token rows
(position len_b - 1) hold different values; the step must overwrite exactly
those rows.  Afterwards every live cache row must equal the oracle's
quantisation of the true inputs bit for bit, and the output must satisfy
|o - ref| <= 2e-3 + 2e-3 |ref| against the fp64 oracle over the dequantised
cache.
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


def _kvq():
    from attention_group_quantized_gb300 import kvq
    return kvq


def _stale_new_rows(x: np.ndarray, lens, seed: int) -> np.ndarray:
    """Copy of x with the row at len_b - 1 of every (b, head) replaced by other values."""
    y = x.copy()
    rng = np.random.default_rng(seed)
    for b, L in enumerate(lens):
        if 1 <= L <= x.shape[2]:
            f = (rng.standard_normal((x.shape[1], x.shape[3])) * 3.0).astype(np.float32)
            y[:, :, L - 1][b] = (f.view(np.uint32) >> 16).astype(np.uint16)
    return y


def _prepared(inp: W.DecodeInputs, seed: int):
    """Caches filled from inputs whose new-token rows are stale; the new rows as device tensors."""
    kvq = _kvq()
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    for c in (kc, vc):
        c.codes.fill_(0xA5)
        c.sz.fill_(-1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = [int(x) for x in inp.seq_lens]
    kvq.quantize(U.to_dev_bf16(_stale_new_rows(inp.k, lens, seed)), kc, 0, status)
    kvq.quantize(U.to_dev_bf16(_stale_new_rows(inp.v, lens, seed + 1)), vc, 0, status)
    pos = [min(max(L - 1, 0), inp.Tcap - 1) for L in lens]
    k_new = np.stack([inp.k[b, :, pos[b]] for b in range(inp.B)])   # [B][Hkv][D]
    v_new = np.stack([inp.v[b, :, pos[b]] for b in range(inp.B)])
    return kc, vc, status, k_new, v_new


def _check(inp: W.DecodeInputs, kc, vc, out, out_dtype):
    lens = inp.seq_lens
    deq = []
    for cache, x in ((kc, inp.k), (vc, inp.v)):
        planes, scale, zero = U.read_cache(cache, inp.Tcap)
        o_planes, o_scale, o_zero, d = U.oracle_quantize(x, inp.head_bits)
        for b, L in enumerate(lens):
            for h in range(inp.Hkv):
                assert np.array_equal(planes[h][b, :L], o_planes[h][b, :L]), (b, h)
            assert np.array_equal(scale[b, :, :L].view(np.uint16), o_scale[b, :, :L].view(np.uint16)), b
            assert np.array_equal(zero[b, :, :L].view(np.uint16), o_zero[b, :, :L].view(np.uint16)), b
        deq.append(d)
    ref = O.decode_attention(inp.q, deq[0], deq[1], lens, inp.softmax_scale)
    return U.assert_close(out, ref, inp.name, out_bf16=out_dtype == 1)


STEP_CASES = [
    # name, seed, B, Hq, Hkv, D, Tcap, lens, bits, out_dtype
    ("step_int8_ragged", 31, 3, 8, 2, 128, 640, [640, 65, 1], "8", 0),
    ("step_mixed_bf16", 32, 2, 16, 4, 128, 512, [300, 512], "mixed", 1),
    ("step_d64_int4", 33, 4, 8, 4, 64, 256, [2, 64, 129, 256], "4", 0),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_decode_step_parity(case):
    name, seed, B, Hq, Hkv, D, Tcap, lens, bits, out_dtype = case
    kvq = _kvq()
    inp = W.make_decode(name, seed, B, Hq, Hkv, D, Tcap, lens=lens, bits=bits,
                        outliers_per_head=2, outlier_head_mult=8.0)
    kc, vc, status, k_new, v_new = _prepared(inp, seed)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    out = kvq.decode_step(U.to_dev_bf16(inp.q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc, sl,
                          inp.softmax_scale, out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(inp, kc, vc, out.float().cpu().numpy(), out_dtype)


@pytest.mark.parametrize("out_dtype,pinned", [(0, True), (1, True), (0, False), (1, False)],
                         ids=["f32_pinned", "bf16_pinned", "f32_pageable", "bf16_pageable"])
def test_decode_step_host_parity(out_dtype, pinned):
    """Pinned buffers take the in-place path (no copy calls), pageable ones the staged copies."""
    kvq = _kvq()
    inp = W.make_decode("step_host", 34, 3, 8, 2, 128, 384, lens=[384, 200, 7], bits="mixed",
                        outliers_per_head=2, outlier_head_mult=8.0)
    kc, vc, status, k_new, v_new = _prepared(inp, 34)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    pin = lambda a: host(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16))
    h_q, h_k, h_v = pin(inp.q), pin(k_new), pin(v_new)
    h_out = host(torch.full((inp.B, inp.Hq, inp.D), 7.0, dtype=torch.float32 if out_dtype == 0 else torch.bfloat16))
    sl = torch.from_numpy(inp.seq_lens).cuda()
    kvq.decode_step_host(h_q, h_k, h_v, kc, vc, sl, h_out, inp.softmax_scale, out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(inp, kc, vc, h_out.float().numpy(), out_dtype)


def test_decode_step_consecutive_steps():
    """Five steps in a row, each appending one token per sequence: every step
    must see the tokens the earlier steps appended."""
    kvq = _kvq()
    T_final = [70, 129, 5]
    inp = W.make_decode("step_seq", 35, 3, 8, 2, 128, 192, lens=T_final, bits="8",
                        outliers_per_head=2, outlier_head_mult=8.0)
    B, Hq, Hkv, D = inp.B, inp.Hq, inp.Hkv, inp.D
    kc = kvq.empty_cache(inp.head_bits, B, inp.Tcap, D)
    vc = kvq.empty_cache(inp.head_bits, B, inp.Tcap, D)
    for c in (kc, vc):
        c.codes.fill_(0xA5)
        c.sz.fill_(-1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_steps = 5
    start = [L - n_steps for L in T_final]
    pre_k, pre_v = inp.k.copy(), inp.v.copy()
    for b, L0 in enumerate(start):
        pre_k[b, :, L0:] = 0
        pre_v[b, :, L0:] = 0
    kvq.quantize(U.to_dev_bf16(pre_k), kc, 0, status)
    kvq.quantize(U.to_dev_bf16(pre_v), vc, 0, status)
    ws = kvq.decode_workspace(B, Hq, Hkv, D, "cuda")
    rng = np.random.default_rng(36)
    deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
    for s in range(n_steps):
        lens = np.array([L0 + s + 1 for L0 in start], dtype=np.int32)
        k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(B)])
        v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(B)])
        q = W._draw_bf16(rng, (B, Hq, D))
        out = kvq.decode_step(U.to_dev_bf16(q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc,
                              torch.from_numpy(lens).cuda(), inp.softmax_scale, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = O.decode_attention(q, deq_k, deq_v, lens, inp.softmax_scale)
        U.assert_close(out.cpu().numpy(), ref, f"step {s}")
    _check(W.DecodeInputs(inp.name, q, inp.k, inp.v, np.array(T_final, np.int32), inp.head_bits,
                          inp.softmax_scale, Hq, Hkv, D, inp.Tcap), kc, vc, out.cpu().numpy(), 0)


def test_decode_step_reports_invalid_length_and_appends_the_rest():
    kvq = _kvq()
    inp = W.make_decode("step_bad_len", 37, 3, 4, 1, 128, 128, lens=[128, 40, 0], bits="8")
    kc, vc, status, k_new, v_new = _prepared(inp, 37)
    codes_before = kc.codes.clone()
    sl = torch.tensor([128, 40, 0], dtype=torch.int32, device="cuda")
    out = kvq.decode_step(U.to_dev_bf16(inp.q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc, sl,
                          inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1          # sequence 2 has no position for its new token
    got = out.cpu().numpy()
    assert np.all(got[2] == 0.0)            # length 0: zero output row
    # sequences 0 and 1 were appended and attended normally
    sub = W.DecodeInputs(inp.name, inp.q[:2], inp.k[:2], inp.v[:2], inp.seq_lens[:2], inp.head_bits,
                         inp.softmax_scale, inp.Hq, inp.Hkv, inp.D, inp.Tcap)
    planes, _, _ = U.read_cache(kc, inp.Tcap)
    o_planes = U.oracle_quantize(inp.k, inp.head_bits)[0]
    for b, L in ((0, 128), (1, 40)):
        assert np.array_equal(planes[0][b, :L], o_planes[0][b, :L]), b
    deq_k = U.oracle_quantize(sub.k, sub.head_bits)[3]
    deq_v = U.oracle_quantize(sub.v, sub.head_bits)[3]
    ref = O.decode_attention(sub.q, deq_k, deq_v, sub.seq_lens, sub.softmax_scale)
    U.assert_close(got[:2], ref, "valid sequences")
    # sequence 2 wrote nothing anywhere in its plane
    R = inp.D
    b2 = kc.codes[2 * inp.Tcap * R:3 * inp.Tcap * R]
    assert torch.equal(b2, codes_before[2 * inp.Tcap * R:3 * inp.Tcap * R])


def test_decode_step_rejects_missing_workspace_without_appending():
    kvq = _kvq()
    inp = W.make_decode("step_ws", 38, 1, 4, 1, 128, 128, lens=[100], bits="8")
    kc, vc, status, k_new, v_new = _prepared(inp, 38)
    before = kc.codes.clone()
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_step(U.to_dev_bf16(inp.q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc,
                        torch.from_numpy(inp.seq_lens).cuda(), 0.0, workspace=ws)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert torch.equal(kc.codes, before)


def test_decode_step_host_prepared_call_matches_the_function():
    """The bound-once call object gives the same bytes as the plain function."""
    kvq = _kvq()
    inp = W.make_decode("step_prepared", 39, 2, 8, 2, 128, 256, lens=[256, 90], bits="8",
                        outliers_per_head=2, outlier_head_mult=8.0)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    outs = []
    for use_obj in (False, True):
        kc, vc, status, k_new, v_new = _prepared(inp, 39)
        h_q, h_k, h_v = pin(inp.q), pin(k_new), pin(v_new)
        h_out = torch.zeros((inp.B, inp.Hq, inp.D), dtype=torch.float32).pin_memory()
        sl = torch.from_numpy(inp.seq_lens).cuda()
        if use_obj:
            # twice: the second call rewrites the same token and reuses the caches' C views
            obj = kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, status=status)
            obj.run(kc, vc)
            obj.run(kc, vc)
        else:
            kvq.decode_step_host(h_q, h_k, h_v, kc, vc, sl, h_out, inp.softmax_scale, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _check(inp, kc, vc, h_out.numpy(), 0)
        outs.append(h_out.numpy().copy())
    assert np.array_equal(outs[0], outs[1])


def test_decode_step_host_repeated_steps_replay_fresh_contents():
    """A serving loop: the same pinned buffers, lengths tensor and caches every
    step, with new contents each time.  From the third identical call on, the
    library launches a graph captured on the second; every step must still
    see that step's lengths, query and new rows.  Two cache pairs take turns,
    so two graphs are kept side by side.  Each output is checked against the
    oracle and against kvq_decode_step on device copies of the same inputs
    (byte for byte: the same kernels on the same data)."""
    kvq = _kvq()
    n_steps = 6
    T_final = [90, 131, 8]
    pairs = []
    for seed in (41, 42):
        inp = W.make_decode(f"step_replay_{seed}", seed, 3, 8, 2, 128, 192, lens=T_final, bits="mixed",
                            outliers_per_head=2, outlier_head_mult=8.0)
        start = [L - n_steps for L in T_final]
        pre_k, pre_v = inp.k.copy(), inp.v.copy()
        for b, L0 in enumerate(start):
            pre_k[b, :, L0:] = 0
            pre_v[b, :, L0:] = 0
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        caches = []
        for copy in range(2):   # [0]: the host-buffer step, [1]: the device-buffer reference
            kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
            vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
            kvq.quantize(U.to_dev_bf16(pre_k), kc, 0, st)
            kvq.quantize(U.to_dev_bf16(pre_v), vc, 0, st)
            caches.append((kc, vc))
        bf = lambda shape: torch.zeros(shape, dtype=torch.bfloat16).pin_memory()
        h_q, h_k, h_v = bf((inp.B, inp.Hq, inp.D)), bf((inp.B, inp.Hkv, inp.D)), bf((inp.B, inp.Hkv, inp.D))
        h_out = torch.zeros((inp.B, inp.Hq, inp.D), dtype=torch.float32).pin_memory()
        sl = torch.zeros(inp.B, dtype=torch.int32, device="cuda")
        call = kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, status=st)
        deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
        deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
        pairs.append(dict(inp=inp, start=start, caches=caches, h=(h_q, h_k, h_v, h_out), sl=sl, call=call,
                          st=st, deq=(deq_k, deq_v), rng=np.random.default_rng(seed + 100)))
    as_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    for s in range(n_steps):
        for pi, P in enumerate(pairs):
            inp = P["inp"]
            B = inp.B
            lens = np.array([L0 + s + 1 for L0 in P["start"]], dtype=np.int32)
            q = W._draw_bf16(P["rng"], (B, inp.Hq, inp.D))
            k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(B)])
            v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(B)])
            h_q, h_k, h_v, h_out = P["h"]
            h_q.copy_(as_bf16(q))
            h_k.copy_(as_bf16(k_new))
            h_v.copy_(as_bf16(v_new))
            h_out.fill_(7.0)
            P["sl"].copy_(torch.from_numpy(lens))
            P["call"].run(*P["caches"][0])
            ref_out = kvq.decode_step(U.to_dev_bf16(q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new),
                                      *P["caches"][1], torch.from_numpy(lens).cuda(), inp.softmax_scale,
                                      status=P["st"])
            torch.cuda.synchronize()
            assert int(P["st"].item()) == 0, (s, pi)
            got = h_out.numpy().copy()
            assert np.array_equal(got, ref_out.cpu().numpy()), (s, pi)
            ref = O.decode_attention(q, P["deq"][0], P["deq"][1], lens, inp.softmax_scale)
            U.assert_close(got, ref, f"replayed step {s} pair {pi}")
    for P in pairs:
        kc, vc = P["caches"][0]
        assert torch.equal(kc.codes, P["caches"][1][0].codes) and torch.equal(vc.sz, P["caches"][1][1].sz)


def _as_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _host_step_buffers(inp):
    bf = lambda shape: torch.zeros(shape, dtype=torch.bfloat16).pin_memory()
    h_q, h_k, h_v = bf((inp.B, inp.Hq, inp.D)), bf((inp.B, inp.Hkv, inp.D)), bf((inp.B, inp.Hkv, inp.D))
    h_out = torch.zeros((inp.B, inp.Hq, inp.D), dtype=torch.float32).pin_memory()
    return h_q, h_k, h_v, h_out


def test_decode_step_host_replay_follows_bit_widths_changed_in_place():
    """The cache's per-head bit widths are part of what a replayed step was
    built from: after the widths change in place (same host array, same
    buffers, re-quantised contents) the next calls must use the new layout."""
    kvq = _kvq()
    lens = [100, 37]
    inp = W.make_decode("step_rebits", 43, 2, 8, 2, 128, 128, lens=lens, bits="8",
                        outliers_per_head=2, outlier_head_mult=8.0)
    kc = kvq.empty_cache([8, 8], inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache([8, 8], inp.B, inp.Tcap, inp.D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_q, h_k, h_v, h_out = _host_step_buffers(inp)
    sl = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    call = kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, status=st)
    k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(inp.B)])
    v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(inp.B)])
    h_q.copy_(_as_bf16(inp.q)); h_k.copy_(_as_bf16(k_new)); h_v.copy_(_as_bf16(v_new))
    for bits in ([8, 8], [8, 4]):
        kc.head_bits[:] = bits
        vc.head_bits[:] = bits
        hb = np.asarray(bits, np.int8)
        kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
        kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
        deq_k = U.oracle_quantize(inp.k, hb)[3]
        deq_v = U.oracle_quantize(inp.v, hb)[3]
        ref = O.decode_attention(inp.q, deq_k, deq_v, np.asarray(lens, np.int32), inp.softmax_scale)
        for s in range(4):   # direct, captured, then replayed
            h_out.fill_(7.0)
            call.run(kc, vc)
            torch.cuda.synchronize()
            assert int(st.item()) == 0, (bits, s)
            U.assert_close(h_out.numpy().copy(), ref, f"bits {bits} call {s}")


def test_decode_step_host_inside_a_captured_graph():
    """A call on a stream that is itself being captured launches its kernels
    into that capture (the library keeps no graph of its own for it); the
    caller's graph then replays the step with each step's contents."""
    kvq = _kvq()
    n_steps = 3
    T_final = [66, 20]
    inp = W.make_decode("step_in_graph", 44, 2, 8, 2, 128, 128, lens=T_final, bits="mixed",
                        outliers_per_head=2, outlier_head_mult=8.0)
    start = [L - n_steps for L in T_final]
    pre_k, pre_v = inp.k.copy(), inp.v.copy()
    for b, L0 in enumerate(start):
        pre_k[b, :, L0:] = 0
        pre_v[b, :, L0:] = 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = []
    for _ in range(2):   # [0]: replayed through the caller's graph, [1]: kvq_decode_step reference
        kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
        vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
        kvq.quantize(U.to_dev_bf16(pre_k), kc, 0, st)
        kvq.quantize(U.to_dev_bf16(pre_v), vc, 0, st)
        caches.append((kc, vc))
    torch.cuda.synchronize()
    h_q, h_k, h_v, h_out = _host_step_buffers(inp)
    sl = torch.zeros(inp.B, dtype=torch.int32, device="cuda")
    cap = torch.cuda.Stream()
    call = kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, status=st, stream=cap)
    rng = np.random.default_rng(45)
    steps = []
    for s in range(n_steps):
        lens = np.array([L0 + s + 1 for L0 in start], dtype=np.int32)
        q = W._draw_bf16(rng, (inp.B, inp.Hq, inp.D))
        k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(inp.B)])
        v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(inp.B)])
        steps.append((lens, q, k_new, v_new))

    def load(step):
        lens, q, k_new, v_new = step
        h_q.copy_(_as_bf16(q)); h_k.copy_(_as_bf16(k_new)); h_v.copy_(_as_bf16(v_new))
        h_out.fill_(7.0)
        sl.copy_(torch.from_numpy(lens))
        torch.cuda.synchronize()

    # one plain call first (the step-0 token, which the first replay writes again)
    load(steps[0])
    with torch.cuda.stream(cap):
        call.run(*caches[0])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        call.run(*caches[0])
    deq_k = U.oracle_quantize(inp.k, inp.head_bits)[3]
    deq_v = U.oracle_quantize(inp.v, inp.head_bits)[3]
    for s, step in enumerate(steps):
        lens, q, k_new, v_new = step
        load(step)
        graph.replay()
        ref_out = kvq.decode_step(U.to_dev_bf16(q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), *caches[1],
                                  torch.from_numpy(lens).cuda(), inp.softmax_scale, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, s
        got = h_out.numpy().copy()
        assert np.array_equal(got, ref_out.cpu().numpy()), s
        U.assert_close(got, O.decode_attention(q, deq_k, deq_v, lens, inp.softmax_scale), f"graph step {s}")


def test_decode_step_host_more_repeated_steps_than_kept_graphs():
    """More distinct repeated steps than the library keeps graphs for (16 per
    process): the steps beyond that launch directly, and every result stays
    byte-equal to kvq_decode_step on device copies of the same inputs."""
    kvq = _kvq()
    lens = [77, 128]
    inp = W.make_decode("step_many_keys", 46, 2, 8, 2, 128, 128, lens=lens, bits="mixed",
                        outliers_per_head=2, outlier_head_mult=8.0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    kvq.quantize(U.to_dev_bf16(inp.k), kc, 0, st)
    kvq.quantize(U.to_dev_bf16(inp.v), vc, 0, st)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    k_new = np.stack([inp.k[b, :, lens[b] - 1] for b in range(inp.B)])
    v_new = np.stack([inp.v[b, :, lens[b] - 1] for b in range(inp.B)])
    ref = kvq.decode_step(U.to_dev_bf16(inp.q), U.to_dev_bf16(k_new), U.to_dev_bf16(v_new), kc, vc, sl,
                          inp.softmax_scale, status=st).cpu().numpy()
    calls = []
    for i in range(20):   # 20 distinct argument sets (own host buffers each)
        h_q, h_k, h_v, h_out = _host_step_buffers(inp)
        h_q.copy_(_as_bf16(inp.q)); h_k.copy_(_as_bf16(k_new)); h_v.copy_(_as_bf16(v_new))
        calls.append((kvq.DecodeStepHost(h_q, h_k, h_v, sl, h_out, inp.softmax_scale, status=st), h_out))
    for rnd in range(3):   # direct, captured (while there is room), replayed
        for i, (call, h_out) in enumerate(calls):
            h_out.fill_(7.0)
            call.run(kc, vc)
            torch.cuda.synchronize()
            assert int(st.item()) == 0, (rnd, i)
            assert np.array_equal(h_out.numpy(), ref), (rnd, i)
