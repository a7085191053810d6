"""Bounded waits and per-call policies on the GPU.

Every wait inside the decode and prefill kernels gives up after the policy's
limit and reports KVQ_ERR_TIMEOUT in the status word.  These tests make a
wait run out on purpose, without any fault: the policy's test-only issue
limit stops the decode's copy issuer after a few tiles (or withholds the
prefill's query load), so the waits for the rest never complete.  The
kernels then return with nothing in flight, and the next call on the same
context, after re-zeroing the decode workspace, must match the oracle.

Decode policies only change how far ahead the cache is fetched, so every
policy must give the same output bytes as the defaults.
"""
import numpy as np
import pytest

from oracle import kvq_oracle as O
import kvq_workloads as W
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TIMEOUT = 5


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_group_quantized_gb300 import kvq as K
    K.lib()
    return K


def _decode_setup(kvq, inp):
    kc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    vc = kvq.empty_cache(inp.head_bits, inp.B, inp.Tcap, inp.D)
    kvq.quantize(U.to_dev_bf16(inp.k), kc)
    kvq.quantize(U.to_dev_bf16(inp.v), vc)
    _, _, _, kd = U.oracle_quantize(inp.k, inp.head_bits)
    _, _, _, vd = U.oracle_quantize(inp.v, inp.head_bits)
    ref = O.decode_attention(inp.q, kd, vd, inp.seq_lens, inp.softmax_scale)
    return kc, vc, ref


@pytest.mark.parametrize("issue_limit", [0, 1, 3])
def test_decode_wait_runs_out_and_the_context_stays_usable(kvq, issue_limit):
    # 4 x 4 segments of up to 128 tiles: every split CTA owns several tiles, so
    # an issue limit of 1 or 3 leaves each of them waiting for a tile
    inp = W.make_decode("timeout", 71, 4, 16, 4, 128, 8192, lens=[8192, 8192, 7000, 8192], bits="mixed")
    kc, vc, ref = _decode_setup(kvq, inp)
    q = U.to_dev_bf16(inp.q)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    ws = kvq.decode_workspace(inp.B, inp.Hq, inp.Hkv, inp.D)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pol = kvq.policy(wait_limit_us=2000, test_issue_limit=issue_limit)
    kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, workspace=ws, status=status, policy=pol)
    torch.cuda.synchronize()
    assert int(status.item()) == TIMEOUT
    # the same context, a zeroed workspace, the default policy: correct again
    ws.zero_()
    status.zero_()
    out = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    U.assert_close(out.cpu().numpy(), ref, "decode after a timed-out call")


def test_prefill_wait_runs_out_and_the_context_stays_usable(kvq):
    inp = W.make_prefill("timeout_prefill", 72, 1, 4, 2, 128, 384, mask_seed=5)
    hb = np.full(inp.Hkv, 8, np.int8)
    kc = kvq.empty_cache(hb, inp.B, inp.S, inp.D)
    vc = kvq.empty_cache(hb, inp.B, inp.S, inp.D)
    q, k, v = U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v)
    mask = torch.from_numpy(inp.tile_mask).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pol = kvq.policy(wait_limit_us=2000, test_issue_limit=0)
    kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, mask, status=status, policy=pol)
    torch.cuda.synchronize()
    assert int(status.item()) == TIMEOUT
    status.zero_()
    out = kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, mask, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    c, s, z = O.quantize_groups(inp.k, 8)
    kd = O.dequantize(c, s, z)
    c, s, z = O.quantize_groups(inp.v, 8)
    vd = O.dequantize(c, s, z)
    got = out.cpu().numpy()
    for h in range(inp.Hq):
        ref = O.prefill_rows(inp.q, kd, vd, 0, h, np.arange(inp.S), inp.tile_mask, inp.softmax_scale)
        U.assert_close(got[0, h], ref, f"prefill after a timed-out call h={h}")


def test_prefill_policy_without_fault_injection_matches_plain_call(kvq):
    inp = W.make_prefill("policy_prefill", 73, 1, 8, 2, 128, 512, mask_seed=6)
    hb = np.full(inp.Hkv, 8, np.int8)
    q, k, v = U.to_dev_bf16(inp.q), U.to_dev_bf16(inp.k), U.to_dev_bf16(inp.v)
    mask = torch.from_numpy(inp.tile_mask).cuda()
    outs = []
    for pol in (None, kvq.policy(wait_limit_us=500_000)):
        kc = kvq.empty_cache(hb, inp.B, inp.S, inp.D)
        vc = kvq.empty_cache(hb, inp.B, inp.S, inp.D)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(kvq.prefill_attention(q, k, v, kc, vc, inp.softmax_scale, mask, status=status, policy=pol))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    assert torch.equal(outs[0], outs[1])


POLICIES = [dict(decode_ring_tiles=2), dict(decode_l2_warm_tiles=0), dict(decode_l2_warm_tiles=16),
            dict(decode_ring_tiles=2, decode_l2_warm_tiles=10)]


@pytest.fixture(scope="module")
def policy_case(kvq):
    # 8 x 8 segments of up to 128 tiles: every split CTA owns a dozen or more
    # tiles, so each ring slot is refilled several times
    inp = W.make_decode("policy", 74, 8, 32, 8, 128, 8192, lens=[8192, 1, 5000, 0, 8192, 7777, 8192, 6000],
                        bits="mixed", outliers_per_head=2, outlier_head_mult=8.0)
    kc, vc, ref = _decode_setup(kvq, inp)
    q = U.to_dev_bf16(inp.q)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    U.assert_close(base.cpu().numpy(), ref, "decode, default policy")
    return inp, kc, vc, q, sl, base


@pytest.mark.parametrize("fields", POLICIES, ids=[",".join(f"{k}={v}" for k, v in p.items()) for p in POLICIES])
def test_decode_policies_give_the_default_bytes(kvq, policy_case, fields):
    """A policy changes only when the cache bytes arrive, never the arithmetic."""
    inp, kc, vc, q, sl, base = policy_case
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = kvq.decode_attention(q, kc, vc, sl, inp.softmax_scale, status=status, policy=kvq.policy(**fields))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(base, got)
