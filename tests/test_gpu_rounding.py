"""GPU parity of the selectable bf16 output rounding (RTNE, RTNA, RTZ).

The MoonMath HIP kernel page measures its bf16 forward kernel in three output
rounding modes.  Here the mode only changes the last fp32 -> bf16 conversion,
so the tests check it three ways:

- exactly, where the fp32 result is known: with scale = 0 and four keys every
  probability is 1 and O is the mean of four integer-valued V rows, a
  multiple of 1/4 that the kernel reaches without rounding, so the bf16
  output must equal the oracle's rounding of the exact mean bit for bit
  (many of these quarters are exact ties between two bf16 neighbours);
- through the merge entry point, whose output is a plain rounding of the fp32
  partial when there is one split;
- on random inputs, against the oracle within the usual tolerance, and
  against each other: the three modes round the same fp32 value, so RTNE and
  RTNA are RTZ or one unit further from zero, and differ only on ties.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

MODES = ("rtne", "rtna", "rtz")


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()
    return attn


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check_modes_consistent(n, a, z, what):
    """n, a, z: uint16 bf16 patterns of the same fp32 values in RTNE, RTNA, RTZ."""
    sign = lambda x: x & 0x8000
    mag = lambda x: (x & 0x7FFF).astype(np.int32)
    assert np.array_equal(sign(n), sign(z)) and np.array_equal(sign(a), sign(z)), f"{what}: sign differs"
    for name, x in (("rtne", n), ("rtna", a)):
        step = mag(x) - mag(z)
        assert ((step == 0) | (step == 1)).all(), f"{what}: {name} is not RTZ or one unit away from it"
    differ = n != a
    # where the nearest modes disagree the value was a tie: RTNE kept the even
    # neighbour, RTNA went one unit away from zero
    assert ((mag(n)[differ] & 1) == 0).all(), f"{what}: RTNE picked an odd neighbour on a tie"
    assert (mag(a)[differ] == mag(n)[differ] + 1).all(), f"{what}: RTNA did not round a tie away from zero"
    return differ.mean(), (n != z).mean()


@pytest.mark.parametrize("layout,B,Hq,Hkv,Sq", [("bshd", 2, 4, 2, 130), ("bhsd", 1, 2, 2, 200)])
def test_exact_quarters_round_bitwise_like_the_oracle(A, layout, B, Hq, Hkv, Sq):
    Sk = 4
    g = torch.Generator().manual_seed(81)
    w = inputs.PrefillWorkload("quarters", B, Hq, Hkv, Sq, Sk, layout=layout, seed=81)
    q, k, _ = inputs.make_prefill(w)
    # integer V in [-256, 256] (exact in bf16); means of four are multiples of 1/4
    v = torch.randint(-256, 257, tuple(k.shape), generator=g).to(torch.bfloat16)
    ref_o, ref_l = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, layout=layout, scale=0.0)
    assert np.array_equal(ref_o * 4, np.round(ref_o * 4)), "oracle mean is not a multiple of 1/4"
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    want = {m: oracle.round_bf16_array(ref_o, m) for m in MODES}
    ties = (want["rtne"] != want["rtna"]).mean()
    assert ties > 0.05, f"the inputs give too few ties ({ties:.3f}) to test the modes"
    for m in MODES:
        out, lse = A.fwd(dq, dk, dv, scale=0.0, layout=layout, rounding=m)
        torch.cuda.synchronize()
        got = _bits(out)
        bad = np.flatnonzero(got.reshape(-1) != want[m].reshape(-1))
        assert bad.size == 0, (f"{m}: {bad.size} elements differ, first at {bad[0]}: got {got.reshape(-1)[bad[0]]:#06x}"
                               f" want {want[m].reshape(-1)[bad[0]]:#06x} (exact {ref_o.reshape(-1)[bad[0]]})")
        check_lse(lse, ref_l, f"quarters {m}")
    assert A.device_status()[0] == 0


@pytest.mark.parametrize("mode", MODES)
def test_merge_rounds_each_partial_like_the_oracle(A, mode):
    rows, d = 96, 128
    g = torch.Generator().manual_seed(82)
    x = torch.randn(rows, d, generator=g) * torch.exp(torch.randn(rows, d, generator=g) * 6)
    # exact ties of the bf16 grid, values past the largest bf16, zeros of both signs
    x[0, :8] = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 64.25, -64.75, 3.0e38, 3.4e38,
                             -3.4e38])
    x[1, :2] = torch.tensor([0.0, -0.0])
    x = x.to(torch.float32)
    # split 0 holds the value with lse 0; split 1 has lse -inf and weight 0
    o_parts = torch.stack([x, torch.randn(rows, d, generator=g)], dim=1).contiguous()
    lse_parts = torch.tensor([0.0, float("-inf")]).repeat(rows, 1).contiguous()
    out, lse = A.lse_merge(o_parts.cuda(), lse_parts.cuda(), rounding=mode)
    torch.cuda.synchronize()
    # the merge sums w * o_part from +0, so a -0 partial comes out as +0 (IEEE -0 + 0 = +0)
    want = oracle.round_bf16_array(x.numpy().astype(np.float64) + 0.0, mode)
    np.testing.assert_array_equal(_bits(out), want)
    assert torch.equal(lse.cpu(), torch.zeros(rows))


def test_modes_on_random_inputs_match_oracle_and_each_other(A):
    w = inputs.PrefillWorkload("modes", 2, 8, 2, 300, 300, causal=True, seed=83)
    q, k, v = inputs.make_prefill(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    ref_o, ref_l = oracle.attention(q, k, v, B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, causal=True,
                                    scale=w.scale)
    res = {}
    for m in MODES:
        out, lse = A.fwd(dq, dk, dv, causal=True, scale=w.scale, rounding=m)
        torch.cuda.synchronize()
        check_out(out, ref_o, f"random {m}")
        check_lse(lse, ref_l, f"random {m}")
        res[m] = (_bits(out), lse.cpu())
    assert torch.equal(res["rtne"][1], res["rtna"][1]) and torch.equal(res["rtne"][1], res["rtz"][1])
    assert np.array_equal(res["rtne"][0], _bits(A.fwd(dq, dk, dv, causal=True, scale=w.scale)[0]))
    tie_frac, rz_frac = _check_modes_consistent(res["rtne"][0], res["rtna"][0], res["rtz"][0], "random")
    assert 0.3 < rz_frac < 0.7, f"RTZ differs from RTNE on {rz_frac:.3f} of the elements"
    assert tie_frac < 0.01
    assert A.device_status()[0] == 0


def test_modes_through_the_tail_split_merge(A):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hq, Hkv, Sq, Sk = sms + 8, 1, 1, 256, 2048
    need = A.fwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, causal=False)
    assert need > 0
    w = inputs.PrefillWorkload("modes-split", B, Hq, Hkv, Sq, Sk, seed=84)
    q, k, v = inputs.make_prefill(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    res = {}
    try:
        A.set_workspace(ws)
        for m in MODES:
            out, _ = A.fwd(dq, dk, dv, scale=w.scale, rounding=m)
            torch.cuda.synchronize()
            res[m] = _bits(out[B - 16:])   # the split units are among the last 16 batches
    finally:
        A.set_workspace(None)
    rows = np.array([(b, 0, i) for b in range(B - 16, B) for i in range(0, Sq, 5)], dtype=np.int64)
    ref_o, _ = oracle.attention_rows(q, k, v, rows, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, scale=w.scale)
    for m in MODES:
        got = torch.from_numpy(res[m].view(np.int16)).view(torch.bfloat16)
        sel = got[torch.from_numpy(rows[:, 0] - (B - 16)), torch.from_numpy(rows[:, 2]), 0]
        check_out(sel, ref_o, f"split {m}")
    _, rz_frac = _check_modes_consistent(res["rtne"], res["rtna"], res["rtz"], "split")
    assert 0.3 < rz_frac < 0.7
    assert A.device_status()[0] == 0
