"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Every comparison is element-wise at |O - O_ref| <= 4e-3 + 8e-3 |O_ref| and
|lse - lse_ref| <= 1e-3.  Small shapes and the full-size workloads are both
compared in full: every output element and every lse.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs
from parity_util import ATOL, RTOL, check_lse, check_out, gather_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()  # raises loudly if the library was not built
    return attn


def _run(A, w, q, k, v, fn="fwd"):
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    out, lse = getattr(A, fn)(dq, dk, dv, causal=w.causal, scale=w.scale, layout=w.layout)
    torch.cuda.synchronize()
    code, site = A.device_status()
    assert code == 0, f"{w.name}: device status {code} at wait site {site}"
    return out, lse


def _oracle_full(w, q, k, v):
    return oracle.attention(q, k, v, B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, d=w.d, layout=w.layout,
                            causal=w.causal, scale=w.scale)


# ---------------------------------------------------------------- tensor-core layouts

def test_umma_layout_selftest(A):
    g = torch.Generator().manual_seed(7)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    da, db = a.cuda(), b.cuda()
    c0 = A.selftest_umma(da, db, 0).cpu().double()
    c1 = A.selftest_umma(da, db, 1).cpu().double()
    ref0 = a.double() @ b.double().T
    ref1 = a.double() @ b.double()
    np.testing.assert_allclose(c0.numpy(), ref0.numpy(), rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(c1.numpy(), ref1.numpy(), rtol=1e-5, atol=1e-4)


# ---------------------------------------------------------------- small shapes, full comparison

SMALL = [
    # name, B, Hq, Hkv, Sq, Sk, layout, causal
    ("tiny_bhsd", 1, 2, 2, 256, 256, "bhsd", False),
    ("gqa_causal_5tiles", 2, 8, 2, 640, 640, "bshd", True),
    ("mqa_causal_ragged", 1, 4, 1, 333, 333, "bshd", True),
    ("cross_ragged", 1, 4, 4, 300, 517, "bshd", False),
    ("odd_group_causal_sq_lt_sk", 1, 3, 1, 200, 700, "bhsd", True),
    ("causal_sq_gt_sk_masked_rows", 1, 2, 2, 700, 200, "bshd", True),
    ("odd_group_bhsd", 2, 6, 2, 129, 129, "bhsd", True),
    ("single_query", 1, 2, 1, 1, 1000, "bshd", False),
    ("single_key", 1, 2, 2, 77, 1, "bshd", False),
    ("bhsd_gqa_causal", 1, 4, 2, 1024, 1024, "bhsd", True),
    ("three_row_blocks_g1", 1, 2, 2, 384, 384, "bshd", False),
    ("short_causal_g1", 1, 1, 1, 130, 130, "bshd", True),
    # five row blocks in pairs: the last pair's second tile lies past the end
    ("odd_row_blocks_g1_causal", 2, 2, 2, 640, 640, "bhsd", True),
    # more units than SMs, so each CTA loops over several: units whose rows see
    # no key (causal, Sq > Sk) between ordinary ones, and an odd group size
    ("looping_units_masked_rows", 4, 32, 8, 2048, 512, "bshd", True),
    ("looping_units_odd_group", 8, 6, 2, 1000, 1000, "bhsd", True),
    # GQA head packing with short query lengths (a tile: 128 / G positions x G heads)
    ("packed_short_q_g8_causal", 8, 32, 4, 16, 4096, "bshd", True),
    ("packed_short_q_g32_bhsd", 2, 32, 1, 5, 700, "bhsd", False),
    ("packed_g8_ragged_causal", 3, 16, 2, 70, 300, "bshd", True),
    ("packed_g4_ragged_bhsd", 2, 8, 2, 45, 130, "bhsd", True),
    ("packed_looping_units", 40, 32, 8, 40, 600, "bshd", True),   # 320 packed units: every CTA loops
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes_full(A, case):
    name, B, Hq, Hkv, Sq, Sk, layout, causal = case
    w = inputs.PrefillWorkload(name, B, Hq, Hkv, Sq, Sk, layout=layout, causal=causal, seed=100 + len(name))
    q, k, v = inputs.make_prefill(w)
    out, lse = _run(A, w, q, k, v)
    ref_o, ref_l = _oracle_full(w, q, k, v)
    check_out(out, ref_o, name)
    check_lse(lse, ref_l, name)


@pytest.mark.parametrize("case", SMALL[:4], ids=[c[0] for c in SMALL[:4]])
def test_simple_kernel_full(A, case):
    name, B, Hq, Hkv, Sq, Sk, layout, causal = case
    w = inputs.PrefillWorkload(name, B, Hq, Hkv, Sq, Sk, layout=layout, causal=causal, seed=100 + len(name))
    q, k, v = inputs.make_prefill(w)
    out, lse = _run(A, w, q, k, v, fn="fwd_simple")
    ref_o, ref_l = _oracle_full(w, q, k, v)
    check_out(out, ref_o, name + "/simple")
    check_lse(lse, ref_l, name + "/simple")


def test_tiny_workload_deterministic(A):
    w = inputs.TINY_BHSD
    q, k, v = inputs.make_prefill(w)
    outs = [_run(A, w, q, k, v) for _ in range(3)]
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    ref_o, ref_l = _oracle_full(w, q, k, v)
    check_out(outs[0][0], ref_o, w.name)
    check_lse(outs[0][1], ref_l, w.name)


# ---------------------------------------------------------------- closed forms and invariants on the GPU

def test_single_key_returns_value_exactly(A):
    w = inputs.PrefillWorkload("sk1", 1, 4, 2, 300, 1, seed=5)
    q, k, v = inputs.make_prefill(w)
    out, lse = _run(A, w, q, k, v)
    want = v.cuda().repeat_interleave(2, dim=2).expand(1, 300, 4, 128)
    assert torch.equal(out, want)


def test_identical_keys_give_mean_value(A):
    B, S, H, d = 1, 512, 2, 128
    g = torch.Generator().manual_seed(9)
    q = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, H, d, generator=g).to(torch.bfloat16).expand(B, S, H, d).contiguous()
    v = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    out, lse = A.fwd(q.cuda(), k.cuda(), v.cuda(), scale=0.088)
    mean_v = v.double().mean(dim=1, keepdim=True).expand(B, S, H, d)
    check_out(out, mean_v.numpy(), "identical keys")
    s = 0.088 * torch.einsum("bihc,hc->bhi", q.double(), k[0, 0].double())
    check_lse(lse, (s + math.log(S)).numpy(), "identical keys")


def test_zero_scale_causal_counts(A):
    w = inputs.PrefillWorkload("z", 1, 2, 2, 400, 400, causal=True, seed=6)
    q, k, v = inputs.make_prefill(w)
    out, lse = A.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=0.0)
    n = torch.arange(1, 401, dtype=torch.float64)
    check_lse(lse, torch.log(n).expand(1, 2, 400).numpy(), "zero scale")
    prefix_mean = v.double().cumsum(dim=1) / n[None, :, None, None]
    check_out(out, prefix_mean.numpy(), "zero scale")


def test_gqa_equals_replicated_heads_bitwise(A):
    w = inputs.PrefillWorkload("g", 2, 8, 2, 512, 512, causal=True, seed=8)
    q, k, v = inputs.make_prefill(w)
    o1, l1 = _run(A, w, q, k, v)
    kr, vr = k.repeat_interleave(4, dim=2).contiguous(), v.repeat_interleave(4, dim=2).contiguous()
    o2, l2 = _run(A, w.with_(Hkv=8), q, kr, vr)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_layouts_bitwise_identical(A):
    w = inputs.PrefillWorkload("l", 1, 4, 2, 300, 300, layout="bshd", causal=True, seed=10)
    q, k, v = inputs.make_prefill(w)
    o1, l1 = _run(A, w, q, k, v)
    w2 = w.with_(layout="bhsd")
    q2, k2, v2 = inputs.make_prefill(w2)
    o2, l2 = _run(A, w2, q2, k2, v2)
    assert torch.equal(o1, o2.permute(0, 2, 1, 3)) and torch.equal(l1, l2)


def test_output_guard_regions_untouched(A):
    w = inputs.PrefillWorkload("guard", 1, 2, 1, 333, 333, causal=True, seed=12)
    q, k, v = inputs.make_prefill(w)
    n = q.numel()
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), device="cuda", dtype=torch.bfloat16)
    out = buf[guard:guard + n].view_as(q)
    lbuf = torch.full((w.Hq * w.Sq + 2 * guard,), 12345.0, device="cuda")
    lse = lbuf[guard:guard + w.Hq * w.Sq].view(1, w.Hq, w.Sq)
    A.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + n:]).all()
    assert (lbuf[:guard] == 12345.0).all() and (lbuf[guard + w.Hq * w.Sq:] == 12345.0).all()
    ref_o, ref_l = _oracle_full(w, q, k, v)
    check_out(out, ref_o, "guard")
    check_lse(lse, ref_l, "guard")


# ---------------------------------------------------------------- full-size workloads, every output

FULL = [inputs.TINY_BHSD, inputs.GQA_CAUSAL, inputs.MQA_CAUSAL, inputs.RAGGED_SELF, inputs.RAGGED_CROSS,
        inputs.GQA_SHORT_QUERY]


def _run_as_benched(A, w, q, k, v):
    """One call in the launch configuration the benchmark times: the tail-split
    workspace registered whenever the shape gets a split on this device."""
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    n = A.fwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.causal)
    ws = torch.empty(n, device="cuda", dtype=torch.uint8) if n else None
    A.set_workspace(ws)
    try:
        out, lse = A.fwd(dq, dk, dv, causal=w.causal, scale=w.scale, layout=w.layout)
        torch.cuda.synchronize()
    finally:
        A.set_workspace(None)
    return out, lse, n


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_every_output(A, w):
    """Every element of O and every lse of the full-size workloads against the
    fp64 oracle (its matmul form, all host cores), plus a cross-check of that
    form against the row-by-row oracle on sampled rows at the same size."""
    q, k, v = inputs.make_prefill(w)
    out, lse, ws_bytes = _run_as_benched(A, w, q, k, v)
    assert A.device_status()[0] == 0
    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, d=w.d, layout=w.layout, causal=w.causal, scale=w.scale)
    ref_o, ref_l = oracle.attention_matmul(q, k, v, **kw)
    out_c, lse_c = out.cpu(), lse.cpu()
    for b in range(w.B):   # one batch at a time keeps the host copies small
        check_out(out_c[b], ref_o[b], f"{w.name} batch {b} (tail split: {bool(ws_bytes)})")
        check_lse(lse_c[b], ref_l[b], f"{w.name} batch {b}")
    rows = sample_rows(w.B, w.Hq, w.Sq, w.Hq // w.Hkv, seed=w.seed)
    row_o, row_l = oracle.attention_rows(q, k, v, rows, **kw)
    mm_o, mm_l = gather_rows(torch.from_numpy(ref_o), torch.from_numpy(ref_l), rows, w.layout)
    np.testing.assert_allclose(mm_o.numpy(), row_o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(mm_l.numpy(), row_l, rtol=0, atol=1e-10)


def test_gqa_workload_deterministic(A):
    w = inputs.GQA_CAUSAL
    q, k, v = (t.cuda() for t in inputs.make_prefill(w))
    o0, l0 = A.fwd(q, k, v, causal=True, scale=w.scale)
    for _ in range(2):
        o1, l1 = A.fwd(q, k, v, causal=True, scale=w.scale)
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


# ---------------------------------------------------------------- paged decode

def _decode(A, w, seqlens=None):
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=seqlens)
    out, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), scale=w.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_paged(q, kp, vp, table, lens, scale=w.scale)
    return out, lse, ref_o, ref_l


def test_paged_decode_workload_full(A):
    w = inputs.PAGED_DECODE
    out, lse, ref_o, ref_l = _decode(A, w)
    check_out(out, ref_o, w.name)
    check_lse(lse, ref_l, w.name)
    assert A.device_status()[0] == 0


@pytest.mark.parametrize("lens", [[0, 1, 15, 16], [17, 31, 32, 33], [8192, 4097, 511, 512], [1, 0, 0, 513]])
def test_paged_decode_edge_lengths(A, lens):
    w = inputs.DecodeWorkload("edge", B=4, Hq=8, Hkv=2, max_blocks=512, seed=7)
    out, lse, ref_o, ref_l = _decode(A, w, seqlens=lens)
    check_out(out, ref_o, f"decode {lens}")
    check_lse(lse, ref_l, f"decode {lens}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (6, 2), (16, 2), (32, 1)])
def test_paged_decode_group_sizes(A, Hq, Hkv):
    w = inputs.DecodeWorkload("groups", B=3, Hq=Hq, Hkv=Hkv, max_blocks=100, len_lo=1, len_hi=1600, seed=8)
    out, lse, ref_o, ref_l = _decode(A, w)
    check_out(out, ref_o, f"decode G={Hq // Hkv}")
    check_lse(lse, ref_l, f"decode G={Hq // Hkv}")


def test_paged_decode_ignores_garbage_past_sequence_end(A):
    # The unused slots of each sequence's last page may hold anything (here
    # NaN and Inf); only keys below seqlen take part in the result.
    w = inputs.DecodeWorkload("garbage", B=4, Hq=8, Hkv=2, max_blocks=64, seed=13)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[17, 33, 1000, 1])
    kp2, vp2 = kp.clone(), vp.clone()
    for b, L in enumerate(lens.tolist()):
        last = int(table[b, (L - 1) // 16])
        kp2[last, L % 16 or 16:] = float("nan")
        vp2[last, L % 16 or 16:] = float("inf")
    out, lse = A.decode_paged(q.cuda(), kp2.cuda(), vp2.cuda(), table.cuda(), lens.cuda(), scale=w.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_paged(q, kp, vp, table, lens, scale=w.scale)
    check_out(out, ref_o, "garbage past the end")
    check_lse(lse, ref_l, "garbage past the end")


def test_paged_decode_long_context(A):
    # 65 536 keys (4096 pages: the split plan's floor of 16 pages a split gives
    # 256 splits, all of them full) beside a 3-token sequence whose splits are
    # all empty but the first.
    w = inputs.DecodeWorkload("long", B=2, Hq=8, Hkv=2, max_blocks=4096, seed=29)
    out, lse, ref_o, ref_l = _decode(A, w, seqlens=[65536, 3])
    check_out(out, ref_o, "decode, 65536 keys")
    check_lse(lse, ref_l, "decode, 65536 keys")
    assert A.device_status()[0] == 0


def test_paged_decode_dominant_keys(A):
    # Two keys per sequence score far above the rest for the first head of
    # each KV group (about 34 and 33.7 in natural-log units) and carry opposite
    # values u and -u: that head's output is u times the difference of their
    # two weights, so a lost or misrounded weight on the largest key moves it
    # by about |u| times the error.  The other heads of the group see those
    # keys at scores of a few units.
    w = inputs.DecodeWorkload("dominant", B=4, Hq=8, Hkv=2, max_blocks=256, seed=23)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[4000, 1, 17, 4096])
    gen = torch.Generator().manual_seed(5)
    G = w.Hq // w.Hkv
    u = (2.0 * torch.randn(w.Hkv, w.d, generator=gen)).to(vp.dtype)
    for b, L in enumerate(lens.tolist()):
        for j, t in enumerate(torch.randperm(L, generator=gen)[:2].tolist()):
            page, slot = int(table[b, t // 16]), t % 16
            for kvh in range(w.Hkv):
                kp[page, slot, kvh] = (3.0 * (1.0 - 0.01 * j) * q[b, kvh * G].float()).to(kp.dtype)
                vp[page, slot, kvh] = u[kvh] if j == 0 else -u[kvh]
    out, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), scale=w.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_paged(q, kp, vp, table, lens, scale=w.scale)
    check_out(out, ref_o, "dominant keys")
    check_lse(lse, ref_l, "dominant keys")


def test_paged_decode_deterministic(A):
    w = inputs.PAGED_DECODE
    q, kp, vp, table, lens = (t.cuda() for t in inputs.make_decode(w))
    o0, l0 = A.decode_paged(q, kp, vp, table, lens, scale=w.scale)
    o1, l1 = A.decode_paged(q, kp, vp, table, lens, scale=w.scale)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_paged_decode_bad_block_table_is_reported(A):
    w = inputs.DecodeWorkload("bad", B=2, Hq=4, Hkv=2, max_blocks=8, seed=9)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[40, 40])
    table[1, 1] = kp.shape[0] + 5          # out of the pool
    assert A.device_status()[0] == 0
    out, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), scale=w.scale)
    code, site = A.device_status()
    assert code == 6  # ATTN_ERR_DEVICE_BOUNDS
    # sequence 0 is unaffected
    ref_o, ref_l = oracle.decode_paged(q[:1], kp, vp, table[:1], lens[:1], scale=w.scale)
    check_out(out[:1], ref_o, "bad table, good row")
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("bad_len", [-1, 8 * 16 + 1, -(2 ** 31)])
def test_paged_decode_bad_length_is_reported(A, bad_len):
    # A length outside [0, 16 * max_blocks] is neither clamped nor read past:
    # it is reported and that sequence's rows come back as zeros and -inf.
    w = inputs.DecodeWorkload("badlen", B=3, Hq=8, Hkv=2, max_blocks=8, seed=19)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[40, 128, 7])
    bad = lens.clone()
    bad[1] = bad_len
    assert A.device_status()[0] == 0
    out, lse = A.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bad.cuda(), scale=w.scale)
    code, site = A.device_status()
    assert code == 6 and site == 16  # ATTN_ERR_DEVICE_BOUNDS at the length check
    assert torch.equal(out[1].cpu(), torch.zeros_like(out[1].cpu()))
    assert torch.isneginf(lse[1]).all()
    keep = [0, 2]
    ref_o, ref_l = oracle.decode_paged(q[keep], kp, vp, table[keep], lens[keep], scale=w.scale)
    check_out(out[keep], ref_o, "bad length, good rows")
    check_lse(lse[keep], ref_l, "bad length, good rows")


def test_lse_merge_matches_oracle(A):
    g = torch.Generator().manual_seed(11)
    rows, nsplit, d = 37, 5, 128
    lse_s = (torch.randn(rows, nsplit, generator=g) * 3).double()
    lse_s[3, :] = -math.inf
    lse_s[4, 1:] = -math.inf
    o_s = torch.randn(rows, nsplit, d, generator=g).double()
    out, lse = A.lse_merge(o_s.float().cuda(), lse_s.float().cuda())
    ref_o, ref_l = oracle.lse_merge(lse_s.float().double().numpy().T.copy(),
                                    o_s.float().double().numpy().transpose(1, 0, 2).copy())
    check_out(out, ref_o, "merge")
    check_lse(lse, ref_l, "merge")
