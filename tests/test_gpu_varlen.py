"""GPU parity of attention over packed variable-length batches (attn_fwd_varlen).

Every sequence of the packed batch must equal plain attention over its own
rows and keys (the oracle runs it sequence by sequence).  Lengths are chosen
around the 128-row tile: 0, 1, 127, 128, 129, 255, 256, 257 and a few longer
ones, with per-sequence key lengths that differ from the query lengths
(including queries with no keys, and causal rows that see none), group sizes
even (two heads per work unit) and odd (two row blocks per unit).  Rows of
no sequence must be left untouched, an equal-length packed batch must equal
the dense batch bit for bit, and bad offsets must be reported without a fault.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()
    return attn


def _run(A, w, **kw):
    q, k, v, cu_q, cu_k = inputs.make_varlen(w)
    out = torch.full(q.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.Hq, q.shape[0]), SENTINEL, dtype=torch.float32, device="cuda")
    A.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), causal=w.causal, scale=w.scale, out=out,
                 lse=lse, **kw)
    torch.cuda.synchronize()
    return (q, k, v, cu_q, cu_k), out.cpu(), lse.cpu()


def _compare_all(w, data, out, lse, what):
    q, k, v, cu_q, cu_k = data
    ref_o, ref_l = oracle.attention_varlen(q, k, v, cu_q, cu_k, Hq=w.Hq, Hkv=w.Hkv, causal=w.causal, scale=w.scale)
    owned = ~np.isnan(ref_l[0])
    check_out(out[torch.from_numpy(owned)], ref_o[owned], what)
    check_lse(lse[:, torch.from_numpy(owned)], ref_l[:, owned], what)
    # rows of no sequence keep what the caller put there
    assert (out[torch.from_numpy(~owned)].float() == SENTINEL).all(), f"{what}: rows outside the sequences written"
    assert (lse[:, torch.from_numpy(~owned)] == SENTINEL).all(), f"{what}: lse outside the sequences written"


EDGE_Q = (0, 1, 127, 128, 129, 255, 256, 257, 600, 1000)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (3, 1)])
def test_edge_lengths_match_oracle(A, causal, Hq, Hkv):
    w = inputs.VarlenWorkload("edges", len(EDGE_Q), Hq, Hkv, causal=causal, seed=91, lens_q=EDGE_Q, pad_q=5)
    data, out, lse = _run(A, w)
    _compare_all(w, data, out, lse, f"edges causal={causal} G={Hq // Hkv}")
    assert A.device_status()[0] == 0


@pytest.mark.parametrize("causal", [False, True])
def test_cross_lengths_match_oracle(A, causal):
    # key lengths differ per sequence: none, fewer than the queries (causal
    # rows that see no key), more, and ragged against the 128-key tile
    lq = (300, 64, 200, 1, 129, 500)
    lk = (0, 300, 77, 1000, 129, 383)
    w = inputs.VarlenWorkload("cross", len(lq), 4, 4, causal=causal, seed=92, lens_q=lq, lens_k=lk)
    data, out, lse = _run(A, w)
    _compare_all(w, data, out, lse, f"cross causal={causal}")
    assert A.device_status()[0] == 0


def test_unit_order_does_not_change_the_result(A):
    # Keys at least twice as long as the queries switch the launch to the
    # sequence-and-KV-head unit order; a larger stated key bound selects it
    # for the same data, which must give the same bits.
    lq = (300, 64, 200, 129)
    lk = (500, 300, 77, 383)
    w = inputs.VarlenWorkload("order", len(lq), 8, 2, causal=True, seed=96, lens_q=lq, lens_k=lk)
    q, k, v, cu_q, cu_k = (t.cuda() for t in inputs.make_varlen(w))
    o_row, l_row = A.fwd_varlen(q, k, v, cu_q, cu_k, max_seqlen_q=300, max_seqlen_k=500, causal=True,
                                scale=w.scale)
    o_kv, l_kv = A.fwd_varlen(q, k, v, cu_q, cu_k, max_seqlen_q=300, max_seqlen_k=sum(lk), causal=True,
                              scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    assert torch.equal(o_row, o_kv) and torch.equal(l_row, l_kv)


def test_equal_lengths_equal_the_dense_batch_bitwise(A):
    B, L, Hq, Hkv = 3, 300, 8, 2
    w = inputs.PrefillWorkload("dense", B, Hq, Hkv, L, L, causal=True, seed=93)
    q, k, v = (t.cuda() for t in inputs.make_prefill(w))
    o_dense, l_dense = A.fwd(q, k, v, causal=True, scale=w.scale)
    cu = torch.arange(0, (B + 1) * L, L, dtype=torch.int32, device="cuda")
    o_var, l_var = A.fwd_varlen(q.reshape(B * L, Hq, 128), k.reshape(B * L, Hkv, 128), v.reshape(B * L, Hkv, 128),
                                cu, cu, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_var, o_dense.reshape(B * L, Hq, 128))
    assert torch.equal(l_var, l_dense.permute(1, 0, 2).reshape(Hq, B * L))


def test_rounding_mode_applies(A):
    w = inputs.VarlenWorkload("round", 3, 4, 2, causal=True, seed=94, lens_q=(130, 7, 260))
    _, o_ne, _ = _run(A, w)
    _, o_z, _ = _run(A, w, rounding="rtz")
    mag = lambda t: (t.view(torch.int16).numpy().view(np.uint16) & 0x7FFF).astype(np.int32)
    step = mag(o_ne) - mag(o_z)
    assert ((step == 0) | (step == 1)).all() and (step == 1).mean() > 0.3


def test_bad_offsets_are_reported_without_a_fault(A):
    w = inputs.VarlenWorkload("bad", 3, 4, 2, seed=95, lens_q=(100, 50, 80))
    q, k, v, cu_q, cu_k = inputs.make_varlen(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    bad_q = cu_q.clone()
    bad_q[2] = bad_q[1] - 10                    # sequence 1 runs backwards
    out = torch.full(q.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    A.fwd_varlen(dq, dk, dv, bad_q.cuda(), cu_k.cuda(), max_seqlen_q=100, max_seqlen_k=100, scale=w.scale, out=out)
    code, site = A.device_status()
    assert code == 6 and site == 12, (code, site)
    # a length past the stated maximum is caught the same way
    A.fwd_varlen(dq, dk, dv, cu_q.cuda(), cu_k.cuda(), max_seqlen_q=90, max_seqlen_k=100, scale=w.scale)
    assert A.device_status()[0] == 6
    # and the context still computes correctly
    data, out, lse = _run(A, w)
    _compare_all(w, data, out, lse, "after bad offsets")
    assert A.device_status()[0] == 0


def test_full_workload_every_output(A):
    w = inputs.VARLEN_CAUSAL
    q, k, v, cu_q, cu_k = inputs.make_varlen(w)
    out, lse = A.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    ref_o, ref_l = oracle.attention_varlen(q, k, v, cu_q, cu_k, Hq=w.Hq, Hkv=w.Hkv, causal=True, scale=w.scale,
                                           dense=oracle.attention_matmul)
    assert not np.isnan(ref_l).any()   # the workload's sequences cover every row
    check_out(out.cpu(), ref_o, w.name)
    check_lse(lse.cpu(), ref_l, w.name)
