"""GPU parity of the prefill tail split (last-wave key-range split + log-sum-exp merge).

The shapes are built from the device's SM count so that the work units leave
a partial last wave: B = num_SMs + 8 batches of one unit each (or two with a
head pair), non-causal, 16 K/V tiles, or 8 (short units, whose first copies
the kernel issues before its CTA-wide barrier).  With a workspace registered, the last
units run as key-range parts whose fp32 partials are merged; every row of the
split units and a sample of the others is compared with the oracle, and the
split result is checked against the unsplit one and for determinism.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs
from parity_util import check_lse, check_out, gather_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()
    return attn


@pytest.mark.parametrize("Sk", [2048, 1024])
@pytest.mark.parametrize("layout,Hq,Hkv", [("bshd", 1, 1), ("bhsd", 2, 1)])
def test_tail_split_matches_oracle_and_unsplit(A, layout, Hq, Hkv, Sk):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Sq = sms + 8, 256
    w = inputs.PrefillWorkload("tail", B, Hq, Hkv, Sq, Sk, layout=layout, seed=71)
    need = A.fwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, causal=False)
    assert need > 0, "this shape is meant to get a tail split"
    assert A.fwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, causal=True) == 0
    q, k, v = inputs.make_prefill(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o_whole, l_whole = A.fwd(dq, dk, dv, scale=w.scale, layout=layout)
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    try:
        A.set_workspace(ws)
        o_split, l_split = A.fwd(dq, dk, dv, scale=w.scale, layout=layout)
        o_again, l_again = A.fwd(dq, dk, dv, scale=w.scale, layout=layout)
        torch.cuda.synchronize()
    finally:
        A.set_workspace(None)
    assert A.device_status()[0] == 0
    assert torch.equal(o_split, o_again) and torch.equal(l_split, l_again)
    # The split units are among the last 16 batches (with a head pair, the
    # units of the upper row block of the last 16 batches): compare all their
    # rows, and every 16th row of a sample of the others, with the oracle.
    tail_b = 16
    rows = [(b, h, i) for b in range(B - tail_b, B) for h in range(Hq) for i in range(Sq)]
    rows += [(b, h, i) for b in range(0, B - tail_b, 37) for h in range(Hq) for i in range(0, Sq, 16)]
    rows = np.array(rows, dtype=np.int64)
    ref_o, ref_l = oracle.attention_rows(q, k, v, rows, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, layout=layout,
                                         scale=w.scale)
    o_rows, l_rows = gather_rows(o_split, l_split, rows, layout)
    check_out(o_rows, ref_o, f"tail split {layout}")
    check_lse(l_rows, ref_l, f"tail split {layout}")
    # units that were not split are bitwise the same as without a workspace
    head = slice(0, B - tail_b)
    assert torch.equal(o_split[head], o_whole[head]) and torch.equal(l_split[head], l_whole[head])
    # and the split units agree with the unsplit result to within the tolerance
    check_out(o_split[B - tail_b:], o_whole[B - tail_b:].double().cpu().numpy(), "split vs whole")


def test_tail_split_with_dead_second_tiles(A):
    # One head (G = 1) and 300 query rows: each batch has a unit of row blocks
    # 0 and 1 and a unit of row block 2 whose second tile lies wholly past the
    # end.  The second kind come last in the unit order, so the split tail
    # units are of that kind: their dead tile passes its turns and its parts
    # carry nothing.  Every output element is compared with the oracle.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Sq, Sk = sms + 8, 300, 2048
    w = inputs.PrefillWorkload("tail_dead", B, 1, 1, Sq, Sk, seed=73)
    need = A.fwd_workspace_bytes(B, 1, 1, Sq, Sk, causal=False)
    assert need > 0, "this shape is meant to get a tail split"
    q, k, v = inputs.make_prefill(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o_whole, l_whole = A.fwd(dq, dk, dv, scale=w.scale)
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    try:
        A.set_workspace(ws)
        o_split, l_split = A.fwd(dq, dk, dv, scale=w.scale)
        o_again, l_again = A.fwd(dq, dk, dv, scale=w.scale)
        torch.cuda.synchronize()
    finally:
        A.set_workspace(None)
    assert A.device_status()[0] == 0
    assert torch.equal(o_split, o_again) and torch.equal(l_split, l_again)
    ref_o, ref_l = oracle.attention(q, k, v, B=B, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=w.d, layout=w.layout, causal=False,
                                    scale=w.scale)
    check_out(o_split, ref_o, "tail split, dead second tiles")
    check_lse(l_split, ref_l, "tail split, dead second tiles")
    check_out(o_whole, ref_o, "no split, dead second tiles")
