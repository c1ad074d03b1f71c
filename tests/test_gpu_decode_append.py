"""GPU parity of the fused KV-cache append + decode step (attn_decode_paged_append).

The new token's K/V must land in exactly its slot (the pools are compared
bit for bit with the oracle's), and every query must attend over the old keys
plus the new one.  Lengths before the append sit around the 16-token page
(including an empty cache and a full table), stale NaN in the slot being
written and past it must never reach the result, and a missing page is
reported without a fault.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()
    return attn


def _case(lens, Hq=32, Hkv=8, seed=111, max_blocks=512):
    w = inputs.PAGED_DECODE.with_(B=len(lens), Hq=Hq, Hkv=Hkv, seed=seed, max_blocks=max_blocks)
    q, kp, vp, table, _ = inputs.make_decode(w, seqlens=[L + 1 for L in lens])   # pages for L + 1 keys
    g = torch.Generator().manual_seed(seed + 1)
    k_new = torch.randn(len(lens), Hkv, 128, generator=g).to(torch.bfloat16)
    v_new = torch.randn(len(lens), Hkv, 128, generator=g).to(torch.bfloat16)
    return w, q, kp, vp, table, torch.tensor(lens, dtype=torch.int32), k_new, v_new


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


EDGE = [0, 1, 15, 16, 17, 31, 32, 100, 1000, 8191]


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (6, 2), (32, 4)])
def test_append_and_decode_match_oracle(A, Hq, Hkv):
    w, q, kp, vp, table, lens, k_new, v_new = _case(EDGE, Hq, Hkv)
    ref_o, ref_l, ref_kp, ref_vp = oracle.decode_paged_append(q, k_new, v_new, kp, vp, table, lens, scale=w.scale)
    dkp, dvp = kp.cuda(), vp.cuda()
    out, lse = A.decode_paged_append(q.cuda(), k_new.cuda(), v_new.cuda(), dkp, dvp, table.cuda(), lens.cuda(),
                                     scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    check_out(out, ref_o, f"append G={Hq // Hkv}")
    check_lse(lse, ref_l, f"append G={Hq // Hkv}")
    assert torch.equal(_bits(dkp), _bits(ref_kp)) and torch.equal(_bits(dvp), _bits(ref_vp))


def test_fused_equals_append_then_decode(A):
    lens_l = [5, 16, 300, 4095, 2000, 64]
    w, q, kp, vp, table, lens, k_new, v_new = _case(lens_l, seed=112)
    dq, dt = q.cuda(), table.cuda()
    dkp, dvp = kp.cuda(), vp.cuda()
    o_f, l_f = A.decode_paged_append(dq, k_new.cuda(), v_new.cuda(), dkp, dvp, dt, lens.cuda(), scale=w.scale)
    # the same step in two: append with torch, then plain decode over L + 1 keys
    kp2, vp2 = kp.clone(), vp.clone()
    for b, L in enumerate(lens_l):
        kp2[int(table[b, L // 16]), L % 16] = k_new[b]
        vp2[int(table[b, L // 16]), L % 16] = v_new[b]
    o_2, l_2 = A.decode_paged(dq, kp2.cuda(), vp2.cuda(), dt, (lens + 1).cuda(), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(_bits(dkp), _bits(kp2)) and torch.equal(_bits(dvp), _bits(vp2))
    check_out(o_f, o_2.double().cpu().numpy(), "fused vs two-step")
    check_lse(l_f, l_2.double().cpu().numpy(), "fused vs two-step")
    # and a second fused call (same slot, same bits) gives the same result bitwise
    o_g, l_g = A.decode_paged_append(dq, k_new.cuda(), v_new.cuda(), dkp, dvp, dt, lens.cuda(), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_f, o_g) and torch.equal(l_f, l_g)


def test_stale_nan_in_and_past_the_new_slot(A):
    lens_l = [0, 7, 16, 33, 1000]
    w, q, kp, vp, table, lens, k_new, v_new = _case(lens_l, seed=113)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    for b, L in enumerate(lens_l):
        page = int(table[b, L // 16])
        kp[page, L % 16:] = nan     # the slot being written and the rest of its page
        vp[page, L % 16:] = nan
    ref_o, ref_l, ref_kp, ref_vp = oracle.decode_paged_append(q, k_new, v_new, kp, vp, table, lens, scale=w.scale)
    dkp, dvp = kp.cuda(), vp.cuda()
    out, lse = A.decode_paged_append(q.cuda(), k_new.cuda(), v_new.cuda(), dkp, dvp, table.cuda(), lens.cuda(),
                                     scale=w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    check_out(out, ref_o, "stale NaN")
    check_lse(lse, ref_l, "stale NaN")
    assert torch.equal(_bits(dkp), _bits(ref_kp)) and torch.equal(_bits(dvp), _bits(ref_vp))


def test_missing_page_for_the_new_token_is_reported(A):
    lens_l = [16, 20]
    w, q, kp, vp, table, lens, k_new, v_new = _case(lens_l, seed=114)
    table[0, 1] = -1                     # sequence 0 needs a new page for token 16: none given
    dkp = kp.cuda()
    out, lse = A.decode_paged_append(q.cuda(), k_new.cuda(), v_new.cuda(), dkp, vp.cuda(), table.cuda(),
                                     lens.cuda(), scale=w.scale)
    code, site = A.device_status()
    assert code == 6 and site == 15, (code, site)
    # sequence 1's token was written; sequence 0's pages are as they were
    assert torch.equal(_bits(dkp[int(table[1, 1])][4]), _bits(k_new[1]))
    assert torch.equal(_bits(dkp[int(table[0, 0])]), _bits(kp[int(table[0, 0])]))


def test_append_long_context(A):
    # The new token lands at position 65 535, the last slot of the last of
    # 4096 pages, of a sequence split 256 ways; the short sequence appends to
    # its first page.  Split 0 of each sequence attends to the new token.
    w, q, kp, vp, table, lens, k_new, v_new = _case([65535, 3], Hq=8, Hkv=2, seed=113, max_blocks=4096)
    ref_o, ref_l, ref_kp, ref_vp = oracle.decode_paged_append(q, k_new, v_new, kp, vp, table, lens, scale=w.scale)
    dkp, dvp = kp.cuda(), vp.cuda()
    out, lse = A.decode_paged_append(q.cuda(), k_new.cuda(), v_new.cuda(), dkp, dvp, table.cuda(), lens.cuda(),
                                     scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    check_out(out, ref_o, "append, 65536 keys")
    check_lse(lse, ref_l, "append, 65536 keys")
    assert torch.equal(_bits(dkp), _bits(ref_kp)) and torch.equal(_bits(dvp), _bits(ref_vp))
