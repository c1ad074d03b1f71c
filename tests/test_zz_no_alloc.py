"""attn_decode_paged_noalloc: the decode step for callers that cannot allocate.

Such callers (an operator interface that hands a kernel only its inputs and
outputs with no workspace hook, or an engine that has reserved all of HBM and
forbids further cudaMalloc) get the split partials kept in a library-owned
device array instead of a workspace they would have to allocate.  This checks,
through the C ABI, that two calls in a row of the allocation-free entry point
give bit for bit the output of the workspace-taking attn_decode_paged (the
same split plan, kernels and merge order), that each also matches the fp64
oracle within the parity tolerance, and that a shape too large for the array
is refused.

Kept in its own file, named to be collected last, so that a failure here never
stops a run before the other tests have run.
"""
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


def _device_inputs(w, seqlens=None):
    return [t.cuda() for t in inputs.make_decode(w, seqlens=seqlens)]


def test_noalloc_decode_matches_workspace_decode_twice(A):
    cases = [
        (inputs.PAGED_DECODE, None),
        # a different, smaller shape second, so the array still holds the
        # first call's partials when the second call reads its own
        (inputs.DecodeWorkload("noalloc_second", B=5, Hq=16, Hkv=4, max_blocks=200, len_lo=0, len_hi=3000,
                               seed=31), [0, 1, 3000, 17, 1024]),
    ]
    for w, lens in cases:
        assert A.decode_workspace_bytes(w.B, w.Hq, w.d, w.max_blocks) <= 16 * 1024 * 1024
        host = inputs.make_decode(w, seqlens=lens)
        q, kp, vp, table, seqlens = (t.cuda() for t in host)
        ref_out, ref_lse = A.decode_paged(q, kp, vp, table, seqlens, scale=w.scale)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq), float("nan"), device=q.device, dtype=torch.float32)
        A.decode_paged_noalloc(q, kp, vp, table, seqlens, scale=w.scale, out=out, lse=lse)
        torch.cuda.synchronize()
        # Same plan, kernels and merge order as the workspace call: bit for bit.
        assert torch.equal(out, ref_out), f"noalloc {w.name}: output differs from attn_decode_paged"
        assert torch.equal(lse, ref_lse), f"noalloc {w.name}: lse differs from attn_decode_paged"
        # And against the fp64 oracle directly.
        o_ref, l_ref = oracle.decode_paged(*host, scale=w.scale)
        check_out(out, o_ref, f"noalloc {w.name} vs oracle")
        check_lse(lse, l_ref, f"noalloc {w.name} vs oracle")
        assert A.device_status()[0] == 0


def test_noalloc_decode_refuses_shapes_beyond_its_array(A):
    # 64 x 64 heads x 8192 pages per sequence needs far more than 16 MiB of partials
    B, Hq, Hkv, maxb = 64, 64, 8, 8192
    assert A.decode_workspace_bytes(B, Hq, 128, maxb) > 16 * 1024 * 1024
    q = torch.zeros((B, Hq, 128), device="cuda", dtype=torch.bfloat16)
    kp = torch.zeros((4, 16, Hkv, 128), device="cuda", dtype=torch.bfloat16)
    table = torch.zeros((B, maxb), device="cuda", dtype=torch.int32)
    seqlens = torch.zeros((B,), device="cuda", dtype=torch.int32)
    with pytest.raises(A.AttnError) as err:
        A.decode_paged_noalloc(q, kp, kp, table, seqlens, scale=0.1)
    assert err.value.code == 5  # ATTN_ERR_WORKSPACE
