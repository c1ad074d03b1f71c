"""Failure detection without a GPU fault: a bounded wait that runs out.

attn_debug_inject(1) makes the next prefill launch's load-issuing warp issue
nothing, so the flag the other warps wait for is never set.  With a short wait
budget their bounded waits expire; the kernel records ATTN_ERR_TIMEOUT and a
site in the device status word, releases tensor memory and exits.  No trap,
no hang, nothing left in flight: the same context then runs a normal call
that must still match the oracle.
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


def test_expired_wait_is_reported_and_context_survives(A):
    w = inputs.PrefillWorkload("inject", 1, 2, 2, 128, 256, seed=61)   # a single work unit
    q, k, v = inputs.make_prefill(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    assert A.device_status()[0] == 0
    A.set_wait_budget_ns(50_000_000)          # 50 ms
    try:
        A.debug_inject(1)
        A.fwd(dq, dk, dv, scale=w.scale)
        code, site = A.device_status()       # synchronises
        assert code == 4, f"expected ATTN_ERR_TIMEOUT, got {code}"
        # a wait of the MMA-issuing, softmax or store side gave up: for its
        # work item (19), its Q tile (1), a K/V tile (2), a score tile (4, 5,
        # 6) or a store command (20)
        assert site in (1, 2, 4, 5, 6, 19, 20), site
        assert A.device_status()[0] == 0      # reading clears it
    finally:
        A.debug_inject(0)
        A.set_wait_budget_ns(0)
    out, lse = A.fwd(dq, dk, dv, scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    ref_o, ref_l = oracle.attention(q, k, v, B=1, Hq=2, Hkv=2, Sq=128, Sk=256, scale=w.scale)
    check_out(out, ref_o, "after injected timeout")
    check_lse(lse, ref_l, "after injected timeout")
