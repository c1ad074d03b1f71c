"""GPU parity of the host-memory entry point attn_fwd_host.

The call copies host inputs to a device workspace in batch chunks, runs the
forward kernel on each chunk and copies the results back; each batch is
computed exactly as attn_fwd would compute it, so the result must equal the
device call bit for bit (no tail-split workspace is registered here) and the
oracle within the tolerance.  Shapes cover one chunk per batch, several
batches per chunk with a short last chunk (B = 10), longer causal rows
(including Sk > Sq and an odd group size), both layouts and a missing lse.
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


@pytest.mark.parametrize("layout,B,Hq,Hkv,S,Sk,causal", [
    ("bshd", 3, 8, 2, 300, 300, True), ("bhsd", 2, 4, 4, 200, 200, False), ("bshd", 10, 2, 1, 130, 130, True),
    # longer causal rows: paired and unpaired heads, Sk > Sq
    ("bshd", 2, 8, 2, 1000, 1000, True), ("bshd", 1, 3, 1, 600, 700, True), ("bshd", 5, 4, 2, 520, 520, True)])
def test_host_call_equals_device_call_and_oracle(A, layout, B, Hq, Hkv, S, Sk, causal):
    w = inputs.PrefillWorkload("host", B, Hq, Hkv, S, Sk, layout=layout, causal=causal, seed=121)
    q, k, v = (t.pin_memory() for t in inputs.make_prefill(w))
    out, lse = A.fwd_host(q, k, v, causal=causal, scale=w.scale, layout=layout)
    torch.cuda.synchronize()
    assert out.device.type == "cpu" and lse.device.type == "cpu"
    o_dev, l_dev = A.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(out, o_dev.cpu()) and torch.equal(lse, l_dev.cpu())
    ref_o, ref_l = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=S, Sk=Sk, layout=layout, causal=causal,
                                    scale=w.scale)
    check_out(out, ref_o, f"host {layout} B={B}")
    check_lse(lse, ref_l, f"host {layout} B={B}")
    assert A.device_status()[0] == 0


def test_host_call_without_lse_and_with_a_given_workspace(A):
    w = inputs.PrefillWorkload("host2", 2, 4, 2, 256, 384, seed=122)
    q, k, v = (t.pin_memory() for t in inputs.make_prefill(w))
    ws = torch.empty(A.fwd_host_workspace_bytes(2, 4, 2, 256, 384), device="cuda", dtype=torch.uint8)
    out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    o, l = A.fwd_host(q, k, v, scale=w.scale, out=out, lse=False, workspace=ws)
    torch.cuda.synchronize()
    assert l is None and o is out
    ref_o, _ = oracle.attention(q, k, v, B=2, Hq=4, Hkv=2, Sq=256, Sk=384, scale=w.scale)
    check_out(out, ref_o, "host without lse")
