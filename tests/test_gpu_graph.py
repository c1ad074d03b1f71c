"""The entry points are asynchronous on the caller's stream and capturable
into a CUDA graph: a graph of one prefill (with its tail-split merge), one
varlen prefill and one paged decode step (with its merge, launched as a
programmatic dependent) replays to exactly the eager results."""
import pytest
import torch

from exact_attention_forward_06_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_06_gb300 as attn
    attn.load()
    return attn


def test_graph_replay_equals_eager(A):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wp = inputs.PrefillWorkload("graph", sms + 8, 1, 1, 256, 2048, seed=131)   # gets a tail split
    q, k, v = (t.cuda() for t in inputs.make_prefill(wp))
    wv = inputs.VarlenWorkload("graph-varlen", 3, 8, 2, causal=True, seed=132, lens_q=(100, 300, 7))
    vq, vk, vv, cu_q, cu_k = (t.cuda() for t in inputs.make_varlen(wv))
    wd = inputs.PAGED_DECODE.with_(B=4, max_blocks=64, len_lo=1, len_hi=1000, seed=133)
    dq, kp, vp, table, lens = (t.cuda() for t in inputs.make_decode(wd))
    need = A.fwd_workspace_bytes(wp.B, 1, 1, 256, 2048)
    assert need > 0
    fws = torch.empty(need, device="cuda", dtype=torch.uint8)
    dws = torch.empty(A.decode_workspace_bytes(wd.B, wd.Hq, 128, wd.max_blocks), device="cuda", dtype=torch.uint8)
    out, lse = torch.empty_like(q), torch.empty((wp.B, 1, 256), device="cuda")
    vout, vlse = torch.empty_like(vq), torch.empty((8, vq.shape[0]), device="cuda")
    dout, dlse = torch.empty_like(dq), torch.empty((wd.B, wd.Hq), device="cuda")
    s = torch.cuda.Stream()

    def step():
        A.fwd(q, k, v, scale=wp.scale, out=out, lse=lse, stream=s)
        A.fwd_varlen(vq, vk, vv, cu_q, cu_k, max_seqlen_q=300, max_seqlen_k=300, causal=True, out=vout, lse=vlse,
                     stream=s)
        A.decode_paged(dq, kp, vp, table, lens, scale=wd.scale, out=dout, lse=dlse, workspace=dws, stream=s)

    try:
        A.set_workspace(fws)
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        eager = [t.clone() for t in (out, lse, vout, vlse, dout, dlse)]
        for t in (out, lse, vout, vlse, dout, dlse):
            t.zero_()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
    finally:
        A.set_workspace(None)
    for got, want in zip((out, lse, vout, vlse, dout, dlse), eager):
        assert torch.equal(got, want)
    assert A.device_status()[0] == 0
