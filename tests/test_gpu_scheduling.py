"""The persistent prefill grid's unit hand-out, on the GPU.

With more work units than SMs each CTA takes the next free unit from a
device counter that the launch owns (one of a pool of counter pairs handed
out in turn; the launch's last CTA sets its pair back to zero).  These tests
check that results do not depend on that: launches in flight at the same
time on two streams, long runs of launches that reuse every counter pair,
and graph replays all give the one-launch result bit for bit.
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


def _case(name, B, Hq, Hkv, S, causal, seed):
    w = inputs.PrefillWorkload(name, B, Hq, Hkv, S, S, causal=causal, seed=seed)
    q, k, v = inputs.make_prefill(w)
    return w, (q, k, v), tuple(t.cuda() for t in (q, k, v))


def test_concurrent_launches_on_two_streams(A):
    # Two different problems, each with more units than SMs, launched many
    # times on two streams with no ordering between them.
    wa, host_a, (qa, ka, va) = _case("two_streams_a", 8, 16, 4, 1024, True, 71)
    wb, host_b, (qb, kb, vb) = _case("two_streams_b", 4, 8, 8, 2048, False, 72)
    ref_a = A.fwd(qa, ka, va, causal=True, scale=wa.scale)
    ref_b = A.fwd(qb, kb, vb, causal=False, scale=wb.scale)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for i in range(24):
        with torch.cuda.stream(s1):
            outs.append(("a",) + A.fwd(qa, ka, va, causal=True, scale=wa.scale))
        with torch.cuda.stream(s2):
            outs.append(("b",) + A.fwd(qb, kb, vb, causal=False, scale=wb.scale))
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    for tag, o, l in outs:
        ro, rl = ref_a if tag == "a" else ref_b
        assert torch.equal(o, ro) and torch.equal(l, rl), f"stream result {tag} differs from the single launch"
    o_ref, l_ref = oracle.attention(*host_a, B=wa.B, Hq=wa.Hq, Hkv=wa.Hkv, Sq=wa.Sq, Sk=wa.Sk, causal=True,
                                    scale=wa.scale)
    check_out(ref_a[0], o_ref, "two streams a")
    check_lse(ref_a[1], l_ref, "two streams a")


def test_every_counter_pair_reused(A):
    # More launches than the pool has counter pairs, so every pair is used
    # again after its previous launch reset it; small and large problems mixed.
    w1, _, (q1, k1, v1) = _case("reuse_small", 1, 2, 2, 300, True, 73)      # fewer units than SMs
    w2, _, (q2, k2, v2) = _case("reuse_large", 8, 8, 2, 1024, True, 74)     # more units than SMs
    r1 = A.fwd(q1, k1, v1, causal=True, scale=w1.scale)
    r2 = A.fwd(q2, k2, v2, causal=True, scale=w2.scale)
    for i in range(600):
        o, l = A.fwd(q2, k2, v2, causal=True, scale=w2.scale)
        if i % 97 == 0:
            A.fwd(q1, k1, v1, causal=True, scale=w1.scale)
        if i % 50 == 0:
            torch.cuda.synchronize()
            assert torch.equal(o, r2[0]) and torch.equal(l, r2[1]), f"launch {i} differs"
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    o1, l1 = A.fwd(q1, k1, v1, causal=True, scale=w1.scale)
    assert torch.equal(o1, r1[0]) and torch.equal(l1, r1[1])


def test_graph_replays_of_a_persistent_launch(A):
    w, _, (q, k, v) = _case("graph_persistent", 4, 32, 8, 1024, True, 75)
    ref = A.fwd(q, k, v, causal=True, scale=w.scale)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), device="cuda", dtype=torch.float32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A.fwd(q, k, v, causal=True, scale=w.scale, out=out, lse=lse)   # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            A.fwd(q, k, v, causal=True, scale=w.scale, out=out, lse=lse, stream=s)
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    assert A.device_status()[0] == 0
