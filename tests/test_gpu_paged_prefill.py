"""GPU parity of chunked prefill against a paged KV cache (attn_fwd_paged).

Each sequence's query chunk must equal plain attention over the keys gathered
from its pages (the oracle gathers them one token at a time).  Chunk and
context lengths sit around the 16-token page and the 128-key tile; the cache's
unused slots and pages are filled with NaN to show they never reach the
result; a pool laid out in order must give exactly the packed-batch result;
bad table entries are reported without a fault.
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


def _poison_unused_slots(kp, vp, table, lens):
    """NaN in every pool slot that holds no key of any sequence."""
    used = torch.zeros(kp.shape[0], kp.shape[1], dtype=torch.bool)
    for b, L in enumerate(lens.tolist()):
        for t in range(L):
            used[int(table[b, t // 16]), t % 16] = True
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    kp[~used] = nan
    vp[~used] = nan


def _run_and_compare(A, w, data, what):
    q, kp, vp, table, lens, cu_q = data
    out = torch.full(q.shape, SENTINEL, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.Hq, q.shape[0]), SENTINEL, dtype=torch.float32, device="cuda")
    A.fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), cu_q.cuda(), causal=w.causal,
                scale=w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    ref_o, ref_l = oracle.attention_paged(q, kp, vp, table, lens, cu_q, Hq=w.Hq, Hkv=w.Hkv, causal=w.causal,
                                          scale=w.scale)
    owned = torch.from_numpy(~np.isnan(ref_l[0]))
    check_out(out.cpu()[owned], ref_o[owned.numpy()], what)
    check_lse(lse.cpu()[:, owned], ref_l[:, owned.numpy()], what)
    return out.cpu(), lse.cpu()


CHUNKS = (1, 1, 16, 17, 127, 128, 129, 300, 5)
CONTEXTS = (0, 15, 16, 0, 1, 127, 200, 1000, 0)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (3, 1)])
def test_edge_chunks_and_contexts_match_oracle(A, causal, Hq, Hkv):
    w = inputs.PagedPrefillWorkload("edges", len(CHUNKS), Hq, Hkv, chunks=CHUNKS, contexts=CONTEXTS, causal=causal,
                                    seed=101, max_blocks=96)
    _run_and_compare(A, w, inputs.make_paged_prefill(w), f"paged edges causal={causal} G={Hq // Hkv}")


def test_nan_in_unused_slots_never_reaches_the_result(A):
    w = inputs.PagedPrefillWorkload("nan", 6, 8, 2, chunks=(3, 40, 129, 1, 77, 200), contexts=(5, 0, 30, 17, 250, 9),
                                    seed=102, max_blocks=40)
    q, kp, vp, table, lens, cu_q = inputs.make_paged_prefill(w)
    _poison_unused_slots(kp, vp, table, lens)
    assert torch.isnan(vp.float()).any()
    out, _ = _run_and_compare(A, w, (q, kp, vp, table, lens, cu_q), "paged with NaN in unused slots")
    assert torch.isfinite(out.float()).all()


def test_in_order_pool_equals_the_packed_batch_bitwise(A):
    # sequences of whole pages laid out in order: the pool, read as one packed
    # K/V tensor, is exactly the varlen call's input
    lq, lk = (100, 256, 17), (160, 256, 48)
    Hq, Hkv, d = 8, 2, 128
    g = torch.Generator().manual_seed(103)
    total_k = sum(lk)
    kp = torch.randn(total_k // 16, 16, Hkv, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(total_k // 16, 16, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(lq), Hq, d, generator=g).to(torch.bfloat16)
    table = torch.full((3, 16), -1, dtype=torch.int32)
    start = 0
    for b, L in enumerate(lk):
        table[b, :L // 16] = torch.arange(start, start + L // 16, dtype=torch.int32)
        start += L // 16
    cu_q = torch.tensor([0, 100, 356, 373], dtype=torch.int32)
    cu_k = torch.tensor([0, 160, 416, 464], dtype=torch.int32)
    dq, dkp, dvp = q.cuda(), kp.cuda(), vp.cuda()
    o_p, l_p = A.fwd_paged(dq, dkp, dvp, table.cuda(), torch.tensor(lk, dtype=torch.int32).cuda(), cu_q.cuda(),
                           causal=True)
    o_v, l_v = A.fwd_varlen(dq, dkp.reshape(total_k, Hkv, d), dvp.reshape(total_k, Hkv, d), cu_q.cuda(),
                            cu_k.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_v) and torch.equal(l_p, l_v)


def test_bad_table_entry_is_reported_without_a_fault(A):
    w = inputs.PagedPrefillWorkload("bad", 3, 4, 2, chunks=(10, 20, 30), contexts=(40, 50, 60), seed=104,
                                    max_blocks=8)
    q, kp, vp, table, lens, cu_q = inputs.make_paged_prefill(w)
    bad = table.clone()
    bad[1, 2] = kp.shape[0] + 5
    A.fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), bad.cuda(), lens.cuda(), cu_q.cuda())
    code, site = A.device_status()
    assert code == 6 and site == 13, (code, site)
    bad_lens = lens.clone()
    bad_lens[0] = 8 * 16 + 1                  # longer than the table row
    A.fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), bad_lens.cuda(), cu_q.cuda())
    assert A.device_status()[0] == 6
    _run_and_compare(A, w, (q, kp, vp, table, lens, cu_q), "after bad table")


def test_full_workload_every_output(A):
    w = inputs.PAGED_PREFILL
    q, kp, vp, table, lens, cu_q = inputs.make_paged_prefill(w)
    out, lse = A.fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(), cu_q.cuda(), causal=True,
                           scale=w.scale)
    torch.cuda.synchronize()
    assert A.device_status()[0] == 0
    ref_o, ref_l = oracle.attention_paged(q, kp, vp, table, lens, cu_q, Hq=w.Hq, Hkv=w.Hkv, causal=True,
                                          scale=w.scale, dense=oracle.attention_matmul)
    assert not np.isnan(ref_l).any()
    check_out(out.cpu(), ref_o, w.name)
    check_lse(lse.cpu(), ref_l, w.name)


def test_runs_of_consecutive_pages_mixed_with_scattered_ones(A):
    # A tile whose 8 table entries are consecutive pool pages is loaded as one
    # run; here some tiles are runs, some have one page out of order, and one
    # run ends at the last page of the pool.
    w = inputs.PagedPrefillWorkload("runs", 3, 8, 2, chunks=(100, 300, 129), contexts=(412, 1000, 127), seed=106,
                                    max_blocks=96)
    q, kp, vp, table, lens, cu_q = inputs.make_paged_prefill(w)
    n_pages = [(int(L) + 15) // 16 for L in lens]
    order = torch.arange(sum(n_pages), dtype=torch.int32)
    t2 = torch.full_like(table, -1)
    off = 0
    for b, n in enumerate(n_pages):
        t2[b, :n] = order[off:off + n]
        off += n
    t2[1, 10], t2[1, 11] = t2[1, 11].clone(), t2[1, 10].clone()     # one tile of sequence 1 is not a run
    # keep the data of every (sequence, token): move pages to the new ids
    kp2, vp2 = kp.clone(), vp.clone()
    for b, n in enumerate(n_pages):
        kp2[t2[b, :n].long()] = kp[table[b, :n].long()]
        vp2[t2[b, :n].long()] = vp[table[b, :n].long()]
    _run_and_compare(A, w, (q, kp2, vp2, t2, lens, cu_q), "paged runs")
