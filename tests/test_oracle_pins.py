"""Pins for the CPU oracle: closed forms, invariants, brute force and a library routine.

None of these re-types the oracle's formula.  Each checks the oracle against
something fixed from outside it: a hand-worked example, a closed form that a
special input reduces to, an invariance the definition implies, torch's own
scaled-dot-product attention in fp64 (an independent library routine), or a
different algorithm (the tiled online-softmax recurrence, the log-sum-exp
merge) that the pages say reaches the same result.  The mutation tests at
the bottom plant plausible mistakes in a copy of the oracle's C source and
check that at least one pin fails for each.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_06_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _scalar(s: str) -> float:
    table = {"ln3": math.log(3.0), "ln4": math.log(4.0), "1": 1.0, "0": 0.0,
             "1+ln3": 1.0 + math.log(3.0)}
    return table[s]


# ---------------------------------------------------------------- golden, hand-worked

def test_golden_hand_worked():
    data = json.load(open(os.path.join(HERE, "golden", "hand_worked.json")))
    for case in data["cases"]:
        q = bf16(case["q"])[None, :, None, :]   # [B=1, Sq, H=1, d]
        k = bf16(case["k"])[None, :, None, :]
        v = bf16(case["v"])[None, :, None, :]
        Sq, Sk, d = q.shape[1], k.shape[1], q.shape[3]
        out, lse = oracle.attention(q, k, v, B=1, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=d,
                                    causal=case["causal"], scale=_scalar(case["scale"]))
        np.testing.assert_allclose(out[0, :, 0, :], np.array(case["out"]), rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse[0, 0], [_scalar(s) for s in case["lse"]], rtol=0, atol=1e-12,
                                   err_msg=case["name"])


# ---------------------------------------------------------------- library routine

def _sdpa_reference(q, k, v, causal, scale, layout="bshd"):
    """torch.nn.functional.scaled_dot_product_attention in fp64, bottom-right causal mask."""
    if layout == "bshd":
        q, k, v = (t.permute(0, 2, 1, 3) for t in (q, k, v))
    q, k, v = (t.to(torch.float64) for t in (q, k, v))
    Hq, Hkv = q.shape[1], k.shape[1]
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    v = v.repeat_interleave(Hq // Hkv, dim=1)
    Sq, Sk = q.shape[2], k.shape[2]
    mask = None
    if causal:
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        mask = j <= i + (Sk - Sq)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    if layout == "bshd":
        o = o.permute(0, 2, 1, 3)
    return o.numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,causal,layout", [
    (1, 2, 2, 17, 17, False, "bshd"),
    (2, 4, 2, 33, 33, True, "bshd"),
    (1, 4, 1, 5, 40, False, "bhsd"),
    (1, 6, 3, 24, 31, True, "bhsd"),   # Sk > Sq causal: bottom-right
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, Sq, Sk, causal, layout):
    d = 32
    w = inputs.PrefillWorkload("t", B, Hq, Hkv, Sq, Sk, d=d, layout=layout, causal=causal, seed=11)
    q, k, v = inputs.make_prefill(w)
    scale = 1.0 / math.sqrt(d)
    out, _ = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d, layout=layout,
                              causal=causal, scale=scale)
    ref = _sdpa_reference(q, k, v, causal, scale, layout)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- the matmul form of the definition

MATMUL_SHAPES = [
    # B, Hq, Hkv, Sq, Sk, layout, causal
    (2, 8, 2, 70, 70, "bshd", True),      # GQA, causal
    (1, 6, 3, 40, 90, "bhsd", True),      # Sk > Sq: bottom-right alignment
    (1, 2, 2, 50, 20, "bshd", True),      # Sq > Sk: rows that see no key
    (2, 4, 1, 33, 129, "bhsd", False),    # MQA, cross
    (1, 3, 1, 1, 64, "bshd", False),      # one query
    (1, 2, 2, 17, 1, "bshd", False),      # one key
]


def _matmul_vs_c(impl, B, Hq, Hkv, Sq, Sk, layout, causal, row_block=16):
    w = inputs.PrefillWorkload("mm", B, Hq, Hkv, Sq, Sk, d=32, layout=layout, causal=causal, seed=61 + Sq)
    q, k, v = inputs.make_prefill(w)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=32, layout=layout, causal=causal, scale=0.21)
    o1, l1 = impl(q, k, v, row_block=row_block, **kw)
    o2, l2 = oracle.attention(q, k, v, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-13)
    assert (np.isneginf(l1) == np.isneginf(l2)).all()
    fin = np.isfinite(l2)
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", MATMUL_SHAPES, ids=[str(s) for s in MATMUL_SHAPES])
def test_matmul_form_equals_row_by_row_oracle(shape):
    """The matmul form against the row-by-row C oracle (itself pinned by the
    closed forms and SDPA above), with row blocks small enough that every
    shape spans several."""
    _matmul_vs_c(oracle.attention_matmul, *shape)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,causal,layout", [(2, 4, 2, 33, 33, True, "bshd"),
                                                          (1, 6, 3, 24, 31, True, "bhsd")])
def test_matmul_form_matches_torch_sdpa_fp64(B, Hq, Hkv, Sq, Sk, causal, layout):
    w = inputs.PrefillWorkload("t", B, Hq, Hkv, Sq, Sk, d=32, layout=layout, causal=causal, seed=11)
    q, k, v = inputs.make_prefill(w)
    out, _ = oracle.attention_matmul(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=32, layout=layout,
                                     causal=causal, scale=1.0 / math.sqrt(32), row_block=8)
    np.testing.assert_allclose(out, _sdpa_reference(q, k, v, causal, 1.0 / math.sqrt(32), layout),
                               rtol=1e-10, atol=1e-12)


MATMUL_MUTATIONS = {
    "head_map_modulo": ("for h in range(g * G, (g + 1) * G):", "for h in range(g, Hq, Hkv):"),
    "causal_top_left": ("s.masked_fill_(keys[:, :kn] > rows + (Sk - Sq), -math.inf)",
                        "s.masked_fill_(keys[:, :kn] > rows, -math.inf)"),
    "key_range_short": ("kn = min(Sk, r1 + Sk - Sq) if causal else Sk", "kn = min(Sk, r1 - 1 + Sk - Sq) if causal else Sk"),
    "scale_dropped": ("s = (qh[r0:r1] @ kg[:kn].T) * scale", "s = qh[r0:r1] @ kg[:kn].T"),
    "no_normalise": ("o = (p @ vg[:kn]) / l_sum", "o = p @ vg[:kn]"),
    "lse_sign": ("(m_sub + torch.log(l_sum))", "(m_sub - torch.log(l_sum))"),
    "value_of_query_head": ("vg = (v64[b, :, g] if bshd else v64[b, g]).contiguous()",
                            "vg = (v64[b, :, 0] if bshd else v64[b, 0]).contiguous()"),
}


@pytest.mark.parametrize("name", sorted(MATMUL_MUTATIONS))
def test_planted_matmul_form_mistake_is_caught(name):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.attention_matmul))
    old, new = MATMUL_MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new, 1), "<mutated attention_matmul>", "exec"), ns)
    bad = ns["attention_matmul"]
    caught = 0
    for shape in MATMUL_SHAPES:
        try:
            _matmul_vs_c(bad, *shape)
        except AssertionError:
            caught += 1
    assert caught, f"no pin caught the planted mistake {name}"


# ---------------------------------------------------------------- packed variable-length batches

@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_sdpa_per_sequence(causal):
    d, Hq, Hkv = 32, 4, 2
    lq, lk = (5, 0, 17, 1, 33, 6), (9, 4, 17, 1, 20, 0)
    w = inputs.VarlenWorkload("v", len(lq), Hq, Hkv, causal=causal, seed=13, lens_q=lq, lens_k=lk, d=d, pad_q=3)
    q, k, v, cu_q, cu_k = inputs.make_varlen(w)
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, Hq=Hq, Hkv=Hkv, d=d, causal=causal, scale=scale)
    for b in range(len(lq)):
        q0, k0 = int(cu_q[b]), int(cu_k[b])
        if lq[b] == 0:
            continue
        o_b = out[q0:q0 + lq[b]]
        if lk[b] == 0:
            assert (o_b == 0).all() and (lse[:, q0:q0 + lq[b]] == -np.inf).all()
            continue
        ref = _sdpa_reference(q[q0:q0 + lq[b]][None], k[k0:k0 + lk[b]][None], v[k0:k0 + lk[b]][None], causal,
                              scale)[0]
        # causal rows that see no key (i < Lq - Lk) are O = 0, lse = -inf; SDPA gives NaN there
        blind = max(0, lq[b] - lk[b]) if causal else 0
        np.testing.assert_allclose(o_b[blind:], ref[blind:], rtol=1e-10, atol=1e-12)
        assert (o_b[:blind] == 0).all() and (lse[:, q0:q0 + blind] == -np.inf).all()
        assert np.isfinite(lse[:, q0 + blind:q0 + lq[b]]).all()
    assert np.isnan(out[-3:]).all() and np.isnan(lse[:, -3:]).all()   # rows of no sequence


def test_varlen_equal_lengths_is_the_dense_batch():
    B, L, Hq, Hkv, d = 3, 20, 4, 2, 16
    w = inputs.PrefillWorkload("t", B, Hq, Hkv, L, L, d=d, causal=True, seed=14)
    q, k, v = inputs.make_prefill(w)
    scale = 0.25
    dense_o, dense_l = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=L, Sk=L, d=d, causal=True, scale=scale)
    cu = torch.arange(0, (B + 1) * L, L, dtype=torch.int32)
    vo, vl = oracle.attention_varlen(q.reshape(B * L, Hq, d), k.reshape(B * L, Hkv, d), v.reshape(B * L, Hkv, d),
                                     cu, cu, Hq=Hq, Hkv=Hkv, d=d, causal=True, scale=scale)
    np.testing.assert_array_equal(vo, dense_o.reshape(B * L, Hq, d))
    np.testing.assert_array_equal(vl, dense_l.transpose(1, 0, 2).reshape(Hq, B * L))


# ---------------------------------------------------------------- prefill against a paged cache

@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_of_one_token_is_decode(causal):
    # a chunk of one query per sequence sees its whole cache either way: it is
    # the decode step, which the C oracle gathers from the pages on its own
    w = inputs.PagedPrefillWorkload("p", 5, 4, 2, chunks=(1,) * 5, contexts=(0, 15, 16, 40, 100), seed=15,
                                    max_blocks=8, d=32)
    q, kp, vp, table, lens, cu_q = inputs.make_paged_prefill(w)
    out, lse = oracle.attention_paged(q, kp, vp, table, lens, cu_q, Hq=4, Hkv=2, d=32, causal=causal, scale=0.2)
    ref_o, ref_l = oracle.decode_paged(q, kp, vp, table, lens, scale=0.2)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.T, ref_l, rtol=1e-12, atol=1e-13)


def test_paged_prefill_equals_attention_on_the_scattered_cache():
    # scatter contiguous K, V into pages through a shuffled table; the paged
    # prefill must equal plain attention on the contiguous tensors
    d, Hq, Hkv, ps = 16, 4, 2, 16
    lq, lk = (7, 20, 1), (30, 20, 17)
    g = torch.Generator().manual_seed(16)
    npages = [(L + ps - 1) // ps for L in lk]
    perm = torch.randperm(sum(npages) + 3, generator=g)          # three unused pages
    kp = torch.randn(sum(npages) + 3, ps, Hkv, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(sum(npages) + 3, ps, Hkv, d, generator=g).to(torch.bfloat16)
    table = torch.full((3, 4), -1, dtype=torch.int32)
    ks, vs, off = [], [], 0
    for b, L in enumerate(lk):
        k_b = torch.randn(L, Hkv, d, generator=g).to(torch.bfloat16)
        v_b = torch.randn(L, Hkv, d, generator=g).to(torch.bfloat16)
        for t in range(L):
            page = int(perm[off + t // ps])
            table[b, t // ps] = page
            kp[page, t % ps] = k_b[t]
            vp[page, t % ps] = v_b[t]
        off += npages[b]
        ks.append(k_b)
        vs.append(v_b)
    q = torch.randn(sum(lq), Hq, d, generator=g).to(torch.bfloat16)
    cu_q = torch.tensor([0, 7, 27, 28], dtype=torch.int32)
    out, lse = oracle.attention_paged(q, kp, vp, table, torch.tensor(lk), cu_q, Hq=Hq, Hkv=Hkv, d=d, causal=True,
                                      scale=0.3)
    for b in range(3):
        q0 = int(cu_q[b])
        ref = _sdpa_reference(q[q0:q0 + lq[b]][None], ks[b][None], vs[b][None], True, 0.3)[0]
        np.testing.assert_allclose(out[q0:q0 + lq[b]], ref, rtol=1e-10, atol=1e-12)


def test_paged_gather_rejects_a_bad_table_entry():
    kp = torch.zeros(2, 16, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.gather_pages(kp, [0, 5], 20)


# ---------------------------------------------------------------- append + decode

def test_append_then_decode_writes_one_slot_and_attends_over_it():
    d, Hq, Hkv = 16, 4, 2
    w = inputs.DecodeWorkload("a", B=4, Hq=Hq, Hkv=Hkv, d=d, max_blocks=4, seed=17)
    lens = [0, 15, 16, 40]
    q, kp, vp, table, sl = inputs.make_decode(w, seqlens=[L + 1 for L in lens])   # pages for L + 1 tokens
    g = torch.Generator().manual_seed(18)
    k_new = torch.randn(4, Hkv, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(4, Hkv, d, generator=g).to(torch.bfloat16)
    out, lse, kp2, vp2 = oracle.decode_paged_append(q, k_new, v_new, kp, vp, table, lens, scale=0.25)
    changed = (kp2.view(torch.int16) != kp.view(torch.int16)).any(dim=(2, 3))
    for b, L in enumerate(lens):
        # the gathered cache's token L is the new one, and nothing else moved
        assert torch.equal(oracle.gather_pages(kp2, table[b], L + 1)[L], k_new[b])
        assert torch.equal(oracle.gather_pages(vp2, table[b], L + 1)[L], v_new[b])
        assert torch.equal(oracle.gather_pages(kp2, table[b], L), oracle.gather_pages(kp, table[b], L))
    assert int(changed.sum()) <= len(lens)
    # attention over L + 1 keys, checked against SDPA on the gathered keys
    for b, L in enumerate(lens):
        kb = oracle.gather_pages(kp2, table[b], L + 1)[None]
        vb = oracle.gather_pages(vp2, table[b], L + 1)[None]
        ref = _sdpa_reference(q[b][None, None], kb, vb, False, 0.25)[0, 0]
        np.testing.assert_allclose(out[b], ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_v():
    B, H, S, d = 1, 2, 37, 16
    q = rand_bf16((B, S, H, d), 1)
    k0 = rand_bf16((1, 1, H, d), 2)
    k = k0.expand(B, S, H, d).contiguous()
    v = rand_bf16((B, S, H, d), 3)
    scale = 0.3
    out, lse = oracle.attention(q, k, v, B=B, Hq=H, Hkv=H, Sq=S, Sk=S, d=d, scale=scale)
    mean_v = f64(v).mean(axis=1)                       # [B, H, d]
    np.testing.assert_allclose(out, np.broadcast_to(mean_v[:, None], out.shape), rtol=0, atol=1e-12)
    s = scale * np.einsum("bihc,hc->bhi", f64(q), f64(k0)[0, 0])
    np.testing.assert_allclose(lse, s + math.log(S), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,Sq,Sk", [(False, 9, 13), (True, 13, 13), (True, 5, 13)])
def test_zero_scale_counts_visible_keys(causal, Sq, Sk):
    d = 8
    q, k, v = rand_bf16((1, Sq, 1, d), 4), rand_bf16((1, Sk, 1, d), 5), rand_bf16((1, Sk, 1, d), 6)
    out, lse = oracle.attention(q, k, v, B=1, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=d, causal=causal, scale=0.0)
    vv = f64(v)[0, :, 0, :]
    for i in range(Sq):
        n = min(Sk, i + 1 + Sk - Sq) if causal else Sk
        np.testing.assert_allclose(out[0, i, 0], vv[:n].mean(axis=0), rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-12


def test_dominant_score_selects_its_value_row():
    d, Sk = 16, 20
    q = bf16(np.eye(1, d, 0))[None, :, None, :]                # q = e0
    k = np.zeros((Sk, d), np.float32)
    k[:, 1] = 1.0
    jstar = 7
    k[jstar, 0] = 64.0                                          # score gap of 64 * scale
    v = rand_bf16((1, Sk, 1, d), 7)
    scale = 1.0
    out, lse = oracle.attention(q, bf16(k)[None, :, None, :], v, B=1, Hq=1, Hkv=1, Sq=1, Sk=Sk,
                                d=d, scale=scale)
    np.testing.assert_allclose(out[0, 0, 0], f64(v)[0, jstar, 0], rtol=0, atol=1e-20)
    assert abs(lse[0, 0, 0] - 64.0) < 1e-12


def test_causal_row_zero_is_first_value():
    B, H, S, d = 2, 3, 19, 16
    q, k, v = rand_bf16((B, S, H, d), 8), rand_bf16((B, S, H, d), 9), rand_bf16((B, S, H, d), 10)
    scale = 0.25
    out, lse = oracle.attention(q, k, v, B=B, Hq=H, Hkv=H, Sq=S, Sk=S, d=d, causal=True, scale=scale)
    np.testing.assert_array_equal(out[:, 0], f64(v)[:, 0])
    s00 = scale * np.einsum("bhc,bhc->bh", f64(q)[:, 0], f64(k)[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-12)


def test_single_key_returns_it_for_every_row():
    Sq, d = 11, 16
    q, k, v = rand_bf16((1, Sq, 2, d), 11), rand_bf16((1, 1, 2, d), 12), rand_bf16((1, 1, 2, d), 13)
    out, _ = oracle.attention(q, k, v, B=1, Hq=2, Hkv=2, Sq=Sq, Sk=1, d=d, scale=0.7)
    np.testing.assert_array_equal(out, np.broadcast_to(f64(v)[:, :1], out.shape))


def test_constant_value_vector_is_returned():
    S, d = 23, 16
    q, k = rand_bf16((1, S, 2, d), 14, std=3.0), rand_bf16((1, S, 2, d), 15, std=3.0)
    c = rand_bf16((d,), 16)
    v = c.expand(1, S, 2, d).contiguous()
    out, _ = oracle.attention(q, k, v, B=1, Hq=2, Hkv=2, Sq=S, Sk=S, d=d, causal=True, scale=0.5)
    np.testing.assert_allclose(out, np.broadcast_to(f64(c), out.shape), rtol=1e-14, atol=0)


def test_probability_rows_sum_to_one():
    S, d = 29, 16
    q, k = rand_bf16((1, S, 1, d), 17, std=4.0), rand_bf16((1, S, 1, d), 18, std=4.0)
    for i in (0, 5, 28):
        for causal in (False, True):
            p = oracle.attention_probs_row(q, k, 0, 0, i, B=1, Hq=1, Hkv=1, Sq=S, Sk=S, d=d,
                                           causal=causal, scale=0.5)
            assert abs(p.sum() - 1.0) < 1e-12
            assert (p >= 0).all()
            if causal:
                assert (p[i + 1:] == 0).all()


def _sdpa_weights(q, k, causal, scale):
    """Attention weights P from torch's scaled_dot_product_attention in fp64:
    with the identity matrix as V (one value column per key) its output row
    is the row of P itself.  q [Sq, d], k [Sk, d]; bottom-right causal mask."""
    q, k = q.to(torch.float64), k.to(torch.float64)
    Sq, Sk = q.shape[0], k.shape[0]
    eye = torch.eye(Sk, dtype=torch.float64)
    mask = None
    if causal:
        mask = torch.arange(Sk)[None, :] <= torch.arange(Sq)[:, None] + (Sk - Sq)
    return torch.nn.functional.scaled_dot_product_attention(q[None, None], k[None, None], eye[None, None],
                                                            attn_mask=mask, scale=scale)[0, 0].numpy()


@pytest.mark.parametrize("Sq,Sk,causal,scale", [(29, 29, False, 0.5), (29, 29, True, 0.5), (7, 40, True, 0.13),
                                                  (12, 9, False, 1.7)])
def test_probability_row_matches_sdpa_weights(Sq, Sk, causal, scale):
    d, Hq, Hkv = 16, 4, 2
    q, k = rand_bf16((1, Sq, Hq, d), 41, std=3.0), rand_bf16((1, Sk, Hkv, d), 42, std=3.0)
    for h in (0, 1, 3):     # h = 1 tells h / G from h % Hkv apart
        ref = _sdpa_weights(q[0, :, h], k[0, :, h // 2], causal, scale)
        for i in (0, Sq // 2, Sq - 1):
            p = oracle.attention_probs_row(q, k, 0, h, i, B=1, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d,
                                           causal=causal, scale=scale)
            np.testing.assert_allclose(p, ref[i], rtol=1e-10, atol=1e-14, err_msg=f"h={h} i={i}")


def test_fully_masked_rows_are_zero_with_minus_inf_lse():
    Sq, Sk, d = 10, 4, 8          # causal with Sq > Sk: rows i < Sq - Sk see no key
    q, k, v = rand_bf16((1, Sq, 1, d), 19), rand_bf16((1, Sk, 1, d), 20), rand_bf16((1, Sk, 1, d), 21)
    out, lse = oracle.attention(q, k, v, B=1, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=d, causal=True, scale=1.0)
    for i in range(Sq):
        if i < Sq - Sk:
            assert (out[0, i, 0] == 0).all() and lse[0, 0, i] == -math.inf
        else:
            assert np.isfinite(lse[0, 0, i])
    # the last row sees every key: equals the non-causal last row
    ref, _ = oracle.attention(q, k, v, B=1, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=d, causal=False, scale=1.0)
    np.testing.assert_array_equal(out[0, -1], ref[0, -1])


# ---------------------------------------------------------------- invariants

def test_gqa_equals_replicated_kv_heads():
    B, Hq, Hkv, S, d = 2, 8, 2, 21, 16
    w = inputs.PrefillWorkload("g", B, Hq, Hkv, S, S, d=d, causal=True, seed=22)
    q, k, v = inputs.make_prefill(w)
    out, lse = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=S, Sk=S, d=d, causal=True, scale=0.2)
    G = Hq // Hkv
    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    out2, lse2 = oracle.attention(q, kr, vr, B=B, Hq=Hq, Hkv=Hq, Sq=S, Sk=S, d=d, causal=True, scale=0.2)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_layouts_agree_after_permute():
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 13, 17, 16
    w = inputs.PrefillWorkload("l", B, Hq, Hkv, Sq, Sk, d=d, layout="bshd", causal=True, seed=23)
    q, k, v = inputs.make_prefill(w)
    q2, k2, v2 = inputs.make_prefill(w.with_(layout="bhsd"))
    assert torch.equal(q.permute(0, 2, 1, 3), q2)
    o1, l1 = oracle.attention(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d, layout="bshd",
                              causal=True, scale=0.3)
    o2, l2 = oracle.attention(q2, k2, v2, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d, layout="bhsd",
                              causal=True, scale=0.3)
    np.testing.assert_array_equal(o1, o2.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(l1, l2)


def test_key_permutation_invariance_noncausal():
    S, Sk, d = 7, 31, 16
    q, k, v = rand_bf16((1, S, 2, d), 24), rand_bf16((1, Sk, 2, d), 25), rand_bf16((1, Sk, 2, d), 26)
    perm = torch.randperm(Sk, generator=torch.Generator().manual_seed(27))
    o1, l1 = oracle.attention(q, k, v, B=1, Hq=2, Hkv=2, Sq=S, Sk=Sk, d=d, scale=0.4)
    o2, l2 = oracle.attention(q, k[:, perm].contiguous(), v[:, perm].contiguous(), B=1, Hq=2, Hkv=2,
                              Sq=S, Sk=Sk, d=d, scale=0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (3, 3), (17, 17), (128, 128), (130, 130), (3, 17), (17, 130)])
@pytest.mark.parametrize("tile", [1, 5, 64])
def test_tiled_online_softmax_equals_full(Sq, Sk, tile):
    d = 16
    causal = Sq == Sk and Sq % 2 == 1
    q, k, v = rand_bf16((1, Sq, 1, d), 30, 2.0), rand_bf16((1, Sk, 1, d), 31, 2.0), rand_bf16((1, Sk, 1, d), 32)
    rows = [(0, 0, i) for i in range(Sq)]
    kw = dict(B=1, Hq=1, Hkv=1, Sq=Sq, Sk=Sk, d=d, causal=causal, scale=0.6)
    o_full, l_full = oracle.attention_rows(q, k, v, rows, **kw)
    o_tile, l_tile = oracle.attention_tiled_rows(q, k, v, rows, tile=tile, **kw)
    np.testing.assert_allclose(o_tile, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_tile, l_full, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_split_and_merge_equals_unsplit(nsplit):
    Sq, Sk, d = 9, 50, 16
    q, k, v = rand_bf16((1, Sq, 2, d), 33, 2.0), rand_bf16((1, Sk, 2, d), 34, 2.0), rand_bf16((1, Sk, 2, d), 35)
    rows = [(0, h, i) for h in range(2) for i in range(Sq)]
    kw = dict(B=1, Hq=2, Hkv=2, Sq=Sq, Sk=Sk, d=d, causal=True, scale=0.5)
    o_full, l_full = oracle.attention_rows(q, k, v, rows, **kw)
    bounds = np.linspace(0, Sk, nsplit + 1).astype(int)
    parts = [oracle.attention_rows(q, k, v, rows, key_range=(bounds[s], bounds[s + 1]), **kw)
             for s in range(nsplit)]
    o_m, l_m = oracle.lse_merge(np.stack([p[1] for p in parts]), np.stack([p[0] for p in parts]))
    np.testing.assert_allclose(o_m, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_m, l_full, rtol=0, atol=1e-12)


def test_merge_of_empty_partials():
    lse_s = np.array([[-np.inf], [-np.inf]])
    o_s = np.zeros((2, 1, 4))
    o, l = oracle.lse_merge(lse_s, o_s)
    assert l[0] == -np.inf and (o == 0).all()


# ---------------------------------------------------------------- paged decode

def _gather_contiguous(k_pages, v_pages, table, seqlens, b):
    L = int(seqlens[b])
    ids = [int(table[b, t // 16]) for t in range(L)]
    slots = [t % 16 for t in range(L)]
    k = k_pages[ids, slots][None]   # [1, L, Hkv, d]
    v = v_pages[ids, slots][None]
    return k.contiguous(), v.contiguous()


def test_paged_decode_equals_contiguous_prefill_oracle():
    w = inputs.DecodeWorkload("small", B=3, Hq=8, Hkv=2, d=16, max_blocks=8, len_lo=1, len_hi=120, seed=40)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[1, 17, 128])
    out, lse = oracle.decode_paged(q, kp, vp, table, lens, scale=0.3)
    for b in range(w.B):
        k, v = _gather_contiguous(kp, vp, table, lens, b)
        L = int(lens[b])
        qb = q[b][None, None]             # [1, Sq=1, Hq, d]
        o2, l2 = oracle.attention(qb, k, v, B=1, Hq=w.Hq, Hkv=w.Hkv, Sq=1, Sk=L, d=w.d, scale=0.3)
        np.testing.assert_array_equal(out[b], o2[0, 0])
        np.testing.assert_array_equal(lse[b], l2[0, :, 0])


def test_paged_decode_zero_length_and_padding():
    w = inputs.DecodeWorkload("z", B=2, Hq=4, Hkv=4, d=16, max_blocks=4, seed=41)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[0, 16])
    assert (table[0] == -1).all() and (table[1, 1:] == -1).all()
    out, lse = oracle.decode_paged(q, kp, vp, table, lens, scale=0.3)
    assert (out[0] == 0).all() and (lse[0] == -np.inf).all()
    assert np.isfinite(lse[1]).all()


def test_paged_decode_rejects_bad_block_table():
    w = inputs.DecodeWorkload("z", B=1, Hq=4, Hkv=4, d=16, max_blocks=4, seed=42)
    q, kp, vp, table, lens = inputs.make_decode(w, seqlens=[20])
    table[0, 1] = kp.shape[0]           # one past the pool
    with pytest.raises(ValueError):
        oracle.decode_paged(q, kp, vp, table, lens, scale=0.3)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rtne_matches_torch_on_float_values():
    g = torch.Generator().manual_seed(50)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(20000, generator=g) * 8)
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16_rtne(float(t)) for t in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_rtne_ties_go_to_even():
    assert oracle.round_bf16_rtne(1.0) == 0x3F80
    assert oracle.round_bf16_rtne(1.0 + 2.0 ** -8) == 0x3F80          # tie, even stays
    assert oracle.round_bf16_rtne(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie, rounds up to even
    assert oracle.round_bf16_rtne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81   # just above the tie
    assert oracle.round_bf16_rtne(-2.0) == 0xC000
    assert oracle.round_bf16_rtne(float("inf")) == 0x7F80


def _random_float32(seed, n=20000):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, generator=g, dtype=torch.float32) * torch.exp(torch.randn(n, generator=g) * 8)
    extra = torch.tensor([1e-39, -3e-40, 1.5e-45, 3.3e38, -3.39e38, 0.0, -0.0], dtype=torch.float32)
    return torch.cat([x, extra]).numpy()


def test_bf16_rtz_is_truncation_of_the_float32_pattern():
    # For a binary32 value, dropping the low 16 bits of its pattern is rounding
    # the magnitude toward zero at bf16 precision.
    x = _random_float32(51)
    want = (x.view(np.uint32) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(oracle.round_bf16_array(x.astype(np.float64), "rtz"), want)


def test_bf16_rtna_is_half_unit_added_to_the_float32_magnitude():
    # Adding half a bf16 unit (0x8000) to the magnitude bits and dropping the low
    # 16 bits rounds to nearest with ties away from zero (a carry moves the exponent).
    x = _random_float32(52)
    u = x.view(np.uint32).astype(np.uint64)
    want = (((u & 0x7FFFFFFF) + 0x8000) >> 16).astype(np.uint16) | ((u >> 16) & 0x8000).astype(np.uint16)
    np.testing.assert_array_equal(oracle.round_bf16_array(x.astype(np.float64), "rtna"), want)


def test_bf16_rtne_array_matches_torch():
    x = _random_float32(53)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.round_bf16_array(x.astype(np.float64), "rtne"), want)
    assert all(oracle.round_bf16(float(t), "rtne") == oracle.round_bf16_rtne(float(t)) for t in x[:200])


@pytest.mark.parametrize("x,rtne,rtna,rtz", [
    (1.0 + 2.0 ** -8, 0x3F80, 0x3F81, 0x3F80),            # tie below an odd neighbour
    (1.0 + 3 * 2.0 ** -8, 0x3F82, 0x3F82, 0x3F81),        # tie below an even neighbour
    (-(1.0 + 2.0 ** -8), 0xBF80, 0xBF81, 0xBF80),         # sign-symmetric
    (64.25, 0x4280, 0x4281, 0x4280),                      # quarter steps at 64: spacing 0.5
    (-64.75, 0xC282, 0xC282, 0xC281),
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81, 0x3F81, 0x3F80),  # just above a tie: one rounding, from the double
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80, 0x3F80, 0x3F80),  # just below
    (3.0e38, 0x7F62, 0x7F62, 0x7F61),
    (3.4e38, 0x7F80, 0x7F80, 0x7F7F),                     # past the largest bf16: RTZ saturates
    (1e300, 0x7F80, 0x7F80, 0x7F7F),
    (float("inf"), 0x7F80, 0x7F80, 0x7F80),
    (float("-inf"), 0xFF80, 0xFF80, 0xFF80),
    (float("nan"), 0x7FC0, 0x7FC0, 0x7FC0),
    (2.0 ** -133, 0x0001, 0x0001, 0x0001),                # smallest bf16 subnormal
    (1.5 * 2.0 ** -133, 0x0002, 0x0002, 0x0001),          # subnormal tie
])
def test_bf16_modes_hand_worked(x, rtne, rtna, rtz):
    assert oracle.round_bf16(x, "rtne") == rtne
    assert oracle.round_bf16(x, "rtna") == rtna
    assert oracle.round_bf16(x, "rtz") == rtz


# ---------------------------------------------------------------- mutation tests

MUTATIONS = {
    # wrong GQA head map
    "head_map_modulo": ("const int64_t g = h / (p->Hq / p->Hkv);", "const int64_t g = h % p->Hkv;"),
    # top-left causal alignment instead of bottom-right
    "causal_top_left": ("int64_t lim = i + Sk - Sq;", "int64_t lim = i;"),
    # sign error in the exponent
    "exp_sign": ("oreal w = exp(scores[j] - M);", "oreal w = exp(M - scores[j]);"),
    # dropped normalisation
    "no_normalise": ("for (int64_t c = 0; c < d; ++c) o[c] = acc[c] / L;",
                     "for (int64_t c = 0; c < d; ++c) o[c] = acc[c];"),
    # lse off by the log term
    "lse_sign": ("*lse = M + log(L);", "*lse = M - log(L);"),
    # transposed operand: key index used for the value row
    "value_from_query_row": (
        "acc[c] += w * (oreal)bf16_to_double(p->v[offset_of(p->layout, b, j, g, c, p->Sk, p->Hkv, d)]);",
        "acc[c] += w * (oreal)bf16_to_double(p->v[offset_of(p->layout, b, i < p->Sk ? i : 0, g, c, p->Sk, p->Hkv, d)]);"),
}


def _pin_suite():
    """The pins that exercise the whole-row path, run against whichever oracle is loaded."""
    failures = []
    for fn in (test_golden_hand_worked,
               lambda: test_matches_torch_sdpa_fp64(1, 6, 3, 24, 31, True, "bhsd"),
               lambda: test_matches_torch_sdpa_fp64(2, 4, 2, 33, 33, True, "bshd"),
               test_identical_keys_give_mean_of_v,
               lambda: test_zero_scale_counts_visible_keys(True, 5, 13),
               test_gqa_equals_replicated_kv_heads):
        try:
            fn()
        except AssertionError:
            failures.append(fn)
    return failures


ROUNDING_MUTATIONS = {
    "rtna_ties_to_even": ("mode == 1 ? round(units)", "mode == 1 ? nearbyint(units)"),
    "rtz_rounds_to_nearest": ("mode == 2 ? trunc(units)", "mode == 2 ? round(units)"),
    "rtz_overflows": ("if (mode == 2 && r > 0x1.fep127) r = 0x1.fep127;", ";"),
    "quantum_off_by_one": ("int qexp = e - 8;", "int qexp = e - 9;"),
}


def _rounding_pin_suite():
    failures = []
    cases = [(1.0 + 2.0 ** -8, 0x3F80, 0x3F81, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82, 0x3F82, 0x3F81),
             (3.4e38, 0x7F80, 0x7F80, 0x7F7F), (64.25, 0x4280, 0x4281, 0x4280), (1e300, 0x7F80, 0x7F80, 0x7F7F)]
    for fn in (test_bf16_rtz_is_truncation_of_the_float32_pattern,
               test_bf16_rtna_is_half_unit_added_to_the_float32_magnitude,
               test_bf16_rtne_array_matches_torch,
               *[(lambda c=c: test_bf16_modes_hand_worked(*c)) for c in cases]):
        try:
            fn()
        except AssertionError:
            failures.append(fn)
    return failures


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(ROUNDING_MUTATIONS))
def test_planted_rounding_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = ROUNDING_MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(old, new, 1))
    so = tmp_path / "libbad.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(bad), "-lm"], check=True)
    with oracle.use_library(str(so)):
        failures = _rounding_pin_suite()
    assert failures, f"no pin caught the planted mistake {name}"
    assert not _rounding_pin_suite()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(old, new, 1))
    so = tmp_path / "libbad.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(bad), "-lm"], check=True)
    with oracle.use_library(str(so)):
        failures = _pin_suite()
    assert failures, f"no pin caught the planted mistake {name}"
    # and the real oracle passes the same suite
    assert not _pin_suite()


PROBS_MUTATIONS = {
    # scale dropped from the probability row's scores
    "probs_no_scale": ("probs[j] = scale * dot;", "probs[j] = dot;"),
    # wrong head map in the probability row
    "probs_head_map": ("const int64_t g = h / (Hq / Hkv);\n    int64_t last", "const int64_t g = h % Hkv;\n    int64_t last"),
    # unnormalised probabilities
    "probs_no_normalise": ("probs[j] = exp(probs[j] - M) / L;", "probs[j] = exp(probs[j] - M);"),
}


def _probs_pin_suite():
    failures = []
    for fn in (lambda: test_probability_row_matches_sdpa_weights(29, 29, True, 0.5),
               lambda: test_probability_row_matches_sdpa_weights(7, 40, True, 0.13)):
        try:
            fn()
        except AssertionError:
            failures.append(fn)
    return failures


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(PROBS_MUTATIONS))
def test_planted_probability_row_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = PROBS_MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(old, new, 1))
    so = tmp_path / "libbad.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(bad), "-lm"], check=True)
    with oracle.use_library(str(so)):
        failures = _probs_pin_suite()
    assert failures, f"no pin caught the planted mistake {name}"
    assert not _probs_pin_suite()


# ---------------------------------------------------------------- the oracle's own numerics

@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_fp32_build_agrees_with_fp64_far_inside_the_tolerance(tmp_path):
    """The same oracle source built with ORACLE_REAL=float: on workload-like
    inputs (unit normal, and peaked rows from keys scaled by 8) its results
    differ from the fp64 build by at most 5% of the parity tolerance
    (4e-3 + 8e-3 |O|, 1e-3 on lse); the fp64 build's own rounding error is
    about 2^29 times smaller still, so it cannot decide a parity verdict."""
    so = tmp_path / "liboracle32.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-DORACLE_REAL=float", "-o", str(so),
                    os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c"), "-lm"], check=True)
    cases = [inputs.PrefillWorkload("f32a", 1, 4, 2, 700, 700, causal=True, seed=51),
             inputs.PrefillWorkload("f32b", 1, 2, 2, 300, 1500, causal=False, seed=52)]
    for w in cases:
        q, k, v = inputs.make_prefill(w)
        if w.name == "f32b":       # a few keys scaled by 8: peaked softmax rows
            k = k.float()
            k[:, ::97] *= 8
            k = k.to(torch.bfloat16)
        kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, d=w.d, layout=w.layout, causal=w.causal, scale=w.scale)
        o64, l64 = oracle.attention(q, k, v, **kw)
        with oracle.use_library(str(so)):
            o32, l32 = oracle.attention(q, k, v, **kw)
        assert not np.array_equal(o32, o64), "the float build should round differently"
        excess = np.abs(o32 - o64) / (4e-3 + 8e-3 * np.abs(o64))
        # at most 5% of either tolerance
        assert excess.max() < 0.05, f"{w.name}: fp32 build uses {excess.max():.3g} of the tolerance"
        assert np.abs(l32 - l64).max() < 5e-5, f"{w.name}: lse differs by {np.abs(l32 - l64).max():.3g}"
