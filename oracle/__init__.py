"""Plain fp64 CPU oracle for exact attention and paged decode.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the CUDA
library and its Python binding) never imports this package, and this package
never imports the product: they share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision,
OpenMP over rows); this module compiles it with gcc on first use and wraps it
with numpy.  Inputs are bf16 bit patterns (``numpy.uint16``), widened to
double exactly inside the C code.  One function is written here instead:
``attention_matmul``, the same definition with its two contractions as fp64
matrix products (plain torch CPU ops), for checking whole full-size outputs;
it shares no code with the C functions and is pinned against them.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double
_p = ctypes.c_void_p


class use_library:
    """Temporarily route every oracle call to another compiled copy (tests only).

    The mutation tests compile deliberately broken copies of attn_oracle.c and
    check that the pins notice; this swaps the loaded library for the duration
    of a ``with`` block.
    """

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in dir(self.saved):
            if name.startswith("oracle_"):
                f, g = getattr(self.saved, name), getattr(lib, name)
                g.argtypes, g.restype = f.argtypes, f.restype
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (gcc, -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_num_threads.restype = _int
            lib.oracle_attention.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                             _int, _int, _dbl, _p, _p]
            lib.oracle_attention_rows.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                                  _int, _int, _dbl, _i64, _p, _i64, _i64, _p, _p]
            lib.oracle_attention_probs_row.argtypes = [_p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                                       _int, _int, _dbl, _i64, _i64, _i64, _p]
            lib.oracle_attention_tiled_rows.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                                        _int, _int, _dbl, _i64, _i64, _p, _p, _p]
            lib.oracle_lse_merge.argtypes = [_i64, _i64, _i64, _p, _p, _p, _p]
            lib.oracle_decode_paged.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64,
                                                _i64, _i64, _i64, _dbl, _p, _p]
            lib.oracle_round_bf16_rtne.argtypes = [_dbl]
            lib.oracle_round_bf16_rtne.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [_dbl, _int]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16_array.argtypes = [_p, _p, _i64, _int]
            lib.oracle_round_bf16_array.restype = _int
            for name in ("oracle_attention", "oracle_attention_rows", "oracle_attention_probs_row",
                         "oracle_attention_tiled_rows", "oracle_lse_merge", "oracle_decode_paged"):
                getattr(lib, name).restype = _int
            _lib = lib
    return _lib


LAYOUTS = {"bshd": 0, "bhsd": 1}


def _bits(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 bit array (accepts torch bf16 or uint16 numpy)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch  # local: only needed when handed a torch tensor
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected its arguments (code {rc})")


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return _load().oracle_num_threads()


def attention(q, k, v, *, B, Hq, Hkv, Sq, Sk, d=128, layout="bshd", causal=False, scale):
    """Full softmax(Q K^T * scale [+causal]) V in fp64.

    Returns (out, lse): out in q's layout as float64, lse as [B, Hq, Sq] float64.
    """
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    lay = LAYOUTS[layout]
    shape = (B, Sq, Hq, d) if lay == 0 else (B, Hq, Sq, d)
    out = np.empty(shape, np.float64)
    lse = np.empty((B, Hq, Sq), np.float64)
    _check(lib.oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Sk, d, lay,
                                int(bool(causal)), float(scale), _ptr(out), _ptr(lse)), "attention")
    return out, lse


def _f64_tensor(a):
    """bf16 data (a torch bf16 tensor or uint16 bit patterns) as a float64 CPU tensor (exact)."""
    import torch
    if isinstance(a, torch.Tensor):
        return a.detach().cpu().to(torch.float64)
    bits = np.ascontiguousarray(a)
    if bits.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {bits.dtype}")
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)


def attention_matmul(q, k, v, *, B, Hq, Hkv, Sq, Sk, d=128, layout="bshd", causal=False, scale, row_block=1024):
    """The definition attention() computes, with its two contractions done as
    fp64 matrix products on the CPU (torch, all cores): for each batch b, head h
    (kv head g = h // (Hq / Hkv)) and block of query rows,

        S   = scale * Q K_g^T, with S[i, j] = -inf where key j is not visible to
              row i (causal: j > i + Sk - Sq, bottom-right alignment),
        M   = max_j S[i, j],      P = exp(S - M),      L = sum_j P[i, j],
        O   = (P V_g) / L,        lse = M + ln L,

    and a row that sees no key gives O = 0, lse = -inf.  The matrix product is
    a library step of the definition; a block of rows is only a batch of
    independent rows, and its product runs over the keys [0, kn) that some
    row of the block may see (the rest would only be masked); nothing is
    tiled over keys or reordered.  It exists for
    parity checks of whole full-size outputs, where the row-by-row C code would
    take minutes.  Returns (out in q's layout, lse [B, Hq, Sq]) as float64 numpy.
    """
    import torch
    q64, k64, v64 = _f64_tensor(q), _f64_tensor(k), _f64_tensor(v)
    bshd = LAYOUTS[layout] == 0
    G = Hq // Hkv
    out = torch.empty((B, Sq, Hq, d) if bshd else (B, Hq, Sq, d), dtype=torch.float64)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float64)
    keys = torch.arange(Sk)[None, :]
    for b in range(B):
        for g in range(Hkv):
            kg = (k64[b, :, g] if bshd else k64[b, g]).contiguous()   # [Sk, d]
            vg = (v64[b, :, g] if bshd else v64[b, g]).contiguous()
            for h in range(g * G, (g + 1) * G):
                qh = (q64[b, :, h] if bshd else q64[b, h]).contiguous()  # [Sq, d]
                for r0 in range(0, Sq, row_block):
                    r1 = min(Sq, r0 + row_block)
                    # keys [0, kn) are the ones any row of the block may see
                    kn = min(Sk, r1 + Sk - Sq) if causal else Sk
                    if kn <= 0:
                        if bshd:
                            out[b, r0:r1, h] = 0.0
                        else:
                            out[b, h, r0:r1] = 0.0
                        lse[b, h, r0:r1] = -math.inf
                        continue
                    s = (qh[r0:r1] @ kg[:kn].T) * scale
                    if causal:
                        rows = torch.arange(r0, r1)[:, None]
                        s.masked_fill_(keys[:, :kn] > rows + (Sk - Sq), -math.inf)
                    m = s.amax(dim=1, keepdim=True)
                    none = torch.isneginf(m)                       # rows that see no key
                    m_sub = torch.where(none, torch.zeros_like(m), m)
                    p = s.sub_(m_sub).exp_()                       # masked keys: exp(-inf) = 0
                    l_sum = p.sum(dim=1, keepdim=True)
                    o = (p @ vg[:kn]) / l_sum
                    o[none[:, 0]] = 0.0
                    if bshd:
                        out[b, r0:r1, h] = o
                    else:
                        out[b, h, r0:r1] = o
                    lse[b, h, r0:r1] = (m_sub + torch.log(l_sum))[:, 0]
    return out.numpy(), lse.numpy()


def attention_varlen(q, k, v, cu_q, cu_k, *, Hq, Hkv, d=128, causal=False, scale, seqs=None, dense=None):
    """A packed variable-length batch, one sequence at a time.

    q [total_q, Hq, d], k and v [total_k, Hkv, d] (bf16); sequence b owns rows
    cu_q[b] .. cu_q[b+1]-1 of q and cu_k[b] .. cu_k[b+1]-1 of k and v, and its
    rows attend only to its own keys: each sequence is the plain attention
    above with B = 1, Sq = its query length and Sk = its key length (causal
    alignment bottom-right within the sequence).  A sequence with queries but
    no keys gives O = 0 and lse = -inf (a row that sees no key).

    Returns (out [total_q, Hq, d] float64, lse [Hq, total_q] float64); rows
    that belong to no sequence (or to a sequence not in `seqs`, when given)
    are NaN.  `dense` picks the dense implementation used per sequence:
    attention (default) or attention_matmul.
    """
    dense = attention if dense is None else dense
    cu_q = [int(x) for x in cu_q]
    cu_k = [int(x) for x in cu_k]
    total_q = q.shape[0]
    out = np.full((total_q, Hq, d), np.nan)
    lse = np.full((Hq, total_q), np.nan)
    for b in (range(len(cu_q) - 1) if seqs is None else seqs):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0:
            continue
        if k1 == k0:
            out[q0:q1] = 0.0
            lse[:, q0:q1] = -np.inf
            continue
        o_b, l_b = dense(q[q0:q1][None], k[k0:k1][None], v[k0:k1][None], B=1, Hq=Hq, Hkv=Hkv,
                         Sq=q1 - q0, Sk=k1 - k0, d=d, causal=causal, scale=scale)
        out[q0:q1] = o_b[0]
        lse[:, q0:q1] = l_b[0]
    return out, lse


def gather_pages(pages, block_table_row, L, page_size=16):
    """The first L tokens of one sequence out of a page pool [num_pages, page_size, H, d]:
    token t lives in slot t % page_size of page block_table_row[t // page_size].
    Returns [L, H, d] in the pool's dtype; raises if a needed table entry is out of range."""
    idx = np.arange(L)
    phys = np.asarray(block_table_row, dtype=np.int64)[idx // page_size]
    if L and (phys.min() < 0 or phys.max() >= pages.shape[0]):
        raise ValueError("block table entry outside the page pool")
    return pages[phys, idx % page_size]


def attention_paged(q, k_pages, v_pages, block_table, seqlens_k, cu_q, *, Hq, Hkv, d=128, causal=False, scale,
                    page_size=16, seqs=None, dense=None):
    """Prefill of packed query chunks against a paged KV cache.

    Sequence b has seqlens_k[b] cached keys, key t at slot t % 16 of page
    block_table[b][t // 16] of the pools, and query rows cu_q[b] .. cu_q[b+1]-1
    of q [total_q, Hq, d]; causal alignment is bottom-right (the chunk is the
    cache's last tokens).  Each sequence is gathered into contiguous K, V and
    run through the plain attention above.  Returns (out [total_q, Hq, d],
    lse [Hq, total_q]) in float64, NaN for rows of no sequence.  `dense` as in
    attention_varlen."""
    dense = attention if dense is None else dense
    cu_q = [int(x) for x in cu_q]
    lens = [int(x) for x in seqlens_k]
    bt = np.asarray(block_table)
    total_q = q.shape[0]
    out = np.full((total_q, Hq, d), np.nan)
    lse = np.full((Hq, total_q), np.nan)
    for b in (range(len(lens)) if seqs is None else seqs):
        q0, q1, Lk = cu_q[b], cu_q[b + 1], lens[b]
        if q1 == q0:
            continue
        if Lk == 0:
            out[q0:q1] = 0.0
            lse[:, q0:q1] = -np.inf
            continue
        k_b = gather_pages(k_pages, bt[b], Lk, page_size)
        v_b = gather_pages(v_pages, bt[b], Lk, page_size)
        o_b, l_b = dense(q[q0:q1][None], k_b[None], v_b[None], B=1, Hq=Hq, Hkv=Hkv, Sq=q1 - q0, Sk=Lk, d=d,
                         causal=causal, scale=scale)
        out[q0:q1] = o_b[0]
        lse[:, q0:q1] = l_b[0]
    return out, lse


def attention_rows(q, k, v, rows, *, B, Hq, Hkv, Sq, Sk, d=128, layout="bshd", causal=False,
                   scale, key_range=None):
    """Selected rows (an [n, 3] array of (b, h, i)), optionally over keys [lo, hi).

    Returns (out [n, d], lse [n]) in float64.
    """
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    lo, hi = (0, Sk) if key_range is None else key_range
    out = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    _check(lib.oracle_attention_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Sk, d,
                                     LAYOUTS[layout], int(bool(causal)), float(scale), n,
                                     _ptr(rows), int(lo), int(hi), _ptr(out), _ptr(lse)),
           "attention_rows")
    return out, lse


def attention_probs_row(q, k, b, h, i, *, B, Hq, Hkv, Sq, Sk, d=128, layout="bshd",
                        causal=False, scale):
    """The softmax probabilities of one query row over all Sk keys (0 where masked)."""
    lib = _load()
    qb, kb = _bits(q), _bits(k)
    probs = np.empty((Sk,), np.float64)
    _check(lib.oracle_attention_probs_row(_ptr(qb), _ptr(kb), B, Hq, Hkv, Sq, Sk, d,
                                          LAYOUTS[layout], int(bool(causal)), float(scale),
                                          b, h, i, _ptr(probs)), "attention_probs_row")
    return probs


def attention_tiled_rows(q, k, v, rows, *, tile, B, Hq, Hkv, Sq, Sk, d=128, layout="bshd",
                         causal=False, scale):
    """The online-softmax recurrence over key tiles of `tile` keys, for selected rows."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    _check(lib.oracle_attention_tiled_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Sk, d,
                                           LAYOUTS[layout], int(bool(causal)), float(scale),
                                           int(tile), n, _ptr(rows), _ptr(out), _ptr(lse)),
           "attention_tiled_rows")
    return out, lse


def lse_merge(lse_parts, o_parts):
    """Merge key-range partials: lse_parts [S, n], o_parts [S, n, d] -> (out [n, d], lse [n])."""
    lib = _load()
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    S, n = lse_parts.shape
    d = o_parts.shape[2]
    out = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    _check(lib.oracle_lse_merge(S, n, d, _ptr(lse_parts), _ptr(o_parts), _ptr(out), _ptr(lse)),
           "lse_merge")
    return out, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, *, scale, page_size=16):
    """Paged-KV decode.  q [B, Hq, d]; pools [num_pages, page_size, Hkv, d];
    block_table [B, max_blocks] int32; seqlens [B] int32.  Returns (out [B, Hq, d], lse [B, Hq])."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_pages), _bits(v_pages)
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    B, Hq, d = qb.shape
    num_pages, ps, Hkv, d2 = kb.shape
    if ps != page_size or d2 != d or vb.shape != kb.shape:
        raise ValueError("page pool shape mismatch")
    out = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    _check(lib.oracle_decode_paged(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(sl), B, Hq, Hkv, d,
                                   page_size, num_pages, bt.shape[1], float(scale), _ptr(out),
                                   _ptr(lse)), "decode_paged")
    return out, lse


def decode_paged_append(q, k_new, v_new, k_pages, v_pages, block_table, seqlens, *, scale, page_size=16):
    """Append one token per sequence to a paged cache, then decode over it.

    k_new, v_new [B, Hkv, d] are written at position L = seqlens[b] of sequence
    b, i.e. slot L % page_size of page block_table[b][L // page_size]; then each
    query attends over the L + 1 keys.  Returns (out [B, Hq, d], lse [B, Hq],
    k_pages', v_pages') with the pools as copies after the append."""
    kp = k_pages.clone()
    vp = v_pages.clone()
    lens = [int(x) for x in seqlens]
    bt = np.asarray(block_table)
    for b, L in enumerate(lens):
        page = int(bt[b][L // page_size])
        if page < 0 or page >= kp.shape[0]:
            raise ValueError("block table has no page for the appended token")
        kp[page, L % page_size] = k_new[b]
        vp[page, L % page_size] = v_new[b]
    out, lse = decode_paged(q, kp, vp, block_table, np.asarray(lens, dtype=np.int32) + 1, scale=scale,
                            page_size=page_size)
    return out, lse, kp, vp


def round_bf16_rtne(x: float) -> int:
    """Bit pattern of the bf16 nearest to x, ties to even."""
    return int(_load().oracle_round_bf16_rtne(float(x)))


ROUNDING_MODES = {"rtne": 0, "rtna": 1, "rtz": 2}


def round_bf16(x: float, mode: str = "rtne") -> int:
    """Bit pattern of x rounded to bf16: "rtne" (nearest, ties to even), "rtna"
    (nearest, ties away from zero) or "rtz" (toward zero)."""
    return int(_load().oracle_round_bf16(float(x), ROUNDING_MODES[mode]))


def round_bf16_array(x, mode: str = "rtne") -> np.ndarray:
    """Element-wise round_bf16 over an array of doubles; uint16 bit patterns, same shape."""
    xd = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xd.shape, dtype=np.uint16)
    _check(_load().oracle_round_bf16_array(_ptr(xd), _ptr(out), xd.size, ROUNDING_MODES[mode]), "round_bf16_array")
    return out
