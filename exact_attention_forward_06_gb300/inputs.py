"""Seeded synthetic inputs for attention prefill and paged decode.

This module only draws random numbers and arranges them into the shapes the
workloads use; it holds none of the attention arithmetic.  Both sides of a
parity check (the CUDA library and the CPU oracle) receive the same bf16
bytes from here.

Recipe (the same for every workload):
  * values are drawn with ``torch.randn`` in fp32 from a CPU
    ``torch.Generator`` seeded per workload, in the order q, k, v, then cast
    to bf16 (round to nearest even);
  * tensors are generated in BSHD order ``[B, S, H, d]``; the BHSD form is a
    permuted copy, so an element (b, s, h, c) has the same value in both;
  * the long-sequence MQA workload scales 1% of the key positions
    (``ceil(0.01 * Sk)`` positions from a seeded permutation) by 8 in fp32
    before the cast, which makes some softmax rows sharply peaked;
  * paged decode draws per-sequence lengths uniformly from [lo, hi], gives each
    sequence ceil(L / 16) pages, assigns physical page ids by a seeded random
    permutation of the whole pool, and pads block-table rows with -1.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int = 128
    layout: str = "bshd"
    causal: bool = False
    seed: int = 0
    spike_frac: float = 0.0
    spike_scale: float = 8.0

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded once to fp32."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    @property
    def flops(self) -> float:
        """Matmul flops 4*B*Hq*Sq*Sk*d, halved for causal (the usual convention)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.d
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int = 32
    Hq: int = 32
    Hkv: int = 8
    d: int = 128
    page_size: int = 16
    max_blocks: int = 512
    len_lo: int = 1024
    len_hi: int = 8192
    seed: int = 5

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    def with_(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """A packed variable-length batch: sequence b owns rows cu_q[b] .. cu_q[b+1]-1
    of q [total_q, Hq, d] and rows cu_k[b] .. cu_k[b+1]-1 of k, v [total_k, Hkv, d].

    Query lengths are drawn U[len_lo, len_hi] (or given in lens_q); key lengths
    equal them unless lens_k is given (cross-attention per sequence)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    len_lo: int = 1
    len_hi: int = 1
    causal: bool = False
    seed: int = 0
    lens_q: tuple = None
    lens_k: tuple = None
    d: int = 128
    pad_q: int = 0   # unused rows after the last sequence (outputs there are left alone)

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    def lengths(self):
        gen = torch.Generator().manual_seed(self.seed)
        if self.lens_q is None:
            lq = torch.randint(self.len_lo, self.len_hi + 1, (self.B,), generator=gen, dtype=torch.int64).tolist()
        else:
            lq = list(self.lens_q)
        lk = list(lq) if self.lens_k is None else list(self.lens_k)
        assert len(lq) == self.B and len(lk) == self.B
        return lq, lk

    @property
    def flops(self) -> float:
        """4 * Hq * d * Lq * Lk per sequence, halved when causal (the dense convention)."""
        lq, lk = self.lengths()
        f = sum(4.0 * self.Hq * self.d * a * b for a, b in zip(lq, lk))
        return f / 2 if self.causal else f


def make_varlen(w: VarlenWorkload):
    """(q [total_q, Hq, d], k, v [total_k, Hkv, d] CPU bf16, cu_q, cu_k [B+1] int32)."""
    lq, lk = w.lengths()
    cu_q = torch.zeros(w.B + 1, dtype=torch.int32)
    cu_k = torch.zeros(w.B + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(lq, dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor(lk, dtype=torch.int64), 0).to(torch.int32)
    gen = torch.Generator().manual_seed(w.seed + 1000)
    total_q = int(cu_q[-1]) + w.pad_q
    total_k = int(cu_k[-1])
    q = _randn_bf16((total_q, w.Hq, w.d), gen)
    k = _randn_bf16((max(total_k, 1), w.Hkv, w.d), gen)
    v = _randn_bf16((max(total_k, 1), w.Hkv, w.d), gen)
    return q, k, v, cu_q, cu_k


# The five workloads: a tiny BHSD case, GQA causal, long MQA causal with
# peaked rows, ragged non-causal self- and cross-attention, and paged decode.
TINY_BHSD = PrefillWorkload("tiny_bhsd_1x2x256", 1, 2, 2, 256, 256, layout="bhsd", seed=1)
GQA_CAUSAL = PrefillWorkload("gqa_causal_4x32q8kv_4096", 4, 32, 8, 4096, 4096, causal=True, seed=2)
MQA_CAUSAL = PrefillWorkload("mqa_causal_1x32q1kv_16384", 1, 32, 1, 16384, 16384, causal=True,
                             seed=3, spike_frac=0.01)
RAGGED_SELF = PrefillWorkload("ragged_self_2x12_32760", 2, 12, 12, 32760, 32760, seed=4)
RAGGED_CROSS = PrefillWorkload("ragged_cross_2x12_32760x512", 2, 12, 12, 32760, 512, seed=40)
PAGED_DECODE = DecodeWorkload("paged_decode_32seq_32q8kv")

# A short query chunk against a long context (a speculative-decoding verify
# step): not one of the benchmark's configurations; shows GQA head packing.
GQA_SHORT_QUERY = PrefillWorkload("gqa_short_query_32x32q4kv_16x4096", 32, 32, 4, 16, 4096, seed=41)

PREFILL_WORKLOADS = {w.name: w for w in (TINY_BHSD, GQA_CAUSAL, MQA_CAUSAL, RAGGED_SELF, RAGGED_CROSS,
                                         GQA_SHORT_QUERY)}
# A packed batch of 16 GQA sequences of mixed lengths, causal (the varlen case).
VARLEN_CAUSAL = VarlenWorkload("varlen_causal_16seq_32q8kv", 16, 32, 8, len_lo=256, len_hi=8192, causal=True,
                               seed=6)
VARLEN_WORKLOADS = {VARLEN_CAUSAL.name: VARLEN_CAUSAL}


def _randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_prefill(w: PrefillWorkload):
    """(q, k, v) as CPU bf16 tensors in w.layout: BSHD [B,S,H,d] or BHSD [B,H,S,d]."""
    gen = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.Sq, w.Hq, w.d), generator=gen, dtype=torch.float32)
    k = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=gen, dtype=torch.float32)
    v = torch.randn((w.B, w.Sk, w.Hkv, w.d), generator=gen, dtype=torch.float32)
    if w.spike_frac > 0:
        n = math.ceil(w.spike_frac * w.Sk)
        pos = torch.randperm(w.Sk, generator=gen)[:n]
        k[:, pos] *= w.spike_scale
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    if w.layout == "bhsd":
        q, k, v = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))
    elif w.layout != "bshd":
        raise ValueError(f"unknown layout {w.layout!r}")
    return q, k, v


def to_layout(t: torch.Tensor, src: str, dst: str) -> torch.Tensor:
    """Re-arrange a [B,S,H,d] / [B,H,S,d] tensor between layouts (a plain permute)."""
    if src == dst:
        return t
    return t.permute(0, 2, 1, 3).contiguous()


def make_decode(w: DecodeWorkload, seqlens=None):
    """(q [B,Hq,d], k_pages, v_pages [P,page,Hkv,d], block_table [B,max_blocks] int32, seqlens [B] int32).

    `seqlens` overrides the drawn lengths (for edge cases); the pool still gets
    ceil(L/page) pages per sequence, with permuted physical ids.
    """
    gen = torch.Generator().manual_seed(w.seed)
    if seqlens is None:
        lens = torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=gen, dtype=torch.int64)
    else:
        lens = torch.as_tensor(seqlens, dtype=torch.int64)
        assert lens.numel() == w.B
    if int(lens.max()) > w.page_size * w.max_blocks:
        raise ValueError("a sequence is longer than the block table allows")
    npages = [(int(L) + w.page_size - 1) // w.page_size for L in lens]
    total = max(1, sum(npages))
    perm = torch.randperm(total, generator=gen).to(torch.int32)
    table = torch.full((w.B, w.max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[off:off + n]
        off += n
    q = _randn_bf16((w.B, w.Hq, w.d), gen)
    k_pages = _randn_bf16((total, w.page_size, w.Hkv, w.d), gen)
    v_pages = _randn_bf16((total, w.page_size, w.Hkv, w.d), gen)
    return q, k_pages, v_pages, table, lens.to(torch.int32)


@dataclasses.dataclass(frozen=True)
class PagedPrefillWorkload:
    """Chunked prefill against a paged KV cache: sequence b has a cache of
    Lk = context + chunk tokens (the chunk's own keys already appended) in
    16-token pages, and a packed query chunk of its last `chunk` tokens."""
    name: str
    B: int
    Hq: int
    Hkv: int
    chunk_lo: int = 1
    chunk_hi: int = 1
    ctx_lo: int = 0
    ctx_hi: int = 0
    causal: bool = True
    seed: int = 0
    d: int = 128
    page_size: int = 16
    max_blocks: int = 512
    chunks: tuple = None     # explicit chunk lengths (overrides the draw)
    contexts: tuple = None   # explicit context lengths (overrides the draw)

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    def lengths(self):
        """(chunk lengths Lq, cache lengths Lk) per sequence."""
        gen = torch.Generator().manual_seed(self.seed)
        lq = torch.randint(self.chunk_lo, self.chunk_hi + 1, (self.B,), generator=gen).tolist()
        ctx = torch.randint(self.ctx_lo, self.ctx_hi + 1, (self.B,), generator=gen).tolist()
        if self.chunks is not None:
            lq = list(self.chunks)
        if self.contexts is not None:
            ctx = list(self.contexts)
        return lq, [a + c for a, c in zip(lq, ctx)]

    @property
    def flops(self) -> float:
        """4 * Hq * d per visible (query, key) pair; causal counts Lq*(Lk-Lq) + Lq^2/2 pairs."""
        lq, lk = self.lengths()
        pairs = sum((a * (b - a) + a * a / 2) if self.causal else a * b for a, b in zip(lq, lk))
        return 4.0 * self.Hq * self.d * pairs


def make_paged_prefill(w: PagedPrefillWorkload):
    """(q [total_q, Hq, d], k_pages, v_pages [P, page, Hkv, d], block_table [B, max_blocks] int32 (-1 padded),
    seqlens_k [B] int32, cu_q [B+1] int32), CPU tensors.  Physical page ids are a seeded permutation."""
    lq, lk = w.lengths()
    if max(lk) > w.page_size * w.max_blocks:
        raise ValueError("a sequence is longer than the block table allows")
    gen = torch.Generator().manual_seed(w.seed + 2000)
    npages = [(L + w.page_size - 1) // w.page_size for L in lk]
    total = max(1, sum(npages))
    perm = torch.randperm(total, generator=gen).to(torch.int32)
    table = torch.full((w.B, w.max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[off:off + n]
        off += n
    cu_q = torch.zeros(w.B + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(lq, dtype=torch.int64), 0).to(torch.int32)
    q = _randn_bf16((max(1, int(cu_q[-1])), w.Hq, w.d), gen)
    k_pages = _randn_bf16((total, w.page_size, w.Hkv, w.d), gen)
    v_pages = _randn_bf16((total, w.page_size, w.Hkv, w.d), gen)
    return q, k_pages, v_pages, table, torch.tensor(lk, dtype=torch.int32), cu_q


def decode_kv_bytes(seqlens, Hkv: int, d: int) -> int:
    """Algorithmic K+V bytes one decode pass must read: 2 tensors * 2 B * Hkv * d per token."""
    return int(sum(int(L) for L in seqlens)) * Hkv * d * 2 * 2


# Chunked prefill of 16 GQA sequences against a paged cache: chunks of
# U[256, 2048] new tokens on contexts of U[0, 6144] cached tokens, causal.
PAGED_PREFILL = PagedPrefillWorkload("paged_prefill_16seq_32q8kv", 16, 32, 8, chunk_lo=256, chunk_hi=2048,
                                     ctx_lo=0, ctx_hi=6144, seed=7)
PAGED_PREFILL_WORKLOADS = {PAGED_PREFILL.name: PAGED_PREFILL}
