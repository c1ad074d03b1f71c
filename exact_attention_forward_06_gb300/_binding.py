"""ctypes binding of libattn.so (the C ABI in include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch owns the device memory and the stream; tensors are passed by
``data_ptr()`` and the current stream by handle.  If the compiled library is
missing this module raises immediately -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
                4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_WORKSPACE", 6: "ATTN_ERR_DEVICE_BOUNDS"}
LAYOUTS = {"bshd": 0, "bhsd": 1}

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")


def load():
    """Load libattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY_PATH):
                raise RuntimeError(
                    f"{LIBRARY_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIBRARY_PATH)
            fwd_args = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p]
            lib.attn_fwd.argtypes = fwd_args
            lib.attn_fwd_simple.argtypes = fwd_args
            lib.attn_fwd_rounded.argtypes = fwd_args[:-1] + [_i, _p]
            lib.attn_fwd_host.argtypes = fwd_args[:-1] + [_i, _p, _sz, _p]
            lib.attn_fwd_host.restype = _i
            lib.attn_fwd_host_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i]
            lib.attn_fwd_host_workspace_bytes.restype = _sz
            lib.attn_fwd_varlen.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                                            _i, _p]
            lib.attn_fwd_paged.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                           _f, _i, _p]
            lib.attn_fwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
            lib.attn_fwd_workspace_bytes.restype = _sz
            lib.attn_set_workspace.argtypes = [_p, _sz]
            lib.attn_set_workspace.restype = _i
            lib.attn_decode_workspace_bytes.argtypes = [_i, _i, _i, _i]
            lib.attn_decode_workspace_bytes.restype = _sz
            lib.attn_decode_paged.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p,
                                              _sz, _p]
            lib.attn_decode_paged_append.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                                     _i, _f, _p, _sz, _p]
            lib.attn_decode_paged_append.restype = _i
            lib.attn_decode_paged_noalloc.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                                                      _f, _p]
            lib.attn_decode_paged_noalloc.restype = _i
            lib.attn_lse_merge.argtypes = [_p, _p, _p, _p, _i, _i, _i, _i, _p]
            lib.attn_get_device_status.argtypes = [_p, ctypes.POINTER(_i)]
            lib.attn_set_wait_budget_ns.argtypes = [_u64]
            lib.attn_debug_inject.argtypes = [_i]
            lib.attn_selftest_umma.argtypes = [_p, _p, _p, _i, _p]
            lib.attn_status_string.argtypes = [_i]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_version.restype = _i
            for name in ("attn_fwd", "attn_fwd_simple", "attn_fwd_rounded", "attn_fwd_varlen", "attn_fwd_paged",
                         "attn_decode_paged",
                         "attn_lse_merge",
                         "attn_get_device_status", "attn_set_wait_budget_ns", "attn_debug_inject",
                         "attn_selftest_umma"):
                getattr(lib, name).restype = _i
            _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev_tensor(t: torch.Tensor, name: str, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q, k, layout):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    if layout == "bshd":
        B, Sq, Hq, d = q.shape
        _, Sk, Hkv, _ = k.shape
    elif layout == "bhsd":
        B, Hq, Sq, d = q.shape
        _, Hkv, Sk, _ = k.shape
    else:
        raise ValueError(f"layout must be 'bshd' or 'bhsd', got {layout!r}")
    return B, Hq, Hkv, Sq, Sk, d


ROUNDING = {"rtne": 0, "rtna": 1, "rtz": 2}


def _fwd_call(fn_name, q, k, v, causal, scale, layout, out, lse, stream, rounding="rtne"):
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev_tensor(t, n, torch.bfloat16)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    B, Hq, Hkv, Sq, Sk, d = _dims(q, k, layout)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    elif lse is not False:
        _dev_tensor(lse, "lse", torch.float32)
    lse_ptr = None if lse is False else lse.data_ptr()
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv, Sq, Sk, d, LAYOUTS[layout],
            int(bool(causal)), float(scale)]
    if rounding != "rtne":
        if fn_name != "attn_fwd":
            raise ValueError(f"{fn_name} rounds its output to nearest even only")
        fn_name = "attn_fwd_rounded"
        args.append(ROUNDING[rounding])
    rc = getattr(lib, fn_name)(*args, _stream(stream))
    _check(rc, fn_name)
    return out, (None if lse is False else lse)


def fwd(q, k, v, *, causal=False, scale=None, layout="bshd", out=None, lse=None, stream=None, rounding="rtne"):
    """Fused exact attention forward: returns (out bf16 in q's layout, lse fp32 [B, Hq, Sq]).

    Pass ``lse=False`` to skip the log-sum-exp output.  ``rounding`` selects how
    the fp32 result is rounded to the bf16 output: "rtne" (nearest, ties to
    even; C entry point attn_fwd), "rtna" (nearest, ties away from zero) or
    "rtz" (toward zero), the latter two through attn_fwd_rounded.
    """
    if rounding not in ROUNDING:
        raise ValueError(f"rounding must be one of {sorted(ROUNDING)}, got {rounding!r}")
    return _fwd_call("attn_fwd", q, k, v, causal, scale, layout, out, lse, stream, rounding)


def fwd_host_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int = 128) -> int:
    """Device workspace bytes fwd_host needs for this shape."""
    return int(load().attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d))


def fwd_host(q, k, v, *, causal=False, scale=None, layout="bshd", out=None, lse=None, workspace=None, stream=None,
             rounding="rtne"):
    """The forward pass from and to host memory (C entry point attn_fwd_host).

    q, k, v: CPU bf16 tensors (pin them for asynchronous copies); out/lse: CPU
    tensors to write (allocated pinned when omitted; ``lse=False`` skips it).
    workspace: a CUDA uint8 tensor of at least fwd_host_workspace_bytes(...)
    bytes (allocated when omitted).  Returns (out, lse); they are complete once
    ``stream`` (default: the current stream) has reached this point.
    """
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU bfloat16 tensor")
    if rounding not in ROUNDING:
        raise ValueError(f"rounding must be one of {sorted(ROUNDING)}, got {rounding!r}")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    B, Hq, Hkv, Sq, Sk, d = _dims(q, k, layout)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32).pin_memory()
    need = fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device="cuda", dtype=torch.uint8)
    _dev_tensor(workspace, "workspace", torch.uint8)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv, Sq, Sk, d,
                           LAYOUTS[layout], int(bool(causal)), float(scale), ROUNDING[rounding], workspace.data_ptr(),
                           workspace.numel(), _stream(stream))
    _check(rc, "attn_fwd_host")
    return out, (None if lse is False else lse)


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q=None, max_seqlen_k=None, causal=False,
               scale=None, out=None, lse=None, stream=None, rounding="rtne"):
    """Attention over a packed batch of variable-length sequences.

    q [total_q, Hq, d], k and v [total_k, Hkv, d] bf16; cu_seqlens_q/k int32 [B+1]
    on the device.  Returns (out [total_q, Hq, d] bf16, lse [Hq, total_q] fp32).
    max_seqlen_q/k bound the sequence lengths; when omitted they are read from
    the offsets, which copies them to the host (a synchronisation).  Rows of
    ``out``/``lse`` outside every sequence are left as given.
    """
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev_tensor(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    if rounding not in ROUNDING:
        raise ValueError(f"rounding must be one of {sorted(ROUNDING)}, got {rounding!r}")
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape:
        raise ValueError("q must be [total_q, Hq, d] and k, v [total_k, Hkv, d]")
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1 or B < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 entries, B >= 1")
    if max_seqlen_q is None:
        max_seqlen_q = max(1, int(torch.diff(cu_seqlens_q).max()))
    if max_seqlen_k is None:
        max_seqlen_k = max(1, int(torch.diff(cu_seqlens_k).max()))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), device=q.device, dtype=torch.float32)
    elif lse is not False:
        _dev_tensor(lse, "lse", torch.float32)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                             cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Hq, Hkv, total_q, total_k,
                             int(max_seqlen_q), int(max_seqlen_k), d, int(bool(causal)), float(scale),
                             ROUNDING[rounding], _stream(stream))
    _check(rc, "attn_fwd_varlen")
    return out, (None if lse is False else lse)


def fwd_paged(q, k_pages, v_pages, block_table, seqlens_k, cu_seqlens_q, *, max_seqlen_q=None, causal=True,
              scale=None, out=None, lse=None, stream=None, rounding="rtne"):
    """Prefill of packed query chunks against a paged KV cache (chunked prefill).

    q [total_q, Hq, d] bf16; k_pages, v_pages [num_pages, 16, Hkv, d] bf16; block_table [B, max_blocks]
    int32; seqlens_k [B] int32 (cache lengths, chunk included); cu_seqlens_q [B+1] int32 -- all on the
    device.  Returns (out [total_q, Hq, d] bf16, lse [Hq, total_q] fp32).  max_seqlen_q, when omitted,
    is read from the offsets (a synchronisation).
    """
    lib = load()
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _dev_tensor(t, n, torch.bfloat16)
    for t, n in ((block_table, "block_table"), (seqlens_k, "seqlens_k"), (cu_seqlens_q, "cu_seqlens_q")):
        _dev_tensor(t, n, torch.int32)
    if rounding not in ROUNDING:
        raise ValueError(f"rounding must be one of {sorted(ROUNDING)}, got {rounding!r}")
    if q.dim() != 3 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise ValueError("q must be [total_q, Hq, d] and the pools [num_pages, 16, Hkv, d]")
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    B = seqlens_k.numel()
    if cu_seqlens_q.numel() != B + 1 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_q must have B + 1 entries and block_table B rows")
    if max_seqlen_q is None:
        max_seqlen_q = max(1, int(torch.diff(cu_seqlens_q).max()))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), device=q.device, dtype=torch.float32)
    elif lse is not False:
        _dev_tensor(lse, "lse", torch.float32)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_fwd_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                            seqlens_k.data_ptr(), cu_seqlens_q.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv,
                            total_q, int(max_seqlen_q), d, page_size, num_pages, block_table.shape[1],
                            int(bool(causal)), float(scale), ROUNDING[rounding], _stream(stream))
    _check(rc, "attn_fwd_paged")
    return out, (None if lse is False else lse)


def fwd_simple(q, k, v, *, causal=False, scale=None, layout="bshd", out=None, lse=None, stream=None):
    """The same operation through the plain SIMT kernel (debugging cross-check; slow)."""
    return _fwd_call("attn_fwd_simple", q, k, v, causal, scale, layout, out, lse, stream)


def fwd_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, d: int = 128, causal: bool = False) -> int:
    """Workspace bytes that let attn_fwd split its last wave of work for this shape (current device)."""
    return int(load().attn_fwd_workspace_bytes(B, Hq, Hkv, Sq, Sk, d, int(bool(causal))))


def set_workspace(buf=None):
    """Register a CUDA uint8 tensor (or None to clear) as the current device's attn_fwd workspace.

    The caller keeps ownership and must keep the tensor alive while it is registered.
    """
    if buf is None:
        _check(load().attn_set_workspace(None, 0), "attn_set_workspace")
        return
    _dev_tensor(buf, "workspace", torch.uint8)
    _check(load().attn_set_workspace(buf.data_ptr(), buf.numel()), "attn_set_workspace")


def decode_workspace_bytes(B: int, Hq: int, d: int, max_blocks_per_seq: int) -> int:
    return int(load().attn_decode_workspace_bytes(B, Hq, d, max_blocks_per_seq))


def decode_paged(q, k_pages, v_pages, block_table, seqlens, *, scale=None, out=None, lse=None, workspace=None,
                 stream=None):
    """One decode step over a paged KV cache.

    q [B, Hq, d] bf16; k_pages/v_pages [num_pages, 16, Hkv, d] bf16; block_table [B, max_blocks] int32;
    seqlens [B] int32 (device).  Returns (out [B, Hq, d] bf16, lse [B, Hq] fp32).
    """
    lib = load()
    _dev_tensor(q, "q", torch.bfloat16)
    _dev_tensor(k_pages, "k_pages", torch.bfloat16)
    _dev_tensor(v_pages, "v_pages", torch.bfloat16)
    _dev_tensor(block_table, "block_table", torch.int32)
    _dev_tensor(seqlens, "seqlens", torch.int32)
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    need = decode_workspace_bytes(B, Hq, d, max_blocks)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                               seqlens.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv, d, page_size, num_pages,
                               max_blocks, float(scale), workspace.data_ptr(), workspace.numel(),
                               _stream(stream))
    _check(rc, "attn_decode_paged")
    return out, (None if lse is False else lse)


def decode_paged_append(q, k_new, v_new, k_pages, v_pages, block_table, seqlens, *, scale=None, out=None, lse=None,
                        workspace=None, stream=None):
    """Append k_new/v_new [B, Hkv, d] at position seqlens[b] of each sequence's pages and decode over the
    seqlens[b] + 1 keys, in one launch.  seqlens (the lengths before the append) is not modified.
    Returns (out [B, Hq, d] bf16, lse [B, Hq] fp32); k_pages and v_pages are updated in place."""
    lib = load()
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _dev_tensor(t, n, torch.bfloat16)
    _dev_tensor(block_table, "block_table", torch.int32)
    _dev_tensor(seqlens, "seqlens", torch.int32)
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    if k_new.shape != (B, Hkv, d) or v_new.shape != (B, Hkv, d):
        raise ValueError("k_new and v_new must be [B, Hkv, d]")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    need = decode_workspace_bytes(B, Hq, d, max_blocks)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_decode_paged_append(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(),
                                      v_pages.data_ptr(), block_table.data_ptr(), seqlens.data_ptr(), out.data_ptr(),
                                      lse_ptr, B, Hq, Hkv, d, page_size, num_pages, max_blocks, float(scale),
                                      workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(rc, "attn_decode_paged_append")
    return out, (None if lse is False else lse)


def decode_paged_noalloc(q, k_pages, v_pages, block_table, seqlens, *, scale=None, out=None, lse=None,
                         stream=None):
    """decode_paged for callers that cannot allocate device memory.

    Same arguments and results as ``decode_paged`` minus the workspace: the
    split partials live in a fixed 16 MiB device array owned by the library
    (shared by every call, so calls must not overlap on the GPU).  ``out`` and
    ``lse`` must be passed by a caller that cannot allocate; when they are
    omitted this wrapper allocates them with torch for convenience.
    """
    lib = load()
    _dev_tensor(q, "q", torch.bfloat16)
    _dev_tensor(k_pages, "k_pages", torch.bfloat16)
    _dev_tensor(v_pages, "v_pages", torch.bfloat16)
    _dev_tensor(block_table, "block_table", torch.int32)
    _dev_tensor(seqlens, "seqlens", torch.int32)
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    lse_ptr = None if lse is False else lse.data_ptr()
    rc = lib.attn_decode_paged_noalloc(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                       block_table.data_ptr(), seqlens.data_ptr(), out.data_ptr(), lse_ptr, B, Hq,
                                       Hkv, d, page_size, num_pages, block_table.shape[1], float(scale),
                                       _stream(stream))
    _check(rc, "attn_decode_paged_noalloc")
    return out, (None if lse is False else lse)


def lse_merge(o_parts, lse_parts, *, out=None, lse=None, stream=None, rounding="rtne"):
    """Merge key-range partials: o_parts [rows, nsplit, d] fp32, lse_parts [rows, nsplit] fp32.

    ``rounding`` ("rtne", "rtna" or "rtz") selects the fp32 -> bf16 rounding of out.
    """
    if rounding not in ROUNDING:
        raise ValueError(f"rounding must be one of {sorted(ROUNDING)}, got {rounding!r}")
    lib = load()
    _dev_tensor(o_parts, "o_parts", torch.float32)
    _dev_tensor(lse_parts, "lse_parts", torch.float32)
    rows, nsplit, d = o_parts.shape
    if out is None:
        out = torch.empty((rows, d), device=o_parts.device, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty((rows,), device=o_parts.device, dtype=torch.float32)
    rc = lib.attn_lse_merge(o_parts.data_ptr(), lse_parts.data_ptr(), out.data_ptr(), lse.data_ptr(), rows, nsplit,
                            d, ROUNDING[rounding], _stream(stream))
    _check(rc, "attn_lse_merge")
    return out, lse


def device_status(stream=None):
    """Synchronise the stream, read and clear the device status word: (code, site)."""
    site = _i(0)
    rc = load().attn_get_device_status(_stream(stream), ctypes.byref(site))
    return rc, site.value


def set_wait_budget_ns(ns: int):
    _check(load().attn_set_wait_budget_ns(int(ns)), "attn_set_wait_budget_ns")


def debug_inject(mode: int):
    _check(load().attn_debug_inject(int(mode)), "attn_debug_inject")


def selftest_umma(a, b, mode: int, stream=None):
    """128x128x128 tensor-core layout check: mode 0 -> a @ b.T, mode 1 -> a @ b (fp32 [128, 128])."""
    _dev_tensor(a, "a", torch.bfloat16)
    _dev_tensor(b, "b", torch.bfloat16)
    c = torch.empty((128, 128), device=a.device, dtype=torch.float32)
    _check(load().attn_selftest_umma(a.data_ptr(), b.data_ptr(), c.data_ptr(), int(mode), _stream(stream)),
           "attn_selftest_umma")
    return c


def status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


def version() -> int:
    return int(load().attn_version())
