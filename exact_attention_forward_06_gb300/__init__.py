"""GB300-native (sm_103a) exact attention: fused prefill forward and paged-KV decode.

The computation lives in the CUDA library ``libattn.so`` (C ABI, include/attn.h);
this package is its thin Python binding.  Importing the package does not load
the library; the first call does, and raises if it has not been built.
"""
from ._binding import (AttnError, LIBRARY_PATH, debug_inject, decode_paged, decode_paged_append, decode_paged_noalloc,
                       decode_workspace_bytes, fwd_workspace_bytes, set_workspace,
                       device_status, fwd, fwd_host, fwd_host_workspace_bytes, fwd_paged, fwd_simple, fwd_varlen, load, lse_merge, selftest_umma, set_wait_budget_ns,
                       status_string, version)

__all__ = ["AttnError", "LIBRARY_PATH", "debug_inject", "decode_paged", "decode_paged_append", "decode_paged_noalloc",
           "decode_workspace_bytes", "device_status", "fwd_workspace_bytes", "set_workspace",
           "fwd", "fwd_host", "fwd_host_workspace_bytes", "fwd_paged", "fwd_simple", "fwd_varlen", "load", "lse_merge", "selftest_umma", "set_wait_budget_ns", "status_string",
           "version"]
