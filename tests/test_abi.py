"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import exact_attention_forward_06_gb300 as A
from exact_attention_forward_06_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_binding.LIBRARY_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return A.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_bytes", "attn_lse_merge",
                 "attn_get_device_status", "attn_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_binding.LIBRARY_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(lib):
    for code, name in _binding.STATUS_NAMES.items():
        assert A.status_string(code) == name
    assert A.version() >= 100


def _fwd(lib, **kw):
    args = dict(q=16, k=16, v=16, out=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, d=128, layout=0, causal=0,
                scale=0.1)
    args.update(kw)
    return lib.attn_fwd(args["q"], args["k"], args["v"], args["out"], args["lse"], args["B"], args["Hq"],
                        args["Hkv"], args["Sq"], args["Sk"], args["d"], args["layout"], args["causal"],
                        args["scale"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(q=24), 1), (dict(B=0), 1), (dict(Sq=0), 1), (dict(Sk=-1), 1),
    (dict(Hq=3, Hkv=2), 1), (dict(layout=2), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=-1.0), 1), (dict(d=64), 2), (dict(lse=18), 1),
])
def test_fwd_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert _fwd(lib, **kw) == code
    # the simple kernel shares the validation
    args = dict(q=16, k=16, v=16, out=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, d=128, layout=0, causal=0,
                scale=0.1)
    args.update(kw)
    assert lib.attn_fwd_simple(*[args[n] for n in ("q", "k", "v", "out", "lse", "B", "Hq", "Hkv", "Sq", "Sk",
                                                   "d", "layout", "causal", "scale")], None) == code


def test_decode_workspace_is_a_pure_function_of_shape(lib):
    a = A.decode_workspace_bytes(32, 32, 128, 512)
    assert a == A.decode_workspace_bytes(32, 32, 128, 512) and a > 0
    # non-decreasing in the table width, and larger once the splits are capped
    assert A.decode_workspace_bytes(32, 32, 128, 513) >= a
    assert A.decode_workspace_bytes(32, 32, 128, 8192) > a
    assert A.decode_workspace_bytes(32, 32, 64, 512) == 0
    assert A.decode_workspace_bytes(0, 32, 128, 512) == 0


def _decode(lib, **kw):
    a = dict(q=16, kp=16, vp=16, bt=16, sl=16, out=16, lse=None, B=2, Hq=4, Hkv=2, d=128, page=16, npages=10,
             maxb=4, scale=0.1, ws=256, wsb=1 << 20)
    a.update(kw)
    return lib.attn_decode_paged(a["q"], a["kp"], a["vp"], a["bt"], a["sl"], a["out"], a["lse"], a["B"], a["Hq"],
                                 a["Hkv"], a["d"], a["page"], a["npages"], a["maxb"], a["scale"], a["ws"],
                                 a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(bt=None), 1), (dict(bt=18), 1), (dict(Hq=5), 1), (dict(npages=0), 1),
    (dict(maxb=0), 1), (dict(scale=float("nan")), 1), (dict(page=32), 2), (dict(d=256), 2),
    (dict(ws=None), 5), (dict(ws=272), 5), (dict(wsb=16), 5),
])
def test_decode_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert _decode(lib, **kw) == code


def _decode_noalloc(lib, **kw):
    a = dict(q=16, kp=16, vp=16, bt=16, sl=16, out=16, lse=None, B=2, Hq=4, Hkv=2, d=128, page=16, npages=10,
             maxb=4, scale=0.1)
    a.update(kw)
    return lib.attn_decode_paged_noalloc(a["q"], a["kp"], a["vp"], a["bt"], a["sl"], a["out"], a["lse"], a["B"],
                                         a["Hq"], a["Hkv"], a["d"], a["page"], a["npages"], a["maxb"], a["scale"],
                                         None)


# 64 sequences x 64 heads x 8192 pages: far more partials than the 16 MiB array holds
_HUGE = dict(B=64, Hq=64, Hkv=8, maxb=8192)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(bt=18), 1), (dict(Hq=5), 1), (dict(scale=float("nan")), 1), (dict(d=256), 2),
    # the argument checks come before the array's size limit
    (dict(q=None, **_HUGE), 1), (dict(out=24, **_HUGE), 1), (dict(page=32, **_HUGE), 2),
    (dict(_HUGE), 5),
])
def test_decode_noalloc_checks_arguments_before_its_size_limit(lib, kw, code):
    assert _decode_noalloc(lib, **kw) == code


def test_merge_rejects_bad_arguments(lib):
    assert lib.attn_lse_merge(None, 16, 16, None, 4, 2, 128, 0, None) == 1
    assert lib.attn_lse_merge(16, 16, 16, None, 0, 2, 128, 0, None) == 1
    assert lib.attn_lse_merge(16, 16, 16, None, 4, 2, 64, 0, None) == 2
    assert lib.attn_lse_merge(16, 16, 16, None, 4, 2, 128, 3, None) == 1     # no such rounding mode
    assert lib.attn_lse_merge(16, 16, 16, None, 4, 2, 128, -1, None) == 1


@pytest.mark.parametrize("kw,code", [(dict(q=None), 1), (dict(d=64), 2), (dict(mode=3), 1), (dict(mode=-1), 1)])
def test_fwd_rounded_validates_before_any_launch(lib, kw, code):
    a = dict(q=16, mode=1, d=128)
    a.update(kw)
    assert lib.attn_fwd_rounded(a["q"], 16, 16, 16, None, 1, 2, 2, 8, 8, a["d"], 0, 0, 0.1, a["mode"], None) == code


def test_python_rounding_names_are_checked(lib):
    with pytest.raises(ValueError):
        A.fwd(None, None, None, rounding="rtn")


def test_debug_controls(lib):
    assert lib.attn_debug_inject(7) == 1
    assert lib.attn_debug_inject(0) == 0
    assert lib.attn_set_wait_budget_ns(0) == 0


def test_fwd_workspace_query_and_registration_validate(lib):
    assert lib.attn_fwd_workspace_bytes(0, 1, 1, 8, 8, 128, 0) == 0
    assert lib.attn_fwd_workspace_bytes(1, 3, 2, 8, 8, 128, 0) == 0
    assert lib.attn_fwd_workspace_bytes(1, 2, 2, 8, 8, 64, 0) == 0
    assert lib.attn_set_workspace(264, 1024) == 1     # not 256-byte aligned


def _varlen(lib, **kw):
    a = dict(q=16, k=16, v=16, out=16, lse=None, cq=64, ck=64, B=2, Hq=4, Hkv=2, tq=100, tk=100, mq=60, mk=60,
             d=128, causal=0, scale=0.1, mode=0)
    a.update(kw)
    return lib.attn_fwd_varlen(a["q"], a["k"], a["v"], a["out"], a["lse"], a["cq"], a["ck"], a["B"], a["Hq"],
                               a["Hkv"], a["tq"], a["tk"], a["mq"], a["mk"], a["d"], a["causal"], a["scale"],
                               a["mode"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cq=None), 1), (dict(ck=None), 1), (dict(cq=66), 1), (dict(q=24), 1), (dict(B=0), 1),
    (dict(tq=0), 1), (dict(tk=0), 1), (dict(mq=0), 1), (dict(mq=101), 1), (dict(mk=101), 1),
    (dict(Hq=3), 1), (dict(d=64), 2), (dict(mode=5), 1), (dict(scale=float("nan")), 1),
])
def test_fwd_varlen_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert _varlen(lib, **kw) == code


def _paged(lib, **kw):
    a = dict(q=16, kp=16, vp=16, bt=64, sl=64, cq=64, out=16, lse=None, B=2, Hq=4, Hkv=2, tq=100, mq=60, d=128,
             page=16, npages=10, maxb=4, causal=1, scale=0.1, mode=0)
    a.update(kw)
    return lib.attn_fwd_paged(a["q"], a["kp"], a["vp"], a["bt"], a["sl"], a["cq"], a["out"], a["lse"], a["B"],
                              a["Hq"], a["Hkv"], a["tq"], a["mq"], a["d"], a["page"], a["npages"], a["maxb"],
                              a["causal"], a["scale"], a["mode"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=None), 1), (dict(sl=None), 1), (dict(cq=None), 1), (dict(bt=66), 1), (dict(kp=24), 1),
    (dict(B=0), 1), (dict(tq=0), 1), (dict(mq=0), 1), (dict(mq=101), 1), (dict(npages=0), 1), (dict(maxb=0), 1),
    (dict(Hq=3), 1), (dict(d=64), 2), (dict(page=32), 2), (dict(mode=3), 1), (dict(scale=-1.0), 1),
])
def test_fwd_paged_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert _paged(lib, **kw) == code


def test_decode_append_rejects_bad_arguments(lib):
    args = [16, 16, 16, 16, 16, 64, 64, 16, None, 2, 4, 2, 128, 16, 10, 4, 0.1, 256, 1 << 20, None]
    assert lib.attn_decode_paged_append(*args[:1], None, *args[2:]) == 1        # no k_new
    assert lib.attn_decode_paged_append(*args[:2], 24, *args[3:]) == 1          # misaligned v_new
    bad = list(args)
    bad[13] = 32                                                                # page size
    assert lib.attn_decode_paged_append(*bad) == 2
    bad = list(args)
    bad[17] = None                                                              # workspace
    assert lib.attn_decode_paged_append(*bad) == 5


def test_fwd_host_rejects_bad_arguments_before_any_copy(lib):
    args = [16, 16, 16, 16, None, 2, 4, 2, 64, 64, 128, 0, 1, 0.1, 0, 256, 1 << 30, None]
    assert lib.attn_fwd_host(None, *args[1:]) == 1
    bad = list(args); bad[10] = 64
    assert lib.attn_fwd_host(*bad) == 2
    bad = list(args); bad[15] = None
    assert lib.attn_fwd_host(*bad) == 5
    bad = list(args); bad[16] = 1024                       # too small
    assert lib.attn_fwd_host(*bad) == 5
    bad = list(args); bad[11] = 3                          # layout
    assert lib.attn_fwd_host(*bad) == 1
    assert lib.attn_fwd_host_workspace_bytes(2, 4, 2, 64, 64, 128) > 0
    assert lib.attn_fwd_host_workspace_bytes(2, 3, 2, 64, 64, 128) == 0


def _header_prototypes():
    """{name: [kind, ...]} from include/*.h, kinds 'ptr', 'int', 'float', 'u64'."""
    protos = {}
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for ret, name, params in re.findall(r"([\w\s\*]+?)\b(attn_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
            kinds = []
            for prm in [x.strip() for x in params.split(",")]:
                if prm in ("", "void"):
                    continue
                if "*" in prm:
                    kinds.append("ptr")
                elif prm.startswith("float"):
                    kinds.append("float")
                elif prm.startswith("size_t"):
                    kinds.append("u64")  # LP64: size_t is a 64-bit unsigned, as ctypes' c_size_t
                elif prm.startswith("uint64_t"):
                    kinds.append("u64")
                else:
                    # plain ints and the header's enums (passed as int)
                    assert prm.split()[0] in ("int", "int32_t", "attn_status_t", "attn_layout_t", "attn_round_t"), \
                        f"{name}: unexpected parameter {prm!r}"
                    kinds.append("int")
            protos[name] = kinds
    return protos


def test_binding_argtypes_match_the_header(lib):
    # The ctypes declarations of the binding must follow include/attn.h
    # parameter for parameter (a mismatch would pass garbage silently).
    kind_of = {ctypes.c_void_p: "ptr", ctypes.c_int: "int", ctypes.c_float: "float", ctypes.c_size_t: "u64",
               ctypes.c_uint64: "u64"}
    protos = _header_prototypes()
    assert set(protos) == set(declared_functions())
    for name, kinds in protos.items():
        argtypes = getattr(lib, name).argtypes
        got = [] if argtypes is None else [
            "ptr" if (t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "contents") or
                      getattr(t, "_type_", None) is not None and t.__name__.startswith("LP_")) else kind_of.get(t, repr(t))
            for t in argtypes]
        assert got == kinds, f"{name}: binding {got} vs header {kinds}"
