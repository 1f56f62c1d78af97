"""C-ABI library checks that need no GPU: it builds, loads and exports every
entry point include/lfattn.h declares; host-side argument validation runs
before any device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lfattn.h")


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    names = re.findall(r"LF_API\s+[\w\s\*]+?\b(lf_\w+)\s*\(", text)
    assert names, "no LF_API declarations found"
    return names


@pytest.fixture(scope="module")
def lib():
    from long_sequence_sparse_lf_b300 import build
    build.build()
    from long_sequence_sparse_lf_b300 import load_library
    return load_library()


def test_header_declares_expected_calls():
    names = set(declared_symbols())
    for n in ("lf_attn_fwd", "lf_attn_fwd_f32", "lf_attn_pairs", "lf_last_error",
              "lf_attn_get_status", "lf_plan_cache_clear"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_exports_match_header_exactly(lib):
    """No undeclared lf_* entry point is exported."""
    import subprocess
    from long_sequence_sparse_lf_b300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.split()[1:2] == ["T"]}
    exported = {s for s in exported if s.startswith("lf_")}
    assert exported == set(declared_symbols())


def test_version(lib):
    assert lib.lf_version() >= 100


def _pairs_call(lib, H, L, w, dil, G):
    from long_sequence_sparse_lf_b300._binding import _i32_array
    total = ctypes.c_int64(-1)
    st = lib.lf_attn_pairs(H, L, w, _i32_array(dil), _i32_array(G), len(G), None, None, 0,
                           ctypes.byref(total), None)
    return st, lib.lf_last_error().decode()


@pytest.mark.parametrize("args,frag", [
    ((0, 16, 2, [1], []), "H="),
    ((1, 0, 2, [1], []), "L=0"),
    ((1, 16, -1, [1], []), "window"),
    ((1, 16, 2, [0], []), "dilation[0]"),
    ((1, 16, 2, [1], [3, 3]), "strictly increasing"),
    ((1, 16, 2, [1], [16]), "out of"),
    ((1, 16, 2, [1], [-1]), "out of"),
])
def test_pairs_argument_validation(lib, args, frag):
    """Invalid patterns are rejected on the host before any device call."""
    st, msg = _pairs_call(lib, *args)
    assert st == 1, (st, msg)
    assert frag in msg


def test_pairs_null_row_ptr_rejected(lib):
    st, msg = _pairs_call(lib, 1, 16, 2, [1], [])
    assert st == 1 and "row_ptr" in msg


def _fwd_call(lib, fn, B, H, L, D, w, dil, G, scale, ptr=16):
    from long_sequence_sparse_lf_b300._binding import _i32_array
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    st = getattr(lib, fn)(p, p, p, p, B, H, L, D, w, _i32_array(dil), _i32_array(G), len(G),
                          scale, None)
    return st, lib.lf_last_error().decode()


@pytest.mark.parametrize("fn", ["lf_attn_fwd", "lf_attn_fwd_f32"])
@pytest.mark.parametrize("args,code,frag", [
    ((0, 1, 128, 64, 2, [1], [], 0.125), 1, "B="),
    ((1, 1, 128, 64, 2, [1], [], float("nan")), 1, "scale"),
    ((1, 1, 128, 64, 2, [1], [], 0.0), 1, "scale"),
    ((1, 1, 128, 64, 2, [1], [], -1.0), 1, "scale"),
    ((1, 1, 128, 32, 2, [1], [], 0.125), 2, "D=32"),
    ((1, 1, 130, 64, 2, [4], [], 0.125), 2, "multiple"),
    ((1, 2, 128, 64, 2, [1, 0], [], 0.125), 1, "dilation[1]"),
    ((1, 1, 128, 64, 2, [1], [5, 2], 0.125), 1, "strictly"),
])
def test_fwd_argument_validation(lib, fn, args, code, frag):
    st, msg = _fwd_call(lib, fn, *args)
    assert st == code, (st, msg)
    assert frag in msg


def test_fwd_rejects_null_and_misaligned(lib):
    st, msg = _fwd_call(lib, "lf_attn_fwd", 1, 1, 128, 64, 2, [1], [], 0.125, ptr=None)
    assert st == 1 and "NULL" in msg
    st, msg = _fwd_call(lib, "lf_attn_fwd", 1, 1, 128, 64, 2, [1], [], 0.125, ptr=24)
    assert st == 1 and "aligned" in msg


def test_binding_raises_without_cuda_tensors():
    import torch
    from long_sequence_sparse_lf_b300 import lf_attn_fwd
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lf_attn_fwd(q, q, q, q.clone(), 2, [1], [], 0.125)


def _prototypes():
    """name -> (return type, [parameter declarations]) of every LF_API call."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"LF_API\s+([\w\s\*]+?)\b(lf_\w+)\s*\(([^)]*)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        protos[name] = (ret, plist)
    return protos


def _ctype_kind(decl: str) -> str:
    """'ptr', 'i32', 'i64', 'u64', 'f32' or 'other' of a C parameter or return type."""
    d = decl.replace("const", " ").strip()
    if "*" in d or re.search(r"\blf_stream_t\b", d):
        return "ptr"
    if re.search(r"\b(int64_t|long long)\b", d):
        return "i64"
    if re.search(r"\buint64_t\b", d):
        return "u64"
    if re.search(r"\b(int|int32_t|lf_status)\b", d):
        return "i32"
    if re.search(r"\bfloat\b", d):
        return "f32"
    return "other"


def _ctypes_kind(t) -> str:
    if t is None:
        return "void"
    if t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "_type_") and isinstance(
            getattr(t, "_type_", None), type):
        return "ptr"
    return {ctypes.c_int32: "i32", ctypes.c_int: "i32", ctypes.c_int64: "i64",
            ctypes.c_longlong: "i64", ctypes.c_uint64: "u64", ctypes.c_float: "f32"}.get(t, "other")


def test_binding_signatures_match_header(lib):
    """Every call the header declares has ctypes argtypes of the same length
    and kinds (pointer / int32 / int64 / uint64 / float) and the same return
    kind, so the binding and the library cannot drift apart."""
    protos = _prototypes()
    assert set(protos) == set(declared_symbols())
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        got = [_ctypes_kind(t) for t in fn.argtypes]
        want = [_ctype_kind(p) for p in params]
        assert got == want, f"{name}: binding {got} vs header {want}"
        want_ret = "void" if ret == "void" else _ctype_kind(ret)
        assert _ctypes_kind(fn.restype) == want_ret, f"{name}: return {fn.restype} vs {ret}"
