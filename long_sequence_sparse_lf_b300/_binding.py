"""ctypes binding of liblfattn: argument marshalling only.

Every function has the name of the C entry point it calls.  Tensors are
torch tensors (torch supplies device memory and streams); all computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the
library is missing or the device is not a B300 the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblfattn.so")

LF_OK = 0
STATUS_NAMES = {0: "LF_OK", 1: "LF_ERR_INVALID_ARG", 2: "LF_ERR_UNSUPPORTED",
                3: "LF_ERR_CUDA", 4: "LF_ERR_NOMEM", 5: "LF_ERR_TIMEOUT"}

_lib = None


class LfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load_library() -> ctypes.CDLL:
    """Load liblfattn.so (built in-tree); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m long_sequence_sparse_lf_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    ip = ctypes.POINTER(ctypes.c_int32)
    fwd_args = [vp, vp, vp, vp, i32, i32, i32, i32, i32, ip, ip, i32, f32, vp]
    lib.lf_attn_fwd.argtypes = fwd_args
    lib.lf_attn_fwd.restype = i32
    lib.lf_attn_fwd_f32.argtypes = fwd_args
    lib.lf_attn_fwd_f32.restype = i32
    lib.lf_attn_fwd_noalloc.argtypes = fwd_args
    lib.lf_attn_fwd_noalloc.restype = i32
    lib.lf_attn_fwd_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, ip, ip, i32,
                                     f32, vp]
    lib.lf_attn_fwd_host.restype = i32
    lib.lf_attn_pairs.argtypes = [i32, i32, i32, ip, ip, i32, vp, vp, ctypes.c_int64,
                                  ctypes.POINTER(ctypes.c_int64), vp]
    lib.lf_attn_pairs.restype = i32
    lib.lf_last_error.argtypes = []
    lib.lf_last_error.restype = ctypes.c_char_p
    lib.lf_attn_get_status.argtypes = [vp]
    lib.lf_attn_get_status.restype = i32
    lib.lf_plan_cache_clear.argtypes = []
    lib.lf_plan_cache_clear.restype = None
    lib.lf_launch_count.argtypes = []
    lib.lf_launch_count.restype = ctypes.c_uint64
    lib.lf_selftest_wait_timeout.argtypes = [i32, vp]
    lib.lf_selftest_wait_timeout.restype = i32
    lib.lf_version.argtypes = []
    lib.lf_version.restype = i32
    lib.lf_profile_enable.argtypes = [i32]
    lib.lf_profile_enable.restype = None
    lib.lf_profile_only.argtypes = [ctypes.c_char_p]
    lib.lf_profile_only.restype = None
    lib.lf_profile_reset.argtypes = []
    lib.lf_profile_reset.restype = None
    lib.lf_profile_query.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_uint64)]
    lib.lf_profile_query.restype = i32
    lib.lf_layer_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ip, ip,
                                 i32, f32, f32, vp]
    lib.lf_layer_fwd.restype = i32
    lib.lf_attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ip, ip, i32,
                                    f32, vp]
    lib.lf_attn_fwd_lse.restype = i32
    lib.lf_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ip,
                                ip, i32, f32, vp]
    lib.lf_attn_bwd.restype = i32
    lib.lf_attn_fwd_bias.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ip, ip, i32,
                                     f32, vp]
    lib.lf_attn_fwd_bias.restype = i32
    lib.lf_attn_fwd_blocks.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, ip, ip, i32, vp,
                                       i32, i32, f32, vp]
    lib.lf_attn_fwd_blocks.restype = i32
    _lib = lib
    return lib


def _check(status: int):
    if status != LF_OK:
        msg = load_library().lf_last_error().decode("utf-8", "replace")
        raise LfError(status, msg)


def _i32_array(vals: Sequence[int]):
    vals = [int(x) for x in vals]
    arr = (ctypes.c_int32 * max(len(vals), 1))(*vals)
    return arr


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_qkv(q, k, v, out, dtype, device_kind):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if t.device.type != device_kind:
            raise ValueError(f"{name} must be on {device_kind}, got {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError(f"{name} must be [B,H,L,D] like q, got {tuple(t.shape)}")


def lf_attn_fwd(q, k, v, out, w: int, dilation: Sequence[int],
                global_idx: Sequence[int], scale: float, stream=None):
    """bf16 forward on device tensors [B,H,L,D]; writes ``out``."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    lib = load_library()
    _check(lib.lf_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, D,
                           int(w), _i32_array(dilation), _i32_array(global_idx),
                           len(global_idx), float(scale), _stream_handle(stream)))
    return out


def lf_attn_fwd_f32(q, k, v, out, w: int, dilation: Sequence[int],
                    global_idx: Sequence[int], scale: float, stream=None):
    """fp32 forward on device tensors (inputs rounded to bf16 on device)."""
    _check_qkv(q, k, v, out, torch.float32, "cuda")
    B, H, L, D = q.shape
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    lib = load_library()
    _check(lib.lf_attn_fwd_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L,
                               D, int(w), _i32_array(dilation), _i32_array(global_idx),
                               len(global_idx), float(scale), _stream_handle(stream)))
    return out


def lf_attn_fwd_noalloc(q, k, v, out, w: int, dilation: Sequence[int],
                        global_idx: Sequence[int], scale: float, stream=None):
    """bf16 forward through the entry point that allocates no device memory
    (its scratch is a fixed device array of the library; see lfattn.h)."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    lib = load_library()
    _check(lib.lf_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                   L, D, int(w), _i32_array(dilation), _i32_array(global_idx),
                                   len(global_idx), float(scale), _stream_handle(stream)))
    return out


class PreparedFwd:
    """lf_attn_fwd (bf16) or lf_attn_fwd_f32 (fp32) with its arguments
    marshalled once; calling the object runs the forward on the stream given
    here.  The tensors are referenced, not copied: they must keep their
    storage for as long as the object is used."""

    def __init__(self, q, k, v, out, w: int, dilation: Sequence[int],
                 global_idx: Sequence[int], scale: float, stream=None):
        dtype = q.dtype
        if dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("q must be bf16 or fp32")
        _check_qkv(q, k, v, out, dtype, "cuda")
        B, H, L, D = q.shape
        if len(dilation) != H:
            raise ValueError("dilation must have H entries")
        lib = load_library()
        self._fn = lib.lf_attn_fwd if dtype == torch.bfloat16 else lib.lf_attn_fwd_f32
        dil, gi = _i32_array(dilation), _i32_array(global_idx)
        self._keep = (q, k, v, out, dil, gi)
        self.out = out
        st = _stream_handle(stream)
        self._args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, D,
                      int(w), dil, gi, len(global_idx), float(scale), st)

    def __call__(self):
        status = self._fn(*self._args)
        if status != LF_OK:
            _check(status)
        return self.out


def prepare_fwd(q, k, v, out, w: int, dilation: Sequence[int], global_idx: Sequence[int],
                scale: float, stream=None) -> PreparedFwd:
    """The forward of lf_attn_fwd / lf_attn_fwd_f32, marshalled for repeated calls."""
    return PreparedFwd(q, k, v, out, w, dilation, global_idx, scale, stream)


def lf_attn_fwd_host(q, k, v, out, w: int, dilation: Sequence[int],
                     global_idx: Sequence[int], scale: float, stream=None):
    """Forward on HOST tensors (bf16 or fp32); copies in and out, blocks."""
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32")
    _check_qkv(q, k, v, out, dtype, "cpu")
    B, H, L, D = q.shape
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    lib = load_library()
    _check(lib.lf_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                1 if dtype == torch.float32 else 0, B, H, L, D, int(w),
                                _i32_array(dilation), _i32_array(global_idx), len(global_idx),
                                float(scale), _stream_handle(stream)))
    return out


def lf_attn_pairs(H: int, L: int, w: int, dilation: Sequence[int],
                  global_idx: Sequence[int], count_only: bool = False,
                  device=None, stream=None):
    """Key lists in CSR form: (row_ptr int64 [H*L+1], col_idx int32 or None, total)."""
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    device = torch.device("cuda") if device is None else torch.device(device)
    lib = load_library()
    row_ptr = torch.empty(H * L + 1, dtype=torch.int64, device=device)
    total = ctypes.c_int64(0)
    dil, gi = _i32_array(dilation), _i32_array(global_idx)
    st = _stream_handle(stream)
    _check(lib.lf_attn_pairs(H, L, int(w), dil, gi, len(global_idx), row_ptr.data_ptr(), None, 0,
                             ctypes.byref(total), st))
    if count_only:
        return row_ptr, None, int(total.value)
    col = torch.empty(max(int(total.value), 1), dtype=torch.int32, device=device)
    _check(lib.lf_attn_pairs(H, L, int(w), dil, gi, len(global_idx), row_ptr.data_ptr(),
                             col.data_ptr(), col.numel(), ctypes.byref(total), st))
    return row_ptr, col[:int(total.value)], int(total.value)


def lf_last_error() -> str:
    return load_library().lf_last_error().decode("utf-8", "replace")


def lf_attn_get_status(stream=None) -> int:
    """Synchronises the stream; returns the library status (0 = OK)."""
    return int(load_library().lf_attn_get_status(_stream_handle(stream)))


def lf_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (see lfattn.h)."""
    _check(load_library().lf_selftest_wait_timeout(int(timeout_us), _stream_handle(stream)))


def lf_plan_cache_clear() -> None:
    load_library().lf_plan_cache_clear()


def lf_launch_count() -> int:
    return int(load_library().lf_launch_count())


def lf_version() -> int:
    return int(load_library().lf_version())


def lf_profile_enable(on: bool = True) -> None:
    load_library().lf_profile_enable(1 if on else 0)


def lf_profile_only(name=None) -> None:
    """Trace only the kernels whose name contains ``name`` (None = all)."""
    load_library().lf_profile_only(name.encode() if name else None)


def lf_profile_reset() -> None:
    load_library().lf_profile_reset()


def lf_profile_query(name: str = ""):
    """(total device ms, launches) of the traced kernels whose name contains ``name``."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_uint64(0)
    _check(load_library().lf_profile_query(name.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def attention(q, k, v, w: int, dilation: Sequence[int], global_idx: Sequence[int],
              scale: Optional[float] = None, stream=None):
    """Allocate the output and run the forward that matches q's dtype."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty_like(q)
    if q.dtype == torch.float32:
        return lf_attn_fwd_f32(q, k, v, out, w, dilation, global_idx, scale, stream)
    return lf_attn_fwd(q, k, v, out, w, dilation, global_idx, scale, stream)


def lf_layer_fwd(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, out, H: int, w: int,
                 dilation: Sequence[int], global_idx: Sequence[int], scale: float,
                 eps: float = 1e-5, stream=None):
    """One Longformer layer forward (see lf_layer_fwd in include/lfattn.h).

    x, out: bf16 cuda [B, L, hidden]; w_qkv bf16 [3*hidden, hidden]; b_qkv
    fp32 [3*hidden]; w_ff bf16 [hidden, hidden]; b_ff fp32 [hidden]; ln1, ln2
    fp32 [2*hidden] (gamma, then beta).  Writes ``out``."""
    if x.dim() != 3:
        raise ValueError("x must be [B, L, hidden]")
    B, L, hidden = x.shape
    shapes = (("x", x, torch.bfloat16, (B, L, hidden)),
              ("w_qkv", w_qkv, torch.bfloat16, (3 * hidden, hidden)),
              ("b_qkv", b_qkv, torch.float32, (3 * hidden,)),
              ("w_ff", w_ff, torch.bfloat16, (hidden, hidden)),
              ("b_ff", b_ff, torch.float32, (hidden,)),
              ("ln1", ln1, torch.float32, (2 * hidden,)),
              ("ln2", ln2, torch.float32, (2 * hidden,)),
              ("out", out, torch.bfloat16, (B, L, hidden)))
    for name, t, dt, shp in shapes:
        if not isinstance(t, torch.Tensor) or t.dtype != dt or t.device.type != "cuda":
            raise TypeError(f"{name} must be a {dt} cuda tensor")
        if not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be contiguous with shape {shp}, got {tuple(t.shape)}")
    if len(dilation) != H:
        raise ValueError("dilation must have H entries")
    lib = load_library()
    _check(lib.lf_layer_fwd(x.data_ptr(), w_qkv.data_ptr(), b_qkv.data_ptr(), w_ff.data_ptr(),
                            b_ff.data_ptr(), ln1.data_ptr(), ln2.data_ptr(), out.data_ptr(),
                            B, L, hidden, H, int(w), _i32_array(dilation),
                            _i32_array(global_idx), len(global_idx), float(scale), float(eps),
                            _stream_handle(stream)))


def lf_attn_fwd_lse(q, k, v, out, lse, w: int, dilation: Sequence[int],
                    global_idx: Sequence[int], scale: float, stream=None):
    """bf16 forward that also writes lse (fp32 cuda [B,H,L]), the row's
    log-sum-exp of the scaled scores over its key set."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, L) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,H,L]")
    lib = load_library()
    _check(lib.lf_attn_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), B, H, L, D, int(w), _i32_array(dilation),
                               _i32_array(global_idx), len(global_idx), float(scale),
                               _stream_handle(stream)))


def lf_attn_fwd_bias(q, k, v, out, rel_bias, w: int, dilation: Sequence[int],
                     global_idx: Sequence[int], scale: float, stream=None):
    """bf16 forward with a relative-position bias on the window's scores:
    rel_bias is fp32 cuda [H, 2w+1] with |values| <= 1e4; a non-global row i
    gains rel_bias[h, t + w] on the score of its window key i + d*t."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    if (rel_bias.dtype != torch.float32 or rel_bias.device.type != "cuda"
            or tuple(rel_bias.shape) != (H, 2 * int(w) + 1) or not rel_bias.is_contiguous()):
        raise ValueError("rel_bias must be a contiguous fp32 cuda tensor [H, 2w+1]")
    lib = load_library()
    _check(lib.lf_attn_fwd_bias(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                rel_bias.data_ptr(), B, H, L, D, int(w), _i32_array(dilation),
                                _i32_array(global_idx), len(global_idx), float(scale),
                                _stream_handle(stream)))


def lf_attn_fwd_blocks(q, k, v, out, w: int, dilation: Sequence[int],
                       global_idx: Sequence[int], xblocks, scale: float, stream=None):
    """bf16 forward with extra key blocks per 128-query tile (BigBird random
    or strided blocks): xblocks is an integer table [H, T, R] (host; -1 for
    none) whose row r*nqt + qt lists the key blocks of tile qt of residue
    class r, nqt = ceil(ceil(L/d) / 128)."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    tab = torch.as_tensor(xblocks).to(dtype=torch.int32, device="cpu").contiguous()
    if tab.dim() != 3 or tab.shape[0] != H:
        raise ValueError(f"xblocks must be [H, T, R] with H={H}, got {tuple(tab.shape)}")
    lib = load_library()
    _check(lib.lf_attn_fwd_blocks(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  B, H, L, D, int(w), _i32_array(dilation),
                                  _i32_array(global_idx), len(global_idx), tab.data_ptr(),
                                  int(tab.shape[1]), int(tab.shape[2]), float(scale),
                                  _stream_handle(stream)))


def lf_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, w: int, dilation: Sequence[int],
                global_idx: Sequence[int], scale: float, stream=None):
    """Gradients dq, dk, dv (fp32 cuda [B,H,L,D]) of sum(out * dout); q, k,
    v, out, dout bf16 cuda [B,H,L,D]; lse from lf_attn_fwd_lse."""
    _check_qkv(q, k, v, out, torch.bfloat16, "cuda")
    B, H, L, D = q.shape
    if dout.dtype != torch.bfloat16 or dout.shape != q.shape or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous bf16 tensor like q")
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t.dtype != torch.float32 or t.shape != q.shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 tensor like q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, L) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,H,L]")
    lib = load_library()
    _check(lib.lf_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), B, H, L, D, int(w), _i32_array(dilation),
                           _i32_array(global_idx), len(global_idx), float(scale),
                           _stream_handle(stream)))
