"""The allocation-free forward (lf_attn_fwd_noalloc).

Some callers cannot let a library allocate device memory: engines that plan
all memory at start-up and forbid allocation afterwards, and processes whose
caching allocator already holds the free device memory.  lf_attn_fwd_noalloc
serves them from one fixed device array of the library.  These checks call it
through the C ABI:
  * twice in a row on different problems (so the second call runs on
    whatever the first left in the shared array), each output equal bit for
    bit to lf_attn_fwd's on the same inputs (the same kernels on the same
    work list), and one output against the fp64 oracle on sampled rows;
  * in a fresh process, that a call on a pattern the library has never seen
    leaves the device's free memory unchanged, while lf_attn_fwd on another
    new pattern lowers it, and that the first call leaves a clean status;
  * a problem whose scratch does not fit is rejected.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
REL_L2 = 5e-3
BF16_HALF_ULP = 2.0 ** -8


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


def _close(got, ref, what):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    d = np.abs(g - r) - BF16_HALF_ULP * np.abs(r)
    rel = float(np.linalg.norm((g - r).ravel()) / max(np.linalg.norm(r.ravel()), 1e-300))
    assert float(d.max()) <= MAX_ABS and rel <= REL_L2, \
        f"{what}: max_abs={float(d.max()):.3e} rel_l2={rel:.3e}"


def _problem(wl):
    q, k, v = (t.cuda() for t in W.make_qkv(wl))
    return q, k, v


# a QA-like problem with dilated heads and more than 128 global tokens, and
# the L=4096 workload with one global token
SMALL = W.custom("qa-dilated", 2, 4, 2048, 64, 128, (1, 2, 1, 4), tuple(range(0, 2048, 13)), 21)
BASE = W.CONFIGS["base"]


def test_noalloc_matches_fwd_on_two_calls_in_a_row(lf):
    results = []
    for wl in (SMALL, BASE):
        q, k, v = _problem(wl)
        ref = torch.empty_like(q)
        lf.lf_attn_fwd(q, k, v, ref, wl.w, wl.dilation, wl.global_idx, wl.scale)
        out = torch.full_like(q, float("nan"))
        lf.lf_attn_fwd_noalloc(q, k, v, out, wl.w, wl.dilation, wl.global_idx, wl.scale)
        assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
        results.append((wl, q, k, v, out, ref))
    for wl, q, k, v, out, ref in results:
        assert torch.equal(out, ref), wl.name
    # the first problem against the oracle on sampled rows (dilated heads,
    # 158 global tokens)
    from oracle import lf_oracle as O
    wl, q, k, v, out, _ = results[0]
    rows = sorted(set(range(0, 140)) | set(range(wl.L - 140, wl.L)) |
                  set(np.random.default_rng(3).integers(0, wl.L, 64).tolist()))
    f64 = lambda t: t.cpu().double().numpy()   # noqa: E731
    ref = O.attention(f64(q), f64(k), f64(v), wl.w, wl.dilation, wl.global_idx, wl.scale,
                      rows=rows)
    _close(out[:, :, rows], torch.from_numpy(ref), wl.name + " vs oracle")


def test_noalloc_repeated_call_same_result(lf):
    wl = SMALL
    q, k, v = _problem(wl)
    ref = torch.empty_like(q)
    lf.lf_attn_fwd(q, k, v, ref, wl.w, wl.dilation, wl.global_idx, wl.scale)
    for rep in range(2):
        out = torch.full_like(q, float("nan"))
        lf.lf_attn_fwd_noalloc(q, k, v, out, wl.w, wl.dilation, wl.global_idx, wl.scale)
        assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
        assert torch.equal(out, ref), f"call {rep}"


# Run in a fresh process: the library's module (and with it the fixed
# array) loads on its first use on the device, and the device's free memory
# is read before and after calls on patterns the library has not seen.
_FREE_MEMORY_SCRIPT = r"""
import sys
import torch
sys.path.insert(0, sys.argv[1])
import long_sequence_sparse_lf_b300 as lf
from long_sequence_sparse_lf_b300 import workloads as W
lf.load_library()
torch.cuda.init()

def qkv(wl):
    return [t.cuda() for t in W.make_qkv(wl)]

first = W.custom("first", 1, 2, 1024, 64, 32, (1, 1), (0, 7), 31)
unseen = W.custom("unseen", 2, 4, 2048, 64, 96, (1, 2, 1, 4), tuple(range(0, 2048, 11)), 32)
other = W.custom("other", 2, 16, 4096, 64, 256, (1,) * 16, tuple(range(64)), 33)
a, b, c = qkv(first), qkv(unseen), qkv(other)
outs = [torch.empty_like(x[0]) for x in (a, b, c)]
torch.cuda.synchronize()

# the first call on the device: clean status afterwards
lf.lf_attn_fwd_noalloc(*a, outs[0], first.w, first.dilation, first.global_idx, first.scale)
torch.cuda.synchronize()
assert lf.lf_attn_get_status() == 0, lf.lf_last_error()

free0 = torch.cuda.mem_get_info()[0]
lf.lf_attn_fwd_noalloc(*b, outs[1], unseen.w, unseen.dilation, unseen.global_idx, unseen.scale)
torch.cuda.synchronize()
assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
free1 = torch.cuda.mem_get_info()[0]

lf.lf_attn_fwd(*c, outs[2], other.w, other.dilation, other.global_idx, other.scale)
torch.cuda.synchronize()
assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
free2 = torch.cuda.mem_get_info()[0]
print("free bytes", free0, free1, free2)
assert free1 == free0, ("the allocation-free call changed free memory", free0, free1)
assert free2 < free1, ("lf_attn_fwd on a new pattern did not allocate", free1, free2)
print("ok")
"""


def test_noalloc_allocates_nothing_in_a_fresh_process():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FREE_MEMORY_SCRIPT, root],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_noalloc_rejects_problems_beyond_its_scratch(lf):
    """B=1, H=16, L=65536, D=128 with 16 global tokens needs more scratch
    than the fixed array holds; the call fails before touching any tensor."""
    from long_sequence_sparse_lf_b300._binding import _i32_array
    wl = W.CONFIGS["long"]
    lib = lf.load_library()
    dummy = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    st = lib.lf_attn_fwd_noalloc(p, p, p, p, wl.B, wl.H, wl.L, wl.D, wl.w,
                                 _i32_array(wl.dilation), _i32_array(wl.global_idx),
                                 len(wl.global_idx), ctypes.c_float(wl.scale), None)
    assert st == 2, (st, lf.lf_last_error())
    msg = lf.lf_last_error()
    assert "bytes of scratch" in msg and str(32 << 20) in msg, msg
    torch.cuda.synchronize()
