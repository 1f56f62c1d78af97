"""The allocation-free forward (lf_attn_fwd_noalloc) against lf_attn_fwd.

Some callers cannot let a library allocate device memory: engines that plan
all memory at start-up and forbid allocation afterwards, and processes whose
caching allocator already holds the free device memory.  lf_attn_fwd_noalloc
serves them from one fixed device array of the library.  These checks call it
through the C ABI, twice in a row on different problems (so the second call
runs on whatever the first left in the shared array), and compare each output
with lf_attn_fwd's on the same inputs, within the parity tolerance of the
other GPU tests.  A problem whose scratch does not fit is rejected.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

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
        results.append((wl.name, out, ref))
    for name, out, ref in results:
        _close(out, ref, name)


def test_noalloc_repeated_call_same_result(lf):
    wl = SMALL
    q, k, v = _problem(wl)
    ref = torch.empty_like(q)
    lf.lf_attn_fwd(q, k, v, ref, wl.w, wl.dilation, wl.global_idx, wl.scale)
    for rep in range(2):
        out = torch.full_like(q, float("nan"))
        lf.lf_attn_fwd_noalloc(q, k, v, out, wl.w, wl.dilation, wl.global_idx, wl.scale)
        assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
        _close(out, ref, f"call {rep}")


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
