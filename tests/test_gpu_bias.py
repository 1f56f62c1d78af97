"""The relative-position-bias forward (lf_attn_fwd_bias) against the oracle's
attention(..., rel_bias=...), on bf16 inputs and an fp32 bias table.

Tolerance as the plain forward's: per element max |gpu - oracle| <= 1e-2
beyond half a bf16 ulp of the output, rel-L2 <= 5e-3.  With a zero table the
biased kernel adds +0.0 to every score, so it must reproduce lf_attn_fwd bit
for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import lf_oracle as O
from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
REL_L2 = 5e-3
BF16_HALF_ULP = 2.0 ** -8
LF_ERR_INVALID_ARG = 1


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


def _assert_close(got, ref, what=""):
    d = np.abs(got - ref) - BF16_HALF_ULP * np.abs(ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))
    assert d.max() <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={d.max():.3e} rel_l2={rel:.3e}"


def _inputs(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(shape, generator=g).to(torch.bfloat16) for _ in range(3))


def _bias(H, w, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    return (sigma * torch.randn((H, 2 * w + 1), generator=g)).float()


def _run_bias(lf, q, k, v, rb, w, dil, G, scale):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = torch.empty_like(qd)
    lf.lf_attn_fwd_bias(qd, kd, vd, out, rb.cuda(), w, dil, G, scale)
    torch.cuda.synchronize()
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    return out


CASES = [
    # B, H, L, D, w, dilation, globals
    (1, 2, 700, 64, 40, (1, 2), (0, 1, 333)),
    (2, 3, 1002, 64, 100, (1, 3, 1), (5, 1001)),
    (1, 2, 900, 128, 64, (2, 1), (0, 450, 899)),
    (1, 2, 513, 64, 300, (1, 1), ()),
    (1, 1, 200, 128, 7, (4,), (17,)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}L{c[2]}D{c[3]}w{c[4]}" for c in CASES])
def test_bias_forward_matches_oracle(lf, case):
    B, H, L, D, w, dil, G = case
    q, k, v = _inputs((B, H, L, D), 40 + L)
    rb = _bias(H, w, 7 + L, sigma=2.0)
    scale = 1.0 / np.sqrt(D)
    got = _run_bias(lf, q, k, v, rb, w, dil, G, scale).float().cpu().double().numpy()
    ref = O.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), w, dil, G, scale,
                      rel_bias=rb.double().numpy())
    _assert_close(got, ref, str(case))


def test_zero_bias_is_bit_identical_to_plain_forward(lf):
    B, H, L, D, w, dil, G = 2, 2, 1500, 64, 128, (1, 2), (0, 64, 1499)
    q, k, v = _inputs((B, H, L, D), 3)
    scale = 0.125
    got = _run_bias(lf, q, k, v, torch.zeros((H, 2 * w + 1)), w, dil, G, scale)
    plain = lf.attention(q.cuda(), k.cuda(), v.cuda(), w, dil, G, scale)
    torch.cuda.synchronize()
    assert torch.equal(got, plain)


def test_bias_keeping_only_offset_zero_returns_v(lf):
    """No globals; every window offset but 0 carries -1e4 (the largest
    magnitude the entry accepts): each row keeps only itself (the others'
    weights fall below 2^-125), so out equals v (bf16 in, bf16 out)."""
    B, H, L, D, w = 1, 2, 642, 64, 50
    q, k, v = _inputs((B, H, L, D), 4)
    rb = torch.full((H, 2 * w + 1), -1e4)
    rb[:, w] = 0.0
    got = _run_bias(lf, q, k, v, rb, w, (1, 3), (), 0.125)
    assert torch.equal(got.cpu(), v)


def test_base_config_sampled_rows(lf):
    """The 4096-token base workload with a random table, sampled rows."""
    wl = W.CONFIGS["base"]
    q, k, v = W.make_qkv(wl)
    rb = _bias(wl.H, wl.w, 11)
    got = _run_bias(lf, q, k, v, rb, wl.w, wl.dilation, wl.global_idx, wl.scale)
    got = got.float().cpu().double().numpy()
    rng = np.random.default_rng(5)
    rows = sorted(set(range(0, 130)) | set(range(wl.L - 130, wl.L)) | set(wl.global_idx)
                  | set(rng.integers(0, wl.L, 128).tolist()))
    ref = O.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), wl.w,
                      wl.dilation, wl.global_idx, wl.scale, rows=rows,
                      rel_bias=rb.double().numpy())
    _assert_close(got[:, :, rows], ref, "base")
    assert np.isfinite(got).all()


def test_bias_argument_errors(lf):
    q, k, v = _inputs((1, 2, 256, 64), 1)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = torch.empty_like(qd)
    with pytest.raises(ValueError):
        lf.lf_attn_fwd_bias(qd, kd, vd, out, torch.zeros((2, 5), device="cuda"), 3, (1, 1), (), 0.1)
    # a null table through the C entry: an argument error, nothing launched
    lib = lf.load_library()
    dil = (ctypes.c_int32 * 2)(1, 1)
    st = lib.lf_attn_fwd_bias(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), None,
                              1, 2, 256, 64, 3, dil, None, 0, 0.1, None)
    assert st == LF_ERR_INVALID_ARG
