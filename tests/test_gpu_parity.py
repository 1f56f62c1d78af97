"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerance, in float64 on the same bf16-rounded inputs:
  * the five workloads (tiny, base, dilated, qa, long): the plain bound,
    max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 5e-3,
    on every output element of tiny, base, dilated and qa, and on a row
    sample of long (edges, around globals, random rows); the measured values
    are printed;
  * the other shapes (randomised, with outputs up to |out| of a few units):
    each element may also differ by the bf16 output's own rounding,
    2^-8 * |oracle| (a bf16 value cannot be nearer the exact result than
    half its step), on top of 1e-2; fp32 outputs get no allowance.
Key lists are compared bit-exactly: in full for tiny, base, dilated and qa,
and for long the totals and a row sample.
"""
import math

import numpy as np
import pytest
import torch

from oracle import lf_oracle as O
from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
REL_L2 = 5e-3


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


BF16_HALF_ULP = 2.0 ** -8


def _errors(got, ref, out_bf16=True):
    d = np.abs(got - ref)
    if out_bf16:
        d = d - BF16_HALF_ULP * np.abs(ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
    return float(d.max()), rel


def _assert_close(got, ref, what="", out_bf16=True):
    mx, rel = _errors(got, ref, out_bf16)
    assert mx <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={mx:.3e} rel_l2={rel:.3e}"
    return mx, rel


def _assert_plain(got, ref, what):
    """The workloads' bound with no allowance for the output's rounding."""
    mx, rel = _errors(got, ref, out_bf16=False)
    print(f"{what}: max_abs={mx:.3e} rel_l2={rel:.3e} elements={got.size}")
    assert mx <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={mx:.3e} rel_l2={rel:.3e}"
    return mx, rel


def _run(lf, q, k, v, w, dil, G, scale):
    """q, k, v: CPU tensors (bf16 or fp32).  Returns the output as float64."""
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = lf.attention(qd, kd, vd, w, dil, G, scale)
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    return out.float().cpu().double().numpy()


def _inputs(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(shape, generator=g).to(dtype) for _ in range(3))


def _f64(t):
    return t.to(torch.bfloat16).double().numpy()


# ------------------------------------------------------------- tiny config

def test_tiny_config_full_parity(lf):
    wl = W.CONFIGS["tiny"]
    q, k, v = W.make_qkv(wl)
    got = _run(lf, q, k, v, wl.w, wl.dilation, wl.global_idx, wl.scale)
    ref = O.attention(_f64(q), _f64(k), _f64(v), wl.w, wl.dilation, wl.global_idx, wl.scale)
    _assert_plain(got, ref, "tiny")


# ------------------------------------------------ closed-form special cases

def test_zero_q_gives_mean_over_key_set(lf):
    """q = 0 makes every attended score equal: out_i = mean of v over K(i)."""
    B, H, L, D, w = 1, 2, 300, 64, 40
    dil, G = [1, 3], (0, 150, 299)
    _, k, v = _inputs((B, H, L, D), 7)
    q = torch.zeros_like(k)
    got = _run(lf, q, k, v, w, dil, G, 0.125)
    vf = _f64(v)
    ref = np.empty_like(vf)
    for h in range(H):
        for i in range(L):
            ks = O.key_set(i, L, w, dil[h], G)
            ref[0, h, i] = vf[0, h, ks].mean(axis=0)
    _assert_close(got, ref, "q=0")


def test_window_zero_no_globals_is_identity(lf):
    B, H, L, D = 2, 2, 256, 64
    q, k, v = _inputs((B, H, L, D), 8)
    got = _run(lf, q, k, v, 0, [1, 2], (), 0.125)
    np.testing.assert_array_equal(got, _f64(v))


def test_full_window_is_full_attention(lf):
    B, H, L, D = 1, 2, 384, 64
    q, k, v = _inputs((B, H, L, D), 9)
    got = _run(lf, q, k, v, L, [1, 1], (), 1 / 8)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(_f64(t)) for t in (q, k, v)), scale=1 / 8).numpy()
    _assert_close(got, ref, "full window")


# ------------------------------------------------------ randomised shapes

SHAPES = [
    # B, H, L, D, w, dilation, globals
    (1, 1, 128, 64, 127, [1], ()),
    (1, 1, 128, 64, 5, [1], ()),
    (1, 2, 1000, 64, 70, [1, 2], (0, 999)),          # ragged tail, even L for d=2
    (2, 1, 777, 64, 64, [1], (3, 400, 776)),
    (1, 2, 640, 128, 100, [1, 1], (0, 1, 2, 3)),
    (1, 3, 768, 64, 33, [1, 2, 3], tuple(range(0, 768, 5))),  # n_g = 154 > 128
    (1, 1, 512, 64, 600, [1], (10,)),                  # w > L
    (1, 2, 256, 128, 0, [1, 4], (100,)),               # w = 0 with a global
    (2, 2, 1024, 64, 256, [1, 1], tuple(range(64))),   # QA-like
    (1, 1, 300, 64, 20, [1], tuple(range(300))),       # every row global
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}L{}D{}w{}".format(*s[:5]))
def test_random_shapes_parity(lf, shape):
    B, H, L, D, w, dil, G = shape
    q, k, v = _inputs((B, H, L, D), 100 + L + w)
    scale = 1 / math.sqrt(D)
    got = _run(lf, q, k, v, w, dil, G, scale)
    ref = O.attention(_f64(q), _f64(k), _f64(v), w, dil, G, scale)
    _assert_close(got, ref, str(shape[:5]))


def test_fp32_path_matches_oracle_on_rounded_inputs(lf):
    """fp32 inputs are rounded to bf16 first, so they match the oracle on the
    rounded values (fp32 output, no final rounding)."""
    B, H, L, D, w = 1, 2, 500, 64, 30
    q, k, v = _inputs((B, H, L, D), 11, dtype=torch.float32)
    got = _run(lf, q, k, v, w, [1, 2], (0, 1), 0.125)
    ref = O.attention(_f64(q), _f64(k), _f64(v), w, [1, 2], (0, 1), 0.125)
    _assert_close(got, ref, "fp32 path", out_bf16=False)


def test_repeat_calls_are_deterministic(lf):
    B, H, L, D, w = 1, 2, 1024, 64, 128
    q, k, v = _inputs((B, H, L, D), 12)
    a = _run(lf, q, k, v, w, [1, 2], (0,), 0.125)
    b = _run(lf, q, k, v, w, [1, 2], (0,), 0.125)
    np.testing.assert_array_equal(a, b)


# -------------------------------------------------------- full-size configs

@pytest.mark.parametrize("name", ["base", "dilated", "qa"])
def test_config_full_size_every_element(lf, name):
    """The full-size workload in the bench's launch configuration, every
    output element against the oracle (about 1e11 to 3e11 fp64 FLOP each on
    the host)."""
    wl = W.CONFIGS[name]
    q, k, v = W.make_qkv(wl)
    got = _run(lf, q, k, v, wl.w, wl.dilation, wl.global_idx, wl.scale)
    ref = O.attention(_f64(q), _f64(k), _f64(v), wl.w, wl.dilation, wl.global_idx, wl.scale)
    _assert_plain(got, ref, name)


def _sample_rows(wl, n_extra, seed):
    L = wl.L
    rows = set(range(0, min(L, 130))) | set(range(max(0, L - 130), L))
    for g in wl.global_idx[:8]:
        rows.update(x for x in (g - 1, g, g + 1, g + wl.w, g - wl.w) if 0 <= x < L)
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, L, n_extra).tolist())
    return sorted(rows)


def test_config_long_sampled_rows(lf):
    """B=1, H=16, L=65536, D=128: the oracle's full cost (3.5e13 fp64 FLOP)
    is out of reach, so a row sample (edges, around globals, random) is
    compared, and every row is checked to be finite."""
    wl = W.CONFIGS["long"]
    q, k, v = W.make_qkv(wl)
    got = _run(lf, q, k, v, wl.w, wl.dilation, wl.global_idx, wl.scale)
    rows = _sample_rows(wl, 64, wl.seed)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    ref = O.attention(qf, kf, vf, wl.w, wl.dilation, wl.global_idx, wl.scale, rows=rows)
    _assert_plain(got[:, :, rows], ref, "long (sampled rows)")
    assert np.isfinite(got).all()


# ------------------------------------------------------------ key lists

PAIR_PATTERNS = [
    (2, 512, 32, [1, 1], (0, 1)),
    (3, 97, 5, [1, 2, 3], (0, 50, 96)),
    (2, 64, 100, [1, 2], ()),
    (1, 40, 0, [4], (7,)),
    (2, 300, 20, [2, 5], tuple(range(0, 300, 3))),
    (1, 33, 3, [1], tuple(range(33))),
]


@pytest.mark.parametrize("pat", PAIR_PATTERNS, ids=lambda p: "H{}L{}w{}".format(*p[:3]))
def test_pairs_bit_exact_small(lf, pat):
    H, L, w, dil, G = pat
    row_ptr, col, total = lf.lf_attn_pairs(H, L, w, dil, G)
    rp_ref, col_ref = O.key_lists(L, w, dil, G)
    assert total == int(rp_ref[-1]) == sum(O.pair_count(L, w, d, G) for d in dil)
    np.testing.assert_array_equal(row_ptr.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(col.cpu().numpy(), col_ref)


@pytest.mark.parametrize("name", ["tiny", "base", "dilated", "qa"])
def test_pairs_configs_full(lf, name):
    """Every key list of the workload's pattern, bit-exact against the
    oracle's enumeration, and the total against the closed form."""
    wl = W.CONFIGS[name]
    row_ptr, col, total = lf.lf_attn_pairs(wl.H, wl.L, wl.w, wl.dilation, wl.global_idx)
    rp_ref, col_ref = O.key_lists(wl.L, wl.w, wl.dilation, wl.global_idx)
    assert total == int(rp_ref[-1]) == O.total_pairs(wl.L, wl.w, wl.dilation, wl.global_idx)
    np.testing.assert_array_equal(row_ptr.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(col.cpu().numpy(), col_ref)


def test_pairs_long_total_and_sampled_rows(lf):
    """long: the whole CSR is built on the device (1.1e9 entries, 4.4 GB);
    the total is checked against the closed form and a sample of rows
    (edges, globals, random) bit-exactly against the oracle's lists."""
    wl = W.CONFIGS["long"]
    H = wl.H
    row_ptr, col, total = lf.lf_attn_pairs(H, wl.L, wl.w, wl.dilation, wl.global_idx)
    assert total == O.total_pairs(wl.L, wl.w, wl.dilation, wl.global_idx)
    rp = row_ptr.cpu().numpy()
    rng = np.random.default_rng(5)
    rows = [(h, i) for h in range(H) for i in
            sorted(set(rng.integers(0, wl.L, 40).tolist()) | {0, 1, wl.L - 2, wl.L - 1}
                   | set(wl.global_idx[:3]))]
    _, col_ref = O.key_lists(wl.L, wl.w, wl.dilation, wl.global_idx, rows=rows)
    got = torch.cat([col[int(rp[h * wl.L + i]):int(rp[h * wl.L + i + 1])] for h, i in rows])
    np.testing.assert_array_equal(got.cpu().numpy(), col_ref)
    del col
    torch.cuda.empty_cache()


def test_pairs_capacity_error(lf):
    import ctypes
    lib = lf.load_library()
    from long_sequence_sparse_lf_b300._binding import _i32_array
    rp = torch.empty(2 * 100 + 1, dtype=torch.int64, device="cuda")
    col = torch.empty(10, dtype=torch.int32, device="cuda")
    total = ctypes.c_int64(0)
    st = lib.lf_attn_pairs(2, 100, 3, _i32_array([1, 1]), _i32_array([]), 0, rp.data_ptr(),
                           col.data_ptr(), 10, ctypes.byref(total), None)
    assert st == 1
    assert total.value == 2 * O.pair_count(100, 3, 1, ())
