"""The forward with extra key blocks per query tile (lf_attn_fwd_blocks:
BigBird random blocks or a strided choice) against the oracle's
attention(..., xblocks=...), bf16 in and out.

Tolerance as the plain forward's: per element max |gpu - oracle| <= 1e-2
beyond half a bf16 ulp of the output, rel-L2 <= 5e-3.  A table of -1 only
must reproduce lf_attn_fwd bit for bit (no block is added, and the order of
the remaining arithmetic is the same).
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


def _run(lf, q, k, v, w, dil, G, tab, scale):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = torch.empty_like(qd)
    lf.lf_attn_fwd_blocks(qd, kd, vd, out, w, dil, G, tab, scale)
    torch.cuda.synchronize()
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    return out


def _ref(q, k, v, w, dil, G, tab, scale, rows=None):
    return O.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), w, dil, G,
                       scale, rows=rows, xblocks=np.asarray(tab))


CASES = [
    # B, H, L, D, w, dilation, globals, table
    (1, 2, 700, 64, 40, (1, 2), (0, 1, 333), ("random", 3)),
    (2, 3, 1002, 64, 100, (1, 3, 1), (5, 600, 1001), ("random", 2)),
    (1, 2, 900, 128, 64, (2, 1), (0, 450, 899), ("random", 3)),
    (1, 2, 1536, 64, 32, (1, 2), (700,), ("strided", 3)),
    (1, 2, 513, 64, 300, (1, 1), (), ("random", 4)),
    (1, 1, 2048, 128, 8, (4,), (17, 1000), ("random", 2)),
]


def _table(kind, L, dil, seed):
    if kind[0] == "random":
        return W.random_blocks(L, dil, kind[1], seed)
    return W.strided_blocks(L, dil, kind[1])


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}L{c[2]}D{c[3]}w{c[4]}{c[7][0]}"
                                             for c in CASES])
def test_blocks_forward_matches_oracle(lf, case):
    B, H, L, D, w, dil, G, kind = case
    q, k, v = _inputs((B, H, L, D), 60 + L)
    tab = _table(kind, L, dil, 9 + L)
    scale = 1.0 / np.sqrt(D)
    got = _run(lf, q, k, v, w, dil, G, tab, scale).float().cpu().double().numpy()
    _assert_close(got, _ref(q, k, v, w, dil, G, tab, scale), str(case))


def test_duplicate_and_in_window_entries(lf):
    """Entries repeated within a row and blocks inside the window (dropped
    by the planner, or masked column by column) add each key once."""
    B, H, L, D, w, dil, G = 1, 2, 1024, 64, 150, (1, 2), (3, 520)
    q, k, v = _inputs((B, H, L, D), 5)
    T = W.block_table_rows(L, dil)
    tab = torch.full((H, T, 4), -1, dtype=torch.int32)
    for h, d in enumerate(dil):
        nqt = W.tiles_per_class(L, d)
        for row in range(d * nqt):
            qt = row % nqt
            # the tile's own block twice, its neighbour, and the last block
            tab[h, row] = torch.tensor([qt, qt, min(qt + 1, nqt - 1), nqt - 1])
    got = _run(lf, q, k, v, w, dil, G, tab, 0.125).float().cpu().double().numpy()
    _assert_close(got, _ref(q, k, v, w, dil, G, tab, 0.125), "duplicates")


def test_empty_table_is_bit_identical_to_plain_forward(lf):
    B, H, L, D, w, dil, G = 2, 2, 1500, 64, 128, (1, 2), (0, 64, 1499)
    q, k, v = _inputs((B, H, L, D), 3)
    tab = torch.full((H, W.block_table_rows(L, dil), 2), -1, dtype=torch.int32)
    got = _run(lf, q, k, v, w, dil, G, tab, 0.125)
    plain = lf.attention(q.cuda(), k.cuda(), v.cuda(), w, dil, G, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(got, plain)


def test_every_block_listed_is_dense_attention(lf):
    """d = 1, no globals, every tile listing every block: dense softmax
    attention, checked against torch on the same bf16 values."""
    B, H, L, D, w = 1, 2, 1000, 64, 20
    q, k, v = _inputs((B, H, L, D), 8)
    nqt = W.tiles_per_class(L, 1)
    tab = torch.arange(nqt, dtype=torch.int32).repeat(H, nqt, 1)
    got = _run(lf, q, k, v, w, (1, 1), (), tab, 0.125).float().cpu().double()
    qf, kf, vf = (t.double() for t in (q, k, v))
    want = torch.softmax(0.125 * qf @ kf.transpose(-1, -2), dim=-1) @ vf
    _assert_close(got.numpy(), want.numpy(), "dense")


def test_base_config_random_blocks_sampled_rows(lf):
    """The 4096-token base workload with BigBird-style random blocks
    (3 per tile), sampled rows."""
    wl = W.CONFIGS["base"]
    q, k, v = W.make_qkv(wl)
    tab = W.random_blocks(wl.L, wl.dilation, 3, 21)
    got = _run(lf, q, k, v, wl.w, wl.dilation, wl.global_idx, tab, wl.scale)
    got = got.float().cpu().double().numpy()
    rng = np.random.default_rng(6)
    rows = sorted(set(range(0, 130)) | set(range(wl.L - 130, wl.L)) | set(wl.global_idx)
                  | set(rng.integers(0, wl.L, 128).tolist()))
    ref = _ref(q, k, v, wl.w, wl.dilation, wl.global_idx, tab, wl.scale, rows=rows)
    _assert_close(got[:, :, rows], ref, "base")
    assert np.isfinite(got).all()


def test_many_tables_evict_and_stay_correct(lf):
    """40 distinct random tables in a row (past the 32 the library caches, so
    the cached ones are freed once on the way); outputs stay right, and an
    evicted table works again when it comes back."""
    B, H, L, D, w, dil, G = 1, 2, 768, 64, 24, (1, 2), (5,)
    q, k, v = _inputs((B, H, L, D), 12)
    tabs = [W.random_blocks(L, dil, 2, 100 + n) for n in range(40)]
    outs = [_run(lf, q, k, v, w, dil, G, t, 0.125).float().cpu().double().numpy()
            for t in tabs]
    for n in (0, 31, 32, 39):
        _assert_close(outs[n], _ref(q, k, v, w, dil, G, tabs[n], 0.125), f"table {n}")
    again = _run(lf, q, k, v, w, dil, G, tabs[0], 0.125).float().cpu().double().numpy()
    assert np.array_equal(again, outs[0])


def test_table_errors(lf):
    q, k, v = _inputs((1, 2, 512, 64), 1)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = torch.empty_like(qd)
    lib = lf.load_library()
    dil = (ctypes.c_int32 * 2)(1, 1)

    def call(tab):
        tab = torch.as_tensor(tab, dtype=torch.int32).contiguous()
        return lib.lf_attn_fwd_blocks(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                      out.data_ptr(), 1, 2, 512, 64, 8, dil, None, 0,
                                      tab.data_ptr(), tab.shape[1], tab.shape[2], 0.1, None)

    assert call(torch.zeros((2, 4, 1))) == 0                 # 4 tiles of 128
    torch.cuda.synchronize()
    assert call(torch.zeros((2, 3, 1))) == LF_ERR_INVALID_ARG     # T too small
    assert call(torch.full((2, 4, 1), 4)) == LF_ERR_INVALID_ARG   # block 4 of 4
    assert call(torch.full((2, 4, 1), -2)) == LF_ERR_INVALID_ARG
