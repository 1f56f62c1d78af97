"""The Longformer layer forward (lf_layer_fwd) against the layer oracle.

The GPU path stores q, k, v, the attention output, x1 and the result in bf16
at the same points as oracle.longformer_layer(store_bf16=True); its products
accumulate in fp32 (the GEMMs and the attention) where the oracle uses
float64.  Tolerance, beyond half a bf16 step of the reference value:
  - the attention step's own error (within 1e-2 max-abs against float64,
    typically a few 1e-3);
  - LayerNorm's division by the row's spread (about 1) and gamma (about 1);
  - an occasional one-step bf16 difference where an fp32 and a float64
    intermediate fall on either side of a rounding boundary.
The result stays within max-abs 2e-2 and rel-L2 1e-2.
"""
import numpy as np
import pytest
import torch

from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 1e-2
BF16_HALF_ULP = 2.0 ** -8


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


def _run(lf, lw, inputs):
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = (t.cuda() for t in inputs)
    out = torch.full_like(x, float("nan"))
    lf.lf_layer_fwd(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, out, lw.H, lw.w, lw.dilation,
                    lw.global_idx, lw.scale, lw.eps)
    torch.cuda.synchronize()
    assert lf.lf_attn_get_status() == 0
    return out.float().cpu().double().numpy()


def _oracle(lw, inputs, rows=None):
    import oracle as O
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = (t.double().numpy() for t in inputs)
    return O.longformer_layer(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, lw.H, lw.w, lw.dilation,
                              lw.global_idx, lw.scale, lw.eps, store_bf16=True, rows=rows)


def _close(got, ref, what):
    d = np.abs(got - ref) - BF16_HALF_ULP * np.abs(ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))
    assert float(d.max()) <= MAX_ABS and rel <= REL_L2, \
        f"{what}: max_abs={float(d.max()):.3e} rel_l2={rel:.3e}"


SMALL = [
    W.LAYER_CONFIGS["layer-tiny"],
    W.LayerWorkload("d128-dilated", 1, 768, 2, 128, 40, (1, 2), (0, 100, 767), 12),
    W.LayerWorkload("h4-ragged", 2, 1000, 4, 64, 70, (1, 1, 2, 1), (3, 500), 13),
]


@pytest.mark.parametrize("lw", SMALL, ids=[c.name for c in SMALL])
def test_layer_matches_oracle(lf, lw):
    inputs = W.make_layer_inputs(lw)
    _close(_run(lf, lw, inputs), _oracle(lw, inputs), lw.name)


def test_layer_base_size_sampled_rows(lf):
    lw = W.LAYER_CONFIGS["layer-base"]
    inputs = W.make_layer_inputs(lw)
    got = _run(lf, lw, inputs)
    rows = sorted({0, 1, 127, 128, 255, 256, 2047, 2048, 4094, 4095} |
                  set(np.random.default_rng(7).integers(0, lw.L, 22).tolist()))
    _close(got[:, rows], _oracle(lw, inputs, rows=rows), "layer-base rows")


def test_layer_rejects_unsupported_width_and_misaligned_pointers(lf):
    from long_sequence_sparse_lf_b300._binding import LfError
    lw = W.LayerWorkload("h3", 1, 256, 3, 64, 8, (1, 1, 1), (), 14)   # hidden 192
    inputs = [t.cuda() for t in W.make_layer_inputs(lw)]
    out = torch.empty_like(inputs[0])
    with pytest.raises(LfError, match="UNSUPPORTED"):
        lf.lf_layer_fwd(*inputs, out, lw.H, lw.w, lw.dilation, lw.global_idx, lw.scale)
    lib = lf.load_library()
    from long_sequence_sparse_lf_b300._binding import _i32_array
    ptrs = [t.data_ptr() for t in inputs]
    st = lib.lf_layer_fwd(ptrs[0] + 2, *ptrs[1:], out.data_ptr(), 1, 256, 192, 3, 8,
                          _i32_array([1, 1, 1]), None, 0, 0.125, 1e-5, None)
    assert st == 1, lf.lf_last_error()
    torch.cuda.synchronize()
