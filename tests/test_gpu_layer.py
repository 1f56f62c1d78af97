"""The Longformer layer forward (lf_layer_fwd) against the layer oracle.

Primary check: the plain float64 layer (oracle.longformer_layer with
store_bf16=False), which is pinned to a dense torch layer by the CPU tests.
The GPU path stores q, k, v (product plus bias, rounded once), the attention
output, x1 and the result in bf16 (the storage points its header documents)
and accumulates its products in fp32.  Tolerance against float64, derived
from those points (bf16 unit roundoff u = 2^-8):
  - the final bf16 store: u * |y| per element, allowed on top of the bound;
  - upstream, to first order: the q/k/v roundings (2u relative) move the
    attention output by about 1e-3 rms, the stored attention output and x1
    add u * |a| and u * |x1|, and the feed-forward map carries x1's error
    through (rms about u * rms(x1)); after LayerNorm (dividing by a row
    spread of about sqrt(2)) the result's upstream error is about 2.5e-3 rms,
    about 1.3e-2 at five standard deviations over the 6.3M outputs of the
    largest case;
  - so: |gpu - ref| <= 3e-2 + u * |ref| per element, and rel-L2 <= 1e-2.
Second check, tighter: the oracle with the same bf16 storage points
(store_bf16=True), which isolates the accumulation-order and attention-kernel
error: |gpu - ref| <= 2e-2 + u * |ref|, rel-L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS_F64 = 3e-2      # against the float64 layer (see above)
MAX_ABS_STORED = 2e-2   # against the layer with the same bf16 storage points
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


def _oracle(lw, inputs, rows=None, store_bf16=False):
    import oracle as O
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = (t.double().numpy() for t in inputs)
    return O.longformer_layer(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, lw.H, lw.w, lw.dilation,
                              lw.global_idx, lw.scale, lw.eps, store_bf16=store_bf16,
                              rows=rows)


def _close(got, ref, what, max_abs):
    d = np.abs(got - ref) - BF16_HALF_ULP * np.abs(ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))
    print(f"{what}: max(|err| - u|ref|)={float(d.max()):.3e} "
          f"max|err|={float(np.abs(got - ref).max()):.3e} rel_l2={rel:.3e}")
    assert float(d.max()) <= max_abs and rel <= REL_L2, \
        f"{what}: max_abs={float(d.max()):.3e} rel_l2={rel:.3e}"


def _check(got, lw, inputs, what, rows=None):
    _close(got, _oracle(lw, inputs, rows=rows), what + " (float64 layer)", MAX_ABS_F64)
    _close(got, _oracle(lw, inputs, rows=rows, store_bf16=True),
           what + " (bf16 storage points)", MAX_ABS_STORED)


SMALL = [
    W.LAYER_CONFIGS["layer-tiny"],
    W.LayerWorkload("d128-dilated", 1, 768, 2, 128, 40, (1, 2), (0, 100, 767), 12),
    W.LayerWorkload("h4-ragged", 2, 1000, 4, 64, 70, (1, 1, 2, 1), (3, 500), 13),
    # hidden 64: 64-column q/k/v and feed-forward tiles; hidden 384: 128-wide
    # q/k/v tiles and a cluster of three feed-forward CTAs; hidden 2048:
    # 256-column feed-forward tiles in clusters of eight
    W.LayerWorkload("h1-narrow", 1, 300, 1, 64, 20, (1,), (0,), 15),
    W.LayerWorkload("h6-cluster3", 1, 512, 6, 64, 30, (1, 2, 1, 1, 2, 1), (7, 8, 9), 16),
    W.LayerWorkload("h16-wide", 1, 256, 16, 128, 16, (1,) * 16, (0,), 17),
]


@pytest.mark.parametrize("lw", SMALL, ids=[c.name for c in SMALL])
def test_layer_matches_oracle(lf, lw):
    inputs = W.make_layer_inputs(lw)
    _check(_run(lf, lw, inputs), lw, inputs, lw.name)


def test_layer_base_size_sampled_rows(lf):
    lw = W.LAYER_CONFIGS["layer-base"]
    inputs = W.make_layer_inputs(lw)
    got = _run(lf, lw, inputs)
    rows = sorted({0, 1, 127, 128, 255, 256, 2047, 2048, 4094, 4095} |
                  set(np.random.default_rng(7).integers(0, lw.L, 22).tolist()))
    _check(got[:, rows], lw, inputs, "layer-base rows", rows=rows)


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
