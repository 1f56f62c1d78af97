"""The forward's log-sum-exp (lf_attn_fwd_lse) and the backward (lf_attn_bwd)
against the oracle, on bf16 inputs (the oracle computes in float64 on the
same bf16 values).

Tolerances:
  - lse: the forward's probabilities are fp32 sums of ex2.approx terms, so lse
    stays within 1e-3 (absolute, in natural-log units) of the float64 value.
  - gradients: the GPU rounds p and ds to bf16 before their products (a
    relative step of 2^-8 at most, 2^-9 on average) and reads delta from the
    bf16 output; fp32 accumulation.  Per tensor, rel-L2 <= 1e-2, and every
    element within 0.05 * max|ref| (this catches a missing class of pairs,
    which moves whole rows by a large part of their size).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LSE_ABS = 1e-3
REL_L2 = 1e-2
MAX_FRAC = 0.05


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


def _inputs(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(shape, generator=g).to(torch.bfloat16) for _ in range(4)]


CASES = [
    # B, H, L, D, w, dilation, globals
    (1, 2, 512, 64, 32, (1, 2), (0, 1, 300)),
    (2, 2, 1000, 64, 70, (1, 1), (3, 500)),
    (1, 2, 768, 128, 40, (1, 2), (0, 100, 767)),
    (1, 1, 256, 64, 16, (1,), ()),
    # more than 128 global tokens (two global-key tiles per head), dilated heads
    (1, 2, 1024, 64, 24, (1, 2), tuple(range(0, 1024, 7))),
    (1, 2, 640, 128, 20, (2, 1), tuple(range(5, 640, 4))),
    # L not a multiple of the query block, globals at both ends
    (1, 3, 333, 64, 50, (1, 1, 1), (0, 332)),
    # the prep kernel's global-key pass at its limit (4 global tokens) and
    # the global-key tiles just past it (5), D = 128 with dilation
    (2, 2, 512, 64, 30, (1, 2), (10, 11, 200, 511)),
    (1, 2, 512, 128, 30, (2, 1), (0, 64, 65, 300, 400)),
    # one query tile per head
    (1, 2, 128, 64, 4, (1, 1), (3,)),
]


def _run_fwd_bwd(lf, q, k, v, dout, w, dil, G, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, dout))
    B, H, L, D = q.shape
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    lf.lf_attn_fwd_lse(qd, kd, vd, out, lse, w, dil, G, scale)
    grads = [torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    lf.lf_attn_bwd(qd, kd, vd, out, lse, dod, *grads, w, dil, G, scale)
    torch.cuda.synchronize()
    assert lf.lf_attn_get_status() == 0
    return lse.cpu().double().numpy(), [t.cpu().double().numpy() for t in grads]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}L{c[2]}D{c[3]}w{c[4]}" for c in CASES])
def test_lse_and_gradients_match_oracle(lf, case):
    import oracle as O
    B, H, L, D, w, dil, G = case
    q, k, v, dout = _inputs((B, H, L, D), 20 + L)
    scale = 1.0 / np.sqrt(D)
    lse, (dq, dk, dv) = _run_fwd_bwd(lf, q, k, v, dout, w, dil, G, scale)
    qf, kf, vf, df = (t.double().numpy() for t in (q, k, v, dout))
    ref_lse = O.attention_lse(qf, kf, w, dil, G, scale)
    assert np.abs(lse - ref_lse).max() <= LSE_ABS
    refs = O.attention_backward(qf, kf, vf, df, w, dil, G, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        rel = float(np.linalg.norm((got - ref).ravel()) / np.linalg.norm(ref.ravel()))
        mx = float(np.abs(got - ref).max())
        assert rel <= REL_L2 and mx <= MAX_FRAC * float(np.abs(ref).max()), \
            f"{name}: rel_l2={rel:.3e} max_abs={mx:.3e} (ref max {np.abs(ref).max():.3e})"
