"""The host-buffer forward (lf_attn_fwd_host) against the device-buffer one.

lf_attn_fwd_host splits a problem into chunks of whole heads of one batch
element and pipelines their copies and computation over two streams.  Each
head's attention is independent of the others and the kernels' work per
head does not depend on how many heads a call holds, so its output must
equal lf_attn_fwd's (or lf_attn_fwd_f32's) on the same inputs bit for bit:
with dilation varying across chunk boundaries, global tokens, a ragged
length, both head sizes, and pinned as well as pageable host memory.
"""
import pytest
import torch

from long_sequence_sparse_lf_b300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


CASES = [
    # name, B, H, L, D, w, dilation, globals, seed, in_dtype
    W.custom("b2-dil-ragged", 2, 5, 1000, 64, 50, (1, 2, 1, 4, 2), (0, 17, 999), 41),
    W.custom("b1-d128", 1, 9, 768, 128, 100, (1, 1, 2, 1, 3, 1, 1, 2, 1), (5,), 42),
    W.custom("b4-noglobals", 4, 2, 512, 64, 32, (1, 2), (), 43),
    W.custom("b1-f32", 1, 6, 512, 64, 40, (1, 2, 1, 1, 4, 1), (0, 1), 44, "fp32"),
]


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_forward_equals_device_forward(lf, wl, pinned):
    q, k, v = W.make_qkv(wl)
    f32 = q.dtype == torch.float32
    ref = torch.empty_like(q, device="cuda")
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    if f32:
        lf.lf_attn_fwd_f32(qd, kd, vd, ref, wl.w, wl.dilation, wl.global_idx, wl.scale)
    else:
        lf.lf_attn_fwd(qd, kd, vd, ref, wl.w, wl.dilation, wl.global_idx, wl.scale)
    if pinned:
        q, k, v = (t.contiguous().pin_memory() for t in (q, k, v))
    out = torch.full_like(q, float("nan"))
    if pinned:
        out = out.pin_memory()
    lf.lf_attn_fwd_host(q, k, v, out, wl.w, wl.dilation, wl.global_idx, wl.scale)
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    assert torch.equal(out, ref.cpu()), wl.name


def test_host_forward_rejects_bad_pattern_before_copying(lf):
    from long_sequence_sparse_lf_b300._binding import LfError
    wl = CASES[0]
    q, k, v = W.make_qkv(wl)
    out = torch.empty_like(q)
    with pytest.raises(LfError, match="INVALID_ARG"):
        lf.lf_attn_fwd_host(q, k, v, out, wl.w, wl.dilation, (5, 3), wl.scale)   # not sorted
