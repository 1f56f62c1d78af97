"""Device-side failure detection, exercised without faulting the GPU.

Every wait of the attention kernel is bounded; when one runs out the kernel
records a timeout in a status word, leaves its loops and returns, and
lf_attn_get_status reports it.  The self-test kernel runs that same wait code
on a barrier nothing completes (no copy or tensor-core work in flight), so
the timeout path runs for real while the GPU and the context stay healthy.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lf():
    import long_sequence_sparse_lf_b300 as lf
    from long_sequence_sparse_lf_b300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    lf.load_library()
    return lf


def test_wait_runs_out_and_is_reported(lf):
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    lf.lf_selftest_wait_timeout(2000)          # 2 ms
    assert lf.lf_attn_get_status() == 5        # LF_ERR_TIMEOUT
    assert "wait ran out" in lf.lf_last_error()
    assert lf.lf_attn_get_status() == 0        # the record was cleared


def test_forward_works_after_a_timeout(lf):
    lf.lf_selftest_wait_timeout(500)
    assert lf.lf_attn_get_status() == 5
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn((1, 1, 256, 64), generator=g).to(torch.bfloat16).cuda()
               for _ in range(3))
    out = lf.attention(q, k, v, 0, [1], [], 0.125)   # w = 0: out = v
    assert lf.lf_attn_get_status() == 0, lf.lf_last_error()
    np.testing.assert_array_equal(out.float().cpu().numpy(), v.float().cpu().numpy())


def test_selftest_rejects_bad_timeouts(lf):
    from long_sequence_sparse_lf_b300._binding import LfError
    for bad in (0, -5, 10 ** 7):
        with pytest.raises(LfError):
            lf.lf_selftest_wait_timeout(bad)
