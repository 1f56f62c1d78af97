"""Pins of the backward oracle (oracle.attention_backward, oracle.attention_lse).

  - finite differences: the gradient's inner product with a random direction
    equals the central difference of sum(out * dout) along it;
  - torch.autograd through a dense attention with the boolean mask of the
    brute-force key sets (oracle.key_set), float64;
  - w = 0 and no globals: out = v, so dv = dout and dq = dk = 0;
  - lse equals torch.logsumexp of the masked scores, and the softmax weights
    exp(s - lse) of every row sum to one.
"""
import numpy as np
import pytest
import torch

import oracle as O


def _inputs(B, H, L, D, seed):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, H, L, D)) for _ in range(4)]


def _mask(L, w, dil, G):
    H = len(dil)
    m = np.zeros((H, L, L), dtype=bool)
    for h in range(H):
        for i in range(L):
            m[h, i, O.key_set(i, L, w, dil[h], G)] = True
    return m


def test_backward_matches_finite_differences():
    B, H, L, D, w = 1, 2, 24, 8, 3
    dil, G, scale = [1, 2], [0, 13], 0.3
    q, k, v, dout = _inputs(B, H, L, D, 1)
    dq, dk, dv = O.attention_backward(q, k, v, dout, w, dil, G, scale)
    g = np.random.default_rng(2)
    f = lambda q_, k_, v_: float((O.attention(q_, k_, v_, w, dil, G, scale) * dout).sum())
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        direc = g.standard_normal(q.shape)
        args_p = {"q": q, "k": k, "v": v}
        args_m = dict(args_p)
        args_p[name] = args_p[name] + eps * direc
        args_m[name] = args_m[name] - eps * direc
        fd = (f(args_p["q"], args_p["k"], args_p["v"]) -
              f(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        assert abs(fd - float((grad * direc).sum())) <= 1e-6 * max(1.0, abs(fd)), name


def test_backward_matches_torch_autograd_on_masked_dense_attention():
    B, H, L, D, w = 2, 2, 40, 16, 4
    dil, G, scale = [1, 2], [0, 7, 31], 0.25
    q, k, v, dout = _inputs(B, H, L, D, 3)
    dq, dk, dv = O.attention_backward(q, k, v, dout, w, dil, G, scale)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = torch.as_tensor(_mask(L, w, dil, G))[None]
    s = (tq @ tk.transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    out = torch.softmax(s, dim=-1) @ tv
    (out * torch.as_tensor(dout)).sum().backward()
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-11)


def test_backward_window_zero_is_identity():
    B, H, L, D = 1, 1, 12, 4
    q, k, v, dout = _inputs(B, H, L, D, 4)
    dq, dk, dv = O.attention_backward(q, k, v, dout, 0, [1], [], 0.5)
    np.testing.assert_allclose(dv, dout, rtol=0, atol=1e-15)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0


@pytest.mark.parametrize("dil,G", [([1, 1], [0]), ([2, 1], [3, 10, 29])])
def test_lse_is_the_log_sum_exp_of_the_masked_scores(dil, G):
    B, H, L, D, w = 2, 2, 32, 8, 3
    q, k, _, _ = _inputs(B, H, L, D, 5)
    scale = 0.4
    lse = O.attention_lse(q, k, w, dil, G, scale)
    mask = torch.as_tensor(_mask(L, w, dil, G))[None]
    s = (torch.as_tensor(q) @ torch.as_tensor(k).transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)
    p = torch.exp(s - torch.as_tensor(lse)[..., None])
    np.testing.assert_allclose(p.sum(-1).numpy(), 1.0, rtol=1e-12)
