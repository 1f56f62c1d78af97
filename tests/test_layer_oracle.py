"""Pins of the layer oracle (oracle.longformer_layer and its helpers).

Each check compares against something computed another way:
  - bf16_round against torch's own float64 -> bfloat16 conversion, and on
    hand-picked ties;
  - layer_norm against torch.nn.functional.layer_norm, and its invariants;
  - the whole layer, with a window covering every key and no globals, against
    a dense layer written with torch.nn.functional (linear, scaled dot-product
    attention, layer_norm) in float64;
  - the whole layer with dilation and global tokens against the same torch
    layer with an explicit boolean mask built from oracle.key_set (the
    brute-force per-query key lists);
  - a zero feed-forward map: LN2 of an already normalised row (gamma 1,
    beta 0) returns the row;
  - the stored (bf16) form against the masked torch layer rounding with
    torch's own bf16 conversion at the same four storage points, element for
    element, and not equal to a form that also rounds the q/k/v product
    before its bias.
The layer follows "基于Block-Sparse Attention的Longformer" §6.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O


def _rng_layer(B, L, H, D, seed):
    g = np.random.default_rng(seed)
    h = H * D
    x = g.standard_normal((B, L, h))
    w_qkv = g.standard_normal((3 * h, h)) / np.sqrt(h)
    b_qkv = 0.02 * g.standard_normal(3 * h)
    w_ff = g.standard_normal((h, h)) / np.sqrt(h)
    b_ff = 0.02 * g.standard_normal(h)
    ln1 = np.concatenate([1 + 0.1 * g.standard_normal(h), 0.1 * g.standard_normal(h)])
    ln2 = np.concatenate([1 + 0.1 * g.standard_normal(h), 0.1 * g.standard_normal(h)])
    return x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2


def _torch_bf16(t):
    """torch's own round-to-nearest-even conversion to bfloat16, back in float64."""
    return t.to(torch.bfloat16).to(torch.float64)


def _torch_layer(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, H, scale, eps, mask=None,
                 store=lambda t: t, store_product=False):
    """Dense reference with torch library routines, float64.  mask: bool
    [H, L, L] (True = attended) or None for full attention.  store: applied
    where the layer stores a tensor (q, k, v; the attention output; x1; the
    result); store_product also applies it to x W_qkv^T before the bias."""
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.float64)
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = map(t, (x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2))
    B, L, h = x.shape
    D = h // H
    if store_product:
        y = store(store(F.linear(x, w_qkv)) + b_qkv)
    else:
        y = store(F.linear(x, w_qkv, b_qkv))                        # [B, L, 3h]
    q, k, v = (y[..., s * h:(s + 1) * h].reshape(B, L, H, D).transpose(1, 2) for s in range(3))
    am = None if mask is None else torch.as_tensor(mask)[None]     # [1, H, L, L]
    a = F.scaled_dot_product_attention(q, k, v, attn_mask=am, scale=scale)
    a = store(a.transpose(1, 2).reshape(B, L, h))
    x1 = store(F.layer_norm(x + a, (h,), ln1[:h], ln1[h:], eps))
    f = F.linear(x1, w_ff, b_ff)
    return store(F.layer_norm(x1 + f, (h,), ln2[:h], ln2[h:], eps)).numpy()


def test_bf16_round_matches_torch_conversion():
    g = np.random.default_rng(1)
    vals = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-6, 6, 20000),
                           [0.0, -0.0, 1.0, -1.0, 65504.0, 3.0e38]])
    want = torch.as_tensor(vals, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_round(vals), want)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is half way between 1 and 1 + 2^-7: the even one (1) wins;
    # 1 + 3*2^-8 is half way between 1 + 2^-7 and 1 + 2^-6: 1 + 2^-6 wins
    assert O.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert O.bf16_round(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0


def test_layer_norm_matches_torch_and_normalises():
    g = np.random.default_rng(2)
    x = g.standard_normal((3, 5, 96)) * 3 + 1.5
    gamma, beta = 1 + 0.1 * g.standard_normal(96), 0.1 * g.standard_normal(96)
    got = O.layer_norm(x, gamma, beta, 1e-5)
    want = F.layer_norm(torch.as_tensor(x), (96,), torch.as_tensor(gamma),
                        torch.as_tensor(beta), 1e-5).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    plain = O.layer_norm(x, np.ones(96), np.zeros(96), 0.0)
    np.testing.assert_allclose(plain.mean(-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(plain.var(-1), 1.0, atol=1e-12)


@pytest.mark.parametrize("H,D", [(1, 64), (2, 32)])
def test_layer_full_window_is_a_dense_layer(H, D):
    B, L = 2, 40
    args = _rng_layer(B, L, H, D, 3)
    scale = 1 / np.sqrt(D)
    got = O.longformer_layer(*args, H=H, w=L, dilation=[1] * H, G=[], scale=scale, eps=1e-5,
                             store_bf16=False)
    want = _torch_layer(*args, H=H, scale=scale, eps=1e-5)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-9)


def test_layer_band_dilation_globals_against_masked_dense_layer():
    B, L, H, D, w = 1, 48, 2, 16, 3
    dil, G = [1, 2], [0, 17, 30]
    args = _rng_layer(B, L, H, D, 4)
    scale = 0.25
    mask = np.zeros((H, L, L), dtype=bool)
    for h in range(H):
        for i in range(L):
            mask[h, i, O.key_set(i, L, w, dil[h], G)] = True
    got = O.longformer_layer(*args, H=H, w=w, dilation=dil, G=G, scale=scale, eps=1e-5,
                             store_bf16=False)
    want = _torch_layer(*args, H=H, scale=scale, eps=1e-5, mask=mask)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-9)
    rows = [0, 5, 17, 47]
    sub = O.longformer_layer(*args, H=H, w=w, dilation=dil, G=G, scale=scale, eps=1e-5,
                             store_bf16=False, rows=rows)
    np.testing.assert_allclose(sub, want[:, rows], rtol=1e-9, atol=1e-9)


def test_zero_feed_forward_returns_the_normalised_row():
    B, L, H, D = 1, 32, 2, 16
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = _rng_layer(B, L, H, D, 5)
    h = H * D
    ln1 = np.concatenate([np.ones(h), np.zeros(h)])
    ln2 = np.concatenate([np.ones(h), np.zeros(h)])
    y = O.longformer_layer(x, w_qkv, b_qkv, np.zeros((h, h)), np.zeros(h), ln1, ln2, H=H, w=4,
                           dilation=[1, 1], G=[0], scale=0.25, eps=0.0, store_bf16=False)
    x1 = O.layer_norm(x + O.attention(*[
        (x @ w_qkv.T + b_qkv).reshape(B, L, 3, H, D).transpose(2, 0, 3, 1, 4)[s]
        for s in range(3)], 4, [1, 1], [0], 0.25).transpose(0, 2, 1, 3).reshape(B, L, h),
        ln1[:h], ln1[h:], 0.0)
    np.testing.assert_allclose(y, x1, rtol=1e-9, atol=1e-9)


def test_stored_bf16_layer_stays_close_to_float64_layer():
    B, L, H, D = 1, 64, 2, 32
    args = _rng_layer(B, L, H, D, 6)
    kw = dict(H=H, w=5, dilation=[1, 2], G=[0, 9], scale=1 / np.sqrt(D), eps=1e-5)
    exact = O.longformer_layer(*args, store_bf16=False, **kw)
    stored = O.longformer_layer(*args, store_bf16=True, **kw)
    assert np.all(O.bf16_round(stored) == stored)
    # four bf16 stores of values of size ~1 (relative step 2^-8) move the
    # result by well under 0.1
    assert np.abs(stored - exact).max() < 0.1


def test_stored_bf16_layer_against_torch_bf16_storage():
    """The stored form against the masked dense torch layer that rounds with
    torch's own bf16 conversion at the same four points (q, k, v after the
    bias; the attention output; x1; the result).  The pre-rounding values of
    the two agree to float64 rounding, so every element must match; rounding
    the q/k/v product once more before its bias (a different storage
    reading) must not."""
    B, L, H, D, w = 2, 48, 2, 32, 4
    dil, G = [1, 2], [0, 17, 30]
    args = _rng_layer(B, L, H, D, 7)
    scale = 1 / np.sqrt(D)
    mask = np.zeros((H, L, L), dtype=bool)
    for h in range(H):
        for i in range(L):
            mask[h, i, O.key_set(i, L, w, dil[h], G)] = True
    got = O.longformer_layer(*args, H=H, w=w, dilation=dil, G=G, scale=scale, eps=1e-5,
                             store_bf16=True)
    want = _torch_layer(*args, H=H, scale=scale, eps=1e-5, mask=mask, store=_torch_bf16)
    assert np.array_equal(got, want), np.abs(got - want).max()
    other = _torch_layer(*args, H=H, scale=scale, eps=1e-5, mask=mask, store=_torch_bf16,
                         store_product=True)
    assert not np.array_equal(got, other)
