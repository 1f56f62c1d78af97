"""Pins of the relative-position-bias variant of the oracle (attention with
rel_bias): s_ij += rel_bias[h, t + w] for a non-global row i and a key
j = i + d*t of its window.

  - a zero bias changes nothing;
  - with no global tokens every key of a row is a window key, so a bias that
    is constant per head shifts a row's scores uniformly and the softmax (and
    the output) are unchanged;
  - a bias of -1e30 everywhere but offset 0 (no globals) leaves each row only
    itself: out = v;
  - a scalar brute force (math.exp, math.fsum over oracle.key_set) with
    dilation and global tokens.
"""
import math

import numpy as np
import pytest

import oracle as O


def _qkv(B, H, L, D, seed):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, H, L, D)) for _ in range(3)]


def test_zero_bias_changes_nothing():
    q, k, v = _qkv(1, 2, 48, 8, 1)
    a = O.attention(q, k, v, 4, [1, 2], [0, 30], 0.3)
    b = O.attention(q, k, v, 4, [1, 2], [0, 30], 0.3, rel_bias=np.zeros((2, 9)))
    assert np.array_equal(a, b)


def test_constant_bias_cancels_without_globals():
    q, k, v = _qkv(2, 2, 40, 8, 2)
    a = O.attention(q, k, v, 3, [1, 2], [], 0.3)
    b = O.attention(q, k, v, 3, [1, 2], [], 0.3, rel_bias=np.array([[5.0] * 7, [-3.0] * 7]))
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)


def test_bias_that_keeps_only_offset_zero_returns_v():
    q, k, v = _qkv(1, 1, 32, 8, 3)
    w = 3
    rb = np.full((1, 2 * w + 1), -1e30)
    rb[0, w] = 0.0
    out = O.attention(q, k, v, w, [1], [], 0.3, rel_bias=rb)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dil,G", [([1, 2], [0, 17]), ([2, 1], [5])])
def test_bias_against_scalar_brute_force(dil, G):
    B, H, L, D, w = 1, 2, 36, 6, 3
    q, k, v = _qkv(B, H, L, D, 4)
    rb = np.random.default_rng(5).standard_normal((H, 2 * w + 1))
    scale = 0.4
    got = O.attention(q, k, v, w, dil, G, scale, rel_bias=rb)
    for h in range(H):
        d = dil[h]
        for i in range(L):
            keys = O.key_set(i, L, w, d, G)
            s = []
            for j in keys:
                x = scale * math.fsum(q[0, h, i, e] * k[0, h, j, e] for e in range(D))
                t = (j - i) // d
                if i not in G and abs(j - i) <= d * w and (j - i) % d == 0:
                    x += rb[h, t + w]
                s.append(x)
            mx = max(s)
            ex = [math.exp(x - mx) for x in s]
            z = math.fsum(ex)
            for c in range(D):
                want = math.fsum(ex[n] * v[0, h, j, c] for n, j in enumerate(keys)) / z
                assert abs(got[0, h, i, c] - want) <= 1e-12
