"""Property tests of the oracle's extended forms and of bench.py's pair count,
on random small patterns (hypothesis, bounded example counts):

  - the dense mask with an extra-block table equals the key sets built here
    from the definition (band ∪ G ∪ the tile's listed blocks, in residue
    space; everything for a global row);
  - attention with a table and a bias equals a scalar softmax over those key
    sets (math.exp, math.fsum);
  - bench.extra_block_pairs equals the number of keys the table adds to
    band ∪ G, counted from the masks.
"""
import math

import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import bench
import oracle as O
from long_sequence_sparse_lf_b300 import workloads as W

SETTINGS = settings(max_examples=25, deadline=None,
                    suppress_health_check=[HealthCheck.too_slow])


@st.composite
def patterns(draw):
    d = draw(st.integers(1, 3))
    L = d * draw(st.integers(40, 300 // d))
    w = draw(st.integers(0, 40))
    n_g = draw(st.integers(0, 4))
    G = sorted(set(draw(st.lists(st.integers(0, L - 1), min_size=n_g, max_size=n_g))))
    nqt = O.tiles_per_class(L, d)
    R = draw(st.integers(1, 3))
    tab = np.array(draw(st.lists(st.integers(-1, nqt - 1), min_size=d * nqt * R,
                                 max_size=d * nqt * R))).reshape(1, d * nqt, R)
    return L, w, d, G, tab


def _key_set_from_definition(i, L, w, d, G, tab_h):
    if i in G:
        return set(range(L))
    keys = {i + d * t for t in range(-w, w + 1) if 0 <= i + d * t < L} | set(G)
    r, t = i % d, i // d
    n_tiles = -(-(-(-L // d)) // 128)
    for kb in tab_h[r * n_tiles + t // 128]:
        if kb >= 0:
            keys |= {r + d * tt for tt in range(128 * kb, 128 * kb + 128) if r + d * tt < L}
    return keys


@SETTINGS
@given(patterns())
def test_mask_with_table_matches_definition(pat):
    L, w, d, G, tab = pat
    m = O.mask_rows(np.arange(L), L, w, d, G, tab[0])
    for i in range(0, L, max(1, L // 25)):
        assert set(np.nonzero(m[i])[0].tolist()) == _key_set_from_definition(i, L, w, d, G, tab[0])


@SETTINGS
@given(patterns(), st.integers(0, 2 ** 31 - 1))
def test_attention_with_table_and_bias_matches_scalar_softmax(pat, seed):
    L, w, d, G, tab = pat
    D, scale = 3, 0.6
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((1, 1, L, D)) for _ in range(3))
    rb = rng.standard_normal((1, 2 * w + 1))
    rows = sorted(set(rng.integers(0, L, 6).tolist()))
    got = O.attention(q, k, v, w, [d], G, scale, rows=rows, xblocks=tab, rel_bias=rb)
    for n, i in enumerate(rows):
        keys = sorted(_key_set_from_definition(i, L, w, d, G, tab[0]))
        s = []
        for j in keys:
            x = scale * math.fsum(q[0, 0, i, e] * k[0, 0, j, e] for e in range(D))
            if i not in G and abs(j - i) <= d * w and (j - i) % d == 0:
                x += rb[0, (j - i) // d + w]
            s.append(x)
        mx = max(s)
        ex = [math.exp(x - mx) for x in s]
        z = math.fsum(ex)
        for c in range(D):
            want = math.fsum(ex[m] * v[0, 0, j, c] for m, j in enumerate(keys)) / z
            assert abs(got[0, 0, n, c] - want) <= 1e-11


@SETTINGS
@given(patterns(), st.integers(1, 2))
def test_bench_extra_pairs_match_masks(pat, B):
    L, w, d, G, tab = pat
    wl = W.custom("p", B, 1, L, 64, w, (d,), G, 0)
    with_tab = int(O.mask_rows(np.arange(L), L, w, d, G, tab[0]).sum())
    without = int(O.mask_rows(np.arange(L), L, w, d, G).sum())
    assert bench.extra_block_pairs(wl, tab) == (with_tab - without) * B
