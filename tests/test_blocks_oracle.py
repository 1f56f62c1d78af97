"""Pins of the extra-key-block form of the oracle (BigBird random / strided
blocks): attention(..., xblocks=table) with table [H, T, R] listing, per
128-query tile of a residue class, key blocks of 128 keys of that class.

  - a table of -1 changes nothing;
  - d = 1, no globals, every tile listing every block: every row sees every
    key, so the output is dense softmax attention (torch.softmax);
  - a scalar brute force (math.exp, math.fsum) whose key sets are written
    here from the definition, with dilation, globals, ragged classes and
    duplicate / window-overlapping entries;
  - the tile indexing: a block listed only for tile 1 of class 1 reaches
    exactly the rows of that tile.
"""
import math

import numpy as np
import torch

import oracle as O


def _qkv(B, H, L, D, seed):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, H, L, D)) for _ in range(3)]


def test_empty_table_changes_nothing():
    q, k, v = _qkv(1, 2, 300, 4, 1)
    tab = -np.ones((2, 4, 2), dtype=np.int64)             # T = 2 classes x 2 tiles
    a = O.attention(q, k, v, 5, [1, 2], [0, 77], 0.5)
    b = O.attention(q, k, v, 5, [1, 2], [0, 77], 0.5, xblocks=tab)
    assert np.array_equal(a, b)


def test_every_block_listed_is_dense_attention():
    L, D = 300, 8
    q, k, v = _qkv(1, 1, L, D, 2)
    nqt = O.tiles_per_class(L, 1)
    tab = np.tile(np.arange(nqt), (1, nqt, 1))           # [1, nqt, nqt]
    got = O.attention(q, k, v, 3, [1], [], 0.3, xblocks=tab)
    qt, kt, vt = (torch.from_numpy(x[0, 0]) for x in (q, k, v))
    want = torch.softmax(0.3 * qt @ kt.T, dim=-1) @ vt
    np.testing.assert_allclose(got[0, 0], want.numpy(), rtol=1e-12, atol=1e-12)


def _in_key_set(i, j, L, w, d, G, tab_h):
    if i in G or j in G:
        return True
    if abs(j - i) <= d * w and (j - i) % d == 0:
        return True
    if j % d != i % d:
        return False
    n_tiles = -(-(-(-L // d)) // 128)
    listed = tab_h[(i % d) * n_tiles + (i // d) // 128]
    return any(kb >= 0 and (j // d) // 128 == kb for kb in listed)


def test_scalar_brute_force_with_dilation_and_globals():
    B, H, L, D, w = 1, 2, 515, 3, 4
    dil, G = [1, 2], [3, 260]
    q, k, v = _qkv(B, H, L, D, 3)
    rng = np.random.default_rng(4)
    T = max(d * O.tiles_per_class(L, d) for d in dil)
    tab = rng.integers(-1, 5, size=(H, T, 3))
    tab[0, 0] = [0, 0, 2]                                 # duplicate, and the own window block
    scale = 0.7
    rows = [0, 1, 2, 3, 127, 128, 129, 255, 256, 257, 260, 383, 384, 511, 512, 513, 514]
    got = O.attention(q, k, v, w, dil, G, scale, rows=rows, xblocks=tab)
    for h in range(H):
        d = dil[h]
        for n, i in enumerate(rows):
            keys = [j for j in range(L) if _in_key_set(i, j, L, w, d, G, tab[h])]
            s = [scale * math.fsum(q[0, h, i, e] * k[0, h, j, e] for e in range(D)) for j in keys]
            mx = max(s)
            ex = [math.exp(x - mx) for x in s]
            z = math.fsum(ex)
            for c in range(D):
                want = math.fsum(ex[m] * v[0, h, j, c] for m, j in enumerate(keys)) / z
                assert abs(got[0, h, n, c] - want) <= 1e-12


def test_tile_indexing():
    """d = 2, L = 600: class 1 has 300 positions, tiles of 128 (3 per class).
    Listing block 2 (class-1 keys 513, 515, ..., 599) for tile 1 of class 1
    (queries 257, 259, ..., 511) adds those keys to those rows only."""
    L, d, w = 600, 2, 3
    nqt = O.tiles_per_class(L, d)
    assert nqt == 3
    tab = -np.ones((2 * nqt, 1), dtype=np.int64)
    tab[1 * nqt + 1, 0] = 2
    added = set(range(513, 600, 2))
    for i in range(L):
        extra = set(O.extra_block_keys(i, L, d, tab))
        in_tile = i % 2 == 1 and 128 <= i // 2 < 256
        assert extra == (added if in_tile else set())
        ks = set(O.key_set(i, L, w, d, [], tab))
        assert ks == set(O.band_offsets(i, L, w, d)) | extra
