"""The pair count bench.py turns into useful FLOPs for the extra-block
workloads, against the oracle's key sets (dense masks) on small workloads:
extra_block_pairs, the pairs a table of extra key blocks adds to band ∪ G.
"""
import numpy as np
import pytest

import bench
import oracle as O
from long_sequence_sparse_lf_b300 import workloads as W

SHAPES = [
    # B, L, w, dilation, globals
    (1, 300, 5, (1, 2), (0, 77)),
    (2, 515, 40, (1, 3), (3, 260, 514)),
    (1, 1024, 150, (2,), ()),
    (1, 700, 200, (1,), tuple(range(0, 700, 97))),
]


def _mask_total(wl, h, xb_h=None, rows=None):
    rows = np.arange(wl.L) if rows is None else rows
    return int(O.mask_rows(rows, wl.L, wl.w, wl.dilation[h], wl.global_idx, xb_h).sum())


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind", ["random", "strided"])
def test_extra_block_pairs_matches_masks(shape, kind):
    B, L, w, dil, G = shape
    wl = W.custom("t", B, len(dil), L, 64, w, dil, G, 0)
    tab = (W.random_blocks(L, dil, 3, 11) if kind == "random"
           else W.strided_blocks(L, dil, 2)).numpy()
    want = 0
    for h in range(len(dil)):
        want += _mask_total(wl, h, tab[h]) - _mask_total(wl, h)
    assert bench.extra_block_pairs(wl, tab) == want * B
