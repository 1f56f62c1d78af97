"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: values printed on
the pages (tests/golden/), closed forms, library routines (torch's
scaled_dot_product_attention and scipy's softmax in float64) and brute force
on tiny inputs.  ``test_planted_mistakes_are_caught`` plants plausible
mistakes into copies of the oracle's functions and checks that the pins fail.
"""
import math
import os

import numpy as np
import pytest
import torch
import scipy.special

from oracle import lf_oracle as O


# ---------------------------------------------------------------- helpers

def _rand(shape, seed):
    g = np.random.default_rng(seed)
    # bf16-representable values, like the real inputs
    x = torch.from_numpy(g.standard_normal(shape)).to(torch.bfloat16)
    return x.to(torch.float64).numpy()


def _sdpa(q, k, v, scale):
    """Full softmax attention from the library routine, float64."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, scale=scale).numpy()


def _read_golden(path):
    rows = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line)
    return rows


def _parse_offsets(tok):
    out = []
    for t in tok.split():
        if ".." in t:
            a, b = t.split("..")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(t))
    return out


GRID_L = [1, 2, 5, 17, 40, 64]
GRID_W = [0, 1, 3, 8, 50]
GRID_D = [1, 2, 3, 5]


def _grid_globals(L):
    cands = [(), (0,), (L - 1,), (0, L - 1), (L // 2,),
             tuple(range(0, L, 7)), tuple(sorted({1, L // 3, L - 2} & set(range(L))))]
    out = []
    for G in cands:
        G = tuple(sorted(set(g for g in G if 0 <= g < L)))
        if G not in out:
            out.append(G)
    return out


# ------------------------------------------------------------ pin checks

def check_page_counts(pair_count, golden_dir):
    """Full attention (window covering the sequence, no dilation, no globals)
    reproduces the dense entry counts the pages print."""
    for line in _read_golden(os.path.join(golden_dir, "page_counts.txt")):
        parts = line.split()
        L, printed, exact = int(parts[0]), int(parts[1]), int(parts[2])
        n = pair_count(L, L, 1, ())
        assert n == L * L
        if exact:
            assert n == printed
        else:
            # the pages round to two or three significant digits
            assert abs(n - printed) / printed < 0.05, (L, n, printed)


def check_window_examples(key_set, golden_dir):
    for line in _read_golden(os.path.join(golden_dir, "window_examples.txt")):
        body = line.split("|")
        head = body[0].split()
        w, d = int(head[0]), int(head[1])
        inside = _parse_offsets(" ".join(head[2:]))
        outside = _parse_offsets(body[1])
        L = 8 * d * w + 1
        i = L // 2
        ks = set(key_set(i, L, w, d, ()))
        for o in inside:
            assert i + o in ks, (w, d, o)
        for o in outside:
            assert i + o not in ks, (w, d, o)
        if d == 1:
            assert len(ks) == 2 * w + 1


def check_counts_bruteforce(pair_count, key_set, mask_rows, key_lists):
    for L in GRID_L:
        for w in GRID_W:
            for d in GRID_D:
                for G in _grid_globals(L):
                    brute = sum(len(key_set(i, L, w, d, G)) for i in range(L))
                    assert pair_count(L, w, d, G) == brute, (L, w, d, G)
                    m = mask_rows(np.arange(L), L, w, d, G)
                    assert int(m.sum()) == brute
                    for i in range(L):
                        assert np.flatnonzero(m[i]).tolist() == \
                            sorted(key_set(i, L, w, d, G))
                    ptr, col = key_lists(L, w, [d], G)
                    assert ptr[-1] == brute
                    for i in range(L):
                        assert col[ptr[i]:ptr[i + 1]].tolist() == \
                            sorted(key_set(i, L, w, d, G))


def check_linear_growth(pair_count):
    # O(n*w): past the edges, one more token adds exactly 2w+1 pairs (d=1)
    for w in (0, 3, 64, 256):
        for L in (2 * w + 2, 4 * w + 9, 1000 + 2 * w):
            assert pair_count(L + 1, w, 1, ()) - pair_count(L, w, 1, ()) == 2 * w + 1
            # closed form for d=1, L > w
            assert pair_count(L, w, 1, ()) == L * (2 * w + 1) - w * (w + 1)


def check_full_attention(attention):
    """w >= L-1, d=1, no globals: textbook softmax attention."""
    B, H, L, D = 2, 3, 37, 16
    q, k, v = _rand((B, H, L, D), 1), _rand((B, H, L, D), 2), _rand((B, H, L, D), 3)
    scale = 1.0 / math.sqrt(D)
    ref = _sdpa(q, k, v, scale)
    for w in (L - 1, L, 5 * L):
        out = attention(q, k, v, w, [1] * H, (), scale, chunk=11)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # second library route: scipy softmax over the score matrix
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    ref2 = np.einsum("bhij,bhjd->bhid", scipy.special.softmax(s, axis=-1), v)
    out = attention(q, k, v, L, [1] * H, (), scale)
    np.testing.assert_allclose(out, ref2, rtol=1e-12, atol=1e-12)


def check_global_rows(attention):
    """Rows of global tokens equal full-attention rows ([LF-explained] §2)."""
    B, H, L, D = 1, 2, 45, 8
    q, k, v = _rand((B, H, L, D), 4), _rand((B, H, L, D), 5), _rand((B, H, L, D), 6)
    scale = 0.3
    G = (0, 13, 44)
    ref = _sdpa(q, k, v, scale)
    out = attention(q, k, v, 2, [1, 3], G, scale)
    for g in G:
        np.testing.assert_allclose(out[:, :, g], ref[:, :, g], rtol=1e-12, atol=1e-12)
    # and a non-global row is NOT a full-attention row
    assert np.abs(out[:, :, 20] - ref[:, :, 20]).max() > 1e-3


def check_window_zero(attention):
    B, H, L, D = 1, 2, 19, 4
    q, k, v = _rand((B, H, L, D), 7), _rand((B, H, L, D), 8), _rand((B, H, L, D), 9)
    out = attention(q, k, v, 0, [1, 2], (), 0.7)
    np.testing.assert_array_equal(out, v)


def check_constant_v(attention):
    B, H, L, D = 1, 2, 33, 5
    q, k = _rand((B, H, L, D), 10), _rand((B, H, L, D), 11)
    c = np.arange(D, dtype=np.float64) - 2.5
    v = np.broadcast_to(c, (B, H, L, D)).copy()
    out = attention(q, k, v, 3, [1, 4], (0, 17), 0.5)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-13)


def check_scale_zero_average(attention, key_set):
    """scale = 0: every attended key has the same weight, so out_i is the
    plain mean of v over K(i)."""
    B, H, L, D = 1, 2, 29, 3
    q, k, v = _rand((B, H, L, D), 12), _rand((B, H, L, D), 13), _rand((B, H, L, D), 14)
    dil = [1, 3]
    G = (2, 20)
    w = 2
    out = attention(q, k, v, w, dil, G, 0.0)
    for h in range(H):
        for i in range(L):
            ks = key_set(i, L, w, dil[h], G)
            np.testing.assert_allclose(out[0, h, i], v[0, h, ks].mean(axis=0),
                                       rtol=1e-13, atol=1e-13)


def check_dilation_deinterleave(attention):
    """With no globals, a d=2 head is two independent d=1 problems on the
    even and odd subsequences."""
    B, H, L, D = 2, 1, 40, 8
    q, k, v = _rand((B, H, L, D), 15), _rand((B, H, L, D), 16), _rand((B, H, L, D), 17)
    w = 3
    out = attention(q, k, v, w, [2], (), 0.4)
    for r in range(2):
        sub = attention(q[:, :, r::2], k[:, :, r::2], v[:, :, r::2], w, [1], (), 0.4)
        np.testing.assert_allclose(out[:, :, r::2], sub, rtol=1e-13, atol=1e-13)


def check_bruteforce_rows(attention, key_set_fn=None):
    B, H, L, D = 1, 3, 23, 6
    q, k, v = _rand((B, H, L, D), 18), _rand((B, H, L, D), 19), _rand((B, H, L, D), 20)
    dil = [1, 2, 4]
    G = (5, 22)
    w = 2
    scale = 0.45
    out = attention(q, k, v, w, dil, G, scale, chunk=7)
    for h in range(H):
        for i in range(L):
            ref = O.attention_row_bruteforce(q, k, v, 0, h, i, w, dil[h], G, scale)
            np.testing.assert_allclose(out[0, h, i], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ tests

def test_page_full_attention_counts(golden_dir):
    check_page_counts(O.pair_count, golden_dir)


def test_page_window_examples(golden_dir):
    check_window_examples(O.key_set, golden_dir)


def test_pair_count_closed_form_vs_bruteforce():
    check_counts_bruteforce(O.pair_count, O.key_set, O.mask_rows, O.key_lists)


def test_pair_count_linear_growth():
    check_linear_growth(O.pair_count)


def test_full_attention_special_case():
    check_full_attention(O.attention)


def test_global_rows_equal_full_rows():
    check_global_rows(O.attention)


def test_window_zero_is_identity():
    check_window_zero(O.attention)


def test_constant_v():
    check_constant_v(O.attention)


def test_scale_zero_is_mean_over_key_set():
    check_scale_zero_average(O.attention, O.key_set)


def test_dilation_deinterleave():
    check_dilation_deinterleave(O.attention)


def test_bruteforce_rows():
    check_bruteforce_rows(O.attention)


def test_rows_subset_matches_full():
    B, H, L, D = 2, 2, 70, 8
    q, k, v = _rand((B, H, L, D), 21), _rand((B, H, L, D), 22), _rand((B, H, L, D), 23)
    full = O.attention(q, k, v, 4, [1, 3], (0, 33), 0.3)
    rows = [69, 0, 33, 12, 40]
    sub = O.attention(q, k, v, 4, [1, 3], (0, 33), 0.3, rows=rows)
    np.testing.assert_array_equal(sub, full[:, :, rows])


def test_config_pair_totals_bruteforce_on_mask():
    """Closed-form totals of the two L=4096 patterns equal the mask count."""
    from long_sequence_sparse_lf_b300 import workloads as W
    for name in ("base", "qa"):
        c = W.CONFIGS[name]
        m = O.mask_rows(np.arange(c.L), c.L, c.w, 1, c.global_idx)
        assert int(m.sum()) == O.pair_count(c.L, c.w, 1, c.global_idx)
    c = W.CONFIGS["dilated"]
    m = O.mask_rows(np.arange(c.L), c.L, c.w, 2, c.global_idx)
    assert int(m.sum()) == O.pair_count(c.L, c.w, 2, c.global_idx)


def test_long_config_globals_fixture(golden_dir):
    from long_sequence_sparse_lf_b300 import workloads as W
    with open(os.path.join(golden_dir, "long_globals.txt")) as f:
        vals = [int(x) for x in f.read().split("\n")[-2].split()]
    assert list(W.CONFIGS["long"].global_idx) == vals


# -------------------------------------------------------- planted mistakes

def _mutant_mask_drop_globals(rows, L, w, d, G):
    return O.mask_rows(rows, L, w, d, ())


def _mutant_mask_window_short(rows, L, w, d, G):
    return O.mask_rows(rows, L, max(w - 1, 0), d, G)


def _mutant_mask_no_dilation(rows, L, w, d, G):
    return O.mask_rows(rows, L, w, 1, G)


def _mutant_mask_global_rows_banded(rows, L, w, d, G):
    m = O.mask_rows(rows, L, w, d, ())
    G = np.asarray(G, dtype=np.int64)
    if G.size:
        m[:, G] = True
    return m


def _attention_with_mask(mask_fn):
    def att(q, k, v, w, dilation, G, scale, rows=None, chunk=256):
        q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
        v = np.asarray(v, np.float64)
        B, H, L, D = q.shape
        r = np.arange(L) if rows is None else np.asarray(rows)
        out = np.empty((B, H, r.size, D))
        for h in range(H):
            m = mask_fn(r, L, w, int(dilation[h]), G)
            for b in range(B):
                s = np.where(m, (q[b, h, r] @ k[b, h].T) * scale, -np.inf)
                p = np.exp(s - s.max(1, keepdims=True))
                out[b, h] = (p / p.sum(1, keepdims=True)) @ v[b, h]
        return out
    return att


def _attention_transposed(q, k, v, w, dilation, G, scale, rows=None, chunk=256):
    # plausible mistake: scores built as K Q^T
    return _attention_with_mask(O.mask_rows)(k, q, v, w, dilation, G, scale, rows)


def _attention_no_max_shift_wrong_norm(q, k, v, w, dilation, G, scale, rows=None,
                                       chunk=256):
    # plausible mistake: normalising over all L keys instead of K(i)
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    B, H, L, D = q.shape
    out = np.empty((B, H, L, D))
    for h in range(H):
        m = O.mask_rows(np.arange(L), L, w, int(dilation[h]), G)
        for b in range(B):
            s = (q[b, h] @ k[b, h].T) * scale
            p = np.exp(s - s.max(1, keepdims=True))
            out[b, h] = (np.where(m, p, 0) / p.sum(1, keepdims=True)) @ v[b, h]
    return out


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("mutant", [
    _mutant_mask_drop_globals, _mutant_mask_window_short,
    _mutant_mask_no_dilation, _mutant_mask_global_rows_banded])
def test_planted_mask_mistakes_are_caught(mutant):
    att = _attention_with_mask(mutant)
    caught = (_fails(check_global_rows, att) or _fails(check_scale_zero_average, att, O.key_set)
              or _fails(check_bruteforce_rows, att) or _fails(check_dilation_deinterleave, att)
              or _fails(check_full_attention, att))
    assert caught


@pytest.mark.parametrize("mutant", [_attention_transposed,
                                    _attention_no_max_shift_wrong_norm])
def test_planted_attention_mistakes_are_caught(mutant):
    caught = (_fails(check_full_attention, mutant) or _fails(check_bruteforce_rows, mutant)
              or _fails(check_constant_v, mutant))
    assert caught


def test_planted_count_mistakes_are_caught(golden_dir):
    def count_no_edge_clip(L, w, d, G):
        return L * (2 * w + 1) + len(G) * L

    def count_no_dedupe(L, w, d, G):
        return O.pair_count(L, w, d, ()) + 2 * len(G) * L

    for bad in (count_no_edge_clip, count_no_dedupe):
        assert (_fails(check_page_counts, bad, golden_dir)
                or _fails(check_counts_bruteforce, bad, O.key_set, O.mask_rows, O.key_lists)
                or _fails(check_linear_growth, bad))
