"""Plain fp64 CPU oracle for Longformer sparse self-attention (forward).

TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the bench's
CPU-baseline / reference leg may import or run this module.  It shares no code
with the CUDA library and imports nothing from it.

Sources (web pages; cited by title and section):
  [LF-explained]  "基于自注意力机制的长文本建模算法：Longformer详解"
                  (Longformer explained), sections 2-4.
  [LF-blocksparse] "基于Block-Sparse Attention的Longformer：降低长序列计算复杂度
                  至O(n)的实现" (block-sparse Longformer), sections 2-4.
  [Reformer-hash] "Reformer哈希", section "核心原理" (the attention formula).
  [Eff-survey]    the commentary on "Efficient Transformers: A Survey",
                  section 2.1 (where the cost of dense attention comes from),
                  sections 3.1-3.2 (strided and BigBird random patterns).
  [LF-blocksparse] §6 "Longformer的整体架构" also defines the layer around the
                  attention (``longformer_layer`` below).

What is computed (the plain definition; readings of open points are listed
in the repository's design notes and repeated at each function):

  For head h with dilation d = dilation[h], one-sided window w, sequence
  length L and the sorted global positions G:
    band(i) = { i + d*t : |t| <= w, 0 <= i + d*t < L }
                  ([LF-explained] §2 sliding window; §2 dilated window)
    K(i)    = [0, L)          if i in G      ([LF-explained] §2 global attention)
            = band(i) ∪ G     otherwise      (the union, each key once)
            (∪ X(i), the tile's extra key blocks, when a random / strided
             block table is given: ``extra_block_keys``)
    s_ij    = scale * <q_i, k_j>             ([Reformer-hash] 核心原理 formula)
    p_ij    = exp(s_ij - max_{K(i)} s) / sum_{j' in K(i)} exp(s_ij' - max)
    out_i   = sum_{j in K(i)} p_ij v_j       (one softmax over all of K(i):
                  [LF-explained] §4, the three patterns combined)

All arithmetic is float64 on whatever values are passed in (callers pass the
bf16-rounded inputs).  The dense-masked form below builds full [rows, L] score
blocks and sets every key outside K(i) to -inf, which is exactly the
definition above: exp(-inf) = 0 removes those keys from both sums.

Parity status: every function here is pinned by tests in
``tests/test_oracle.py`` against values the pages print, closed forms,
library routines and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np


# --------------------------------------------------------------------------
# Key sets
# --------------------------------------------------------------------------

def band_offsets(i: int, L: int, w: int, d: int) -> List[int]:
    """band(i): the dilated sliding window of query i, clipped to [0, L).

    [LF-explained] §2: each token attends to a fixed number of neighbours on
    each side (one-sided width w); with dilation d the attended positions are
    i-d*w, ..., i-d, i, i+d, ..., i+d*w.  Positions outside the sequence are
    dropped (no wrap-around, no padding).
    """
    keys = []
    for t in range(-w, w + 1):
        j = i + d * t
        if 0 <= j < L:
            keys.append(j)
    return keys


XBLOCK = 128   # keys per extra block and queries per tile (residue space)


def tiles_per_class(L: int, d: int) -> int:
    """Query tiles of XBLOCK rows in the longest residue class of a head."""
    return -(-(-(-L // d)) // XBLOCK)


def extra_block_keys(i: int, L: int, d: int, xb_h) -> List[int]:
    """X(i): the extra key blocks of query i's tile, as positions.

    BigBird adds random key blocks to window + global attention; the survey
    commentary also names a fixed-stride pattern as the deterministic
    alternative ([Eff-survey] §3.1 fixed patterns, §3.2 combined patterns).
    Neither gives a block size or an indexing, so the reading taken here:
    with r = i mod d and t = i div d (the residue space of the dilated
    window), the row belongs to tile qt = t div 128 of class r, and
    xb_h[r * tiles_per_class(L, d) + qt] lists key blocks kb (-1 = none);
    block kb holds the keys r + d*t' for 128*kb <= t' < 128*kb + 128 of the
    same class, clipped to [0, L).  A random table gives BigBird's random
    blocks, a table listing every s-th block the strided pattern.
    """
    r, t = i % d, i // d
    nqt = tiles_per_class(L, d)
    keys = set()
    for kb in np.asarray(xb_h[r * nqt + t // XBLOCK]).ravel():
        kb = int(kb)
        if kb < 0:
            continue
        for tt in range(kb * XBLOCK, kb * XBLOCK + XBLOCK):
            j = r + d * tt
            if j < L:
                keys.add(j)
    return sorted(keys)


def key_set(i: int, L: int, w: int, d: int, G: Sequence[int], xb_h=None) -> List[int]:
    """K(i) as a sorted list (see the module docstring); ``xb_h`` (one head's
    extra-block table, see :func:`extra_block_keys`) adds X(i) to a
    non-global row."""
    Gs = set(int(g) for g in G)
    if i in Gs:
        # [LF-explained] §2 global attention: a global token sees the whole
        # sequence.
        return list(range(L))
    # Every token also attends to the global tokens ([LF-blocksparse] §4).
    keys = set(band_offsets(i, L, w, d)) | Gs
    if xb_h is not None:
        keys |= set(extra_block_keys(i, L, d, xb_h))
    return sorted(keys)


def mask_rows(rows: np.ndarray, L: int, w: int, d: int,
              G: Sequence[int], xb_h=None) -> np.ndarray:
    """Boolean [len(rows), L] mask, True where key j is in K(row).

    Vectorised form of :func:`key_set`: j is in band(i) iff |i-j| <= d*w and
    d divides i-j (then i-j = d*t with |t| <= w).
    """
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(L, dtype=np.int64)[None, :]
    i = rows[:, None]
    diff = j - i
    m = (np.abs(diff) <= d * w) & (diff % d == 0)
    if xb_h is not None:
        for n, row in enumerate(rows.tolist()):
            m[n, extra_block_keys(row, L, d, xb_h)] = True
    G = np.asarray(G, dtype=np.int64)
    if G.size:
        m[:, G] = True
        is_g = np.isin(rows, G)
        m[is_g, :] = True
    return m


def pair_count(L: int, w: int, d: int, G: Sequence[int]) -> int:
    """Number of attended (query, key) pairs of one head, in closed form.

    Sliding window: sum_i |band(i)| = L + 2 * sum_{t=1..w} max(0, L - t*d)
    (each offset +-t*d is valid for exactly L - t*d queries).  This is the
    exact, edge-clipped form of the O(n*w) count ([LF-explained] §2,
    [LF-blocksparse] §3).  Global rows add n_g*L ([LF-blocksparse] §4, the
    O(n*g) term); each non-global query gains the globals outside its band.
    """
    G = sorted(set(int(g) for g in G))
    band_total = L + 2 * sum(max(0, L - t * d) for t in range(1, w + 1))
    if not G:
        return band_total
    Gset = set(G)
    total = len(G) * L
    # Non-global rows: |band(i)| + |G \ band(i)|.
    band_nonglobal = band_total - sum(_band_size(g, L, w, d) for g in G)
    extra = 0
    for g in G:
        # Number of non-global queries i whose band does NOT contain g:
        # (L - n_g) minus the non-global i with g in band(i).  By symmetry
        # of the relation, g in band(i) iff i in band(g).
        in_band_of_g = [i for i in _band_members(g, L, w, d) if i not in Gset]
        extra += (L - len(G)) - len(in_band_of_g)
    return total + band_nonglobal + extra


def _band_size(i: int, L: int, w: int, d: int) -> int:
    return 1 + min(w, i // d) + min(w, (L - 1 - i) // d)


def _band_members(i: int, L: int, w: int, d: int) -> List[int]:
    lo = max(-w, -(i // d))
    hi = min(w, (L - 1 - i) // d)
    return [i + d * t for t in range(lo, hi + 1)]


def key_lists(L: int, w: int, dilation: Sequence[int], G: Sequence[int],
              rows: Optional[Iterable[Tuple[int, int]]] = None):
    """Per-(head, query) sorted key lists in CSR form.

    Without ``rows`` every (h, i) row in head-major order is listed and the
    result is (row_ptr int64 [H*L+1], col_idx int32 [total]).  With ``rows``
    (an iterable of (h, i)) only those rows are listed, in that order.
    """
    H = len(dilation)
    if rows is None:
        rows = [(h, i) for h in range(H) for i in range(L)]
    rows = list(rows)
    G = np.asarray(sorted(int(g) for g in G), dtype=np.int64)
    Gset = set(G.tolist())
    ptr = [0]
    cols: List[np.ndarray] = []
    for (h, i) in rows:
        d = int(dilation[h])
        if i in Gset:
            c = np.arange(L, dtype=np.int64)
        else:
            lo = max(-w, -(i // d))
            hi = min(w, (L - 1 - i) // d)
            band = i + d * np.arange(lo, hi + 1, dtype=np.int64)
            c = np.union1d(band, G)
        cols.append(c)
        ptr.append(ptr[-1] + c.size)
    col = (np.concatenate(cols) if cols else np.zeros(0, np.int64))
    return np.asarray(ptr, dtype=np.int64), col.astype(np.int32)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, w: int,
              dilation: Sequence[int], G: Sequence[int], scale: float,
              rows: Optional[Sequence[int]] = None,
              chunk: int = 256,
              rel_bias: Optional[np.ndarray] = None,
              xblocks: Optional[np.ndarray] = None) -> np.ndarray:
    """Longformer sparse self-attention forward, dense-masked, float64.

    q, k, v: arrays [B, H, L, D] (any float type; promoted to float64).
    Returns out [B, H, L, D] float64, or [B, H, len(rows), D] when ``rows``
    (a list of query positions shared by all heads) is given.

    For each (b, h) and each chunk of query rows: scores = scale * Q K^T over
    all L keys ([Reformer-hash] 核心原理), keys outside K(i) set to -inf
    (exact exclusion: the reading of "attends only to" in [LF-explained] §2),
    one row softmax ([LF-explained] §4: the patterns share one normalisation),
    then the product with V.

    rel_bias ([H, 2w+1] or None): a relative-position bias on the window's
    scores.  [LF-explained] §5 (position-encoding adaptations) says local
    attention is strengthened by a relative position bias but gives no
    formula.  The form chosen here: for a non-global row i and a key
    j = i + d*t of its window (|t| <= w), s_ij += rel_bias[h, t + w];
    scores of global keys outside the window, and of global rows, carry no
    bias.

    xblocks ([H, T, R] integer table or None): extra key blocks per query
    tile (BigBird random / strided blocks, see :func:`extra_block_keys`),
    added to K(i) of every non-global row.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, L, D = q.shape
    if rows is None:
        rows_arr = np.arange(L, dtype=np.int64)
    else:
        rows_arr = np.asarray(rows, dtype=np.int64)
    out = np.empty((B, H, rows_arr.size, D), dtype=np.float64)
    for h in range(H):
        d = int(dilation[h])
        for c0 in range(0, rows_arr.size, chunk):
            r = rows_arr[c0:c0 + chunk]
            m = mask_rows(r, L, w, d, G, None if xblocks is None else xblocks[h])
            bias = None
            if rel_bias is not None:
                # the window's offsets t = (j - i) / d of each (row, key)
                diff = np.arange(L)[None, :] - r[:, None]
                in_band = (np.abs(diff) <= d * w) & (diff % d == 0)
                in_band &= ~np.isin(r, np.asarray(G, dtype=np.int64))[:, None]
                t = np.clip(diff // d + w, 0, 2 * w)
                bias = np.where(in_band, np.asarray(rel_bias, np.float64)[h][t], 0.0)
            for b in range(B):
                s = (q[b, h, r, :] @ k[b, h].T) * scale
                if bias is not None:
                    s = s + bias
                s = np.where(m, s, -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                p /= p.sum(axis=1, keepdims=True)
                out[b, h, c0:c0 + r.size, :] = p @ v[b, h]
    return out


def attention_row_bruteforce(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                             b: int, h: int, i: int, w: int, d: int,
                             G: Sequence[int], scale: float) -> List[float]:
    """One output row with scalar Python loops over K(i) (tiny inputs only).

    Written directly from the definition with math.exp and math.fsum, as an
    independent check of the dense-masked form.
    """
    L = q.shape[2]
    D = q.shape[3]
    keys = key_set(i, L, w, d, G)
    s = []
    for j in keys:
        acc = math.fsum(float(q[b, h, i, e]) * float(k[b, h, j, e])
                        for e in range(D))
        s.append(scale * acc)
    mx = max(s)
    e = [math.exp(x - mx) for x in s]
    z = math.fsum(e)
    return [math.fsum(e[n] * float(v[b, h, j, c]) for n, j in enumerate(keys)) / z
            for c in range(D)]


def useful_flops(B: int, H: int, D: int, pairs_all_heads: int) -> int:
    """Useful FLOPs of the forward: 2*D for q.k plus 2*D for p*v per pair."""
    return 4 * B * D * pairs_all_heads


def total_pairs(L: int, w: int, dilation: Sequence[int],
                G: Sequence[int]) -> int:
    """Attended pairs summed over heads (batch-independent)."""
    cache = {}
    tot = 0
    for d in dilation:
        d = int(d)
        if d not in cache:
            cache[d] = pair_count(L, w, d, G)
        tot += cache[d]
    return tot


# --------------------------------------------------------------------------
# The layer around the attention
# --------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even) and return float64 values.

    The value is first rounded to float32 (nearest even), then its 32-bit
    pattern is rounded to the upper 16 bits: add 0x7FFF plus the lowest kept
    bit, clear the low 16 bits.  Used only where the layer stores an
    activation in bf16 (see ``longformer_layer``); NaN and infinities do not
    occur in the layer's values.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray,
               eps: float) -> np.ndarray:
    """LayerNorm over the last axis, float64: (x - mean) / sqrt(var + eps)
    * gamma + beta with the biased variance (the mean of squared
    deviations), the normalisation the page's layer applies after each
    residual ([LF-blocksparse] §6, nn.LayerNorm)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + \
        np.asarray(beta, np.float64)


def longformer_layer(x: np.ndarray, w_qkv: np.ndarray, b_qkv: np.ndarray,
                     w_ff: np.ndarray, b_ff: np.ndarray, ln1: np.ndarray,
                     ln2: np.ndarray, H: int, w: int, dilation: Sequence[int],
                     G: Sequence[int], scale: float, eps: float,
                     store_bf16: bool = True,
                     rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """One Longformer layer forward, float64 ([LF-blocksparse] §6).

    The page's layer maps x to q, k and v with three linear maps, applies the
    attention, adds the result to x and normalises (LayerNorm), then applies
    one linear feed-forward map (no activation), adds and normalises again.
    Its attention is read as the sparse attention of ``attention`` (one
    softmax per row over band(i) ∪ G) with the hidden axis split into H
    heads of D = hidden / H; the page's two attention sublayers, each with
    its own residual and norm, are that single attention (the repository's
    design notes list this reading).

    x: [B, L, hidden]; w_qkv: [3*hidden, hidden] (q rows, then k, then v;
    out = x W^T + b as for nn.Linear); b_qkv: [3*hidden]; w_ff: [hidden,
    hidden]; b_ff: [hidden]; ln1, ln2: [2, hidden] or [2*hidden] (gamma, then
    beta).  With store_bf16 (the library's storage), q, k, v (the product
    x W_qkv^T plus its bias, rounded once), the attention output, x1 and the
    result are rounded to bf16 where the layer stores them; everything else
    is float64.  ``rows`` (token positions shared by
    the batch) limits the attention and everything after it to those rows;
    the result is then [B, len(rows), hidden].
    """
    rnd = bf16_round if store_bf16 else (lambda t: np.asarray(t, np.float64))
    x = np.asarray(x, dtype=np.float64)
    B, L, hidden = x.shape
    D = hidden // H
    ln1 = np.asarray(ln1, np.float64).reshape(2, hidden)
    ln2 = np.asarray(ln2, np.float64).reshape(2, hidden)
    y = rnd(x @ np.asarray(w_qkv, np.float64).T + np.asarray(b_qkv, np.float64))
    # [B, L, 3, H, D] -> three [B, H, L, D]
    y = y.reshape(B, L, 3, H, D).transpose(2, 0, 3, 1, 4)
    a = attention(y[0], y[1], y[2], w, dilation, G, scale, rows=rows)   # [B, H, R, D]
    R = a.shape[2]
    a = rnd(a).transpose(0, 2, 1, 3).reshape(B, R, hidden)
    xr = x if rows is None else x[:, np.asarray(rows, dtype=np.int64), :]
    x1 = rnd(layer_norm(xr + a, ln1[0], ln1[1], eps))
    f = x1 @ np.asarray(w_ff, np.float64).T + np.asarray(b_ff, np.float64)
    return rnd(layer_norm(x1 + f, ln2[0], ln2[1], eps))


# --------------------------------------------------------------------------
# Backward of the attention
# --------------------------------------------------------------------------

def attention_lse(q: np.ndarray, k: np.ndarray, w: int, dilation: Sequence[int],
                  G: Sequence[int], scale: float, chunk: int = 256) -> np.ndarray:
    """lse[b, h, i] = ln sum_{j in K(i)} exp(scale * q_i . k_j), float64: the
    normaliser of the softmax of ``attention``, so that its weights are
    p_ij = exp(scale q_i.k_j - lse_i)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, H, L, D = q.shape
    out = np.empty((B, H, L), dtype=np.float64)
    for h in range(H):
        d = int(dilation[h])
        for c0 in range(0, L, chunk):
            r = np.arange(c0, min(L, c0 + chunk))
            m = mask_rows(r, L, w, d, G)
            for b in range(B):
                s = np.where(m, (q[b, h, r, :] @ k[b, h].T) * scale, -np.inf)
                mx = s.max(axis=1, keepdims=True)
                out[b, h, r] = (mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True)))[:, 0]
    return out


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                       w: int, dilation: Sequence[int], G: Sequence[int], scale: float,
                       chunk: int = 256):
    """Gradients (dq, dk, dv) of sum(out * dout) for out = attention(q, k, v),
    float64, dense-masked.  With s_ij = scale q_i.k_j over K(i), the softmax
    p_ij and out_i = sum_j p_ij v_j (the definition of ``attention``), the
    chain rule gives, row by row:
        dv_j  += p_ij dout_i                   (out is linear in v)
        dp_ij  = dout_i . v_j
        ds_ij  = p_ij (dp_ij - sum_j' p_ij' dp_ij')   (the softmax's Jacobian)
        dq_i   = scale sum_j ds_ij k_j,   dk_j += scale ds_ij q_i
    with p_ij = 0 for j outside K(i).  This is the derivative of the plain
    definition, written out; the pages give no backward of their own."""
    q, k, v, dout = (np.asarray(t, dtype=np.float64) for t in (q, k, v, dout))
    B, H, L, D = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(H):
        d = int(dilation[h])
        for c0 in range(0, L, chunk):
            r = np.arange(c0, min(L, c0 + chunk))
            m = mask_rows(r, L, w, d, G)
            for b in range(B):
                s = np.where(m, (q[b, h, r, :] @ k[b, h].T) * scale, -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                p /= p.sum(axis=1, keepdims=True)
                dp = dout[b, h, r, :] @ v[b, h].T
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
                dq[b, h, r, :] = scale * (ds @ k[b, h])
                dk[b, h] += scale * (ds.T @ q[b, h, r, :])
                dv[b, h] += p.T @ dout[b, h, r, :]
    return dq, dk, dv
