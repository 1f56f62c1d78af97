"""Seeded synthetic workloads for Longformer sparse attention.

This module only describes problem shapes and draws random inputs; it holds
none of the attention arithmetic, so both the CUDA path's tests/bench and the
CPU oracle can take their inputs from it without sharing any of the method.

Input recipe (the same for every configuration):
  * ``g = torch.Generator('cpu').manual_seed(seed)``;
  * ``q, k, v = torch.randn((B, H, L, D), generator=g, dtype=torch.float32)``,
    drawn in that order (iid N(0, 1));
  * the arithmetic inputs are those values rounded to bf16 (round to nearest
    even).  Configurations with fp32 inputs keep the fp32 tensors for the
    call, and both sides round them to bf16 before any product.

The window size w is one-sided (2w+1 keys including the query itself), the
dilation is per head, and the global token positions are a sorted list.
Scale is 1/sqrt(D) for every configuration.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    D: int
    w: int
    dilation: tuple          # per head, len H
    global_idx: tuple        # sorted, strictly increasing
    seed: int
    in_dtype: str            # "fp32" or "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def n_global(self) -> int:
        return len(self.global_idx)

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "H": self.H, "L": self.L,
            "D": self.D, "w": self.w, "dilation": list(self.dilation),
            "n_global": self.n_global, "in_dtype": self.in_dtype,
            "seed": self.seed,
        }


def _long_globals(L: int = 65536, n: int = 16, seed: int = 4) -> tuple:
    """16 distinct positions drawn uniformly from [0, L) with a fresh generator."""
    g = torch.Generator().manual_seed(seed)
    return tuple(sorted(torch.randperm(L, generator=g)[:n].tolist()))


# The five synthetic configurations (tiny is the one the oracle finishes in
# well under a second; base is the L=4096 headline workload).
CONFIGS = {
    "tiny": Workload("tiny", 1, 2, 512, 64, 32, (1, 1), (0, 1), 0, "fp32"),
    "base": Workload("base", 2, 12, 4096, 64, 256, (1,) * 12, (0,), 1, "bf16"),
    "dilated": Workload("dilated", 1, 12, 8192, 64, 128, (1,) * 8 + (2,) * 4,
                        (0,), 2, "bf16"),
    "qa": Workload("qa", 4, 16, 4096, 64, 256, (1,) * 16, tuple(range(64)), 3,
                   "bf16"),
    "long": Workload("long", 1, 16, 65536, 128, 512, (1,) * 16,
                     _long_globals(), 4, "bf16"),
}

CONFIG_ORDER = ["tiny", "base", "dilated", "qa", "long"]


def custom(name: str, B: int, H: int, L: int, D: int, w: int,
           dilation: Sequence[int], global_idx: Sequence[int], seed: int,
           in_dtype: str = "bf16") -> Workload:
    return Workload(name, B, H, L, D, w, tuple(int(x) for x in dilation),
                    tuple(int(x) for x in global_idx), seed, in_dtype)


def make_qkv(wl: Workload, generator_device: str = "cpu"):
    """Draw q, k, v for a workload.

    Returns (q, k, v) as CPU tensors of the call dtype: bf16 for bf16
    workloads, fp32 for fp32 ones.  Use :func:`bf16_round_f64` to get the
    exact values the arithmetic sees.
    """
    g = torch.Generator(generator_device).manual_seed(wl.seed)
    shape = (wl.B, wl.H, wl.L, wl.D)
    out = []
    for _ in range(3):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if wl.in_dtype == "bf16":
            t = t.to(torch.bfloat16)
        out.append(t)
    return tuple(out)


def bf16_round_f64(t: torch.Tensor):
    """The bf16-rounded values of ``t`` as a float64 numpy array."""
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def random_globals(L: int, n: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    n = min(n, L)
    return tuple(sorted(torch.randperm(L, generator=g)[:n].tolist()))


# ------------------------------------------------- extra key-block tables
# Tables [H, T, R] of extra key blocks per 128-query tile (BigBird random
# blocks, or a fixed strided choice).  Head h with dilation d has
# nqt = ceil(ceil(L / d) / 128) tiles per residue class and d classes; its
# rows r*nqt + qt are used, the rest are -1.  Only indices are drawn here.

TILE = 128


def tiles_per_class(L: int, d: int) -> int:
    return -(-(-(-L // d)) // TILE)


def block_table_rows(L: int, dilation: Sequence[int]) -> int:
    """T: the table rows that every head's tiles fit in."""
    return max(int(d) * tiles_per_class(L, int(d)) for d in dilation)


def random_blocks(L: int, dilation: Sequence[int], R: int, seed: int) -> torch.Tensor:
    """R distinct key blocks per tile, uniform over the tile's class (fewer,
    padded with -1, when the class has fewer blocks); int32 [H, T, R]."""
    H, T = len(dilation), block_table_rows(L, dilation)
    g = torch.Generator().manual_seed(seed)
    tab = torch.full((H, T, R), -1, dtype=torch.int32)
    for h, d in enumerate(dilation):
        nqt = tiles_per_class(L, int(d))
        for row in range(int(d) * nqt):
            pick = torch.randperm(nqt, generator=g)[:R]
            tab[h, row, :pick.numel()] = pick.to(torch.int32)
    return tab


def strided_blocks(L: int, dilation: Sequence[int], stride: int) -> torch.Tensor:
    """Every tile lists the key blocks 0, stride, 2*stride, ... of its class;
    int32 [H, T, R] with R the longest such list."""
    H, T = len(dilation), block_table_rows(L, dilation)
    lists = [list(range(0, tiles_per_class(L, int(d)), stride)) for d in dilation]
    R = max(len(x) for x in lists)
    tab = torch.full((H, T, R), -1, dtype=torch.int32)
    for h, d in enumerate(dilation):
        nqt = tiles_per_class(L, int(d))
        tab[h, :int(d) * nqt, :len(lists[h])] = torch.tensor(lists[h], dtype=torch.int32)
    return tab


# ------------------------------------------------------------ layer inputs
# Synthetic inputs of one Longformer layer (random-init weights of the
# page's layer shape; no trained weights exist here).  Only random numbers:
#   x      ~ N(0, 1)                 bf16 [B, L, hidden]
#   w_qkv  ~ N(0, 1/hidden)          bf16 [3*hidden, hidden] (q, k, v rows)
#   b_qkv  ~ N(0, 0.02^2)            fp32 [3*hidden]
#   w_ff   ~ N(0, 1/hidden)          bf16 [hidden, hidden]
#   b_ff   ~ N(0, 0.02^2)            fp32 [hidden]
#   ln1/2  gamma ~ 1 + N(0, 0.1^2), beta ~ N(0, 0.1^2), fp32 [2*hidden]
# drawn in that order from one CPU generator seeded with `seed`.

@dataclasses.dataclass(frozen=True)
class LayerWorkload:
    name: str
    B: int
    L: int
    H: int
    D: int
    w: int
    dilation: tuple
    global_idx: tuple
    seed: int
    eps: float = 1e-5

    @property
    def hidden(self) -> int:
        return self.H * self.D

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


LAYER_CONFIGS = {
    "layer-tiny": LayerWorkload("layer-tiny", 1, 512, 2, 64, 32, (1, 1), (0, 1), 10),
    "layer-base": LayerWorkload("layer-base", 2, 4096, 12, 64, 256, (1,) * 12, (0,), 11),
}


def make_layer_inputs(lw: LayerWorkload):
    """CPU tensors (x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2) per the recipe above."""
    g = torch.Generator("cpu").manual_seed(lw.seed)
    h = lw.hidden
    x = torch.randn((lw.B, lw.L, h), generator=g).to(torch.bfloat16)
    w_qkv = (torch.randn((3 * h, h), generator=g) / math.sqrt(h)).to(torch.bfloat16)
    b_qkv = torch.randn((3 * h,), generator=g) * 0.02
    w_ff = (torch.randn((h, h), generator=g) / math.sqrt(h)).to(torch.bfloat16)
    b_ff = torch.randn((h,), generator=g) * 0.02
    ln1 = torch.cat([1 + 0.1 * torch.randn((h,), generator=g), 0.1 * torch.randn((h,), generator=g)])
    ln2 = torch.cat([1 + 0.1 * torch.randn((h,), generator=g), 0.1 * torch.randn((h,), generator=g)])
    return x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2
