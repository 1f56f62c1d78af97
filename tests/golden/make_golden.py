"""Writes tests/golden/long_globals.txt (the long workload's global positions).

The positions are part of the input recipe, not of the method: 16 distinct
positions drawn uniformly from [0, 65536) with torch.randperm on a fresh
generator seeded with 4, then sorted.  Stored so a change of the generator
is noticed.  Run: python tests/golden/make_golden.py
"""
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))

if __name__ == "__main__":
    g = torch.Generator().manual_seed(4)
    vals = sorted(torch.randperm(65536, generator=g)[:16].tolist())
    with open(os.path.join(HERE, "long_globals.txt"), "w") as f:
        f.write("# long workload: sorted(torch.randperm(65536, Generator().manual_seed(4))[:16])\n")
        f.write(" ".join(str(v) for v in vals) + "\n")
