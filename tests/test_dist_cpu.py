"""The multi-process path of bench.py on CPU (gloo, world size 2, 127.0.0.1):
the path shards into independent replicas, so the only cross-rank steps are
the barrier and the maximum of the timings, and the whole-job value counts
every rank's steps.  The reference arm runs on rank 0 only: the other ranks
return without work."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_CODE = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
dist.barrier()
local_ms = [12.5, 30.0][rank]
got = bench.max_over_ranks(local_ms, dist, "cpu")
value = bench.replica_value(2.0e12, 10, dist.get_world_size(), got)
dist.barrier()
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "max_ms": got, "value": value}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code, world=2, extra_env=None, timeout=120):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=timeout)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_and_weak_scaling_value():
    outs = _run_ranks(RANK_CODE.format(root=ROOT))
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    for r in res:
        assert r["max_ms"] == 30.0          # the slower replica sets the job's time
        # 2 ranks x 10 steps x 2 TFLOP in 30 ms
        assert abs(r["value"] - 2 * 10 * 2.0 / 0.030) < 1e-9


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0) == 7.0
    assert abs(bench.replica_value(1e12, 4, 1, 8.0) - 500.0) < 1e-9


def test_reference_arm_other_ranks_exit_without_work():
    code = r"""
import sys
sys.path.insert(0, {root!r})
import argparse, bench
from long_sequence_sparse_lf_b300 import workloads as W
args = argparse.Namespace(steps=2, warmup=3)
print("rc", bench.run_reference(args, W.CONFIGS["base"]))
""".format(root=ROOT)
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "rc 0"
