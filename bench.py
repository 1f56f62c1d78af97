"""Benchmark of the Longformer sparse attention forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config base]

One step = one call of the whole forward (lf_attn_fwd: gather of global rows,
the band + global attention kernel, the global-row combine) on one batch of
the workload.  The default workload is "base" (B=2, H=12, L=4096, D=64,
one-sided window 256, no dilation, one global token at 0), the L=4096
configuration the headline metric is quoted on.  Inputs are seeded
synthetic N(0,1) values rounded to bf16 (see workloads.py).

Timing: W untimed warm-up steps; then K steps, each preceded by an L2 flush
(a 256 MiB device memset outside the timed events), each timed with CUDA
events on the launching stream; barrier + synchronize on both sides; the
maximum over ranks.  Under torchrun every rank runs its own replica of the
workload on its own GPU (the problem shards into independent (b, h) heads,
so there is no exchange on the data path): scaling is weak.

Metric: useful TFLOP/s = 4 * B * H * D * (attended pairs) / time, the pairs
counted by the library's own key-list enumerator (lf_attn_pairs).

--impl reference times the fp64 CPU oracle (the plain dense-masked
definition) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from long_sequence_sparse_lf_b300 import workloads as W  # noqa: E402

METRIC = "banded+global attention fwd useful TFLOP/s & % of BF16 tensor peak (1 B300)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["lf_attn_kernel.cuh", "lf_ptx.cuh", "lf_common.cuh"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "long_sequence_sparse_lf_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of attn_main from the committed ncu summary
    profiles/attn_main_<workload>.md (its "kernel_sha:" and
    "traffic_bytes_per_launch:" lines), if it was taken on the current kernel
    sources; else None."""
    path = os.path.join(ROOT, "profiles", f"attn_main_{workload}.md")
    try:
        with open(path, encoding="utf-8") as f:
            text = f.read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`").strip("-").strip()
        if ":" in line:
            key, _, val = line.partition(":")
            fields[key.strip()] = val.strip().strip("`")
    if fields.get("kernel_sha") != kernel_sha():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def useful_work(wl, pairs_all_heads: int):
    """pairs_all_heads: attended pairs summed over the H heads of one batch
    element (the pattern does not depend on b)."""
    flops = 4 * wl.B * wl.D * pairs_all_heads
    elt = 2  # bf16
    compulsory = 4 * wl.B * wl.H * wl.L * wl.D * elt   # q, k, v read + out write
    return flops, compulsory


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        loaded = [r for r in rows if num(r[4]) >= 50] or rows
        sm = [num(r[1]) for r in loaded if not math.isnan(num(r[1]))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(num(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


# --------------------------------------------------------------- CPU oracle

def oracle_sample(wl, q, k, v, budget_s: float, max_heads=None):
    """Runs the oracle over whole (b, h) heads until the time budget is spent.
    Returns (seconds, useful flops of the heads done, heads done, threads)."""
    from oracle import lf_oracle as O
    qf = q.to(torch.bfloat16).double().numpy()
    kf = k.to(torch.bfloat16).double().numpy()
    vf = v.to(torch.bfloat16).double().numpy()
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    if max_heads is not None:
        heads = heads[:max_heads]
    done, flops = 0, 0
    t0 = time.perf_counter()
    for (b, h) in heads:
        O.attention(qf[b:b + 1, h:h + 1], kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1],
                    wl.w, [wl.dilation[h]], wl.global_idx, wl.scale)
        done += 1
        flops += 4 * wl.D * O.pair_count(wl.L, wl.w, wl.dilation[h], wl.global_idx)
        if time.perf_counter() - t0 > budget_s:
            break
    return time.perf_counter() - t0, flops, done


def oracle_rows_step(wl, qf, kf, vf, rows, b, h):
    from oracle import lf_oracle as O
    O.attention(qf[b:b + 1, h:h + 1], kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1], wl.w,
                [wl.dilation[h]], wl.global_idx, wl.scale, rows=rows)
    pairs = 0
    for i in rows:
        pairs += len(O.key_set(int(i), wl.L, wl.w, wl.dilation[h], wl.global_idx))
    return 4 * wl.D * pairs


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ arms

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, pg=None, device="cpu") -> float:
    """The maximum of x over the ranks of the default process group (x itself
    without one): the job's time is its slowest replica's."""
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_value(flops_per_step: float, steps: int, world_size: int, total_ms: float) -> float:
    """Whole-job useful TFLOP/s of `world_size` replicas, each running `steps`
    steps of the same workload in `total_ms` (the maximum over ranks)."""
    return flops_per_step * world_size * steps / (total_ms * 1e-3) / 1e12


def run_reference(args, wl):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    q, k, v = W.make_qkv(wl)
    qf = q.to(torch.bfloat16).double().numpy()
    kf = k.to(torch.bfloat16).double().numpy()
    vf = v.to(torch.bfloat16).double().numpy()
    # size one step so that all steps end within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    oracle_rows_step(wl, qf, kf, vf, list(range(64)), 0, 0)
    per_row = (time.perf_counter() - t0) / 64
    n_rows = int(max(16, min(wl.L, budget / max(per_row, 1e-9))))
    rng = np.random.default_rng(0)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]

    def one_step(s):
        b, h = heads[s % len(heads)]
        r0 = int(rng.integers(0, max(1, wl.L - n_rows + 1)))
        return oracle_rows_step(wl, qf, kf, vf, list(range(r0, r0 + n_rows)), b, h)

    for s in range(args.warmup):
        one_step(s)
    t0 = time.perf_counter()
    flops = 0
    for s in range(args.steps):
        flops += one_step(s)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"fp64 dense-masked oracle, {args.steps} steps of {n_rows} consecutive query rows "
              f"of one (b,h) head each (heads in turn) of the {wl.name} workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wl.describe(), parallelism="host cores"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Timed steps are queued in batches behind a GPU-side pause (torch.cuda._sleep
# of about 10 ms at 2 GHz), long enough for the host to queue a batch.
QUEUE_BATCH = 100
QUEUE_SLEEP_CYCLES = 20_000_000


def percentiles_us(ms_list):
    """median, p10 and p90 of per-step times, in microseconds."""
    a = sorted(1e3 * x for x in ms_list)
    pick = lambda f: a[min(len(a) - 1, max(0, int(round(f * (len(a) - 1)))))]   # noqa: E731
    return {"median_us": pick(0.5), "p10_us": pick(0.1), "p90_us": pick(0.9), "n": len(a)}


def host_link(qh, kh, vh, oh, dev, reps: int = 3):
    """Time plain pinned copies: q, k, v host->device on one stream while
    the output's bytes go device->host on another (the copy engines work in
    both directions at once).  Returns the best of ``reps``."""
    nb = qh.numel() * qh.element_size()
    dq = torch.empty(3 * qh.numel(), dtype=qh.dtype, device=dev)
    do = torch.empty_like(oh, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = None
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(s_in):
            for x, t in enumerate((qh, kh, vh)):
                dq[x * qh.numel():(x + 1) * qh.numel()].view_as(t).copy_(t, non_blocking=True)
        with torch.cuda.stream(s_out):
            oh.copy_(do, non_blocking=True)
        torch.cuda.synchronize(dev)
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    return {"ms": best * 1e3, "h2d_bytes": 3 * nb, "d2h_bytes": nb,
            "h2d_gbs": 3 * nb / best / 1e9,
            "what": "pinned cudaMemcpyAsync of the same bytes, in and out concurrently"}


def run_ours(args, wl):
    import long_sequence_sparse_lf_b300 as lf
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    lf.load_library()

    q, k, v = W.make_qkv(wl)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # attended pairs from the library's enumerator (one count, not timed)
    _, _, pairs = lf.lf_attn_pairs(wl.H, wl.L, wl.w, wl.dilation, wl.global_idx,
                                   count_only=True, device=dev)
    flops, comp_bytes = useful_work(wl, pairs)

    # the forward with its arguments marshalled once (lf_attn_fwd through the C ABI)
    step = lf.prepare_fwd(qd, kd, vd, out, wl.w, wl.dilation, wl.global_idx, wl.scale, stream)

    # the clock sampler starts (and is given time to take its first sample)
    # before the warm-up, so that the warm-up steps come right before the
    # timed ones: an idle gap there leaves the first timed steps slow
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error after warm-up: " + lf.lf_last_error())

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    lf.lf_profile_reset()
    # events around attn_main only: every traced launch costs the stream an
    # event pair, and only attn_main's duration is used below
    lf.lf_profile_only("attn_main")
    lf.lf_profile_enable(True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    launches0 = lf.lf_launch_count()
    for lo in range(0, args.steps, QUEUE_BATCH):
        # a GPU-side pause ahead of each batch lets the host queue the
        # batch's launches before the GPU reaches them, so that the events
        # time the GPU's work and not the host's launch rate
        torch.cuda._sleep(QUEUE_SLEEP_CYCLES)
        for s in range(lo, min(args.steps, lo + QUEUE_BATCH)):
            flush.zero_()
            evs[s][0].record(stream)
            step()
            evs[s][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = lf.lf_launch_count() - launches0
    if pg:
        pg.barrier()
    clocks = sampler.stop() if sampler else None
    lf.lf_profile_enable(False)
    lf.lf_profile_only(None)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = float(sum(step_ms))
    main_ms, main_n = lf.lf_profile_query("attn_main")
    lf.lf_profile_reset()
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error in timed region: " + lf.lf_last_error())
    total_ms = max_over_ranks(total_ms, pg, dev)

    # ---- a second, L2-warm series (no flush between steps), reported
    # beside the cold headline: the same steps back to back
    wsteps = max(3, min(args.steps, 200))
    wevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(wsteps)]
    for _ in range(3):
        step()
    lf.lf_profile_enable(True)
    lf.lf_profile_only("attn_main")
    torch.cuda.synchronize(dev)
    for lo in range(0, wsteps, QUEUE_BATCH):
        torch.cuda._sleep(QUEUE_SLEEP_CYCLES)
        for s_ in range(lo, min(wsteps, lo + QUEUE_BATCH)):
            wevs[s_][0].record(stream)
            step()
            wevs[s_][1].record(stream)
    torch.cuda.synchronize(dev)
    lf.lf_profile_enable(False)
    lf.lf_profile_only(None)
    warm_ms = [a.elapsed_time(b) for a, b in wevs]
    warm_main_ms, warm_main_n = lf.lf_profile_query("attn_main")
    lf.lf_profile_reset()
    value = replica_value(flops, args.steps, ws, total_ms)
    ms_per_step = total_ms / args.steps

    # ---- end to end through the host-buffer entry point (pinned memory)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lf.lf_attn_fwd_host(qh, kh, vh, oh, wl.w, wl.dilation, wl.global_idx, wl.scale, stream)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        lf.lf_attn_fwd_host(qh, kh, vh, oh, wl.w, wl.dilation, wl.global_idx, wl.scale, stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, pg, dev)
    e2e_value = replica_value(flops, e2e_steps, ws, e2e_s * 1e3)
    io_bytes = qh.numel() * qh.element_size()
    # the host link alone: plain pinned copies of the same bytes, in (q, k,
    # v) and out at the same time on two streams, the bound of the e2e call
    link = host_link(qh, kh, vh, oh, dev)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel (attn_main)
    peaks, peak_src = load_peaks()
    main_avg_s = main_ms / max(main_n, 1) * 1e-3
    ai = flops / comp_bytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_achieved = flops / main_avg_s / 1e12
    hbm_achieved = comp_bytes / main_avg_s / 1e9
    traffic = recorded_traffic(wl.name)
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": hbm_achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": hbm_achieved / peaks["hbm_gbs"]}
    else:
        roof = {"bound": "tensor", "achieved": tensor_achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": tensor_achieved / peaks["bf16_tflops"]}
    roof.update({"traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json)"
                 if peak_src == "measured" else "fallback",
                 "kernel": "attn_main", "kernel_ms": main_avg_s * 1e3,
                 "algorithmic_bytes": comp_bytes, "useful_flops": flops,
                 "arithmetic_intensity": ai, "ridge": ridge,
                 "tensor_achieved_tflops": tensor_achieved,
                 "tensor_frac": tensor_achieved / peaks["bf16_tflops"]})

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": dict(wl.describe(), parallelism=f"replica x{ws}",
                       l2="flushed between timed steps (256 MiB memset)",
                       queue=f"launches queued ahead of the GPU in batches of {QUEUE_BATCH}",
                       pairs=pairs * wl.B),
        "peak_frac_bf16": value / peaks["bf16_tflops"],
        "roofline": roof,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 3 * io_bytes,
                "d2h_bytes_per_step": io_bytes, "steps": e2e_steps,
                "api": "lf_attn_fwd_host (pinned host buffers)",
                "ms_per_step": e2e_s * 1e3 / e2e_steps,
                "host_link": link,
                "link_bound_frac": link["ms"] / (e2e_s * 1e3 / e2e_steps)},
        "series": {
            "cold": dict(percentiles_us(step_ms), attn_main_avg_us=1e3 * main_ms / max(main_n, 1),
                         l2="256 MiB memset before every step"),
            "warm": dict(percentiles_us(warm_ms),
                         attn_main_avg_us=1e3 * warm_main_ms / max(warm_main_n, 1),
                         attn_main_tflops=flops / (warm_main_ms / max(warm_main_n, 1) * 1e-3) / 1e12,
                         steps=wsteps, l2="no flush (back-to-back steps)"),
        },
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        secs, cflops, heads = oracle_sample(wl, q, k, v, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": cflops / secs / 1e12, "unit": UNIT, "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"fp64 dense-masked oracle over {heads} whole (b,h) heads of the "
                      f"{wl.name} workload (time-bounded to ~{args.cpu_budget:.0f} s)"}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


LAYER_KERNELS = ("layer_gemm_qkv", "layer_split_qkv", "gather_globals", "attn_main",
                 "combine_globals", "layer_merge_ln1", "layer_gemm_ff", "layer_ln2")


def run_layer(args):
    """One Longformer layer forward (lf_layer_fwd) on a layer workload: QKV
    GEMM, head split, the sparse attention, residual + LayerNorm, the
    feed-forward GEMM, residual + LayerNorm.  Useful FLOPs = the two GEMMs
    (2*M*h*3h + 2*M*h*h, M = B*L tokens, h = hidden) + the attention's
    4*B*D*pairs; the metric is tokens per second."""
    import long_sequence_sparse_lf_b300 as lf
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lf.load_library()
    lw = W.LAYER_CONFIGS[args.layer]
    host_inputs = W.make_layer_inputs(lw)
    x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2 = (t.to(dev) for t in host_inputs)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    _, _, pairs = lf.lf_attn_pairs(lw.H, lw.L, lw.w, lw.dilation, lw.global_idx,
                                   count_only=True, device=dev)
    M, h = lw.B * lw.L, lw.hidden
    gemm_flops = {"layer_gemm_qkv": 2 * M * h * 3 * h, "layer_gemm_ff": 2 * M * h * h}
    attn_flops = 4 * lw.B * lw.D * pairs
    flops = sum(gemm_flops.values()) + attn_flops

    def step(xin, yout):
        lf.lf_layer_fwd(xin, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, yout, lw.H, lw.w,
                        lw.dilation, lw.global_idx, lw.scale, lw.eps, stream)

    # the clock sampler starts (and is given time to take its first sample)
    # before the warm-up, so that the warm-up steps come right before the
    # timed ones: an idle gap there leaves the first timed steps slow
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush.zero_()
        step(x, out)
    torch.cuda.synchronize(dev)
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error after warm-up: " + lf.lf_last_error())
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    lf.lf_profile_reset()
    # in the timed loop only attn_main (the roofline's kernel) is bracketed by
    # events: each traced launch costs the stream an event pair
    lf.lf_profile_only("attn_main")
    lf.lf_profile_enable(True)
    torch.cuda.synchronize(dev)
    launches0 = lf.lf_launch_count()
    for s_ in range(args.steps):
        flush.zero_()
        evs[s_][0].record(stream)
        step(x, out)
        evs[s_][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = lf.lf_launch_count() - launches0
    clocks = sampler.stop()
    lf.lf_profile_enable(False)
    lf.lf_profile_only(None)
    total_ms = float(sum(a.elapsed_time(b) for a, b in evs))
    attn_ms, attn_n = lf.lf_profile_query("attn_main")
    lf.lf_profile_reset()
    # per-kernel breakdown: a separate loop with every launch traced
    prof_steps = min(args.steps, 20)
    lf.lf_profile_enable(True)
    for _ in range(prof_steps):
        flush.zero_()
        step(x, out)
    torch.cuda.synchronize(dev)
    lf.lf_profile_enable(False)
    per_kernel = {}
    for name in LAYER_KERNELS:
        ms, n = lf.lf_profile_query(name)
        if n:
            per_kernel[name] = ms / prof_steps
    lf.lf_profile_reset()
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error in timed region: " + lf.lf_last_error())
    ms_per_step = total_ms / args.steps
    value = M * args.steps / (total_ms * 1e-3)

    # ---- end to end: x from pinned host memory, the layer, the result back
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    xh = host_inputs[0].contiguous().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    xd, od = torch.empty_like(x), torch.empty_like(out)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        xd.copy_(xh, non_blocking=True)
        step(xd, od)
        oh.copy_(od, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    io_bytes = xh.numel() * xh.element_size()

    # ---- roofline of the layer's largest kernel, the attention (timed in the loop)
    peaks, peak_src = load_peaks()
    attn_s = attn_ms / max(attn_n, 1) * 1e-3
    ach = attn_flops / attn_s / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": None,
            "kernel": "attn_main", "kernel_ms": attn_s * 1e3,
            "peak_source": "measured (MEASURED_PEAKS.json)" if peak_src == "measured"
            else "fallback"}
    line = {
        "metric": "Longformer layer fwd tokens/s (QKV GEMM, sparse attention, LN, FF GEMM, "
                  "LN; 1 B300)",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded inputs and random-init weights of the layer's shape)",
        "config": {"workload": lw.name, "B": lw.B, "L": lw.L, "H": lw.H, "D": lw.D,
                   "hidden": h, "w": lw.w, "n_global": len(lw.global_idx),
                   "l2": "flushed between timed steps (256 MiB memset)",
                   "useful_tflop_per_step": flops / 1e12},
        "useful_tflops": flops * args.steps / (total_ms * 1e-3) / 1e12,
        "kernel_ms_per_step": per_kernel,
        "kernel_ms_note": "from a separate loop of min(steps, 20) steps with every launch "
                          "bracketed by events (not the timed loop)",
        "roofline": roof,
        "gpu_launches": launches,
        "e2e": {"value": M * e2e_steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                "steps": e2e_steps, "api": "lf_layer_fwd with x copied from pinned host "
                                           "memory and the result copied back"},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle as O
        rows = list(range(0, lw.L, max(1, lw.L // 64)))
        xs = [t.double().numpy() for t in host_inputs]
        t0 = time.perf_counter()
        O.longformer_layer(*xs, lw.H, lw.w, lw.dilation, lw.global_idx, lw.scale, lw.eps,
                           store_bf16=True, rows=rows)
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": lw.B * len(rows) / secs, "unit": "tokens/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"fp64 layer oracle for {len(rows)} token rows per batch element "
                      f"(its q/k/v GEMM over all {lw.L} tokens is included)"}
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args, wl):
    """The backward (lf_attn_bwd) on a workload: useful FLOPs = 10*B*D*pairs
    (recomputed S, dP, dV, dK, dQ products per attended pair)."""
    import long_sequence_sparse_lf_b300 as lf
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lf.load_library()
    q, k, v = W.make_qkv(wl)
    g = torch.Generator("cpu").manual_seed(wl.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, dout))
    out = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    lf.lf_attn_fwd_lse(qd, kd, vd, out, lse, wl.w, wl.dilation, wl.global_idx, wl.scale, stream)
    grads = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    _, _, pairs = lf.lf_attn_pairs(wl.H, wl.L, wl.w, wl.dilation, wl.global_idx,
                                   count_only=True, device=dev)
    flops = 10 * wl.B * wl.D * pairs

    def step(bufs):
        lf.lf_attn_bwd(*bufs, wl.w, wl.dilation, wl.global_idx, wl.scale, stream)

    bufs = (qd, kd, vd, out, lse, dod, *grads)
    # the clock sampler starts (and is given time to take its first sample)
    # before the warm-up, so that the warm-up steps come right before the
    # timed ones: an idle gap there leaves the first timed steps slow
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush.zero_()
        step(bufs)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    lf.lf_profile_reset()
    lf.lf_profile_only("bwd_tc")
    lf.lf_profile_enable(True)
    torch.cuda.synchronize(dev)
    launches0 = lf.lf_launch_count()
    for s_ in range(args.steps):
        flush.zero_()
        evs[s_][0].record(stream)
        step(bufs)
        evs[s_][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = lf.lf_launch_count() - launches0
    clocks = sampler.stop()
    lf.lf_profile_enable(False)
    lf.lf_profile_only(None)
    total_ms = float(sum(a.elapsed_time(b) for a, b in evs))
    # the tcgen05 kernel's launches of a step (band tiles, then global-key
    # tiles when the pattern has global tokens) own every attended pair
    tc_ms, _ = lf.lf_profile_query("bwd_tc")
    lf.lf_profile_reset()
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error in timed region: " + lf.lf_last_error())
    value = flops * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end: inputs from pinned host memory, gradients back
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_in = [t.cpu().pin_memory() for t in (qd, kd, vd, out, lse, dod)]
    host_out = [torch.empty(q.shape, dtype=torch.float32).pin_memory() for _ in range(3)]
    dev_in = [torch.empty_like(t) for t in (qd, kd, vd, out, lse, dod)]
    dev_out = [torch.empty_like(t) for t in grads]
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for dd, hh in zip(dev_in, host_in):
            dd.copy_(hh, non_blocking=True)
        step((*dev_in, *dev_out))
        for hh, dd in zip(host_out, dev_out):
            hh.copy_(dd, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    peaks, peak_src = load_peaks()
    tc_s = tc_ms / args.steps * 1e-3
    ach = flops / tc_s / 1e12
    line = {
        "metric": "banded+global attention backward useful TFLOP/s (10*D per attended pair; "
                  "1 B300)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded; dout from seed+1000)",
        "config": dict(wl.describe(), l2="flushed between timed steps (256 MiB memset)",
                       pairs=pairs * wl.B),
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": None,
                     "kernel": "lf_bwd_band_tc_kernel (all launches of a step)",
                     "kernel_ms": tc_s * 1e3, "kernel_useful_flops": flops,
                     "peak_source": "measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback"},
        "gpu_launches": launches,
        "e2e": {"value": flops * e2e_steps / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "lf_attn_bwd with inputs copied from pinned host memory and the "
                       "gradients copied back"},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle as O
        heads = max(1, min(wl.H, 2))
        qf, kf, vf, df = (t[:1, :heads].double().numpy() for t in (q, k, v, dout))
        t0 = time.perf_counter()
        O.attention_backward(qf, kf, vf, df, wl.w, wl.dilation[:heads], wl.global_idx, wl.scale)
        secs = time.perf_counter() - t0
        sample_pairs = pairs * heads / wl.H
        line["cpu_baseline"] = {
            "value": 10 * wl.D * sample_pairs / secs / 1e12, "unit": "TFLOP/s",
            "cores": cpu_threads(), "kind": "oracle",
            "sample": f"fp64 dense-masked backward oracle over {heads} (b,h) heads of the "
                      f"{wl.name} workload"}
    print(json.dumps(line), flush=True)
    return 0

def extra_block_pairs(wl, tab) -> int:
    """Attended pairs that a table of extra key blocks adds, summed over heads
    and batch: per tile, its listed blocks' keys (deduplicated, clipped to the
    class) that are not global, times its non-global rows whose window does
    not already hold them (|t' - t| > w in residue space)."""
    tab = np.asarray(tab)
    L, w = wl.L, wl.w
    isg = np.zeros(L, dtype=bool)
    isg[list(wl.global_idx)] = True
    total = 0
    for h, d in enumerate(wl.dilation):
        nqt = W.tiles_per_class(L, d)
        for r in range(d):
            pos = np.arange(r, L, d)
            Lr = pos.size
            for qt in range(nqt):
                rows = np.arange(qt * W.TILE, min(qt * W.TILE + W.TILE, Lr))
                kbs = sorted(set(int(x) for x in tab[h, r * nqt + qt] if x >= 0))
                if rows.size == 0 or not kbs:
                    continue
                keys = np.concatenate([np.arange(kb * W.TILE, min(kb * W.TILE + W.TILE, Lr))
                                       for kb in kbs])
                keys = keys[~isg[pos[keys]]]
                rows = rows[~isg[pos[rows]]]
                total += int((np.abs(keys[None, :] - rows[:, None]) > w).sum())
    return total * wl.B


def run_variant(args, wl, variant: str):
    """A forward variant on a workload, timed like the plain forward:
      "bias"           lf_attn_fwd_bias, table N(0,1) fp32 [H, 2w+1];
      "blocks-random"  lf_attn_fwd_blocks, 3 random key blocks per tile
                       (BigBird-style), seeded;
      "blocks-strided" lf_attn_fwd_blocks, key blocks 0, 8, 16, ... per tile.
    Useful FLOPs = 4*D per attended pair (the variant's own key sets)."""
    import long_sequence_sparse_lf_b300 as lf
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lf.load_library()
    q, k, v = W.make_qkv(wl)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    _, _, pairs = lf.lf_attn_pairs(wl.H, wl.L, wl.w, wl.dilation, wl.global_idx,
                                   count_only=True, device=dev)
    pairs *= wl.B
    extra_host = []        # host inputs copied each e2e step (besides q, k, v)
    if variant == "bias":
        g = torch.Generator("cpu").manual_seed(wl.seed + 2000)
        rb = torch.randn((wl.H, 2 * wl.w + 1), generator=g)
        rbd = rb.to(dev)
        extra_host = [rb]

        def step(a, b, c, o, dev_extra):
            lf.lf_attn_fwd_bias(a, b, c, o, dev_extra[0], wl.w, wl.dilation, wl.global_idx,
                                wl.scale, stream)
        dev_extra = [rbd]
        metric = ("banded+global attention forward with relative position bias, useful "
                  "TFLOP/s (4*D per attended pair; 1 B300)")
        data = "synthetic (seeded N(0,1), bf16-rounded; bias N(0,1) fp32 from seed+2000)"
        cfg_extra = {"rel_bias": "[H, 2w+1] fp32"}
        kernel = "attn_main (bias build)"
    else:
        if variant == "blocks-random":
            tab = W.random_blocks(wl.L, wl.dilation, 3, wl.seed + 3000)
            cfg_extra = {"extra_blocks": "3 random key blocks of 128 per 128-query tile "
                                         "(seed+3000)"}
        else:
            tab = W.strided_blocks(wl.L, wl.dilation, 8)
            cfg_extra = {"extra_blocks": "key blocks 0, 8, 16, ... of 128 per 128-query tile"}
        pairs += extra_block_pairs(wl, tab)
        # the table is a host argument of the call: it is read on the host every step

        def step(a, b, c, o, dev_extra):
            lf.lf_attn_fwd_blocks(a, b, c, o, wl.w, wl.dilation, wl.global_idx, tab, wl.scale,
                                  stream)
        dev_extra = []
        metric = ("banded+global attention forward with extra key blocks per tile (BigBird "
                  "random / strided), useful TFLOP/s (4*D per attended pair; 1 B300)")
        data = "synthetic (seeded N(0,1), bf16-rounded; block table seeded)"
        kernel = "attn_main (extra-block build)"
    flops = 4 * wl.D * pairs

    # the clock sampler starts (and is given time to take its first sample)
    # before the warm-up, so that the warm-up steps come right before the
    # timed ones: an idle gap there leaves the first timed steps slow
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush.zero_()
        step(qd, kd, vd, out, dev_extra)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    lf.lf_profile_reset()
    lf.lf_profile_only("attn_main")
    lf.lf_profile_enable(True)
    torch.cuda.synchronize(dev)
    launches0 = lf.lf_launch_count()
    for s_ in range(args.steps):
        flush.zero_()
        evs[s_][0].record(stream)
        step(qd, kd, vd, out, dev_extra)
        evs[s_][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = lf.lf_launch_count() - launches0
    clocks = sampler.stop()
    lf.lf_profile_enable(False)
    lf.lf_profile_only(None)
    total_ms = float(sum(a.elapsed_time(b) for a, b in evs))
    main_ms, main_n = lf.lf_profile_query("attn_main")
    lf.lf_profile_reset()
    if lf.lf_attn_get_status(stream) != 0:
        raise SystemExit("device status error in timed region: " + lf.lf_last_error())
    value = flops * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end: q, k, v (and a bias table) from pinned host memory, out back
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_in = [t.pin_memory() for t in (q, k, v, *extra_host)]
    host_out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    dev_in = [torch.empty_like(t, device=dev) for t in host_in]
    dev_out = torch.empty_like(out)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for dd, hh in zip(dev_in, host_in):
            dd.copy_(hh, non_blocking=True)
        step(dev_in[0], dev_in[1], dev_in[2], dev_out, dev_in[3:])
        host_out.copy_(dev_out, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    peaks, peak_src = load_peaks()
    main_s = main_ms / max(main_n, 1) * 1e-3
    ach = flops / main_s / 1e12
    line = {
        "metric": metric,
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": data,
        "config": dict(wl.describe(), l2="flushed between timed steps (256 MiB memset)",
                       pairs=pairs, **cfg_extra),
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": None,
                     "kernel": kernel, "kernel_ms": main_s * 1e3,
                     "peak_source": "measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback"},
        "gpu_launches": launches,
        "e2e": {"value": flops * e2e_steps / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": f"the {variant} forward with its inputs copied from pinned host memory "
                       "and the output copied back"},
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle as O
        rows = list(range(0, wl.L, max(1, wl.L // 256)))
        qf, kf, vf = (t[:1].double().numpy() for t in (q, k, v))
        kw = {"rel_bias": rb.double().numpy()} if variant == "bias" else \
             {"xblocks": np.asarray(tab)}
        t0 = time.perf_counter()
        O.attention(qf, kf, vf, wl.w, wl.dilation, wl.global_idx, wl.scale, rows=rows, **kw)
        secs = time.perf_counter() - t0
        sample_pairs = pairs / wl.B * len(rows) / wl.L
        line["cpu_baseline"] = {
            "value": 4 * wl.D * sample_pairs / secs / 1e12, "unit": "TFLOP/s",
            "cores": cpu_threads(), "kind": "oracle",
            "sample": f"fp64 dense-masked oracle of the {variant} forward, {len(rows)} evenly "
                      f"spaced rows of every head of one batch element of the {wl.name} "
                      "workload"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="base", choices=W.CONFIG_ORDER)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward (lf_attn_bwd) on --config instead of the forward")
    ap.add_argument("--layer", default=None, choices=sorted(W.LAYER_CONFIGS),
                    help="time one Longformer layer forward (lf_layer_fwd) instead of the "
                         "attention alone")
    ap.add_argument("--rel-bias", action="store_true",
                    help="time the relative-position-bias forward (lf_attn_fwd_bias) on --config")
    ap.add_argument("--blocks", default=None, choices=["random", "strided"],
                    help="time the forward with extra key blocks per tile (lf_attn_fwd_blocks): "
                         "3 random blocks, or blocks 0, 8, 16, ...")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.backward:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the backward line has no "
                              "reference arm"}))
            return 0
        return run_backward(args, W.CONFIGS[args.config])
    if args.rel_bias or args.blocks:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the variant lines have no "
                              "reference arm"}))
            return 0
        variant = "bias" if args.rel_bias else "blocks-" + args.blocks
        return run_variant(args, W.CONFIGS[args.config], variant)
    if args.layer is not None:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the layer line has no "
                              "reference arm; time the oracle with the default layer run"}))
            return 0
        return run_layer(args)
    wl = W.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
