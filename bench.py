#!/usr/bin/env python
"""Attention throughput on GB300: TFLOP/s of forward and of forward+backward (bf16, causal).

One step = one pass of the whole path on one batch: fa_fwd (O, LSE) then the three backward
stages (fa_bwd_prepare, fa_bwd_compute, fa_bwd_finalize) on the Llama-3.1-8B-shaped causal
workload B=4, Hq=32, Hkv=8 (GQA 4:1), N=4096, d=128, bf16, inputs N(0,1)*0.5 from seed 2.
FLOPs are algorithmic: 4*d per visible (query, key) pair for the forward (2*d*N*(N+1) per
head, causal), 2.5x that for the backward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). With N > 1 (launched by torch.distributed.run) every rank
runs the same per-GPU workload on its own GPU with no data-path collective (weak scaling);
the timing uses a barrier and the max over ranks. `--impl reference` times the fp64 CPU
oracle on the host cores on bounded samples of the same workload.
`--batch B` shrinks the batch for profiling runs only; such a line is not a bench value.
`--workload softmax_rows|splitkv|window|naive|sweep|long|shape` times one of the extra
workloads instead (the row softmax, split-KV, sliding window, S/P-through-HBM attention, a
sequence-length sweep at B*N = 16384, the N = 131072 long-context forward, or the single shape
given by --shape B,Hq,Hkv,N,d,causal) and prints its own JSON line. The default line also
carries `targets`: the causal d=128 bar at N >= 4096 (forward >= 60 %, backward >= 45 % of the
bf16 peak) on the sweep's shapes and the long-context forward.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd & fwd+bwd (bf16, d=128, causal) and % of dense BF16 peak"
WL = dict(B=4, Hq=32, Hkv=8, N=4096, d=128, causal=True, value_scale=0.5, seed=2)
WORKLOAD_NAME = "llama3.1-8b attention: B=4 Hq=32 Hkv=8 N=4096 d=128 causal bf16, fwd+bwd"
BWD_FACTOR = 2.5
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fa_bwd_compute_llama8b_traffic.txt")
KERNEL_SOURCES = ["online_softmax_09_gb300/csrc/fa_bwd.cu", "online_softmax_09_gb300/csrc/fa_ptx.cuh"]


def fwd_flops(B, Hq, N, d, causal):
    pairs = N * (N + 1) // 2 if causal else N * N
    return 4 * d * pairs * B * Hq


def rows_flops(rows, d, causal, N):
    """fwd+bwd algorithmic FLOPs of a block of query rows of one head."""
    pairs = sum((i + 1) if causal else N for i in rows)
    return 4 * d * pairs * (1 + BWD_FACTOR)


def config_block():
    return {"workload": WORKLOAD_NAME, "B": WL["B"], "Hq": WL["Hq"], "Hkv": WL["Hkv"], "N": WL["N"], "d": WL["d"],
            "causal": WL["causal"], "inputs": "iid N(0,1)*0.5 from seed 2, cast to bf16",
            "l2": "inputs larger than L2: ~0.9 GB touched per step (q,k,v,o,dO,dq,dk,dv,workspace), no flush",
            "parallelism": "replicas (independent per-GPU workload, no collective)"}


def cores_used():
    n = len(os.sched_getaffinity(0))
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return min(n, int(os.environ[var]))
    return n


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes per launch of the backward compute kernel from the committed ncu summary,
    or None when that summary was taken on different kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.loads(f.read().split("\n---\n", 1)[0])
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def rank_max(value, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (the timing rule: the slowest rank sets the time).
    Identity without a process group."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_peak(timed_ms, burst, sustained, src, clocks):
    """The bf16 peak a kernel timed inside `timed_ms` of back-to-back work is held to: the burst
    figure (cuBLAS timed alone) unless the timed region lasts seconds, like the sustained figure's
    own loop; then the sustained one. Returns (peak, explanation)."""
    mhz = clocks.get("sm_mhz") if clocks else None
    clk = f", median SM clock {mhz:.0f} MHz during the timed region" if mhz else ""
    if timed_ms >= 2000.0:
        return sustained, f"{src} bf16_tflops_sustained: timed region {timed_ms / 1e3:.2f} s{clk}"
    return burst, f"{src} bf16_tflops (burst): timed region {timed_ms:.0f} ms, well under the sustained loop{clk}"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------------------------------
# Clock sampling (nvidia-smi) during the timed region.
# --------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------------------------
# Our arm: the CUDA path through the C ABI.
# --------------------------------------------------------------------------------------------
def run_ours(args):
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    B = args.batch if args.batch else WL["B"]
    Hq, Hkv, N, d, causal = WL["Hq"], WL["Hkv"], WL["N"], WL["d"], WL["causal"]

    qh, kh, vh, doh = make_qkv(B, Hq, Hkv, N, d, seed=WL["seed"], value_scale=WL["value_scale"], with_do=True)
    q, k, v, do = (t.to(dev) for t in (qh, kh, vh, doh))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    f_fwd = fwd_flops(B, Hq, N, d, causal)
    f_step = f_fwd * (1 + BWD_FACTOR)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.forward(q, k, v, causal, out=o, lse=lse)
        fa.backward_stages(q, k, v, o, do, lse, dq, dk, dv, ws, causal,
                           between=(lambda i: ev[i + 1].record(stream)) if ev is not None else None)

    for _ in range(args.warmup):
        step()
    fa.check()
    # Tiles the forward computes and skips (fa_fwd_stats, one counted call outside the timed
    # region): the FLOPs the kernels execute, whole 128 x 128 tiles included.
    counters = torch.zeros(3, dtype=torch.int64, device=dev)
    fa.forward(q, k, v, causal, out=o, lse=lse, counters=counters)
    fa.check()
    tiles_done, tiles_skipped = (int(x) for x in counters[:2].tolist())
    tile_fwd_flops = tiles_done * 4 * 128 * 128 * d

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(dev).uuid)) if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clock:
        clock.start()
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = clock.stop() if clock else None
    fa.check()
    total_ms = t0.elapsed_time(t1)
    # evs[i]: 0 before fa_fwd, 1 before prepare, 2 before compute, 3 before finalize, 4 after it
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_compute_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[4]) for e in evs)
    total_ms = rank_max(total_ms, dist, dev)

    e2e = None
    if not args.no_e2e:
        # End to end through the C ABI with host buffers (fa_fwd_bwd_host): every step copies
        # q, k, v, dO from pinned host memory to the device, runs the whole path and copies
        # o, lse, dq, dk, dv back to pinned host memory; the library overlaps the copies of one
        # batch element with the kernels of another.
        hin = [t.pin_memory() for t in (qh, kh, vh, doh)]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
        hws = torch.empty(fa.fwd_bwd_host_workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
        E = max(3, min(K, 50))

        def e2e_step():
            fa.fwd_bwd_host(*hin, causal, out=hout, workspace=hws, stream=stream)

        e2e_step()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        a0.record(stream)
        for _ in range(E):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        fa.check()
        e2e_ms = rank_max(a0.elapsed_time(a1) / E, dist, dev)
        e2e = {"value": round(world * f_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout)}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    burst, sustained, src = load_peaks()
    ms_step = total_ms / K
    value = world * f_step / (ms_step * 1e-3) / 1e12
    achieved = f_fwd * BWD_FACTOR / (bwd_compute_ms * 1e-3) / 1e12
    peak, peak_note = roofline_peak(total_ms, burst, sustained, src, clocks)
    cfg = config_block()
    if B != WL["B"]:
        cfg["workload"] = f"PROFILING CASE (not a bench value): batch {B} instead of {WL['B']}"
        cfg["B"] = B
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": cfg,
        "fwd": {"tflops": round(f_fwd / (fwd_ms * 1e-3) / 1e12, 2), "ms": round(fwd_ms, 4),
                "pct_of_peak_burst": round(100 * f_fwd / (fwd_ms * 1e-3) / 1e12 / burst, 2)},
        "fwd_bwd": {"tflops": round(value / world, 2), "ms": round(fwd_ms + bwd_ms, 4),
                    "pct_of_peak_burst": round(100 * value / world / burst, 2),
                    "bwd_tflops": round(f_fwd * BWD_FACTOR / (bwd_ms * 1e-3) / 1e12, 2),
                    "bwd_pct_of_peak_burst": round(100 * f_fwd * BWD_FACTOR / (bwd_ms * 1e-3) / 1e12 / burst, 2)},
        "roofline": {"kernel": "fa_bwd_main_kernel<128> (fa_bwd_compute)", "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "peak_source": peak_note,
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic(),
                     "algorithmic_flops_per_launch": f_fwd * BWD_FACTOR, "ms_per_launch": round(bwd_compute_ms, 4)},
        "executed": {"tiles_computed": tiles_done, "tiles_skipped": tiles_skipped,
                     "fwd_flops": tile_fwd_flops, "fwd_tflops": round(tile_fwd_flops / (fwd_ms * 1e-3) / 1e12, 2),
                     "fwd_bwd_tflops": round(tile_fwd_flops * (1 + BWD_FACTOR) / (ms_step * 1e-3) / 1e12, 2),
                     "note": "FLOPs of every computed 128x128 tile (diagonal tiles in full), against the "
                             "algorithmic count of visible pairs used everywhere else"},
        "e2e": e2e,
        "gpu_launches": 4 * K,
        "clocks": clocks,
    }
    if world == 1 and not args.no_targets:
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
        line["targets"] = run_targets(burst, src)  # its own launches, outside the timed region
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(qh, kh, vh, doh, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------------------------
# The fp64 CPU oracle on the host cores (reported baseline; never the product path).
# --------------------------------------------------------------------------------------------
def _oracle_blocks(qh, kh, vh, doh, rows_per_block):
    """Endless sequence of (head arrays, rows) samples of the workload: blocks of query rows
    of one head at a time, walking the rows from the end (the longest causal rows first)."""
    from online_softmax_09_gb300.inputs import to_f64

    G = WL["Hq"] // WL["Hkv"]
    N = qh.shape[2]
    heads = [(b, h) for b in range(qh.shape[0]) for h in range(qh.shape[1])]
    cache = {}
    while True:
        for b, h in heads:
            if (b, h) not in cache:
                cache.clear()
                cache[(b, h)] = tuple(to_f64(t) for t in (qh[b, h], kh[b, h // G], vh[b, h // G], doh[b, h]))
            for end in range(N, 0, -rows_per_block):
                yield cache[(b, h)], list(range(max(0, end - rows_per_block), end))


def cpu_baseline(qh, kh, vh, doh, budget_s=15.0, rows_per_block=256):
    import oracle

    scale = 1 / math.sqrt(WL["d"])
    done_flops, done_rows, t_used = 0.0, 0, 0.0
    for arrs, rows in _oracle_blocks(qh, kh, vh, doh, rows_per_block):
        t = time.perf_counter()
        oracle.attention_query_block(*arrs, rows, WL["causal"], scale)
        t_used += time.perf_counter() - t
        done_flops += rows_flops(rows, WL["d"], WL["causal"], WL["N"])
        done_rows += len(rows)
        if t_used >= budget_s:
            break
    return {"value": round(done_flops / t_used / 1e12, 6), "unit": "TFLOP/s", "cores": cores_used(),
            "kind": "oracle",
            "sample": f"fp64 NumPy oracle (S and P materialised), fwd+bwd of {done_rows} query rows starting at "
                      f"head (0,0), {rows_per_block}-row blocks from the last row down, {t_used:.1f} s of host time",
            "small_configs": small_config_timings()}


SMALL_CONFIGS = [  # (name, B, H, N, d, causal, with backward, seed): the two small workload configurations
    ("B=1 H=1 N=256 d=64 non-causal fwd", 1, 1, 256, 64, False, False, 0),
    ("B=2 H=8 N=1024 d=64 causal fwd+bwd", 2, 8, 1024, 64, True, True, 1),
    ("B=2 H=8 N=1024 d=64 non-causal fwd+bwd", 2, 8, 1024, 64, False, True, 1),
]
THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _time_small_configs(repeats=3):
    """Best-of-`repeats` seconds of the fp64 oracle on each small configuration (whole problem)."""
    import oracle
    from online_softmax_09_gb300.inputs import make_qkv, to_f64

    out = []
    for name, B, H, N, d, causal, bwd, seed in SMALL_CONFIGS:
        q, k, v, do = (to_f64(t) for t in make_qkv(B, H, H, N, d, seed=seed, with_do=True))
        scale = 1 / math.sqrt(d)
        best = float("inf")
        for _ in range(repeats):
            t = time.perf_counter()
            oracle.attention_forward(q, k, v, causal, scale)
            if bwd:
                oracle.attention_backward(q, k, v, do, causal, scale)
            best = min(best, time.perf_counter() - t)
        out.append({"config": name, "seconds": round(best, 5)})
    return out


def small_config_timings():
    """The oracle on the small configurations with all host cores, and with one thread (a child
    process started with the BLAS thread variables set to 1, so the setting holds from import)."""
    rows = _time_small_configs()
    env = dict(os.environ, **{v: "1" for v in THREAD_VARS})
    single = None
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--small-configs-child"], env=env,
                           capture_output=True, text=True, timeout=300)
        if r.returncode == 0:
            single = json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.TimeoutExpired, ValueError, IndexError):
        single = None
    for i, row in enumerate(rows):
        row["seconds_all_cores"] = row.pop("seconds")
        row["seconds_1_thread"] = single[i]["seconds"] if single else None
    return {"cores": cores_used(), "rows": rows}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    from online_softmax_09_gb300.inputs import make_qkv

    qh, kh, vh, doh = make_qkv(WL["B"], WL["Hq"], WL["Hkv"], WL["N"], WL["d"], seed=WL["seed"],
                               value_scale=WL["value_scale"], with_do=True)
    scale = 1 / math.sqrt(WL["d"])
    # Size each step so that warm-up + timed steps take about two minutes of host time.
    budget = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    gen = _oracle_blocks(qh, kh, vh, doh, 64)
    arrs, rows = next(gen)
    t = time.perf_counter()
    oracle.attention_query_block(*arrs, rows, WL["causal"], scale)
    per_row = (time.perf_counter() - t) / len(rows)
    rpb = int(max(8, min(WL["N"], budget / max(per_row, 1e-9))))
    gen = _oracle_blocks(qh, kh, vh, doh, rpb)
    for _ in range(args.warmup):
        arrs, rows = next(gen)
        oracle.attention_query_block(*arrs, rows, WL["causal"], scale)
    flops, secs, nrows = 0.0, 0.0, 0
    for _ in range(args.steps):
        arrs, rows = next(gen)
        t = time.perf_counter()
        oracle.attention_query_block(*arrs, rows, WL["causal"], scale)
        secs += time.perf_counter() - t
        flops += rows_flops(rows, WL["d"], WL["causal"], WL["N"])
        nrows += len(rows)
    value = flops / secs / 1e12
    sample = (f"fp64 NumPy oracle, fwd+bwd of up to {rpb} query rows per step ({nrows} rows in total) of the same "
              f"workload, rows walked from the last row of head (0,0) down")
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_block(),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------------
# Extra workloads (not the headline metric): one JSON line each, same timing rules.
# --------------------------------------------------------------------------------------------
def load_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_softmax_rows(args):
    """Online-softmax rows (fa_softmax_rows): 65536 rows x 2048 fp32 logits, N(0,1)*8 from seed 3
    (the shape of the pages' check, scaled up to be HBM-sized: 512 MiB in, 512 MiB out)."""
    import torch

    from online_softmax_09_gb300 import fa

    rows, n = 65536, 2048
    g = torch.Generator().manual_seed(3)
    xh = torch.randn(rows, n, generator=g) * 8.0
    x = xh.cuda()
    p = torch.empty_like(x)
    lse = torch.empty(rows, device=x.device)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        fa.softmax_rows(x, out=p, lse=lse)
    fa.check()
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        fa.softmax_rows(x, out=p, lse=lse)
    t1.record(stream)
    torch.cuda.synchronize()
    fa.check()
    ms = t0.elapsed_time(t1) / K
    nbytes = rows * n * 8 + rows * 4  # read x, write p and lse
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, src = load_hbm_peak()
    print(json.dumps({
        "metric": "online softmax rows GB/s (fp32, 65536 x 2048, read x + write p + lse)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "fa_softmax_rows 65536 x 2048, N(0,1)*8 seed 3",
                   "l2": "inputs larger than L2 (512 MiB), no flush"},
        "roofline": {"kernel": "fa_softmax_warp_rows_kernel<16>", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "peak_source": f"{src} hbm_gbs (copy)",
                     "frac": round(gbs / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": K}), flush=True)


def _time_ms(fn, steps, warmup):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def run_splitkv(args):
    """Split-KV forward against the plain forward on small-batch shapes whose plain grid leaves
    SMs idle or whose longest causal work item runs alone: B=1, Hq=Hkv, d=128; the headline shape
    is H=8, N=2048, causal (8 heads x 8 query-tile pairs = 64 work items for 152 SMs)."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = []
    for H, N, causal in ((8, 2048, True), (2, 8192, True), (4, 4096, True), (8, 2048, False), (16, 1024, True)):
        B, d = 1, 128
        q, k, v, _ = (t.cuda() if t is not None else None for t in make_qkv(B, H, H, N, d, seed=5, value_scale=0.5))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, device=q.device)
        s = fa.splitkv_auto(B, H, H, N, d, causal, sms)
        ws = torch.empty(max(16, fa.lib().fa_fwd_splitkv_workspace_bytes(B, H, H, N, d, s)), dtype=torch.uint8,
                         device=q.device)
        fl = fwd_flops(B, H, N, d, causal)
        t_plain = _time_ms(lambda: fa.forward(q, k, v, causal, out=o, lse=lse), args.steps, args.warmup)
        t_split = _time_ms(lambda: fa.forward_splitkv(q, k, v, causal, 0, out=o, lse=lse, workspace=ws),
                           args.steps, args.warmup)
        fa.check()
        rows.append({"H": H, "N": N, "causal": causal, "splits": s, "plain_ms": round(t_plain, 4),
                     "split_ms": round(t_split, 4), "split_tflops": round(fl / (t_split * 1e-3) / 1e12, 2),
                     "speedup_vs_plain": round(t_plain / t_split, 3)})
    r0 = rows[0]
    print(json.dumps({
        "metric": "split-KV forward TFLOP/s (bf16, B=1 H=8 N=2048 d=128 causal)",
        "value": r0["split_tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r0["split_ms"], "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": "fa_fwd_splitkv (automatic split count) vs fa_fwd, B=1 d=128"},
        "speedup_vs_plain": r0["speedup_vs_plain"], "rows": rows,
        "gpu_launches": sum(1 + (2 if r["splits"] > 1 else 1) for r in rows) * (args.steps + args.warmup)}),
        flush=True)


def run_window(args):
    """Sliding-window attention, fwd + bwd, B=1, Hq=32, Hkv=8, N=32768, d=128, window 4096, against
    full causal attention on the same inputs. FLOPs count visible (query, key) pairs only."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    B, Hq, Hkv, N, d, w = 1, 32, 8, 32768, 128, 4096
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=6, value_scale=0.5, with_do=True))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, N, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=q.device)
    pairs = sum(min(i + 1, w) for i in range(N))
    fl = 4 * d * pairs * B * Hq * (1 + BWD_FACTOR)
    fl_causal = fwd_flops(B, Hq, N, d, True) * (1 + BWD_FACTOR)

    def win():
        fa.forward_window(q, k, v, w, out=o, lse=lse)
        fa.backward_window(q, k, v, o, do, lse, w, dq=dq, dk=dk, dv=dv, workspace=ws)

    def full():
        fa.forward(q, k, v, True, out=o, lse=lse)
        fa.backward(q, k, v, o, do, lse, True, dq=dq, dk=dk, dv=dv, workspace=ws)

    t_win = _time_ms(win, args.steps, args.warmup)
    t_full = _time_ms(full, args.steps, args.warmup)
    fa.check()
    print(json.dumps({
        "metric": "sliding-window attention fwd+bwd TFLOP/s (bf16, N=32768, window 4096, d=128)",
        "value": round(fl / (t_win * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_win, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": "fa_fwd_window + fa_bwd_window, B=1 Hq=32 Hkv=8"},
        "full_causal": {"tflops": round(fl_causal / (t_full * 1e-3) / 1e12, 2), "ms": round(t_full, 4)},
        "time_ratio_full_over_window": round(t_full / t_win, 3), "visible_pair_ratio": round(N * (N + 1) / 2 / pairs, 3),
        "gpu_launches": 8 * args.steps}), flush=True)


def run_naive(args):
    """Standard attention with S and P in HBM (fa_naive_fwd) against the tiled kernel (fa_fwd), the
    comparison of "LLM Architecture Refresh [3]", section 8 (8 heads, d=64, causal, N=512..4096)."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    rows = []
    for N in (512, 1024, 2048, 4096):
        q, k, v, _ = (t.cuda() if t is not None else None for t in make_qkv(1, 8, 8, N, 64, seed=7))
        o = torch.empty_like(q)
        lse = torch.empty(1, 8, N, device=q.device)
        ws = torch.empty(int(fa.lib().fa_naive_workspace_bytes(1, 8, 8, N, 64)), dtype=torch.uint8, device=q.device)
        t_naive = _time_ms(lambda: fa.forward_naive(q, k, v, True, out=o, lse=lse, workspace=ws), args.steps,
                           args.warmup)
        t_tiled = _time_ms(lambda: fa.forward(q, k, v, True, out=o, lse=lse), args.steps, args.warmup)
        fa.check()
        rows.append({"N": N, "naive_ms": round(t_naive, 4), "tiled_ms": round(t_tiled, 4),
                     "speedup": round(t_naive / t_tiled, 2)})
    print(json.dumps({
        "metric": "tiled / naive attention speedup (bf16, B=1 H=8 d=64 causal)", "value": rows[-1]["speedup"],
        "unit": "x at N=4096", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "fa_naive_fwd (S fp32 and P bf16 through HBM, cuBLAS GEMMs) vs fa_fwd"},
        "rows": rows}), flush=True)


def run_long(args):
    """Long context: B=1, Hq=32, Hkv=8, N=131072, d=128, causal, N(0,1)*0.5 from seed 4 (the
    forward streams K and V with no extra device memory). Forward TFLOP/s, the tiles it computed
    and skipped (fa_fwd_stats), the device memory the forward call allocated (none), and the
    backward for reference."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    B, Hq, Hkv, N, d = 1, 32, 8, 131072, 128
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=4, value_scale=0.5, with_do=True))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, N, device=q.device)
    fl = fwd_flops(B, Hq, N, d, True)
    steps, warmup = max(1, min(args.steps, 5)), args.warmup
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.max_memory_allocated()
    t_fwd = _time_ms(lambda: fa.forward(q, k, v, True, out=o, lse=lse), steps, warmup)
    extra = torch.cuda.max_memory_allocated() - before
    counters = torch.zeros(3, dtype=torch.int64, device=q.device)
    fa.forward(q, k, v, True, out=o, lse=lse, counters=counters)
    done, skipped, raised = (int(x) for x in counters.tolist())
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=q.device)
    t_bwd = _time_ms(lambda: fa.backward(q, k, v, o, do, lse, True, dq=dq, dk=dk, dv=dv, workspace=ws), steps, 1)
    fa.check()
    burst, _, _ = load_peaks()
    T = N // 128
    print(json.dumps({
        "metric": "long-context forward TFLOP/s (bf16, B=1 Hq=32 Hkv=8 N=131072 d=128 causal)",
        "value": round(fl / (t_fwd * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": round(t_fwd, 3), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": "fa_fwd at N=131072 (and fa_bwd for reference)"},
        "pct_of_peak_burst": round(100 * fl / (t_fwd * 1e-3) / 1e12 / burst, 2),
        "tiles": {"computed": done, "skipped": skipped, "expected_computed": B * Hq * T * (T + 1) // 2,
                  "skipped_fraction": round(skipped / (done + skipped), 6), "rows_rescaled": raised},
        "forward_extra_device_bytes": int(extra),
        "backward": {"tflops": round(BWD_FACTOR * fl / (t_bwd * 1e-3) / 1e12, 2), "ms": round(t_bwd, 3),
                     "workspace_bytes": ws.numel()},
        "gpu_launches": (steps + warmup + 1) + 3 * (steps + 1)}), flush=True)


def _median_ms_cold(fn, steps, warmup, flush):
    """Median over `steps` single calls of `fn`, each timed alone with CUDA events after a write
    of `flush` (larger than L2), so that every call starts with its inputs in HBM only."""
    import torch

    for _ in range(warmup):
        fn()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(steps):
        flush.zero_()
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times)


TARGET_FWD_FRAC, TARGET_BWD_FRAC = 0.60, 0.45


def run_targets(burst, src, steps=7, warmup=3):
    """The causal bf16 d=128 throughput bar (forward >= 60 %, backward >= 45 % of the dense bf16
    peak at N >= 4096) on the token-count sweep's N >= 4096 shapes (B*N = 16384, Hq = Hkv = 16,
    inputs N(0,1) from seed 3), causal and non-causal, plus the long-context forward (B=1, Hq=32,
    Hkv=8, N=131072, N(0,1)*0.5 from seed 4) with the device memory the forward call added and
    its tile counts. Each time is the median of single calls with L2 flushed before each; the
    backward is the whole of fa_bwd (prepare, compute, finalize)."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    H, d, rows, misses, launches = 16, 128, [], [], 0
    for N in (4096, 8192, 16384):
        B = 16384 // N
        q, k, v, do = (t.cuda() for t in make_qkv(B, H, H, N, d, seed=3, with_do=True))
        o, lse = torch.empty_like(q), torch.empty(B, H, N, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.workspace_bytes(B, H, H, N, d), dtype=torch.uint8, device=q.device)
        for causal in (True, False):
            fl = fwd_flops(B, H, N, d, causal)
            t_f = _median_ms_cold(lambda: fa.forward(q, k, v, causal, out=o, lse=lse), steps, warmup, flush)
            t_b = _median_ms_cold(lambda: fa.backward(q, k, v, o, do, lse, causal, dq=dq, dk=dk, dv=dv, workspace=ws),
                                  steps, warmup, flush)
            fa.check()
            launches += (steps + warmup) * 4
            fwd_tf, bwd_tf = fl / (t_f * 1e-3) / 1e12, BWD_FACTOR * fl / (t_b * 1e-3) / 1e12
            row = {"N": N, "B": B, "causal": causal, "fwd_ms": round(t_f, 4), "fwd_tflops": round(fwd_tf, 1),
                   "fwd_pct_burst": round(100 * fwd_tf / burst, 2), "bwd_ms": round(t_b, 4),
                   "bwd_tflops": round(bwd_tf, 1), "bwd_pct_burst": round(100 * bwd_tf / burst, 2)}
            rows.append(row)
            if causal and fwd_tf < TARGET_FWD_FRAC * burst:
                misses.append(f"forward N={N} causal: {row['fwd_pct_burst']} % < 60 %")
            if causal and bwd_tf < TARGET_BWD_FRAC * burst:
                misses.append(f"backward N={N} causal: {row['bwd_pct_burst']} % < 45 %")
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
    # Long context: the forward alone, its added device memory and its tile counts.
    B, Hq, Hkv, N = 1, 32, 8, 131072
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_qkv(B, Hq, Hkv, N, d, seed=4, value_scale=0.5))
    o, lse = torch.empty_like(q), torch.empty(B, Hq, N, device=q.device)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.max_memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    t_long = _median_ms_cold(lambda: fa.forward(q, k, v, True, out=o, lse=lse), 3, 3, flush)
    extra = torch.cuda.max_memory_allocated() - before
    free_drop = free0 - torch.cuda.mem_get_info()[0]
    counters = torch.zeros(3, dtype=torch.int64, device=q.device)
    fa.forward(q, k, v, True, out=o, lse=lse, counters=counters)
    fa.check()
    launches += 7
    done, skipped = (int(x) for x in counters[:2].tolist())
    T = N // 128
    fl = fwd_flops(B, Hq, N, d, True)
    long_tf = fl / (t_long * 1e-3) / 1e12
    long_row = {"B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "causal": True, "fwd_ms": round(t_long, 3),
                "fwd_tflops": round(long_tf, 1), "fwd_pct_burst": round(100 * long_tf / burst, 2),
                "extra_device_bytes": int(extra), "device_free_bytes_drop": int(free_drop),
                "tiles_computed": done, "tiles_expected": B * Hq * T * (T + 1) // 2,
                "skipped_fraction": round(skipped / (done + skipped), 6),
                "skipped_fraction_expected": round((T - 1) / (2 * T), 6)}
    if long_tf < TARGET_FWD_FRAC * burst:
        misses.append(f"forward N={N} causal (long context): {long_row['fwd_pct_burst']} % < 60 %")
    if extra != 0:
        misses.append(f"long-context forward added {extra} bytes of device memory")
    if done != long_row["tiles_expected"]:
        misses.append("long-context tile count differs from T(T+1)/2 per head")
    del q, k, v, o, lse, flush
    torch.cuda.empty_cache()
    return {"bar": "causal bf16 d=128 at N >= 4096: forward >= 60 %, backward (fa_bwd, all stages) >= 45 % of "
                   f"the {src} bf16 burst peak ({burst} TFLOP/s); non-causal rows for reference",
            "sweep": "B*N = 16384, Hq = Hkv = 16, d = 128, N(0,1) seed 3; median of single calls, L2 flushed",
            "rows": rows, "long_context": long_row, "misses": misses, "launches": launches}


def run_sweep(args):
    """Sequence-length sweep at a fixed token count: B*N = 16384, Hq = Hkv = 16, N = 512..16384,
    d in {64, 128}, causal and non-causal, inputs N(0,1) from seed 3. Per shape: forward,
    backward (all three stages) and forward+backward step, each the median of single calls
    with L2 flushed before each; TFLOP/s from algorithmic FLOPs and HBM GB/s from the
    compulsory bytes (forward: read Q, K, V, write O and LSE; backward: read Q, K, V, O, dO and
    LSE, write dQ, dK, dV)."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    burst, _, peak_src = load_peaks()
    hbm, hbm_src = load_hbm_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    H, rows = 16, []
    for d in (64, 128):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            B = 16384 // N
            q, k, v, do = (t.cuda() for t in make_qkv(B, H, H, N, d, seed=3, with_do=True))
            o = torch.empty_like(q)
            lse = torch.empty(B, H, N, device=q.device)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(fa.workspace_bytes(B, H, H, N, d), dtype=torch.uint8, device=q.device)
            tensor_bytes = B * H * N * d * 2
            fwd_bytes = 4 * tensor_bytes + B * H * N * 4
            bwd_bytes = 8 * tensor_bytes + B * H * N * 4
            for causal in (False, True):
                fl = fwd_flops(B, H, N, d, causal)

                def fwd():
                    fa.forward(q, k, v, causal, out=o, lse=lse)

                def bwd():
                    fa.backward(q, k, v, o, do, lse, causal, dq=dq, dk=dk, dv=dv, workspace=ws)

                def step():
                    fwd()
                    bwd()

                t_f = _median_ms_cold(fwd, args.steps, args.warmup, flush)
                t_b = _median_ms_cold(bwd, args.steps, args.warmup, flush)
                t_s = _median_ms_cold(step, args.steps, args.warmup, flush)
                fa.check()
                rows.append({
                    "d": d, "N": N, "B": B, "causal": causal,
                    "fwd_ms": round(t_f, 4), "fwd_tflops": round(fl / (t_f * 1e-3) / 1e12, 1),
                    "fwd_frac": round(fl / (t_f * 1e-3) / 1e12 / burst, 3),
                    "fwd_hbm_gbs": round(fwd_bytes / (t_f * 1e-3) / 1e9, 1),
                    "bwd_ms": round(t_b, 4), "bwd_tflops": round(BWD_FACTOR * fl / (t_b * 1e-3) / 1e12, 1),
                    "bwd_hbm_gbs": round(bwd_bytes / (t_b * 1e-3) / 1e9, 1),
                    "step_ms": round(t_s, 4), "step_tflops": round((1 + BWD_FACTOR) * fl / (t_s * 1e-3) / 1e12, 1)})
            del q, k, v, do, o, lse, dq, dk, dv, ws
    best = max(r["fwd_tflops"] for r in rows)
    print(json.dumps({
        "metric": "attention TFLOP/s over N at B*N=16384 (bf16, H=16, d=64/128, causal and non-causal)",
        "value": best, "unit": "TFLOP/s (best forward in the sweep)", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "fa_fwd / fa_bwd sweep, B*N=16384, Hq=Hkv=16", "l2": "flushed before each call",
                   "timing": "median of single calls"},
        "peaks": {"bf16_tflops_burst": burst, "bf16_src": peak_src, "hbm_gbs": hbm, "hbm_src": hbm_src},
        "gpu_launches": len(rows) * (args.warmup + args.steps) * 8, "rows": rows}), flush=True)


def run_shape(args):
    """One shape, timed: forward, whole backward (prepare, compute, finalize) and the backward
    compute kernel alone, each the median of single calls with L2 flushed before each, with
    TFLOP/s (algorithmic) and compulsory-byte GB/s. For profiling and for checking one point of the
    sweep; not the headline metric."""
    import torch

    from online_softmax_09_gb300 import fa
    from online_softmax_09_gb300.inputs import make_qkv

    B, Hq, Hkv, N, d, causal = (int(x) for x in args.shape.split(","))
    causal = bool(causal)
    q, k, v, do = (t.cuda() for t in make_qkv(B, Hq, Hkv, N, d, seed=3, with_do=True))
    o, lse = torch.empty_like(q), torch.empty(B, Hq, N, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8, device=q.device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fl = fwd_flops(B, Hq, N, d, causal)
    t_f = _median_ms_cold(lambda: fa.forward(q, k, v, causal, out=o, lse=lse), args.steps, args.warmup, flush)
    t_b = _median_ms_cold(lambda: fa.backward(q, k, v, o, do, lse, causal, dq=dq, dk=dk, dv=dv, workspace=ws),
                          args.steps, args.warmup, flush)
    fa.backward_stages(q, k, v, o, do, lse, dq, dk, dv, ws, causal)
    t_c = _median_ms_cold(lambda: fa.backward_stages(q, k, v, o, do, lse, dq, dk, dv, ws, causal, only=(1,)),
                          args.steps, args.warmup, flush)
    fa.check()
    burst, _, src = load_peaks()
    qb, kvb = B * Hq * N * d * 2, B * Hkv * N * d * 2
    fwd_bytes = 2 * qb + 2 * kvb + B * Hq * N * 4
    bwd_bytes = 3 * qb + 4 * kvb + qb + B * Hq * N * 4
    print(json.dumps({
        "metric": f"attention TFLOP/s on one shape (bf16, B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} causal={causal})",
        "value": round(fl / (t_f * 1e-3) / 1e12, 2), "unit": "TFLOP/s (forward)", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"fa_fwd / fa_bwd, B={B} Hq={Hq} Hkv={Hkv} N={N} d={d} causal={causal}, seed 3",
                   "l2": "flushed before each call", "timing": "median of single calls"},
        "fwd": {"ms": round(t_f, 4), "tflops": round(fl / (t_f * 1e-3) / 1e12, 1),
                "pct_of_peak_burst": round(100 * fl / (t_f * 1e-3) / 1e12 / burst, 2),
                "compulsory_gbs": round(fwd_bytes / (t_f * 1e-3) / 1e9, 1)},
        "bwd": {"ms": round(t_b, 4), "tflops": round(BWD_FACTOR * fl / (t_b * 1e-3) / 1e12, 1),
                "pct_of_peak_burst": round(100 * BWD_FACTOR * fl / (t_b * 1e-3) / 1e12 / burst, 2),
                "compulsory_gbs": round(bwd_bytes / (t_b * 1e-3) / 1e9, 1)},
        "bwd_compute": {"ms": round(t_c, 4), "tflops": round(BWD_FACTOR * fl / (t_c * 1e-3) / 1e12, 1)},
        "peak": {"bf16_tflops_burst": burst, "source": src},
        "gpu_launches": (args.steps + args.warmup) * 5 + 3}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-targets", action="store_true", help="skip the N >= 4096 target shapes")
    ap.add_argument("--batch", type=int, default=0, help="profiling only: override the batch size")
    ap.add_argument("--workload", choices=["attention", "softmax_rows", "splitkv", "window", "naive", "sweep", "long",
                                           "shape"],
                    default="attention",
                    help="attention (the headline metric) or one of the extra workloads")
    ap.add_argument("--shape", default="32,16,16,512,128,1", help="B,Hq,Hkv,N,d,causal for --workload shape")
    ap.add_argument("--small-configs-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.small_configs_child:
        print(json.dumps(_time_small_configs()), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload == "softmax_rows":
        run_softmax_rows(args)
    elif args.workload == "splitkv":
        run_splitkv(args)
    elif args.workload == "window":
        run_window(args)
    elif args.workload == "naive":
        run_naive(args)
    elif args.workload == "sweep":
        run_sweep(args)
    elif args.workload == "long":
        run_long(args)
    elif args.workload == "shape":
        run_shape(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
