"""Benchmark: µs per layer and useful bf16 TFLOP/s of the submanifold 3x3x3
convolution (kernel map + GEMM) on one GB300, with roofline fractions.

One step = build the kernel map of the workload's coordinates (key packing,
mapper, masks, mask sort, compaction) + every layer of the workload through
the packed-weight forward, then free the map.  Inputs are resident in HBM;
the L2 is flushed (256 MB write) before every timed step and every timed
kernel.  ``e2e`` repeats the step through the same public calls from pinned
host buffers, with the copies inside the timed region (the feature upload on a
second stream, overlapping the map build, which needs only the coordinates).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload outdoor]
    python bench.py --impl reference ...      # the CPU oracle on the same workload

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are independent
replicas: every rank runs the whole workload on its own GPU (weak scaling),
with no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "µs/layer and useful bf16 TFLOP/s per subm conv (map+GEMM), 1 GB300, % roofline"
UNIT = "us/layer"
# FlyDSL PR #942, "Performance": 47 µs end to end (mapping included) on an AMD
# gfx950 for N=32,371, C=128 -- another machine's number, quoted as context.
PAGES_US = {"outdoor": 47.0, "large": 178.0}
L2_FLUSH_BYTES = 256 << 20
# GB300 nominal figures, reported beside the measured peaks: HBM3e bandwidth and
# dense bf16 tensor throughput
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
DATA = ("synthetic, seeded: LiDAR-like scan-ring ground plane (2 jittered layers) plus "
        "box/cylinder surfaces, rows shuffled; features N(0,1), weights N(0,1/sqrt(27*C_in)), bf16")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def file_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_key, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key][workload]
    except Exception:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or file_hash(src) != rec["source_hash"]:
        return None
    return rec["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples (100 ms) for the timed window."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        if not self.samples:
            return None
        win = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        where = "timed window"
        if not win:
            win = [p for (_, p) in self.samples]
            where = "whole run (timed window shorter than one 100 ms sample)"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win), "window": where}


# ---------------------------------------------------------------------------
# ranks: independent replicas (weak scaling), one timing for the whole job
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's ``value`` (the job takes as long as its slowest rank)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer(total_ms: float, steps: int, layers: int, world: int) -> float:
    """µs per layer of the whole job: every rank ran ``steps`` steps of ``layers`` layers in ``total_ms``."""
    return total_ms * 1e3 / (steps * layers * world)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, device):
    import submanifold_sparse_convolution_gb300 as sc
    from submanifold_sparse_convolution_gb300 import build as build_mod
    from submanifold_sparse_convolution_gb300 import synthetic as S

    build_mod.build()
    peaks = load_peaks()
    wl = S.make_workload(args.workload, kernel_size=args.kernel_size)
    strided = args.conv == "strided"
    # a strided convolution changes the sites: one layer (the workload's first weights)
    L = 1 if strided else wl.layers
    coords = wl.coords.to(device)
    feats = wl.feats.to(device)
    wps = [sc.wpack_create(w.to(device)) for w in wl.weights]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    launches = [0]

    # events inside the timed steps: per step [start, map done, layer 0 done]
    marks = []
    recording = [False]

    def mark():
        if recording[0]:
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            marks[-1].append(e)

    def layers(m, x):
        y = None
        for li in range(L):
            # the ReLU between layers is fused into the GEMM's store
            y = sc.subm_forward_packed(m, x, wps[li], relu=li + 1 < L)
            launches[0] += sc.last_launch_count()
            if li == 0:
                mark()
            x = y
        return y

    def build(c):
        if strided:
            return sc.build_map_strided(c, wl.spatial_shape, wl.batch_size)
        return sc.build_map(c, wl.spatial_shape, wl.batch_size, kernel_size=args.kernel_size,
                            groups=args.groups, gemm=args.gemm, pipeline=args.pipeline)

    def step():
        m = build(coords)
        launches[0] += sc.last_launch_count()
        mark()
        y = layers(m, feats)
        m.destroy()
        return y

    # map statistics (one synchronising call, outside any timing)
    m0 = build(coords)
    if sc.map_status(m0) != 0:
        raise RuntimeError("map build reported " + sc.status_string(sc.map_status(m0)))
    info = sc.map_info(m0)
    pairs = info["pairs"]
    useful_flops_layer = 2.0 * pairs * wl.c_in * wl.c_out
    # MMA rows the GEMM executes: mask-union tiles, or 128-pair tiles per tap (only each tap's last is ragged)
    tap_major = info["gemm"] == "tap_major"
    if tap_major:
        tap_off = sc.map_export(m0)["tap_off"].cpu().numpy().astype(np.int64)
        executed_rows = int(sum(-(-(tap_off[k + 1] - tap_off[k]) // 128) * 128 for k in range(27)))
    else:
        executed_rows = info["tile_taps"] * 128

    def timed(fn, reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for i in range(reps):
            flush.zero_()
            ev[i][0].record(stream)
            if recording[0]:
                marks.append([ev[i][0]])
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # ---- the timed K steps
    sampler = ClockSampler(device.index if device.index is not None else 0) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    launches[0] = 0
    t0 = time.time()
    recording[0] = True
    step_ms = timed(step, args.steps)
    recording[0] = False
    t1 = time.time()
    gpu_launches = launches[0]
    # map and first-layer GEMM durations of every timed step, from the same events
    map_ms = [mk[0].elapsed_time(mk[1]) for mk in marks]
    gemm_ms = [mk[1].elapsed_time(mk[2]) for mk in marks]
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(step_ms), device)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    clocks = sampler.summary(t0, t1) if sampler else None

    map_launches = None
    m1 = build(coords)
    map_launches = sc.last_launch_count()
    m1.destroy()

    # ---- end to end from pinned host buffers
    coords_h = wl.coords.pin_memory()
    feats_h = wl.feats.pin_memory()
    n_rows = info["n"]   # output sites (the input sites but for a strided convolution)
    out_h = torch.empty((n_rows, wl.c_out), dtype=torch.bfloat16).pin_memory()
    coords_d2 = torch.empty_like(coords)
    feats_d2 = torch.empty_like(feats)
    # the map needs only the coordinates: the features travel on a side stream
    # while it builds, and the first layer waits for them
    side = torch.cuda.Stream(device)
    feats_ready = torch.cuda.Event()

    def e2e_step():
        coords_d2.copy_(coords_h, non_blocking=True)
        side.wait_stream(stream)        # after the step's start mark and the previous step's layers
        with torch.cuda.stream(side):
            feats_d2.copy_(feats_h, non_blocking=True)
            feats_ready.record(side)
        m = build(coords_d2)
        stream.wait_event(feats_ready)
        y = layers(m, feats_d2)
        out_h.copy_(y, non_blocking=True)
        m.destroy()

    e2e_ms = timed(e2e_step, max(args.steps, 5))
    h2d = coords.numel() * 4 + feats.numel() * 2
    d2h = n_rows * wl.c_out * 2

    m0.destroy()
    if rank != 0:
        return None

    layers_total = args.steps * L * world
    us_per_layer = job_us_per_layer(total_ms, args.steps, L, world)
    useful_tflops = useful_flops_layer * layers_total / (total_ms * 1e-3) / 1e12
    gemm_avg_s = statistics.mean(gemm_ms) * 1e-3
    gemm_tflops = useful_flops_layer / gemm_avg_s / 1e12
    n, P = wl.n, pairs
    V, G = info["kernel_size"] ** 3, info["groups"]
    # coordinates read, nbr [rows][V] written, masks and row order per group, pair lists
    map_bytes = 16 * n + 4 * V * n_rows + 8 * G * n_rows + 8 * P
    map_avg_s = statistics.mean(map_ms) * 1e-3
    kernel_name = (f"k_tc_gemm<{256 if wl.c_out > 256 else (128 if wl.c_out > 64 else 64)}, "
                   f"{'tap-major' if tap_major else 'tile-union'}>")
    plain = info["kernel_size"] == 3 and G == 1 and not strided
    traffic = ncu_traffic("k_tc_gemm", args.workload if plain else
                          f"{args.workload}-strided" if strided else f"{args.workload}-k{info['kernel_size']}-g{G}")
    pages_us = PAGES_US.get(args.workload) if plain else None
    out = {
        "metric": METRIC, "value": round(us_per_layer, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": round(us_per_layer / pages_us, 4) if pages_us else None,
        "vs_baseline_note": ("value / the pages' µs on an AMD gfx950 for the same N and C "
                             "(context: other hardware, real scans)") if pages_us else None,
        "dtype": "bf16", "data": DATA,
        "config": {"workload": f"{args.workload}: N={wl.n}, C_in={wl.c_in}, C_out={wl.c_out}, "
                               f"layers={L}, batch={wl.batch_size}, grid={'x'.join(map(str, wl.spatial_shape))}",
                   "conv": args.conv, "output_sites": n_rows,
                   "kernel_size": info["kernel_size"], "groups": G,
                   "pairs": P, "pairs_per_row": round(P / n_rows, 3) if n_rows else None, "mapper": info["mapper"], "pipeline": info["pipeline"], "gemm": info["gemm"],
                   "tile_taps": info["tile_taps"], "l2": "flushed (256 MB write) before every timed step",
                   "weights": "packed once per layer (outside the step)",
                   "relu": "between layers, fused into the GEMM store" if L > 1 else None},
        "useful_tflops": round(useful_tflops, 3),
        "components_us": {"map": round(map_avg_s * 1e6, 3), "gemm_layer0": round(gemm_avg_s * 1e6, 3),
                          "map_launches": map_launches},
        "roofline": {"bound": "tensor", "kernel": kernel_name, "achieved": round(gemm_tflops, 2),
                     "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peaks["bf16"], 4), "traffic": traffic,
                     "frac_of_nominal": round(gemm_tflops / NOMINAL_BF16_TFLOPS, 4),
                     "peak_source": f"{peaks['source']} bf16 dense (burst, kernel timed alone)",
                     "launches_per_layer": G,
                     "executed_over_useful": round(executed_rows / P, 3)},
        "roofline_map": {"bound": "hbm", "achieved": round(map_bytes / map_avg_s / 1e9, 2),
                         "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": round(map_bytes / map_avg_s / 1e9 / peaks["hbm"], 4),
                         "frac_of_nominal": round(map_bytes / map_avg_s / 1e9 / NOMINAL_HBM_GBS, 4),
                         "algorithmic_bytes": map_bytes},
        "e2e": {"value": round(statistics.mean(e2e_ms) * 1e3 / L, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    return out


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def prepare_oracle(workload, kernel_size=3, groups=0, conv="submanifold"):
    import oracle
    from submanifold_sparse_convolution_gb300 import synthetic as S

    oracle.build()
    wl = S.make_workload(workload, kernel_size=kernel_size)
    G = groups if groups > 0 else (1 if kernel_size == 3 else kernel_size)
    return dict(wl=wl, c=wl.coords.numpy(), f=wl.feats.double().numpy(),
                w=wl.weights[0].double().numpy(), K=kernel_size, G=G, conv=conv)


def time_oracle(prep, budget_s):
    """Oracle µs/layer: full map build + fp64 conv on a row sample scaled to N."""
    import oracle

    wl, c, f, w = prep["wl"], prep["c"], prep["f"], prep["w"]
    t = time.perf_counter()
    if prep["conv"] == "strided":
        _, nbr = oracle.strided_map(c, wl.spatial_shape, wl.batch_size)
    else:
        nbr = oracle.kernel_map(c, wl.spatial_shape, wl.batch_size, prep["K"])
    _, _, p = oracle.group_orders(nbr, prep["G"], True)
    oracle.pair_lists(nbr, p)
    n_rows = nbr.shape[0]                   # output sites (strided: fewer than the inputs)
    layers = 1 if prep["conv"] == "strided" else wl.layers
    t_map = time.perf_counter() - t
    # calibrate the conv sample on 256 rows, then size it to the budget
    rows = np.arange(min(256, n_rows), dtype=np.int32)
    t = time.perf_counter()
    oracle.conv_f64(nbr, f, w, rows=rows)
    t_cal = max(time.perf_counter() - t, 1e-6) / max(1, rows.shape[0])
    k = int(min(n_rows, max(256, budget_s / t_cal)))
    rows = np.linspace(0, n_rows - 1, k).astype(np.int32)
    t = time.perf_counter()
    oracle.conv_f64(nbr, f, w, rows=rows)
    t_conv = (time.perf_counter() - t) / max(1, k) * n_rows
    us_per_layer = (t_map + layers * t_conv) / layers * 1e6
    what = "strided map (kernel 3, stride 2)" if prep["conv"] == "strided" else f"full kernel map (K={prep['K']})"
    sample = (f"{what}, masks, order and pair lists ({prep['G']} group(s)) of N={wl.n}; fp64 conv on {k} of "
              f"{n_rows} output rows (evenly spaced) scaled to all; {layers} layer(s)")
    return us_per_layer, oracle.max_threads(), sample


def cpu_baseline(workload, budget_s, kernel_size=3, groups=0, conv="submanifold"):
    us, cores, sample = time_oracle(prepare_oracle(workload, kernel_size, groups, conv), budget_s)
    return {"value": round(us, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}


def run_reference(args):
    prep = prepare_oracle(args.workload, args.kernel_size, args.groups, args.conv)
    wl = prep["wl"]
    # the whole run stays within about two minutes of oracle work
    budget = max(0.05, min(args.ref_budget, 120.0 / (args.steps + args.warmup)))
    per_step = []
    cores, sample = None, None
    for i in range(args.warmup + args.steps):
        us, cores, sample = time_oracle(prep, budget)
        if i >= args.warmup:
            per_step.append(us)
    value = statistics.mean(per_step)
    layers = 1 if args.conv == "strided" else wl.layers
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value * layers / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": {"workload": f"{args.workload}: N={wl.n}, C_in={wl.c_in}, C_out={wl.c_out}, "
                               f"layers={layers}, batch={wl.batch_size}, "
                               f"grid={'x'.join(map(str, wl.spatial_shape))}",
                   "kernel_size": prep["K"], "groups": prep["G"], "conv": prep["conv"]},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="outdoor",
                    choices=["tiny", "outdoor", "deep", "large", "stage"])
    ap.add_argument("--pipeline", default="auto", choices=["auto", "wide", "fused", "multi"],
                    help="kernel-map build pipeline (auto: wide when the keys fit it)")
    ap.add_argument("--gemm", default="auto", choices=["auto", "tile_union", "tap_major"],
                    help="work decomposition of the bf16 GEMM")
    ap.add_argument("--kernel-size", type=int, default=3, choices=[3, 5],
                    help="K of the K x K x K kernel (the workloads are quoted for 3)")
    ap.add_argument("--groups", type=int, default=0,
                    help="offset groups (0: 1 for K = 3, K for K = 5; or K)")
    ap.add_argument("--conv", default="submanifold", choices=["submanifold", "strided"],
                    help="submanifold convolution (the workloads' layers), or one strided layer "
                         "(kernel 3, stride 2, padding 1) on the workload's sites")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle conv work for the cpu_baseline leg (0 disables)")
    ap.add_argument("--ref-budget", type=float, default=2.0,
                    help="seconds of oracle conv work per reference step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    out = run_ours(args, rank, world, device)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0 and out is not None:
        if world == 1 and args.cpu_budget > 0:
            out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_budget, args.kernel_size, args.groups,
                                               args.conv)
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
