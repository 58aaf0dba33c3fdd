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

class StepTimer:
    """Timed repetitions on one stream, the L2 flushed (a 256 MB write) before each;
    ``mark()`` records an event inside the repetition being timed."""

    def __init__(self, stream, flush):
        self.stream = stream
        self.flush = flush
        self.marks = []
        self.recording = False

    def mark(self):
        if self.recording:
            e = torch.cuda.Event(enable_timing=True)
            e.record(self.stream)
            self.marks[-1].append(e)

    def run(self, fn, reps, record=False):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        self.marks = []
        self.recording = record
        for i in range(reps):
            self.flush.zero_()
            ev[i][0].record(self.stream)
            if record:
                self.marks.append([ev[i][0]])
            fn()
            ev[i][1].record(self.stream)
        torch.cuda.synchronize(self.stream.device)
        self.recording = False
        return [a.elapsed_time(b) for a, b in ev]

    def spans(self, a, b):
        """Milliseconds between marks a and b of every recorded repetition."""
        return [mk[a].elapsed_time(mk[b]) for mk in self.marks]


def gemm_bytes(n_in, n_out, c_in, c_out, taps, pairs, elem):
    """Algorithmic bytes of one forward: input rows read once, output rows written once,
    the weights once, and one gather and one scatter index per pair."""
    return elem * (n_in * c_in + n_out * c_out + taps * c_in * c_out) + 8 * pairs


def map_bytes(n_in, n_rows, taps, groups, pairs):
    """Algorithmic bytes of one map build: coordinates read, nbr [rows][taps] written,
    masks and row order per group, the pair lists."""
    return 16 * n_in + 4 * taps * n_rows + 8 * groups * n_rows + 8 * pairs


class Workbench:
    """One workload on the device: its map build and layers, timed per step."""

    def __init__(self, sc, wl, device, timer, build_kw, strided=False):
        self.sc, self.wl, self.device, self.timer = sc, wl, device, timer
        self.strided = strided
        # a strided convolution changes the sites: one layer (the workload's first weights)
        self.L = 1 if strided else wl.layers
        self.coords = wl.coords.to(device)
        self.feats = wl.feats.to(device)
        self.wps = [sc.wpack_create(w.to(device)) for w in wl.weights[:self.L]]
        self.build_kw = build_kw
        self.launches = 0

    def build(self, c, **over):
        kw = dict(self.build_kw, **over)
        if self.strided:
            return self.sc.build_map_strided(c, self.wl.spatial_shape, self.wl.batch_size)
        return self.sc.build_map(c, self.wl.spatial_shape, self.wl.batch_size, **kw)

    def layers(self, m, x):
        y = None
        for li in range(self.L):
            # the ReLU between layers is fused into the GEMM's store
            y = self.sc.subm_forward_packed(m, x, self.wps[li], relu=li + 1 < self.L)
            self.launches += self.sc.last_launch_count()
            if li == 0:
                self.timer.mark()
            x = y
        return y

    def step(self):
        m = self.build(self.coords)
        self.launches += self.sc.last_launch_count()
        self.timer.mark()
        y = self.layers(m, self.feats)
        m.destroy()
        return y

    def info(self):
        """Map statistics (one synchronising call, outside any timing)."""
        m0 = self.build(self.coords)
        st = self.sc.map_status(m0)
        if st != 0:
            raise RuntimeError("map build reported " + self.sc.status_string(st))
        info = self.sc.map_info(m0)
        if info["gemm"] == "tap_major":
            # 128-pair tiles per tap (only each tap's last is ragged)
            tap_off = self.sc.map_export(m0)["tap_off"].cpu().numpy().astype(np.int64)
            V = info["kernel_size"] ** 3
            info["executed_rows"] = int(sum(-(-(tap_off[k + 1] - tap_off[k]) // 128) * 128 for k in range(V)))
        else:
            info["executed_rows"] = info["tile_taps"] * 128
        self.map0 = m0
        m1 = self.build(self.coords)
        info["map_launches"] = self.sc.last_launch_count()
        m1.destroy()
        return info

    def time_steps(self, steps, warmup):
        """The timed steps, then the map/GEMM split from a separate instrumented pass.

        An event recorded between the map build and the first layer serialises
        the two (the layer can no longer launch while the build's last kernel
        runs), so the timed steps carry no such event; the split comes from
        min(steps, 50) more steps that do, and their step time is reported
        beside it."""
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(self.device)
        self.launches = 0
        step_ms = self.timer.run(self.step, steps, record=False)
        launches = self.launches
        istep_ms = self.timer.run(self.step, max(1, min(steps, 50)), record=True)
        split = dict(map_ms=self.timer.spans(0, 1), gemm_ms=self.timer.spans(1, 2), istep_ms=istep_ms)
        self.launches = launches
        return dict(step_ms=step_ms, **split)

    def fused_step(self):
        """The map build and every layer in one fused launch (ReLU between layers)."""
        m = self.build(self.coords)
        self.timer.mark()
        self.sc.subm_forward_layers(m, self.feats, self.wps, relu=[li + 1 < self.L for li in range(self.L)],
                                    outs=self.fused_outs)
        m.destroy()

    def time_fused(self, steps, warmup):
        """Steps with the layers fused into one launch: step ms per step, then (as in
        time_steps) the map's share from an instrumented pass."""
        self.fused_outs = [torch.empty((self.map0.n, self.wl.c_out), dtype=torch.bfloat16, device=self.device)
                           for _ in range(2)] * ((self.L + 1) // 2)
        self.fused_outs = self.fused_outs[:self.L]
        for _ in range(warmup):
            self.fused_step()
        torch.cuda.synchronize(self.device)
        step_ms = self.timer.run(self.fused_step, steps, record=False)
        istep_ms = self.timer.run(self.fused_step, max(1, min(steps, 50)), record=True)
        return dict(step_ms=step_ms, map_ms=self.timer.spans(0, 1), istep_ms=istep_ms)

    def time_map(self, reps, **over):
        """Map build alone (e.g. another mapper), flushed L2, mean ms."""
        for _ in range(3):
            self.build(self.coords, **over).destroy()
        ms = self.timer.run(lambda: self.build(self.coords, **over).destroy(), reps)
        return statistics.mean(ms)

    def time_fp32_layer(self, reps):
        """The first layer in exact fp32 mode (SIMT FFMA) on the built map, mean ms."""
        f32 = self.wl.feats.float().to(self.device)
        w32 = self.wl.weights[0].float().to(self.device)
        out = torch.empty((self.map0.n, self.wl.c_out), dtype=torch.float32, device=self.device)
        for _ in range(3):
            self.sc.subm_forward(self.map0, f32, w32, out=out)
        return statistics.mean(self.timer.run(lambda: self.sc.subm_forward(self.map0, f32, w32, out=out), reps))

    def close(self):
        self.map0.destroy()


def summarise(wb, info, t, peaks, L):
    """µs/layer, component times and roofline fractions of one workload's timed steps."""
    wl = wb.wl
    P, n_rows = info["pairs"], info["n"]
    V, G = info["kernel_size"] ** 3, info["groups"]
    useful = 2.0 * P * wl.c_in * wl.c_out
    map_s = statistics.mean(t["map_ms"]) * 1e-3
    gemm_s = statistics.mean(t["gemm_ms"]) * 1e-3
    us_layer = statistics.mean(t["step_ms"]) * 1e3 / L
    tflops = useful / gemm_s / 1e12
    gbytes = gemm_bytes(wl.n, n_rows, wl.c_in, wl.c_out, V, P, 2)
    mbytes = map_bytes(wl.n, n_rows, V, G, P)
    gather = P * wl.c_in * 2
    return {
        "us_per_layer": round(us_layer, 3), "layers": L,
        "map_us": round(map_s * 1e6, 3), "gemm_us": round(gemm_s * 1e6, 3),
        # the split's own run: an event between map and GEMM serialises them
        "instrumented_us_per_layer": round(statistics.mean(t["istep_ms"]) * 1e3 / L, 3),
        "useful_tflops_gemm": round(tflops, 2),
        "useful_tflops_layer": round(useful * L / (statistics.mean(t["step_ms"]) * 1e-3) / 1e12, 3),
        "gemm_tensor": {"frac": round(tflops / peaks["bf16"], 4), "peak": peaks["bf16"], "unit": "TFLOP/s",
                        "executed_over_useful": round(info["executed_rows"] / P, 3) if P else None},
        # the same GEMM against HBM: what a memory-bound launch of this size would move
        "gemm_hbm": {"algorithmic_bytes": gbytes, "achieved": round(gbytes / gemm_s / 1e9, 2),
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": round(gbytes / gemm_s / 1e9 / peaks["hbm"], 4)},
        # feature rows the gather moves into shared memory (one C_in row per pair, zero rows not counted)
        "gather": {"bytes": gather, "achieved": round(gather / gemm_s / 1e9, 2), "unit": "GB/s"},
        "map_hbm": {"algorithmic_bytes": mbytes, "achieved": round(mbytes / map_s / 1e9, 2),
                    "peak": peaks["hbm"], "unit": "GB/s", "frac": round(mbytes / map_s / 1e9 / peaks["hbm"], 4)},
        "pairs": P, "pairs_per_row": round(P / n_rows, 3) if n_rows else None,
        "mapper": info["mapper"], "pipeline": info["pipeline"], "gemm": info["gemm"],
        "tile_taps": info["tile_taps"], "map_launches": info["map_launches"],
    }


def ffma_peak_tflops(device, sm_mhz):
    """SIMT fp32 peak: SMs x 128 FP32 lanes x 2 FLOP (FFMA) x SM clock."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def workload_config(args, wl, n_rows, pairs, kernel_size, groups, L):
    """The workload as both arms name it (no implementation detail)."""
    return {"workload": f"{args.workload}: N={wl.n}, C_in={wl.c_in}, C_out={wl.c_out}, "
                        f"layers={L}, batch={wl.batch_size}, grid={'x'.join(map(str, wl.spatial_shape))}",
            "conv": args.conv, "output_sites": n_rows, "kernel_size": kernel_size, "groups": groups,
            "pairs": pairs, "pairs_per_row": round(pairs / n_rows, 3) if n_rows else None,
            "l2": "flushed (256 MB write) before every timed step"}


PER_WORKLOAD = ["tiny", "outdoor", "deep", "large", "stage"]


def run_ours(args, rank, world, device):
    import submanifold_sparse_convolution_gb300 as sc
    from submanifold_sparse_convolution_gb300 import build as build_mod
    from submanifold_sparse_convolution_gb300 import synthetic as S

    build_mod.build()
    peaks = load_peaks()
    wl = S.make_workload(args.workload, kernel_size=args.kernel_size)
    strided = args.conv == "strided"
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    timer = StepTimer(stream, flush)
    build_kw = dict(kernel_size=args.kernel_size, groups=args.groups, gemm=args.gemm, pipeline=args.pipeline)
    wb = Workbench(sc, wl, device, timer, build_kw, strided)
    L = wb.L
    info = wb.info()
    pairs = info["pairs"]
    useful_flops_layer = 2.0 * pairs * wl.c_in * wl.c_out

    for _ in range(args.warmup):
        wb.step()
    torch.cuda.synchronize(device)

    # ---- the timed K steps
    sampler = ClockSampler(device.index if device.index is not None else 0) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t0 = time.time()
    t = wb.time_steps(args.steps, 0)
    t1 = time.time()
    gpu_launches = wb.launches
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(t["step_ms"]), device)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    clocks = sampler.summary(t0, t1) if sampler else None

    # ---- end to end from pinned host buffers
    coords_h = wl.coords.pin_memory()
    feats_h = wl.feats.pin_memory()
    n_rows = info["n"]   # output sites (the input sites but for a strided convolution)
    out_h = torch.empty((n_rows, wl.c_out), dtype=torch.bfloat16).pin_memory()
    coords_d2 = torch.empty_like(wb.coords)
    feats_d2 = torch.empty_like(wb.feats)
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
        m = wb.build(coords_d2)
        stream.wait_event(feats_ready)
        y = wb.layers(m, feats_d2)
        out_h.copy_(y, non_blocking=True)
        m.destroy()

    e2e_ms = timer.run(e2e_step, max(args.steps, 5))
    h2d = wb.coords.numel() * 4 + wb.feats.numel() * 2
    d2h = n_rows * wl.c_out * 2

    plain = info["kernel_size"] == 3 and info["groups"] == 1 and not strided
    # the benchmark spec's sorted-key mapper, timed beside the shipped one
    sorted_map_us = None
    if plain and info["mapper"] == "hash" and rank == 0:
        sorted_map_us = round(wb.time_map(max(10, min(args.steps, 50)), mapper="sorted") * 1e3, 3)
    wb.close()
    if rank != 0:
        return None

    summ = summarise(wb, info, t, peaks, L)
    us_per_layer = job_us_per_layer(total_ms, args.steps, L, world)
    layers_total = args.steps * L * world
    useful_tflops = useful_flops_layer * layers_total / (total_ms * 1e-3) / 1e12
    gemm_tflops = summ["useful_tflops_gemm"]
    tap_major = info["gemm"] == "tap_major"
    G = info["groups"]
    kernel_name = (f"k_tc_gemm<{256 if wl.c_out > 256 else (128 if wl.c_out > 64 else 64)}, "
                   f"{'tap-major' if tap_major else 'tile-union'}>")
    traffic = ncu_traffic("k_tc_gemm", args.workload if plain else
                          f"{args.workload}-strided" if strided else f"{args.workload}-k{info['kernel_size']}-g{G}")
    pages_us = PAGES_US.get(args.workload) if plain else None
    config = workload_config(args, wl, n_rows, pairs, info["kernel_size"], G, L)
    out = {
        "metric": METRIC, "value": round(us_per_layer, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": round(us_per_layer / pages_us, 4) if pages_us else None,
        "vs_baseline_note": ("value / the pages' µs on an AMD gfx950 for the same N and C "
                             "(context: other hardware, real scans)") if pages_us else None,
        "dtype": "bf16", "data": DATA, "config": config,
        "impl_config": {"mapper": info["mapper"], "pipeline": info["pipeline"], "gemm": info["gemm"],
                        "tile_taps": info["tile_taps"],
                        "weights": "packed once per layer (outside the step)",
                        "relu": "between layers, fused into the GEMM store" if L > 1 else None},
        "useful_tflops": round(useful_tflops, 3),
        "components_us": {"map": summ["map_us"], "gemm_layer0": summ["gemm_us"],
                          "map_launches": info["map_launches"], "map_sorted_mapper": sorted_map_us,
                          "instrumented_us_per_layer": summ["instrumented_us_per_layer"],
                          "note": ("map and GEMM times from a separate run of min(steps, 50) steps with an "
                                   "event between them, which serialises the two; the timed steps that give "
                                   "value carry no such event, so the GEMM may start during the map's last "
                                   "kernel")},
        "roofline": {"bound": "tensor", "kernel": kernel_name, "achieved": gemm_tflops,
                     "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peaks["bf16"], 4), "traffic": traffic,
                     "frac_of_nominal": round(gemm_tflops / NOMINAL_BF16_TFLOPS, 4),
                     "peak_source": f"{peaks['source']} bf16 dense (burst, kernel timed alone)",
                     "launches_per_layer": G,
                     "executed_over_useful": summ["gemm_tensor"]["executed_over_useful"],
                     "gather": summ["gather"], "hbm": summ["gemm_hbm"]},
        "roofline_map": {"bound": "hbm", "achieved": summ["map_hbm"]["achieved"],
                         "peak": peaks["hbm"], "unit": "GB/s", "frac": summ["map_hbm"]["frac"],
                         "frac_of_nominal": round(summ["map_hbm"]["achieved"] / NOMINAL_HBM_GBS, 4),
                         "algorithmic_bytes": summ["map_hbm"]["algorithmic_bytes"]},
        "e2e": {"value": round(statistics.mean(e2e_ms) * 1e3 / L, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if plain and args.per_workload and world == 1:
        sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
        out["per_workload"] = per_workload(sc, S, args, device, timer, peaks, sm_mhz, {args.workload: summ})
    return out


def per_workload(sc, S, args, device, timer, peaks, sm_mhz, done):
    """Every workload of the metric, timed the same way in this run (fewer steps each)."""
    res = {}
    steps = max(5, min(args.steps, 30))
    for name in PER_WORKLOAD:
        if name in done:
            res[name] = done[name]
            continue
        wl = S.make_workload(name)
        wb = Workbench(sc, wl, device, timer, dict(pipeline=args.pipeline, gemm=args.gemm))
        info = wb.info()
        t = wb.time_steps(steps, 3)
        r = summarise(wb, info, t, peaks, wb.L)
        r["steps"] = steps
        if wb.L > 1:
            # the same layers as one launch over the shared map
            tf = wb.time_fused(steps, 3)
            # the layers' share of each (instrumented) step: step minus map
            fused_layers_ms = statistics.mean(a - b for a, b in zip(tf["istep_ms"], tf["map_ms"]))
            r["fused_layers"] = {"us_per_layer": round(statistics.mean(tf["step_ms"]) * 1e3 / wb.L, 3),
                                 "layers_us_per_layer": round(fused_layers_ms * 1e3 / wb.L, 3),
                                 "separate_layers_us_per_layer": round(
                                     (statistics.mean(t["istep_ms"]) - statistics.mean(t["map_ms"])) * 1e3 / wb.L, 3),
                                 "launches_per_step": 1}
        if name == "stage":
            # the same first layer in exact fp32 (SIMT FFMA, plain ALUs)
            ms = wb.time_fp32_layer(steps)
            flops = 2.0 * info["pairs"] * wl.c_in * wl.c_out
            peak = ffma_peak_tflops(device, sm_mhz)
            b32 = gemm_bytes(wl.n, info["n"], wl.c_in, wl.c_out, 27, info["pairs"], 4)
            r["fp32_layer"] = {"bound": "alu", "us": round(ms * 1e3, 3),
                               "achieved": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                               "peak": round(peak, 2), "frac": round(flops / (ms * 1e-3) / 1e12 / peak, 4),
                               "peak_source": f"SMs x 128 FP32 lanes x 2 x {sm_mhz:.0f} MHz (median SM clock "
                                              "of the timed run)",
                               "hbm_achieved": round(b32 / (ms * 1e-3) / 1e9, 2),
                               "hbm_frac": round(b32 / (ms * 1e-3) / 1e9 / peaks["hbm"], 4)}
        wb.close()
        res[name] = r
        del wb
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in outp.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model", "hardware")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def prepare_oracle(workload, kernel_size=3, groups=0, conv="submanifold"):
    import oracle
    from submanifold_sparse_convolution_gb300 import synthetic as S

    oracle.build()
    wl = S.make_workload(workload, kernel_size=kernel_size)
    G = groups if groups > 0 else (1 if kernel_size == 3 else kernel_size)
    return dict(wl=wl, c=wl.coords.numpy(), f=wl.feats.double().numpy(),
                w=wl.weights[0].double().numpy(), K=kernel_size, G=G, conv=conv)


def oracle_map(prep):
    """The oracle's map build (single-threaded): kernel map, masks, order, pair lists."""
    import oracle

    wl, c = prep["wl"], prep["c"]
    if prep["conv"] == "strided":
        _, nbr = oracle.strided_map(c, wl.spatial_shape, wl.batch_size)
    else:
        nbr = oracle.kernel_map(c, wl.spatial_shape, wl.batch_size, prep["K"])
    _, _, p = oracle.group_orders(nbr, prep["G"], True)
    lists = oracle.pair_lists(nbr, p)
    return nbr, int(lists[0][-1])


def time_oracle(prep, budget_s, threads=0, nbr=None):
    """Oracle µs/layer: the full map build + the fp64 conv on ``threads`` threads (0: all),
    on a row sample scaled to N.  Returns (µs/layer, threads used, sample, nbr, map s)."""
    import oracle

    wl, f, w = prep["wl"], prep["f"], prep["w"]
    t = time.perf_counter()
    if nbr is None:
        nbr, _ = oracle_map(prep)
        t_map = time.perf_counter() - t
    else:
        t_map = prep["t_map"]
    n_rows = nbr.shape[0]                   # output sites (strided: fewer than the inputs)
    layers = 1 if prep["conv"] == "strided" else wl.layers
    # calibrate the conv sample on 256 rows, then size it to the budget
    rows = np.arange(min(256, n_rows), dtype=np.int32)
    t = time.perf_counter()
    oracle.conv_f64(nbr, f, w, rows=rows, threads=threads)
    t_cal = max(time.perf_counter() - t, 1e-6) / max(1, rows.shape[0])
    k = int(min(n_rows, max(256, budget_s / t_cal)))
    rows = np.linspace(0, n_rows - 1, k).astype(np.int32)
    t = time.perf_counter()
    oracle.conv_f64(nbr, f, w, rows=rows, threads=threads)
    t_conv = (time.perf_counter() - t) / max(1, k) * n_rows
    us_per_layer = (t_map + layers * t_conv) / layers * 1e6
    used = threads if threads > 0 else oracle.max_threads()
    what = "strided map (kernel 3, stride 2)" if prep["conv"] == "strided" else f"full kernel map (K={prep['K']})"
    sample = (f"{what}, masks, order and pair lists ({prep['G']} group(s)) of N={wl.n} on one thread; "
              f"fp64 conv on {k} of {n_rows} output rows (evenly spaced) on {used} thread(s), scaled to all; "
              f"{layers} layer(s)")
    return us_per_layer, used, sample, nbr, t_map


def cpu_baseline(workload, budget_s, kernel_size=3, groups=0, conv="submanifold"):
    """The oracle on all host threads and on one, the map build timed once for both."""
    prep = prepare_oracle(workload, kernel_size, groups, conv)
    us, cores, sample, nbr, t_map = time_oracle(prep, budget_s)
    prep["t_map"] = t_map
    us1, _, sample1, _, _ = time_oracle(prep, budget_s / 2, threads=1, nbr=nbr)
    return {"value": round(us, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "value_1thread": round(us1, 3), "sample_1thread": sample1,
            "map_build_s": round(t_map, 4), "cpu_model": cpu_model(), "host_threads": os.cpu_count()}


def run_reference(args):
    prep = prepare_oracle(args.workload, args.kernel_size, args.groups, args.conv)
    wl = prep["wl"]
    # the whole run stays within about two minutes of oracle work
    budget = max(0.05, min(args.ref_budget, 120.0 / (args.steps + args.warmup)))
    per_step = []
    cores, sample, pairs, n_rows = None, None, 0, wl.n
    for i in range(args.warmup + args.steps):
        us, cores, sample, nbr, _ = time_oracle(prep, budget)
        n_rows = nbr.shape[0]
        if i >= args.warmup:
            per_step.append(us)
    _, pairs = oracle_map(prep)
    value = statistics.mean(per_step)
    layers = 1 if args.conv == "strided" else wl.layers
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value * layers / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": workload_config(args, wl, n_rows, pairs, prep["K"], prep["G"], layers),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
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
    ap.add_argument("--per-workload", type=int, default=1,
                    help="also time every other workload in the same run (per_workload key; 0 disables)")
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
