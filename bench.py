#!/usr/bin/env python
"""Benchmark: the dense decode-layer MLP built from the affine-Q4 GEMV on GB300.

One step = for every NB in the sweep (default 1, 2, 4, 8, 16), one decode-layer
MLP on each of L weight sets (default 8, so the 453 MB of weights are larger
than three L2 caches and every layer streams from HBM):
    q4a_gemv_rmsnorm_gate_up_silu  4096 -> 2 x 6144 gate|up with the RMSNorm prologue
                                   and h = fp16(silu(gate) * up) in the epilogue
    q4a_gemv                       12288 -> 4096 down projection (its own synthetic input
                                   x = fp16(silu(a) * b), built once per NB by
                                   q4a_silu_mul_xsum)
The headline value is achieved HBM GB/s over the step: algorithmic bytes of every
launch (packed codes at 0.5 B per weight, bf16 scale + bias per 64 weights,
activations, outputs) divided by the device time of the step.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
N > 1 runs under torch.distributed.run: every rank runs the same workload on its
own GPU (independent replicas: the workload partitions into independent batches
and needs no exchange), value = bytes of all ranks / max step time over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import q4a_workloads as wl  # noqa: E402

HIDDEN, INTER2, INTER = 4096, 12288, 6144         # gate|up = 2 x 6144
DOWN_IN, DOWN_OUT = 12288, 4096
BYTES_PER_WEIGHT = 0.5 + 4.0 / 64.0                # codes + bf16 scale and bias per 64
WORKLOAD = ("dense decode-layer MLP: 4096->2x6144 gate|up (RMSNorm prologue, silu(gate)*up epilogue) + "
            "12288->4096 down; affine-Q4 group 64")
METRIC = "achieved HBM GB/s (and % of roofline) per q4a_gemv call vs NB; us/decode-layer"


def gemv_bytes(out_dim, in_dim, nb, x_bytes_per_el, bits=4):
    """Algorithmic bytes of one product: codes (bits / 8 per weight) plus a bf16 scale and
    bias per 64 weights, the activations and the fp32 outputs."""
    per_weight = bits / 8.0 + 4.0 / 64.0
    return out_dim * in_dim * per_weight + nb * in_dim * x_bytes_per_el + nb * out_dim * 4


def layer_bytes(nb):
    """(fused gate|up, down) algorithmic bytes of one decode layer at NB rows: the gate|up
    reads fp32 x_raw and the bf16 norm weight and writes h in fp16 (no fp32 gate|up output)."""
    gu = INTER2 * HIDDEN * BYTES_PER_WEIGHT + nb * HIDDEN * 4 + HIDDEN * 2 + nb * INTER * 2
    dn = gemv_bytes(DOWN_OUT, DOWN_IN, nb, 2)
    return gu, dn


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's value (every rank gets it); x itself outside a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the bytes every rank moved in one step over the slowest rank's
    step time (weak scaling: each rank runs the same workload on its own GPU)."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None
        self.window = None   # (start, end) wall-clock seconds of the timed region

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        try:
            with open(self.tmp.name) as f:
                rows = [r.split(", ") for r in f.read().strip().splitlines() if r.strip()]
            os.unlink(self.tmp.name)
        except Exception:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        import datetime

        def when(r):
            try:
                return datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except Exception:
                return None

        rows = [r for r in rows if len(r) >= 10]
        if self.window:
            inside = [r for r in rows if when(r) is not None and self.window[0] - 0.05 <= when(r) <= self.window[1] + 0.05]
            rows = inside or rows
        sm = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---- CPU baseline (the oracle as it stands) --------------------------------------------

def oracle_sample(seconds_target: float = 12.0, nbs=(1, 2, 4, 8, 16)):
    """Time the CPU oracle on a bounded sample of the same workload: the decode-layer MLP at
    every NB of the step on a row sample of both projections (128 gate|up rows -- 64 gate, 64
    up -- and 64 down rows), repeated until ~seconds_target. Returns (GB/s, description,
    cores)."""
    import oracle

    rows_gu, rows_dn = 128, 64
    qm_gu = wl.quant_matrix(wl.DENSE_GATE_UP, rows_gu, HIDDEN)
    qm_dn = wl.quant_matrix(wl.DENSE_DOWN, rows_dn, DOWN_IN)
    p_gu, p_dn = oracle.pack(qm_gu.codes), oracle.pack(qm_dn.codes)
    nw = wl.norm_weight(wl.DENSE_GATE_UP, wl.T_NORM_W, HIDDEN)
    total_bytes, t0, reps = 0.0, time.perf_counter(), 0
    while True:
        for nb in nbs:
            a = wl.normal_f32(wl.DENSE_GATE_UP, wl.T_A, (nb, HIDDEN))
            xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6)
            y, _ = oracle.gemv(p_gu, qm_gu.scale, qm_gu.bias, xn)
            h = oracle.silu_mul_f16(y.astype(np.float32))    # 64 gate rows, then 64 up rows
            xd = wl.normal_f16(wl.DENSE_DOWN, wl.T_X, (nb, DOWN_IN))
            oracle.gemv(p_dn, qm_dn.scale, qm_dn.bias, xd)
            # the same accounting as layer_bytes, for the sampled rows
            total_bytes += (rows_gu * HIDDEN * BYTES_PER_WEIGHT + nb * HIDDEN * 4 + HIDDEN * 2 + h.size * 2
                            + gemv_bytes(rows_dn, DOWN_IN, nb, 2))
        reps += 1
        if time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    desc = (f"oracle decode-layer MLP on a row sample ({rows_gu} of {INTER2} gate|up rows, {rows_dn} of "
            f"{DOWN_OUT} down rows) at NB={','.join(str(v) for v in nbs)}, {reps} repetitions, {dt:.1f} s, "
            f"single-threaded fp64")
    return total_bytes / dt / 1e9, desc, 1


def host_info():
    """The host's logical core count and CPU model (the oracle uses one of the cores). Arm hosts
    list no model name in /proc/cpuinfo, only the implementer and part numbers; those are
    reported, with the core's name for the parts known here."""
    model, impl, part = None, None, None
    arm_parts = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                 ("0x41", "0xd0c"): "Arm Neoverse-N1", ("0x41", "0xd49"): "Arm Neoverse-N2"}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" not in line:
                    continue
                key, val = (t.strip() for t in line.split(":", 1))
                key = key.lower()
                if key in ("model name", "cpu model", "hardware") and not model:
                    model = val
                elif key == "cpu implementer" and impl is None:
                    impl = val.lower()
                elif key == "cpu part" and part is None:
                    part = val.lower()
    except Exception:
        pass
    if not model and impl and part:
        name = arm_parts.get((impl, part))
        model = f"{name + ' ' if name else ''}(CPU implementer {impl}, part {part})"
    if not model:
        import platform

        model = platform.processor() or platform.machine()
    return {"host_cores": os.cpu_count(), "cpu_model": model}


def run_reference(args, rank, world):
    if rank != 0:
        return
    steps_bytes, times = [], []
    import oracle  # noqa: F401
    for i in range(args.warmup + args.steps):
        # --ref-seconds in all (a minute by default), whatever --steps and --warmup are (one
        # repetition over every NB takes ~40-60 ms)
        per = max(0.05, args.ref_seconds / max(1, args.warmup + args.steps))
        gbs, desc, cores = oracle_sample(seconds_target=per, nbs=tuple(int(v) for v in args.nbs.split(",")))
        if i >= args.warmup:
            times.append(gbs)
    value = statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "nbs": [int(v) for v in args.nbs.split(",")]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc,
                         **host_info()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the GPU arm ------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch

    import affine_q4_dequant_gb300 as q4a

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    nbs = [int(v) for v in args.nbs.split(",")]
    L = args.layers

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    # weights: L layers of (gate|up, down); layer 0 is the seed-0 workload, layer l uses seed l
    layers = []
    with torch.cuda.stream(stream):
        for l in range(L):
            gu = wl.quant_matrix(wl.DENSE_GATE_UP, INTER2, HIDDEN, seed=l)
            dn = wl.quant_matrix(wl.DENSE_DOWN, DOWN_OUT, DOWN_IN, seed=l)
            layer = {}
            for key, qm in (("gu", gu), ("dn", dn)):
                layer[key] = (q4a.pack(to_dev(qm.codes)), to_dev(qm.scale), to_dev(qm.bias))
            layer["norm_w"] = to_dev(wl.norm_weight(wl.DENSE_GATE_UP, wl.T_NORM_W, HIDDEN, seed=l))
            if args.layer_mode == "decode_mlp":
                # the down projection that matches the fused gate|up: 6144 -> 4096
                dm = wl.quant_matrix(wl.DENSE_DOWN, DOWN_OUT, INTER, seed=l)
                layer["dn_mlp"] = (q4a.pack(to_dev(dm.codes)), to_dev(dm.scale), to_dev(dm.bias))
            layers.append(layer)
        # activations per NB
        acts = {}
        for nb in nbs:
            a = to_dev(wl.normal_f32(wl.DENSE_GATE_UP, wl.T_A, (nb, HIDDEN)))
            ga = wl.normal_f32(wl.DENSE_DOWN, wl.T_A, (nb, DOWN_IN))
            gb = wl.normal_f32(wl.DENSE_DOWN, wl.T_B, (nb, DOWN_IN))
            gate_up_dn = to_dev(np.concatenate([ga, gb], axis=1))
            x_dn, _ = q4a.silu_mul_xsum(gate_up_dn, want_hsum=False)
            acts[nb] = {
                "a": a, "x_dn": x_dn,
                "h": torch.empty((nb, INTER), dtype=torch.float16, device=dev),
                "y_dn": torch.empty((nb, DOWN_OUT), dtype=torch.float32, device=dev),
            }
    torch.cuda.synchronize()

    def gate_up_call(nb, l):
        ly, ac = layers[l], acts[nb]
        w, s_, b_ = ly["gu"]
        q4a.gemv_rmsnorm_gate_up_silu(w, s_, b_, ac["a"], ly["norm_w"], eps=1e-6, out=ac["h"], stream=stream)

    def down_call(nb, l):
        ly, ac = layers[l], acts[nb]
        w, s_, b_ = ly["dn"]
        q4a.gemv(w, s_, b_, ac["x_dn"], out=ac["y_dn"], stream=stream)

    def layer_call(nb, l):
        if args.layer_mode == "separate":
            gate_up_call(nb, l)
            down_call(nb, l)
            return
        ly, ac = layers[l], acts[nb]
        q4a.decode_mlp(*ly["gu"], ac["a"], ly["norm_w"], *ly["dn_mlp"], eps=1e-6, out=ac["y_dn"], h=ac["h"],
                       stream=stream)

    # eager warm-up: first calls fill the library's per-device caches before capture
    with torch.cuda.stream(stream):
        for nb in nbs:
            layer_call(nb, 0)
    stream.synchronize()

    # Graphs per NB (no event nodes inside, so programmatic dependent launch overlaps
    # consecutive kernels): the decode layer over the L weight sets, and one chain per
    # kernel kind (L fused gate|up launches, L down launches) whose replay time gives the
    # per-launch kernel duration.
    kinds = {"layer": layer_call, "gate_up": gate_up_call, "down": down_call}
    graphs = {}
    for nb in nbs:
        for kind, fn in kinds.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for l in range(L):
                    fn(nb, l)
            graphs[(kind, nb)] = g
    torch.cuda.synchronize()

    total_steps = args.warmup + args.steps
    ev = {(k, kind, nb, e): torch.cuda.Event(enable_timing=True)
          for k in range(total_steps) for kind in kinds for nb in nbs for e in (0, 1)}

    def run_step(k):
        for nb in nbs:
            for kind in kinds:
                ev[(k, kind, nb, 0)].record(stream)
                graphs[(kind, nb)].replay()
                ev[(k, kind, nb, 1)].record(stream)

    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            run_step(k)
    stream.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        w0 = time.time()
        t0.record(stream)
        with torch.cuda.stream(stream):
            for k in range(args.warmup, total_steps):
                run_step(k)
        t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        clk.mark(w0, time.time())
    if dist is not None:
        dist.barrier()
    q4a.check_device_error(stream)
    elapsed_ms = t0.elapsed_time(t1)

    timed = range(args.warmup, total_steps)

    def kind_ms(kind, nb):
        return sum(ev[(k, kind, nb, 0)].elapsed_time(ev[(k, kind, nb, 1)]) for k in timed)

    per_nb = {}
    gemv_bytes_total, gemv_ms_total, step_bytes = 0.0, 0.0, 0.0
    n = args.steps * L
    for nb in nbs:
        gu_b, dn_b = layer_bytes(nb)
        gu_ms, dn_ms, lay_ms = (kind_ms(k, nb) for k in ("gate_up", "down", "layer"))
        lay_b = gu_b + (gemv_bytes(DOWN_OUT, INTER, nb, 2) if args.layer_mode == "decode_mlp" else dn_b)
        per_nb[str(nb)] = {
            "layer_us": lay_ms / n * 1e3, "layer_gbs": lay_b / (lay_ms / n * 1e-3) / 1e9,
            "gate_up_us": gu_ms / n * 1e3, "gate_up_gbs": gu_b / (gu_ms / n * 1e-3) / 1e9,
            "down_us": dn_ms / n * 1e3, "down_gbs": dn_b / (dn_ms / n * 1e-3) / 1e9,
        }
        gemv_bytes_total += (gu_b + dn_b) * n
        gemv_ms_total += gu_ms + dn_ms
        step_bytes += 2 * (gu_b + dn_b) * L     # the layer chain + the per-kind chains
    gemv_launches = 2 * n * len(nbs)
    ms_per_step = max_over_ranks(elapsed_ms / args.steps, dev if dist is not None else None)
    value = whole_job_gbs(step_bytes, world, ms_per_step)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if rank == 0 or world > 1:
        e2e = e2e_measure(q4a, torch, layers, nbs, dev, stream, steps=max(3, min(args.steps, 10)))

    peak, peak_kind = load_peaks()
    roofline = None
    if gemv_ms_total > 0:
        achieved = gemv_bytes_total / (gemv_ms_total * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind,
                    "kernel": "gemv_kernel: every q4a_gemv_rmsnorm_gate_up_silu / q4a_gemv launch of the step",
                    "kernel_source_sha256_16": kernel_source_hash(),
                    "launches": gemv_launches, "traffic": load_traffic(),
                    "timing": "CUDA events around graph replays of back-to-back launches of one kind, "
                              "inside the timed region"}

    # every workload of the set, per launch (rank 0 only; after the timed region)
    configs = None
    if rank == 0 and not args.no_per_config:
        configs = per_config(q4a, torch)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xu4->f32", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "step": "per NB: the decode layer on each of the weight sets, then the same "
                           "gate|up and down launches as one back-to-back chain per kind",
                   "nbs": nbs, "layers_cycled": L,
                   "l2": f"weights cycled over {L} layers ({L * 2 * 28.3:.0f} MB > 3 x L2); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_nb": per_nb,
        "us_per_decode_layer": {k: v["layer_us"] for k, v in per_nb.items()},
        "roofline": roofline,
        "per_config": configs,
        "e2e": e2e,
        "gpu_launches": args.steps * len(nbs) * L * 4,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        gbs, desc, cores = oracle_sample(seconds_target=args.cpu_seconds, nbs=tuple(int(v) for v in args.nbs.split(",")))
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc,
                                **host_info()}
    print(json.dumps(line), flush=True)


def kernel_source_hash():
    import hashlib

    h = hashlib.sha256()
    for name in ("q4a_gemv.cu", "q4a_internal.h", "q4a_device.cuh"):
        with open(os.path.join(ROOT, "affine_q4_dequant_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Mean DRAM bytes per GEMV launch of this step from a committed ncu summary; None when
    the summary is missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "gemv_step_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return d.get("traffic_per_launch_bytes")
    except Exception:
        return None


KERNEL_SHAPES = {"gate_up": (INTER2, HIDDEN), "down": (DOWN_OUT, DOWN_IN), "lm_head": (151936, HIDDEN),
                 "small": (256, 512)}


def load_tc_peak():
    """Dense bf16 tensor throughput (burst) from MEASURED_PEAKS.json, in TFLOP/s. The tensor-core
    path runs f16 x f16 -> f32, whose dense rate equals bf16's."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def time_dense(q4a, torch, out_dim, in_dim, nbs, bits=4, reps=60, profile=False):
    """Per-launch time of q4a_gemv (or q4a_gemv_lowbit) on one shape: a CUDA graph of
    back-to-back calls cycling through weight copies that total > 3 x L2, so that every launch
    streams from HBM; median of 5 replays. One record per NB."""
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    wbytes = out_dim * in_dim * (bits / 8.0 + 4.0 / 64.0)
    copies = max(2, int(3 * 130e6 // wbytes) + 1)
    ws = []
    for _ in range(copies):
        codes = torch.randint(0, 16, (out_dim, in_dim), dtype=torch.uint8, device=dev, generator=g)
        w4 = q4a.pack(codes)
        del codes
        # derived low-bit codes (q4 >> 2, q4 >> 1) replace the nibbles when bits < 4
        wc = (w4, None) if bits == 4 else q4a.lowbit_pack(w4, with_lowest=bits == 3)
        if bits != 4:
            del w4
        ws.append((wc, (torch.rand(out_dim, in_dim // 64, device=dev, generator=g) * 0.02).to(torch.bfloat16),
                   (torch.randn(out_dim, in_dim // 64, device=dev, generator=g) * -0.08).to(torch.bfloat16)))
    peak, kind = load_peaks()
    tc_peak, tc_kind = load_tc_peak()
    out = []
    for nb in nbs:
        x = torch.randn(nb, in_dim, device=dev, generator=g).half()
        y = torch.empty(nb, out_dim, device=dev)

        def call(i):
            (w, w_lo), s_, b_ = ws[i % copies]
            if bits == 4:
                q4a.gemv(w, s_, b_, x, out=y)
            else:
                q4a.gemv_lowbit(bits, w, w_lo, s_, b_, x, out=y)

        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        if profile:
            # plain launches for a profiler: no graph, no timing
            for i in range(reps):
                call(3 + i)
            torch.cuda.synchronize()
            out.append({"kernel": "q4a_gemv" if bits == 4 else "q4a_gemv_lowbit", "bits": bits,
                        "shape": f"{in_dim}->{out_dim}", "nb": nb, "profile_launches": reps + 3})
            continue
        n = copies * max(1, reps // copies)
        us = graph_us(torch, call, n)
        nbytes = gemv_bytes(out_dim, in_dim, nb, 2, bits)
        rec = {"kernel": "q4a_gemv" if bits == 4 else "q4a_gemv_lowbit", "bits": bits,
               "shape": f"{in_dim}->{out_dim}", "nb": nb, "us_per_call": us, "gbs": nbytes / us / 1e3,
               "weights_per_s": out_dim * in_dim / (us * 1e-6), "frac_of_peak": nbytes / us / 1e3 / peak,
               "peak": peak, "peak_kind": kind, "launches_timed": n, "weight_copies": copies}
        path = q4a.gemv_kernel_choice(ws[0][1], ws[0][2], nb, out_dim, in_dim) if bits == 4 else "gemv"
        rec["path"] = path
        if path == "tcgen05":
            # the tensor-core path: a contraction, bounded by max(bytes / HBM, flops / tensor peak)
            tflops = 2.0 * out_dim * in_dim * nb / (us * 1e-6) / 1e12
            bound_us = max(nbytes / (peak * 1e3), 2.0 * out_dim * in_dim * nb / (tc_peak * 1e12) * 1e6)
            rec.update({"tflops": tflops, "tc_peak": tc_peak, "tc_peak_kind": tc_kind,
                        "frac_of_tc_peak": tflops / tc_peak, "frac_of_bound": bound_us / us})
        out.append(rec)
    del ws
    torch.cuda.empty_cache()
    return out


def time_fused_gate_up(q4a, torch, nbs, reps=60, profile=False):
    """Per-launch time of q4a_gemv_rmsnorm_gate_up_silu on the 4096 -> 2 x 6144 matrix (the
    decode layer's first half: RMSNorm prologue, silu(gate) * up epilogue), weight copies > 3 x
    L2, graph of back-to-back calls, median of 5 replays."""
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    copies = max(2, int(3 * 130e6 // (INTER2 * HIDDEN * BYTES_PER_WEIGHT)) + 1)
    ws = []
    for _ in range(copies):
        codes = torch.randint(0, 16, (INTER2, HIDDEN), dtype=torch.uint8, device=dev, generator=g)
        ws.append((q4a.pack(codes), (torch.rand(INTER2, HIDDEN // 64, device=dev, generator=g) * 0.02).to(torch.bfloat16),
                   (torch.randn(INTER2, HIDDEN // 64, device=dev, generator=g) * -0.08).to(torch.bfloat16)))
        del codes
    nw = (1.0 + 0.05 * torch.randn(HIDDEN, device=dev, generator=g)).to(torch.bfloat16)
    peak, kind = load_peaks()
    out = []
    for nb in nbs:
        a = torch.randn(nb, HIDDEN, device=dev, generator=g)
        h = torch.empty(nb, INTER, dtype=torch.float16, device=dev)

        def call(i):
            w, s_, b_ = ws[i % copies]
            q4a.gemv_rmsnorm_gate_up_silu(w, s_, b_, a, nw, eps=1e-6, out=h)

        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        if profile:
            for i in range(reps):
                call(3 + i)
            torch.cuda.synchronize()
            out.append({"kernel": "q4a_gemv_rmsnorm_gate_up_silu", "nb": nb, "profile_launches": reps + 3})
            continue
        n = copies * max(1, reps // copies)
        us = graph_us(torch, call, n)
        nbytes = layer_bytes(nb)[0]
        out.append({"kernel": "q4a_gemv_rmsnorm_gate_up_silu", "shape": f"{HIDDEN}->2x{INTER}", "nb": nb,
                    "us_per_call": us, "gbs": nbytes / us / 1e3, "weights_per_s": INTER2 * HIDDEN / (us * 1e-6),
                    "frac_of_peak": nbytes / us / 1e3 / peak, "peak": peak, "peak_kind": kind, "launches_timed": n})
    del ws
    torch.cuda.empty_cache()
    return out


def run_kernel_mode(args):
    """Per-launch time of one GEMV shape (see time_dense)."""
    import torch

    import affine_q4_dequant_gb300 as q4a

    if args.kernel == "fused_gate_up":
        for rec in time_fused_gate_up(q4a, torch, [int(v) for v in args.nbs.split(",")], args.reps, args.profile):
            print(json.dumps(rec), flush=True)
        return
    out_dim, in_dim = KERNEL_SHAPES[args.kernel]
    for rec in time_dense(q4a, torch, out_dim, in_dim, [int(v) for v in args.nbs.split(",")], args.bits, args.reps,
                          args.profile):
        print(json.dumps(rec), flush=True)


def run_prefill_mode(args):
    """The prefill helpers: q4a_quantize on the 12288 x 4096 gate|up weights (fp32 in, packed
    codes + bf16 scales/biases out) and q4a_gemv_f32x on a narrow 64 x 4096 projection at
    NB = 1, 128 and 512 (fp32 activations). Per-call time from CUDA graphs of back-to-back
    calls; GB/s = bytes read and written / time."""
    import torch

    import affine_q4_dequant_gb300 as q4a

    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    peak, kind = load_peaks()
    rows, cols = INTER2, HIDDEN
    w = torch.randn(rows, cols, device=dev, generator=g) * 0.05

    def quant(i):
        q4a.quantize(w)

    quant(0)
    torch.cuda.synchronize()
    us = graph_us(torch, quant, 20)
    nbytes = rows * cols * 4 + rows * cols / 2 + 2 * rows * (cols // 64) * 2
    print(json.dumps({"kernel": "q4a_quantize", "shape": f"{rows}x{cols} fp32", "us_per_call": us,
                      "gbs": nbytes / us / 1e3, "frac_of_peak": nbytes / us / 1e3 / peak, "peak": peak,
                      "peak_kind": kind}), flush=True)
    out_dim = 64
    ws = []
    for _ in range(8):
        codes = torch.randint(0, 16, (out_dim, cols), dtype=torch.uint8, device=dev, generator=g)
        ws.append((q4a.pack(codes), (torch.rand(out_dim, cols // 64, device=dev, generator=g) * 0.02).to(torch.bfloat16),
                   (torch.randn(out_dim, cols // 64, device=dev, generator=g) * -0.08).to(torch.bfloat16)))
    for nb in (1, 128, 512):
        x = torch.randn(nb, cols, device=dev, generator=g)
        y = torch.empty(nb, out_dim, device=dev)

        def proj(i):
            wq, s_, b_ = ws[i % 8]
            q4a.gemv_f32x(wq, s_, b_, x, out=y)

        proj(0)
        torch.cuda.synchronize()
        us = graph_us(torch, proj, 40)
        nbytes = out_dim * cols * BYTES_PER_WEIGHT + nb * cols * 4 + nb * out_dim * 4
        print(json.dumps({"kernel": "q4a_gemv_f32x", "shape": f"{cols}->{out_dim}", "nb": nb, "us_per_call": us,
                          "gbs": nbytes / us / 1e3, "gflops": 2.0 * out_dim * cols * nb / us / 1e3,
                          "peak": peak, "peak_kind": kind}), flush=True)


def graph_us(torch, fn, n, trials=5):
    """Median per-call time of a CUDA graph of n back-to-back fn(i) calls."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n):
            fn(i)
    graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(trials):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / n * 1e3)
    return statistics.median(times)


def time_moe(q4a, torch, reps=60, profile=False):
    """One routed MoE layer on the 64-expert bank (hidden 2048, inter 640, 16 tokens,
    top-8 by N(0,1) logits): q4a_gemv_experts on gate|up with the token map, the
    SiLU*up activation, q4a_gemv_experts on down, and q4a_moe_combine back to one row per
    token (no shared expert in this workload). Bank replicas total > 3 x L2."""
    E, H, I, T = wl.MOE_EXPERTS, wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_TOKENS
    r = wl.route_by_logits(wl.moe_logits(), wl.MOE_TOP_K)
    U, slots = int(r.expert_ids.shape[0]), int(r.token_offsets[-1])
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def bank(rows, cols):
        codes = torch.randint(0, 16, (rows, cols), dtype=torch.uint8, device=dev, generator=g)
        return (q4a.pack(codes), (torch.rand(rows, cols // 64, device=dev, generator=g) * 0.02).to(torch.bfloat16),
                (torch.randn(rows, cols // 64, device=dev, generator=g) * -0.08).to(torch.bfloat16))

    per_expert = (2 * I * H + H * I) * BYTES_PER_WEIGHT
    copies = max(2, int(3 * 130e6 // (E * per_expert)) + 1)
    banks = [(bank(E * 2 * I, H), bank(E * H, I)) for _ in range(copies)]
    x = torch.randn(T, H, device=dev, generator=g).half()
    x_rows = torch.from_numpy(r.x_rows).to(dev)
    y_gu = torch.empty(slots, 2 * I, device=dev)
    h = torch.empty(slots, I, dtype=torch.float16, device=dev)
    hs = torch.empty(slots, I // 64, device=dev)
    y_dn = torch.empty(slots, H, device=dev)
    slot_np, w_np = wl.moe_combine_inputs(r)
    c_slot = torch.from_numpy(slot_np).to(dev)
    c_w = torch.from_numpy(w_np).to(dev)
    out = torch.empty(T, H, device=dev)

    def gate_up(i):
        w, s_, b_ = banks[i % copies][0]
        q4a.gemv_experts(w, s_, b_, x, x_rows, r.expert_ids, r.token_offsets, E, 2 * I, out=y_gu)

    def act(i):
        q4a.silu_mul_xsum(y_gu, h=h, hsum=hs)

    def down(i):
        w, s_, b_ = banks[i % copies][1]
        q4a.gemv_experts(w, s_, b_, h, None, r.expert_ids, r.token_offsets, E, H, out=y_dn)

    def combine(i):
        q4a.moe_combine(y_dn, c_slot, c_w, out=out)

    def layer(i):
        gate_up(i)
        act(i)
        down(i)
        combine(i)

    for i in range(3):
        layer(i)
    torch.cuda.synchronize()
    if profile:
        for i in range(reps):
            layer(3 + i)
        torch.cuda.synchronize()
        q4a.check_device_error()
        return {"kernel": "moe_layer", "profile_layers": reps + 3}
    n = copies * max(1, reps // copies)
    us = {k: graph_us(torch, fn, n) for k, fn in (("gate_up", gate_up), ("act", act), ("down", down),
                                                   ("combine", combine), ("layer", layer))}
    q4a.check_device_error()
    gu_b = U * 2 * I * H * BYTES_PER_WEIGHT + T * H * 2 + slots * 2 * I * 4
    act_b = slots * 2 * I * 4 + slots * I * 2 + slots * (I // 64) * 4
    dn_b = U * H * I * BYTES_PER_WEIGHT + slots * I * 2 + slots * H * 4
    cb_b = slots * H * 4 + T * H * 4 + slots * 8
    peak, kind = load_peaks()
    del banks
    torch.cuda.empty_cache()
    layer_b = gu_b + act_b + dn_b + cb_b
    return {
        "kernel": "moe_layer", "experts": E, "union_experts": U, "slots": slots,
        "touched_weight_bytes": U * per_expert, "us_per_moe_layer": us["layer"],
        "weights_per_s": U * 3 * I * H / (us["layer"] * 1e-6),
        "gate_up_us": us["gate_up"], "gate_up_gbs": gu_b / us["gate_up"] / 1e3,
        "act_us": us["act"], "down_us": us["down"], "down_gbs": dn_b / us["down"] / 1e3,
        "combine_us": us["combine"], "combine_gbs": cb_b / us["combine"] / 1e3,
        "layer_gbs": layer_b / us["layer"] / 1e3, "frac_of_peak": layer_b / us["layer"] / 1e3 / peak,
        "frac_of_peak_gate_up": gu_b / us["gate_up"] / 1e3 / peak,
        "frac_of_peak_down": dn_b / us["down"] / 1e3 / peak, "peak": peak, "peak_kind": kind,
        "launches_timed": n, "bank_copies": copies}


def run_moe_mode(args):
    import torch

    import affine_q4_dequant_gb300 as q4a

    print(json.dumps(time_moe(q4a, torch, args.reps, args.profile)), flush=True)


def per_config(q4a, torch, reps=40):
    """Every workload of the benchmark set, timed per launch on this GPU: the 256 x 512 GEMV,
    the 4096 -> 12288 projection (plain, and fused with the RMSNorm prologue and the
    silu(gate)*up epilogue), the 12288 -> 4096 down projection, the routed MoE layer and the
    151936-row LM head (NB >= 64 on the tensor-core path)."""
    def brief(recs):
        keep = ("nb", "us_per_call", "gbs", "weights_per_s", "frac_of_peak", "path", "tflops", "frac_of_tc_peak",
                "frac_of_bound")
        return [{k: r[k] for k in keep if k in r} for r in recs]

    out = {
        "gemv_256x512": brief(time_dense(q4a, torch, 256, 512, [1], reps=reps)),
        "gate_up_4096x12288": brief(time_dense(q4a, torch, INTER2, HIDDEN, [1, 2, 4, 8, 16, 32, 64], reps=reps)),
        "fused_rmsnorm_gate_up_silu_4096x2x6144": brief(time_fused_gate_up(q4a, torch, [1, 2, 4, 8, 16], reps=reps)),
        "down_12288x4096": brief(time_dense(q4a, torch, DOWN_OUT, DOWN_IN, [1, 4, 8, 16, 32, 64], reps=reps)),
        "lm_head_4096x151936": brief(time_dense(q4a, torch, 151936, HIDDEN, [1, 8, 32, 64, 128], reps=reps)),
    }
    moe = time_moe(q4a, torch, reps=reps)
    out["moe_layer_64x2048x640"] = {k: moe[k] for k in ("union_experts", "slots", "us_per_moe_layer", "layer_gbs",
                                                         "weights_per_s", "frac_of_peak", "gate_up_us", "down_us",
                                                         "act_us", "combine_us")}
    return out


def e2e_measure(q4a, torch, layers, nbs, dev, stream, steps):
    """Public API, host buffers: every step copies all NBs' inputs in from pinned memory (one copy
    of one packed buffer: the fp32 rows of the fused gate|up and the binary16 rows of the down
    projection), runs each NB's decode-layer MLP through the binding -- the same two kernels as
    the device-timed step: q4a.gemv_rmsnorm_gate_up_silu, then q4a.gemv (eager launches, outputs
    into preallocated device buffers) -- and copies the down projections' outputs back (one
    copy)."""
    parts = []
    for nb in nbs:
        a = wl.normal_f32(wl.DENSE_GATE_UP, wl.T_A, (nb, HIDDEN))
        x_dn = wl.normal_f16(wl.DENSE_DOWN, wl.T_A, (nb, DOWN_IN))   # binary16 bit patterns
        parts.append((nb, a, x_dn))
    n_f32 = sum(a.size for _, a, _ in parts)
    n_f16 = sum(x.size for _, _, x in parts)
    host_in = torch.empty(n_f32 * 4 + n_f16 * 2, dtype=torch.uint8).pin_memory()
    hv = host_in.numpy()
    off = 0
    for _, a, _ in parts:
        hv[off:off + a.size * 4] = np.ascontiguousarray(a, np.float32).view(np.uint8).ravel()
        off += a.size * 4
    for _, _, x in parts:
        hv[off:off + x.size * 2] = np.ascontiguousarray(x, np.uint16).view(np.uint8).ravel()
        off += x.size * 2
    # two pinned output buffers: step k + 1 is enqueued before the host reads step k's output
    host_out = [torch.empty(sum(nb * DOWN_OUT for nb in nbs), dtype=torch.float32).pin_memory() for _ in range(2)]
    dev_in = torch.empty(host_in.numel(), dtype=torch.uint8, device=dev)
    dev_out = torch.empty(host_out[0].numel(), dtype=torch.float32, device=dev)
    views, fo, ho, oo = [], 0, n_f32 * 4, 0
    for nb, a, x in parts:
        va = dev_in[fo:fo + a.size * 4].view(torch.float32).view(nb, HIDDEN)
        fo += a.size * 4
        vx = dev_in[ho:ho + x.size * 2].view(torch.float16).view(nb, DOWN_IN)
        ho += x.size * 2
        vo = dev_out[oo:oo + nb * DOWN_OUT].view(nb, DOWN_OUT)
        oo += nb * DOWN_OUT
        h = torch.empty((nb, INTER2 // 2), dtype=torch.float16, device=dev)
        views.append((va, vx, vo, h))
    h2d = host_in.numel()
    d2h = host_out[0].numel() * 4
    L = len(layers)
    done = [torch.cuda.Event(), torch.cuda.Event()]
    seen = []

    def enqueue(k):
        # step k: its inputs in, its kernels, its outputs out (stream order keeps the copies of
        # consecutive steps apart from each other's kernels)
        ly = layers[k % L]
        with torch.cuda.stream(stream):
            dev_in.copy_(host_in, non_blocking=True)
            for va, vx, vo, h in views:
                w, s, b = ly["gu"]
                q4a.gemv_rmsnorm_gate_up_silu(w, s, b, va, ly["norm_w"], eps=1e-6, out=h, stream=stream)
                w, s, b = ly["dn"]
                q4a.gemv(w, s, b, vx, out=vo, stream=stream)
            host_out[k % 2].copy_(dev_out, non_blocking=True)
            done[k % 2].record(stream)

    def read(k):
        # the host waits for step k and reads its outputs
        done[k % 2].synchronize()
        seen.append(float(host_out[k % 2][-1]))

    for k in range(2):
        enqueue(k)
        read(k)
    t0 = time.perf_counter()
    enqueue(0)
    for k in range(1, steps):
        enqueue(k)
        read(k - 1)
    read(steps - 1)
    dt = (time.perf_counter() - t0) / steps
    assert all(v == v for v in seen), "non-finite output in the end-to-end steps"
    step_bytes = sum(sum(layer_bytes(nb)) for nb in nbs)
    # host cost of one call through the binding (argument checks, marshalling, the C ABI's
    # validation, planning and launch): back-to-back calls on a small product, no sync between
    ly = layers[0]
    w, s, b = ly["dn"]
    x1 = torch.zeros((1, DOWN_IN), dtype=torch.float16, device=dev)
    y1 = torch.empty((1, DOWN_OUT), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(20):
            q4a.gemv(w, s, b, x1, out=y1, stream=stream)
        stream.synchronize()
        n_calls = 200
        h0 = time.perf_counter()
        for _ in range(n_calls):
            q4a.gemv(w, s, b, x1, out=y1, stream=stream)
        host_us = (time.perf_counter() - h0) / n_calls * 1e6
        stream.synchronize()
    return {"value": step_bytes / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "host_us_per_call": host_us,
            "note": "per NB per step the step's two kernels (fused RMSNorm + gate|up + silu*up, then the "
                    "down projection), eager launches through the Python binding; every step copies its "
                    "inputs in and its outputs out, and the host reads each step's outputs while the next "
                    "step runs (two steps in flight); host_us_per_call: wall time of one q4a.gemv call on "
                    "the host (launch included)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--nbs", default="1,2,4,8,16")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: total seconds of oracle work over all warm-up and timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload launch timings")
    ap.add_argument("--kernel", choices=sorted(KERNEL_SHAPES) + ["fused_gate_up", "moe", "prefill"], default=None,
                    help="time one GEMV shape per launch instead of the decode-layer step")
    ap.add_argument("--reps", type=int, default=60)
    ap.add_argument("--bits", type=int, choices=[4, 3, 2], default=4,
                    help="with --kernel: code width (3 and 2: derived low-bit codes, q4a_gemv_lowbit)")
    ap.add_argument("--layer-mode", choices=["decode_mlp", "separate"], default="separate",
                    help="separate: the 4096 -> 2 x 6144 fused gate|up and the 12288 -> 4096 down projection "
                         "(both workloads of the set); decode_mlp: q4a_decode_mlp with its matching "
                         "6144 -> 4096 down projection")
    ap.add_argument("--profile", action="store_true",
                    help="with --kernel: eager launches only (a target for ncu), no timing")
    args = ap.parse_args()
    if args.kernel == "moe":
        run_moe_mode(args)
        return
    if args.kernel == "prefill":
        run_prefill_mode(args)
        return
    if args.kernel:
        run_kernel_mode(args)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
