#!/usr/bin/env python
"""Benchmark: the dense decode-layer MLP built from the affine-Q4 GEMV on GB300.

One step = for every NB in the sweep (default 1, 2, 4, 8, 16), one decode-layer
MLP on each of L weight sets (default 8, so the 453 MB of weights are larger
than three L2 caches and every layer streams from HBM):
    q4a_gemv_rmsnorm  4096 -> 12288 fused gate|up with the RMSNorm prologue
    q4a_silu_mul_xsum silu(gate) * up on the 6144-wide halves
    q4a_gemv          12288 -> 4096 down projection (its own synthetic input
                      x = fp16(silu(a) * b), built once per NB by the same kernel)
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
METRIC = "achieved HBM GB/s (and % of roofline) per q4a_gemv call vs NB; us/decode-layer"


def gemv_bytes(out_dim, in_dim, nb, x_bytes_per_el):
    return out_dim * in_dim * BYTES_PER_WEIGHT + nb * in_dim * x_bytes_per_el + nb * out_dim * 4


def layer_bytes(nb):
    gu = gemv_bytes(INTER2, HIDDEN, nb, 4) + HIDDEN * 2           # fp32 x_raw + bf16 norm weight
    act = nb * INTER2 * 4 + nb * INTER * 2 + nb * (INTER // 64) * 4
    dn = gemv_bytes(DOWN_OUT, DOWN_IN, nb, 2)
    return gu, act, dn


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

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
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
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---- CPU baseline (the oracle as it stands) --------------------------------------------

def oracle_sample(seconds_target: float = 12.0):
    """Time the CPU oracle on a bounded sample of the same workload: the decode-layer
    MLP at NB = 1 and 2 on a row sample of both projections (512 gate|up rows, 256
    down rows), repeated until ~seconds_target. Returns (GB/s, description, cores)."""
    import oracle

    rows_gu, rows_dn = 512, 256
    qm_gu = wl.quant_matrix(wl.DENSE_GATE_UP, rows_gu, HIDDEN)
    qm_dn = wl.quant_matrix(wl.DENSE_DOWN, rows_dn, DOWN_IN)
    p_gu, p_dn = oracle.pack(qm_gu.codes), oracle.pack(qm_dn.codes)
    nw = wl.norm_weight(wl.DENSE_GATE_UP, wl.T_NORM_W, HIDDEN)
    total_bytes, t0, reps = 0.0, time.perf_counter(), 0
    while True:
        for nb in (1, 2):
            a = wl.normal_f32(wl.DENSE_GATE_UP, wl.T_A, (nb, HIDDEN))
            xn, _ = oracle.rmsnorm_f16(a, nw, eps=1e-6)
            y, _ = oracle.gemv(p_gu, qm_gu.scale, qm_gu.bias, xn)
            h = oracle.silu_mul_f16(np.concatenate([y, y], axis=1).astype(np.float32))
            xd = wl.normal_f16(wl.DENSE_DOWN, wl.T_X, (nb, DOWN_IN))
            oracle.gemv(p_dn, qm_dn.scale, qm_dn.bias, xd)
            total_bytes += (gemv_bytes(rows_gu, HIDDEN, nb, 4) + gemv_bytes(rows_dn, DOWN_IN, nb, 2)
                            + h.size * 2)
        reps += 1
        if time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    desc = (f"oracle decode-layer MLP on a row sample ({rows_gu} of {INTER2} gate|up rows, {rows_dn} of "
            f"{DOWN_OUT} down rows) at NB=1,2, {reps} repetitions, {dt:.1f} s, single-threaded fp64")
    return total_bytes / dt / 1e9, desc, 1


def run_reference(args, rank, world):
    if rank != 0:
        return
    steps_bytes, times = [], []
    import oracle  # noqa: F401
    for i in range(args.warmup + args.steps):
        per = max(2.0, 60.0 / max(1, args.warmup + args.steps))
        gbs, desc, cores = oracle_sample(seconds_target=per)
        if i >= args.warmup:
            times.append(gbs)
    value = statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "dense decode-layer MLP 4096->12288 gate|up (RMSNorm fused) + silu*up + "
                               "12288->4096 down, affine-Q4 group 64", "nbs": args.nbs},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
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
                "y_gu": torch.empty((nb, INTER2), dtype=torch.float32, device=dev),
                "h": torch.empty((nb, INTER), dtype=torch.float16, device=dev),
                "hsum": torch.empty((nb, INTER // 64), dtype=torch.float32, device=dev),
                "y_dn": torch.empty((nb, DOWN_OUT), dtype=torch.float32, device=dev),
            }
    torch.cuda.synchronize()

    def layer_call(nb, l, evs=None):
        ly, ac = layers[l], acts[nb]
        w, s, b = ly["gu"]
        if evs: evs[0].record(stream)
        q4a.gemv_rmsnorm(w, s, b, ac["a"], ly["norm_w"], eps=1e-6, out=ac["y_gu"], stream=stream)
        if evs: evs[1].record(stream)
        q4a.silu_mul_xsum(ac["y_gu"], h=ac["h"], hsum=ac["hsum"], stream=stream)
        if evs: evs[2].record(stream)
        w, s, b = ly["dn"]
        q4a.gemv(w, s, b, ac["x_dn"], out=ac["y_dn"], stream=stream)
        if evs: evs[3].record(stream)

    # ---- graphs: one per (step, NB), each with event nodes around every launch ----
    total_steps = args.warmup + args.steps

    def new_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None

    # eager warm-up: first calls fill the library's per-device caches before capture
    with torch.cuda.stream(stream):
        for nb in nbs:
            layer_call(nb, 0)
    stream.synchronize()

    graphs, gevents = {}, {}
    use_graph_events = new_event() is not None
    for k in range(total_steps):
        for nb in nbs:
            evs = [[new_event() for _ in range(4)] for _ in range(L)] if use_graph_events else None
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for l in range(L):
                    layer_call(nb, l, evs[l] if evs else None)
            graphs[(k, nb)] = g
            gevents[(k, nb)] = evs
    torch.cuda.synchronize()

    step_start = [torch.cuda.Event(enable_timing=True) for _ in range(total_steps)]
    step_end = [torch.cuda.Event(enable_timing=True) for _ in range(total_steps)]
    nb_start = {(k, nb): torch.cuda.Event(enable_timing=True) for k in range(total_steps) for nb in nbs}
    nb_end = {(k, nb): torch.cuda.Event(enable_timing=True) for k in range(total_steps) for nb in nbs}

    def run_step(k):
        step_start[k].record(stream)
        for nb in nbs:
            nb_start[(k, nb)].record(stream)
            graphs[(k, nb)].replay()
            nb_end[(k, nb)].record(stream)
        step_end[k].record(stream)

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
        t0.record(stream)
        with torch.cuda.stream(stream):
            for k in range(args.warmup, total_steps):
                run_step(k)
        t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    q4a.check_device_error(stream)
    elapsed_ms = t0.elapsed_time(t1)

    # per-NB and per-kernel times from the timed steps
    timed = range(args.warmup, total_steps)
    per_nb = {}
    gemv_bytes_total, gemv_ms_total, gemv_launches = 0.0, 0.0, 0
    for nb in nbs:
        nb_ms = sum(nb_start[(k, nb)].elapsed_time(nb_end[(k, nb)]) for k in timed)
        gu_b, act_b, dn_b = layer_bytes(nb)
        rec = {"layer_us": nb_ms / (args.steps * L) * 1e3}
        if use_graph_events:
            gu_ms = act_ms = dn_ms = 0.0
            for k in timed:
                for ev in gevents[(k, nb)]:
                    gu_ms += ev[0].elapsed_time(ev[1])
                    act_ms += ev[1].elapsed_time(ev[2])
                    dn_ms += ev[2].elapsed_time(ev[3])
            n = args.steps * L
            rec.update({
                "gate_up_us": gu_ms / n * 1e3, "gate_up_gbs": gu_b / (gu_ms / n * 1e-3) / 1e9,
                "act_us": act_ms / n * 1e3,
                "down_us": dn_ms / n * 1e3, "down_gbs": dn_b / (dn_ms / n * 1e-3) / 1e9,
            })
            gemv_bytes_total += (gu_b + dn_b) * n
            gemv_ms_total += gu_ms + dn_ms
            gemv_launches += 2 * n
        per_nb[str(nb)] = rec

    step_bytes = sum(sum(layer_bytes(nb)) for nb in nbs) * L
    ms_per_step = elapsed_ms / args.steps
    if dist is not None:
        import torch.distributed as dist
        t = torch.tensor([ms_per_step], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step = float(t.item())
    value = step_bytes * world / (ms_per_step * 1e-3) / 1e9

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
                    "kernel": "q4a gemv (gemv_kernel, all NB, gate|up with RMSNorm + down)",
                    "launches": gemv_launches, "traffic": load_traffic()}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xu4->f32", "data": "synthetic",
        "config": {"workload": "dense decode-layer MLP: 4096->12288 gate|up (fused RMSNorm) + "
                               "silu*up (6144) + 12288->4096 down; affine-Q4 group 64",
                   "nbs": nbs, "layers_cycled": L,
                   "l2": f"weights cycled over {L} layers ({L * 2 * 28.3:.0f} MB > 3 x L2); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_nb": per_nb,
        "us_per_decode_layer": {k: v["layer_us"] for k, v in per_nb.items()},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * len(nbs) * L * 3,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        gbs, desc, cores = oracle_sample(seconds_target=args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


def load_traffic():
    """Per-launch DRAM bytes of the GEMV kernel from a committed ncu summary, if present."""
    path = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    try:
        with open(path) as f:
            return json.load(f).get("traffic_per_launch_bytes")
    except Exception:
        return None


def e2e_measure(q4a, torch, layers, nbs, dev, stream, steps):
    """Public API, host buffers: every step copies each NB's activations in from pinned
    memory, runs one decode-layer MLP per NB through the binding (eager launches, no
    graph), and copies the down projection's output back."""
    host_in, host_out = {}, {}
    for nb in nbs:
        a = wl.normal_f32(wl.DENSE_GATE_UP, wl.T_A, (nb, HIDDEN))
        ga = wl.normal_f32(wl.DENSE_DOWN, wl.T_A, (nb, DOWN_IN))
        gb = wl.normal_f32(wl.DENSE_DOWN, wl.T_B, (nb, DOWN_IN))
        host_in[nb] = (torch.from_numpy(a).pin_memory(),
                       torch.from_numpy(np.concatenate([ga, gb], axis=1)).pin_memory())
        host_out[nb] = torch.empty((nb, DOWN_OUT), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * 4 for nb in nbs for t in host_in[nb])
    d2h = sum(host_out[nb].numel() * 4 for nb in nbs)
    L = len(layers)

    def one(k):
        ly = layers[k % L]
        with torch.cuda.stream(stream):
            for nb in nbs:
                a = host_in[nb][0].to(dev, non_blocking=True)
                gu_dn = host_in[nb][1].to(dev, non_blocking=True)
                w, s, b = ly["gu"]
                y = q4a.gemv_rmsnorm(w, s, b, a, ly["norm_w"], eps=1e-6, stream=stream)
                q4a.silu_mul_xsum(y, stream=stream)
                x_dn, _ = q4a.silu_mul_xsum(gu_dn, want_hsum=False, stream=stream)
                w, s, b = ly["dn"]
                y_dn = q4a.gemv(w, s, b, x_dn, stream=stream)
                host_out[nb].copy_(y_dn, non_blocking=True)
        stream.synchronize()

    for k in range(2):
        one(k)
    t0 = time.perf_counter()
    for k in range(steps):
        one(k)
    dt = (time.perf_counter() - t0) / steps
    step_bytes = sum(sum(layer_bytes(nb)) for nb in nbs)
    return {"value": step_bytes / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
            "note": "one decode-layer MLP per NB per step, eager launches through the Python binding"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--nbs", default="1,2,4,8,16")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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
