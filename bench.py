"""Benchmark of the int4 affine decode path on one GB300 (or N replicas under torchrun).

Workload (one "step"): one dense decode layer, hidden 5120, FFN 17408, M = 1 -- gate and up
(17408 x 5120 each, one fused launch with the SwiGLU epilogue, h in fp32) followed by down
(5120 x 17408, fp32 h).  Weights are seeded synthetic int4 group-64 data with bf16 scales/biases;
x is bf16 N(0, 1).  Every step reads a different copy of the layer's weights (12 copies, 1.8 GB,
far larger than the 129 MB L2), so weights always come from HBM.

The JSON line reports
  value      effective GB/s of the layer (algorithmic bytes: packed codes + scales + biases + x +
             h + y) with inputs resident in HBM,
  e2e        the same metric through the C-ABI calls with host buffers: each step copies x in from
             pinned host memory and y back out,
  roofline   for the dominant kernel (the fused gate/up SwiGLU GEMV), timed back to back,
  target     the M = 1 GEMV at 5120 x 17408 with bf16 x (us/call, GB/s, fractions of HBM peak),
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same layer.

    python bench.py [--steps K] [--warmup W] [--impl qg|reference]
"""
from __future__ import annotations

import argparse
import hashlib
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

HIDDEN, FFN = 5120, 17408
N_COPIES = 12
NOMINAL_HBM_GBS = 8000.0


def weight_bytes(out, in_dim):
    return out * in_dim // 2 + 2 * 2 * out * (in_dim // 64)


# algorithmic bytes per kernel / per layer
B_GATEUP = 2 * weight_bytes(FFN, HIDDEN) + HIDDEN * 2 + FFN * 4      # gate+up weights, x bf16, h fp32
B_DOWN_H = weight_bytes(HIDDEN, FFN) + FFN * 4 + HIDDEN * 4            # down weights, h fp32, y fp32
B_LAYER = B_GATEUP + B_DOWN_H
B_DOWN_BF16 = weight_bytes(HIDDEN, FFN) + FFN * 2 + HIDDEN * 4         # the headline GEMV, bf16 x


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda") if torch.cuda.is_available() and dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is under load."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "100", "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 7]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------- qg arm
def run_qg(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    from moe_int4_affine_gb300 import build

    build.build()
    from moe_int4_affine_gb300 import inputs as I
    from moe_int4_affine_gb300 import qg

    dev = torch.device("cuda", local_rank)
    gate = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, FFN, HIDDEN), dev)
    up = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, FFN, HIDDEN), dev)
    down = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, HIDDEN, FFN), dev)

    def copy_w(w):
        return qg.Int4Weight(w.packed.clone(), w.scales.clone(), w.biases.clone(), w.out, w.in_dim)

    layers = [(gate, up, down)] + [(copy_w(gate), copy_w(up), copy_w(down)) for _ in range(N_COPIES - 1)]
    x_np = I.bf16_normal(0, I.TID_X, HIDDEN)
    x = qg.to_device(x_np, dev)
    h = torch.empty(FFN, dtype=torch.float32, device=dev)
    y = torch.empty(HIDDEN, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = int(stream.cuda_stream)
    lib, P = qg.lib, qg.ctypes.c_void_p
    import ctypes

    # pre-marshalled C-ABI arguments per copy: the timed loop makes only the two C calls per step
    pairs = []
    for g_, u_, d_ in layers:
        arr = (qg.qg_int4_weight * 2)(g_.struct, u_.struct)
        ys = (P * 2)(h.data_ptr(), None)
        pairs.append((arr, ys, ctypes.byref(d_.struct), d_))
    xp, hp, yp = P(x.data_ptr()), P(h.data_ptr()), P(y.data_ptr())

    def step(i, xptr=xp):
        arr, ys, dref, _ = pairs[i % N_COPIES]
        rc = lib.qgemv_int4_multi(2, arr, xptr, qg.QG_X_BF16, ys, qg.QG_EPI_SWIGLU, s)
        rc |= lib.qgemv_int4(dref, hp, qg.QG_X_F32, yp, s)
        return rc

    qg.qg_set_pdl(not args.no_pdl)
    for i in range(args.warmup):
        assert step(i) == 0
    torch.cuda.synchronize()
    assert qg.qg_device_status() == 0

    # soak under the clock sampler, then the timed region
    sampler = ClockSampler(local_rank) if rank == 0 else None
    t_end = time.time() + args.soak
    i = 0
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    barrier(world)
    ms = max_over_ranks(ms, world)
    clocks = sampler.stop() if sampler else None
    ms_step = ms / args.steps
    value = world * B_LAYER / (ms_step * 1e-3) / 1e9

    # dominant kernel (fused gate/up SwiGLU GEMV), back to back on the same stream
    def time_loop(fn, n):
        for i in range(8):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n  # us per launch

    def gateup(i):
        arr, ys, _, _ = pairs[i % N_COPIES]
        return lib.qgemv_int4_multi(2, arr, xp, qg.QG_X_BF16, ys, qg.QG_EPI_SWIGLU, s)

    def down_bf16(i):
        _, _, dref, _ = pairs[i % N_COPIES]
        return lib.qgemv_int4(dref, xbig, qg.QG_X_BF16, yp, s)

    xbig_t = qg.to_device(I.bf16_normal(0, I.TID_X + 100, FFN), dev)
    xbig = P(xbig_t.data_ptr())
    n_loop = max(50, args.steps)
    us_gateup = time_loop(gateup, n_loop)
    us_down = time_loop(down_bf16, n_loop)
    qg.qg_set_pdl(False)
    us_down_nopdl = time_loop(down_bf16, n_loop)
    qg.qg_set_pdl(not args.no_pdl)

    # end to end: x in from pinned host memory, y back to pinned host memory, every step
    x_host = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    y_host = torch.empty(HIDDEN, dtype=torch.float32).pin_memory()
    x_dev16 = x.view(torch.int16)
    for i in range(args.warmup):
        x_dev16.copy_(x_host, non_blocking=True)
        step(i)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        x_dev16.copy_(x_host, non_blocking=True)
        step(i)
        y_host.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    assert qg.qg_device_status() == 0
    qg.qg_set_pdl(False)

    if rank != 0:
        return None
    peak, peak_kind = peaks()
    achieved = B_GATEUP / (us_gateup * 1e-6) / 1e9
    traffic = None
    tf = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(tf) as f:
            t = json.load(f)
        src = open(os.path.join(ROOT, "moe_int4_affine_gb300", "csrc", "qgemv.cu"), "rb").read()
        if t.get("source_sha256") == hashlib.sha256(src).hexdigest():
            traffic = t.get("gateup_bytes_per_launch")
    except Exception:
        pass
    line = {
        "metric": "int4 dequant-GEMV effective GB/s (dense decode layer M=1, hidden 5120, FFN 17408)",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_layer": round(ms_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4 weights, bf16 x, fp32 accumulate",
        "data": "synthetic (seeded int4 group-64 weights, bf16 scales/biases, x ~ N(0,1))",
        "config": {"workload": "dense decode layer M=1: gate+up 17408x5120 (fused, SwiGLU) -> down 5120x17408",
                   "hidden": HIDDEN, "ffn": FFN, "group_size": 64, "bytes_per_layer": B_LAYER,
                   "l2": f"weights rotate over {N_COPIES} copies ({N_COPIES * B_LAYER / 1e9:.2f} GB), larger than L2",
                   "pdl": not args.no_pdl, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "gemv_kernel (gate+up SwiGLU pair)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "us_per_launch": round(us_gateup, 3),
                     "algorithmic_bytes": B_GATEUP},
        "target": {"gemv": "5120x17408, bf16 x", "us_per_call": round(us_down, 3),
                   "GBps": round(B_DOWN_BF16 / (us_down * 1e-6) / 1e9, 1),
                   "frac_of_8000": round(B_DOWN_BF16 / (us_down * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                   "frac_of_measured": round(B_DOWN_BF16 / (us_down * 1e-6) / 1e9 / peak, 4),
                   "us_per_call_without_pdl": round(us_down_nopdl, 3), "algorithmic_bytes": B_DOWN_BF16},
        "e2e": {"value": round(world * B_LAYER / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": HIDDEN * 2, "d2h_bytes_per_step": HIDDEN * 4,
                "us_per_layer": round(e2e_ms * 1e3, 3)},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    return line


# ---------------------------------------------------------------------------------------------- oracle
def oracle_layer_sample(frac: float, threads: int):
    """Run the fp64 oracle on the first `frac` of each matrix's rows of the decode layer; return
    (seconds, algorithmic bytes of the sample)."""
    import oracle
    from moe_int4_affine_gb300 import inputs as I

    gate = I.int4_weight(0, I.TID_GATE, FFN, HIDDEN)
    up = I.int4_weight(0, I.TID_UP, FFN, HIDDEN)
    down = I.int4_weight(0, I.TID_DOWN, HIDDEN, FFN)
    x = I.bf16_normal(0, I.TID_X, HIDDEN)
    h = I.f32_normal(0, 99, FFN)  # stand-in activations for the down rows' sample (same cost)
    rg = max(1, int(FFN * frac))
    rd = max(1, int(HIDDEN * frac))
    t0 = time.perf_counter()
    oracle.qgemv(gate["packed"], gate["scales"], gate["biases"], x, rows=(0, rg), threads=threads)
    oracle.qgemv(up["packed"], up["scales"], up["biases"], x, rows=(0, rg), threads=threads)
    oracle.qgemv(down["packed"], down["scales"], down["biases"], h, rows=(0, rd), threads=threads)
    dt = time.perf_counter() - t0
    nbytes = 2 * rg * weight_bytes(1, HIDDEN) + rd * weight_bytes(1, FFN) + HIDDEN * 2 + FFN * 4 + rd * 4
    return dt, nbytes


def cpu_baseline(target_s: float = 12.0):
    threads = os.cpu_count() or 1
    dt, nb = oracle_layer_sample(0.002, threads)  # calibration
    frac = min(1.0, 0.002 * target_s / max(dt, 1e-3))
    dt, nb = oracle_layer_sample(frac, threads)
    return {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"first {frac:.4f} of the rows of gate, up and down ({nb / 1e6:.1f} MB), fp64 C oracle, "
                      f"{threads} host threads, {dt:.1f} s"}


def run_reference(args):
    threads = os.cpu_count() or 1
    dt, nb = oracle_layer_sample(0.002, threads)
    frac = min(1.0, 0.002 * 4.0 / max(dt, 1e-3))  # each step about 4 s of oracle work
    for _ in range(args.warmup):
        oracle_layer_sample(frac / 8, threads)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_layer_sample(frac, threads)
        tot_t += dt
        tot_b += nb
    v = tot_b / tot_t / 1e9
    return {"impl": "reference", "metric": "int4 dequant-GEMV effective GB/s (dense decode layer M=1, hidden 5120, "
                                           "FFN 17408)",
            "value": round(v, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "dense decode layer M=1: gate+up 17408x5120 -> down 5120x17408 (row sample)",
                       "sample_fraction": round(frac, 5)},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {frac:.4f} of each matrix's rows per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qg", choices=["qg", "reference"])
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed steps under the clock sampler")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist

        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(run_reference(args)), flush=True)
            return 0
        line = run_qg(args, rank, world, local_rank)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
            print(json.dumps(line), flush=True)
        return 0
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
