"""Benchmark of the int4 affine decode path on one GB300 (or N replicas under torchrun).

Workload (one "step"): one dense decode layer, hidden 5120, FFN 17408, M = 1 -- gate and up
(17408 x 5120 each, one fused launch with the SwiGLU epilogue, h in fp32) followed by down
(5120 x 17408, fp32 h): one dense_layer_int4 call.  Weights are seeded synthetic int4 group-64 data with bf16 scales/biases;
x is bf16 N(0, 1).  Every step reads a different copy of the layer's weights (12 copies, 1.8 GB,
far larger than the 129 MB L2), so weights always come from HBM.

The JSON line reports
  value      effective GB/s of the layer (algorithmic bytes: packed codes + scales + biases + x +
             h + y) with inputs resident in HBM,
  e2e        the same metric through the host-buffer C-ABI call (dense_layer_int4_host): each step
             the GPU reads x from pinned host memory and writes y back into pinned host memory,
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
    y = torch.empty(HIDDEN, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = int(stream.cuda_stream)
    lib, P = qg.lib, qg.ctypes.c_void_p
    import ctypes

    # pre-marshalled C-ABI arguments per copy: the timed loop makes one C call per step
    # (dense_layer_int4: the gate/up SwiGLU launch, then the down launch; h in the workspace)
    ws_bytes = qg.qg_workspace_bytes(qg.QG_OP_LAYER, down, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    h = ws[:4 * FFN].view(torch.float32)
    pairs = []
    for g_, u_, d_ in layers:
        arr = (qg.qg_int4_weight * 2)(g_.struct, u_.struct)
        ys = (P * 2)(h.data_ptr(), None)
        pairs.append((arr, ys, ctypes.byref(d_.struct), ctypes.byref(g_.struct), ctypes.byref(u_.struct)))
    xp, hp, yp, wsp = P(x.data_ptr()), P(h.data_ptr()), P(y.data_ptr()), P(ws.data_ptr())

    def step(i, xptr=xp):
        _, _, dref, gref, uref = pairs[i % N_COPIES]
        return lib.dense_layer_int4(gref, uref, dref, xptr, qg.QG_X_BF16, yp, wsp, ws_bytes, s)

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
    # the timed region: exactly K steps between a barrier and a synchronize on both sides, repeated
    # (at least 5 times and 250 steps in all) and reported as the median over the repeats, with the
    # spread; each repeat's time is the max over ranks
    reps = max(5, -(-250 // args.steps))
    rep_ms = []
    for r in range(reps):
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            step(r * args.steps + i)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        rep_ms.append(max_over_ranks(ev0.elapsed_time(ev1), world))
    clocks = sampler.stop() if sampler else None
    ms = statistics.median(rep_ms)
    ms_step = ms / args.steps
    value = world * B_LAYER / (ms_step * 1e-3) / 1e9
    spread = {"repeats": reps, "steps_per_repeat": args.steps,
              "ms_per_step_min": round(min(rep_ms) / args.steps, 5), "ms_per_step_max": round(max(rep_ms) / args.steps, 5)}

    # dominant kernel (fused gate/up SwiGLU GEMV), back to back on the same stream
    def time_loop(fn, n):  # us per launch: the median of 5 runs of n back-to-back launches
        for i in range(8):
            fn(i)
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        return statistics.median(ts)

    def gateup(i):
        arr, ys = pairs[i % N_COPIES][:2]
        return lib.qgemv_int4_multi(2, arr, xp, qg.QG_X_BF16, ys, qg.QG_EPI_SWIGLU, s)

    def down_bf16(i):
        dref = pairs[i % N_COPIES][2]
        return lib.qgemv_int4(dref, xbig, qg.QG_X_BF16, yp, s)

    xbig_t = qg.to_device(I.bf16_normal(0, I.TID_X + 100, FFN), dev)
    xbig = P(xbig_t.data_ptr())
    n_loop = max(50, args.steps)
    us_gateup = time_loop(gateup, n_loop)
    us_down = time_loop(down_bf16, n_loop)
    qg.qg_set_pdl(False)
    us_down_nopdl = time_loop(down_bf16, n_loop)
    qg.qg_set_pdl(not args.no_pdl)

    configs = None
    if rank == 0 and not args.no_configs:
        try:  # (a failing configuration is reported in the line, not allowed to drop the line)
            configs = measure_configs(qg, I, dev, stream)
        except Exception as e:  # noqa: BLE001
            configs = {"error": f"{type(e).__name__}: {e}"}
    qg.qg_set_pdl(not args.no_pdl)

    # end to end through the host-buffer call: every step the GPU reads x from pinned host memory
    # (a one-block copy kernel) and the down kernel writes y into pinned host memory
    x_host = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    y_host = torch.empty(HIDDEN, dtype=torch.float32).pin_memory()
    wsh_bytes = qg.qg_workspace_bytes(qg.QG_OP_LAYER_HOST, down, HIDDEN)
    wsh = torch.empty(wsh_bytes, dtype=torch.uint8, device=dev)
    xhp, yhp, wshp = P(x_host.data_ptr()), P(y_host.data_ptr()), P(wsh.data_ptr())

    def step_host(i):
        _, _, dref, gref, uref = pairs[i % N_COPIES]
        return lib.dense_layer_int4_host(gref, uref, dref, xhp, qg.QG_X_BF16, yhp, wshp, wsh_bytes, s)

    for i in range(args.warmup):
        assert step_host(i) == 0
    assert step(0) == 0
    torch.cuda.synchronize()
    assert torch.equal(y_host, y.cpu()), "host-buffer layer differs from the device-buffer layer"
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step_host(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    assert qg.qg_device_status() == 0

    # the same layer steps captured once in a CUDA graph and replayed: the host's per-launch work
    # leaves the loop (reported beside the stream-launched number, not instead of it)
    graph = None
    if rank == 0:
        try:
            cap = torch.cuda.Stream(dev)
            cs = int(cap.cuda_stream)
            n_graph = 16  # layer steps per graph, over rotating weight copies
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(stream)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                for i in range(n_graph):
                    _, _, dref, gref, uref = pairs[i % N_COPIES]
                    rc = lib.dense_layer_int4(gref, uref, dref, xp, qg.QG_X_BF16, yp, wsp, ws_bytes, cs)
                    if rc != 0:
                        raise RuntimeError(f"dense_layer_int4 returned {rc} under capture")
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = max(4, args.steps // n_graph)
            cur = torch.cuda.current_stream(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            for _ in range(reps):
                g.replay()
            e1.record(cur)
            torch.cuda.synchronize()
            g_us = e0.elapsed_time(e1) * 1e3 / (reps * n_graph)
            graph = {"us_per_layer": round(g_us, 3), "GBps": round(B_LAYER / (g_us * 1e-6) / 1e9, 1),
                     "steps_per_graph": n_graph, "replays": reps, "pdl_edges": not args.no_pdl}
            assert qg.qg_device_status() == 0
        except Exception as e:  # noqa: BLE001  (reported, not allowed to drop the line)
            graph = {"error": f"{type(e).__name__}: {e}"}
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
        src = open(os.path.join(ROOT, "moe_int4_affine_gb300", "csrc", "gemv_kernel.cuh"), "rb").read()
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
        "timing": dict(spread, how="median over the repeats of exactly `steps` steps, each between a barrier "
                                   "and a device synchronize, CUDA events on the launching stream"),
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
                "us_per_layer": round(e2e_ms * 1e3, 3), "call": "dense_layer_int4_host",
                "transfer": "x read by a GPU copy kernel from pinned host memory, y written by the "
                            "down kernel into pinned host memory (NVLink-C2C), every step",
                "gpu_launches_per_step": 3},
        "graph": graph,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "configs": configs,
    }
    return line


def measure_configs(qg, I, dev, stream):
    """Every configuration of the workload set, timed back to back with CUDA events on `stream`
    (median of 5 runs of at least 50 calls).  Weights rotate over enough copies to exceed L2 unless noted."""
    import ctypes

    import torch

    P, byref = ctypes.c_void_p, ctypes.byref
    s = int(stream.cuda_stream)
    lib = qg.lib
    peak_hbm, _ = peaks()
    peak_tf = _peak_tflops()
    res = {}

    def tl(fn, n):  # the median of 5 runs of at least 50 back-to-back calls
        n = max(n, 50)
        for i in range(6):
            assert fn(i) == 0
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(5):
            e0.record(stream)
            for i in range(n):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        return statistics.median(ts)

    def copies(w, n):
        return [w] + [qg.Int4Weight(w.packed.clone(), w.scales.clone(), w.biases.clone(), w.out, w.in_dim,
                                    w.n_mat, bits=w.bits) for _ in range(n - 1)]

    def gb(nbytes, us):
        return {"us_per_call": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
                "frac_of_8000": round(nbytes / us / 1e3 / NOMINAL_HBM_GBS, 4),
                "frac_of_measured": round(nbytes / us / 1e3 / peak_hbm, 4), "algorithmic_bytes": nbytes}

    # config 0: 256 x 1024 (150 KB: L2-resident, launch-bound)
    w = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_W, 256, 1024), dev)
    x = qg.to_device(I.bf16_normal(0, I.TID_X, 1024), dev)
    y = torch.empty(256, dtype=torch.float32, device=dev)
    us = tl(lambda i: lib.qgemv_int4(byref(w.struct), P(x.data_ptr()), qg.QG_X_BF16, P(y.data_ptr()), s), 200)
    res["c0_gemv_256x1024"] = dict(gb(weight_bytes(256, 1024) + 2048 + 1024, us), l2="hot (one 150 KB weight)")

    # config 2: shared-input multi-projection GEMVs, in = 2048
    for name, outs, ncp in (("c2_quartet_8192_4096_32_32", (8192, 4096, 32, 32), 12),
                            ("c2_triple_4096_512_512", (4096, 512, 512), 28)):
        mats = [qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_MULTI + j, o, 2048), dev) for j, o in enumerate(outs)]
        sets = [mats] + [[copies(m, 2)[1] for m in mats] for _ in range(ncp - 1)]
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 2048), dev)
        ys = [torch.empty(o, dtype=torch.float32, device=dev) for o in outs]
        args = [((qg.qg_int4_weight * len(outs))(*[m.struct for m in st]), (P * len(outs))(*[t.data_ptr() for t in ys]))
                for st in sets]
        n = len(outs)
        us = tl(lambda i: lib.qgemv_int4_multi(n, args[i % ncp][0], P(x.data_ptr()), qg.QG_X_BF16, args[i % ncp][1],
                                               qg.QG_EPI_NONE, s), 100)
        nbytes = sum(weight_bytes(o, 2048) for o in outs) + 2048 * 2 + 4 * sum(outs)
        res[name] = dict(gb(nbytes, us), l2=f"weights rotate over {ncp} copies")

    # config 3: MoE decode T=1 -- router top-8 of 128, gate/up (SwiGLU) and down + residual, one layer
    E, HID, INTER, K = 128, 2048, 768, 8
    g = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, INTER, HID, n_mat=E), dev)
    u = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, INTER, HID, n_mat=E), dev)
    d = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, HID, INTER, n_mat=E), dev)
    logits = [qg.to_device(I.f32_normal(i, I.TID_LOGITS, E), dev) for i in range(16)]
    x = qg.to_device(I.bf16_normal(0, I.TID_X, HID), dev)
    r = qg.to_device(I.bf16_normal(0, I.TID_RESID, HID), dev)
    idx = torch.empty(K, dtype=torch.int32, device=dev)
    pk = torch.empty(K, dtype=torch.float32, device=dev)
    y = torch.empty(HID, dtype=torch.float32, device=dev)
    wsb = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_MOE, d, K), dtype=torch.uint8, device=dev)

    def moe(i):
        rc = lib.moe_router_topk(P(logits[i % 16].data_ptr()), E, K, 1, P(idx.data_ptr()), P(pk.data_ptr()), s)
        return rc | lib.moe_gather_qgemv_int4(byref(g.struct), byref(u.struct), byref(d.struct), P(idx.data_ptr()),
                                              P(pk.data_ptr()), K, P(x.data_ptr()), P(r.data_ptr()), P(y.data_ptr()),
                                              P(wsb.data_ptr()), wsb.numel(), s)
    us = tl(moe, 100)
    nbytes = K * 3 * weight_bytes(INTER, HID) + 2 * HID * 2 + E * 4 + HID * 4
    l2 = f"128-expert pool ({3 * E * weight_bytes(INTER, HID) / 1e6:.0f} MB), router logits rotate over 16 vectors"
    res["c3_moe_layer_T1"] = dict(gb(nbytes, us), kernels=3, call="moe_router_topk + moe_gather_qgemv_int4", l2=l2)

    def moe_fused(i):
        return lib.moe_layer_int4(P(logits[i % 16].data_ptr()), 1, byref(g.struct), byref(u.struct), byref(d.struct),
                                  K, P(x.data_ptr()), P(r.data_ptr()), P(y.data_ptr()), P(idx.data_ptr()),
                                  P(pk.data_ptr()), P(wsb.data_ptr()), wsb.numel(), s)
    us = tl(moe_fused, 100)
    res["c3_moe_layer_T1_fused_router"] = dict(gb(nbytes, us), kernels=2, call="moe_layer_int4", l2=l2)

    # next row N2: the MoE layer for T tokens (prefill), tokens grouped by expert on the tensor cores
    for T in (32, 256):
        lgT = [qg.to_device(I.f32_normal(i, I.TID_LOGITS, (T, E)), dev) for i in range(4)]
        XT = qg.to_device(I.bf16_normal(0, I.TID_X, (T, HID)), dev)
        RT = qg.to_device(I.bf16_normal(0, I.TID_RESID, (T, HID)), dev)
        YT = torch.empty((T, HID), dtype=torch.float32, device=dev)
        iT = torch.empty((T, K), dtype=torch.int32, device=dev)
        pT = torch.empty((T, K), dtype=torch.float32, device=dev)
        wsT = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_MOE_PREFILL, d, T), dtype=torch.uint8, device=dev)
        us = tl(lambda i: lib.moe_prefill_int4(P(lgT[i % 4].data_ptr()), T, 1, byref(g.struct), byref(u.struct),
                                               byref(d.struct), K, P(XT.data_ptr()), P(RT.data_ptr()),
                                               P(YT.data_ptr()), P(iT.data_ptr()), P(pT.data_ptr()),
                                               P(wsT.data_ptr()), wsT.numel(), s), 20)
        hit = int(torch.unique(iT).numel())  # experts whose weights the last call read
        nbytes = hit * 3 * weight_bytes(INTER, HID) + T * HID * (2 + 2 + 4) + T * E * 4
        tf = 2.0 * T * K * 3 * INTER * HID / us / 1e6
        res[f"n2_moe_prefill_T{T}"] = dict(gb(nbytes, us), call="moe_prefill_int4", launches=7, experts_hit=hit,
                                          TFLOPs=round(tf, 1), l2=f"{hit} experts' weights ({hit * 3 * weight_bytes(INTER, HID) / 1e6:.0f} MB) per call")
        del lgT, XT, RT, YT, iT, pT, wsT
    del g, u, d

    # next rows: the RMSNorm-fused gate/up pair (the FFN input after its norm) against the plain
    # pair, and the shared-expert down projection with the sigmoid gate, routed base and residual
    gw = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_GATE, FFN, HIDDEN), dev)
    uw = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_UP, FFN, HIDDEN), dev)
    pairs_ = [(gw, uw)] + [(copies(gw, 2)[1], copies(uw, 2)[1]) for _ in range(5)]
    x = qg.to_device(I.bf16_normal(0, I.TID_X, HIDDEN), dev)
    gam = qg.to_device(I.bf16_normal(1, I.TID_RESID, HIDDEN), dev)
    h = torch.empty(FFN, dtype=torch.float32, device=dev)
    pargs = [((qg.qg_int4_weight * 2)(a_.struct, b_.struct), (P * 2)(h.data_ptr(), None)) for a_, b_ in pairs_]
    nbytes = 2 * weight_bytes(FFN, HIDDEN) + HIDDEN * 2 + HIDDEN * 2 + FFN * 4
    us = tl(lambda i: lib.rmsnorm_qgemv_int4_multi(2, pargs[i % 6][0], P(x.data_ptr()), qg.QG_X_BF16,
                                                   P(gam.data_ptr()), ctypes.c_float(1e-6), pargs[i % 6][1],
                                                   qg.QG_EPI_SWIGLU, s), 60)
    us0 = tl(lambda i: lib.qgemv_int4_multi(2, pargs[i % 6][0], P(x.data_ptr()), qg.QG_X_BF16, pargs[i % 6][1],
                                            qg.QG_EPI_SWIGLU, s), 60)
    res["n1_rmsnorm_gateup_swiglu_17408x5120"] = dict(gb(nbytes, us), call="rmsnorm_qgemv_int4_multi",
                                                      us_without_norm=round(us0, 3),
                                                      l2="weights rotate over 6 copies (1.2 GB)")
    del gw, uw, pairs_
    SD_OUT, SD_IN = 2048, 768  # shared expert of the MoE config: down 2048 x 768
    sd = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_DOWN, SD_OUT, SD_IN), dev)
    sds = copies(sd, 192)
    hx = qg.to_device(I.f32_normal(0, I.TID_X, SD_IN), dev)
    gate = qg.to_device(np.array([0.3], np.float32), dev)
    base = qg.to_device(I.f32_normal(1, I.TID_X, SD_OUT), dev)
    r = qg.to_device(I.bf16_normal(0, I.TID_RESID, SD_OUT), dev)
    y = torch.empty(SD_OUT, dtype=torch.float32, device=dev)
    us = tl(lambda i: lib.qgemv_int4_sigmoid_fma(byref(sds[i % 192].struct), P(hx.data_ptr()), qg.QG_X_F32,
                                                 P(gate.data_ptr()), P(base.data_ptr()), P(r.data_ptr()),
                                                 P(y.data_ptr()), s), 200)
    nbytes = weight_bytes(SD_OUT, SD_IN) + SD_IN * 4 + 4 + SD_OUT * (4 + 2 + 4)
    res["n1_shared_down_sigmoid_fma_2048x768"] = dict(gb(nbytes, us), call="qgemv_int4_sigmoid_fma",
                                                      l2="weights rotate over 192 copies (170 MB, larger than L2)")

    # ... and the gated RMSNorm before the GDN mixer's out-projection: 32 heads of 128 into 2048
    GN_OUT, GN_IN, GN_HD = 2048, 4096, 128
    gn = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_W, GN_OUT, GN_IN), dev)
    gns = copies(gn, 36)
    gy = qg.to_device(I.bf16_normal(0, I.TID_X, GN_IN), dev)
    gz = qg.to_device(I.bf16_normal(1, I.TID_X, GN_IN), dev)
    gg = qg.to_device(I.bf16_normal(0, I.TID_RESID, GN_IN), dev)
    go = torch.empty(GN_OUT, dtype=torch.float32, device=dev)
    gws = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_GATED_NORM, gn, 0), dtype=torch.uint8, device=dev)
    us = tl(lambda i: lib.gated_rmsnorm_qgemv_int4(byref(gns[i % 36].struct), P(gy.data_ptr()), P(gz.data_ptr()),
                                                   qg.QG_X_BF16, P(gg.data_ptr()), ctypes.c_float(1e-6), GN_HD,
                                                   P(go.data_ptr()), P(gws.data_ptr()), gws.numel(), s), 200)
    nbytes = weight_bytes(GN_OUT, GN_IN) + GN_IN * 2 * 3 + GN_IN * 4 * 2 + GN_OUT * 4
    res["n1_gated_rmsnorm_2048x4096_heads128"] = dict(gb(nbytes, us), call="gated_rmsnorm_qgemv_int4", launches=2,
                                                      l2="weights rotate over 36 copies (170 MB)")
    del gn, gns
    del sd, sds

    # next row N3: the affine encoder over the FFN gate's shape (bf16 weights in, Q4_64A / Q2_64A out)
    wq = [qg.to_device(I.bf16_normal(i, I.TID_W, (FFN, HIDDEN)), dev) for i in range(2)]
    for bits in (4, 2):
        pq = torch.empty((FFN, HIDDEN * bits // 32), dtype=torch.int32, device=dev)
        sq = torch.empty((FFN, HIDDEN // 64), dtype=torch.bfloat16, device=dev)
        bq = torch.empty((FFN, HIDDEN // 64), dtype=torch.bfloat16, device=dev)
        us = tl(lambda i: lib.quantize_affine_q64a(P(wq[i % 2].data_ptr()), qg.QG_X_BF16, FFN, HIDDEN, bits,
                                                   P(pq.data_ptr()), P(sq.data_ptr()), P(bq.data_ptr()), s), 30)
        nbytes = FFN * HIDDEN * 2 + FFN * HIDDEN * bits // 8 + FFN * (HIDDEN // 64) * 4
        res[f"n3_quantize_q{bits}_64a_17408x5120"] = dict(gb(nbytes, us), call="quantize_affine_q64a",
                                                         l2="two 178 MB inputs alternate")
    del wq

    # next row N4: the 2-bit (Q2_64A) GEMV on the decode layer's shapes
    def q2w(seed, tid, out, in_dim):
        d = I.int2_weight(seed, tid, out, in_dim)
        t = lambda a: qg.to_device(a, dev)
        return qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, bits=2)

    def q2bytes(out, in_dim):
        return out * in_dim // 4 + 4 * out * (in_dim // 64)
    dq = q2w(0, I.TID_DOWN, HIDDEN, FFN)
    dqs = copies(dq, 24)
    xb = qg.to_device(I.bf16_normal(0, I.TID_X, FFN), dev)
    yq = torch.empty(HIDDEN, dtype=torch.float32, device=dev)
    us = tl(lambda i: lib.qgemv_q2(byref(dqs[i % 24].struct), P(xb.data_ptr()), qg.QG_X_BF16, P(yq.data_ptr()), s), 100)
    res["n4_q2_gemv_5120x17408"] = dict(gb(q2bytes(HIDDEN, FFN) + FFN * 2 + HIDDEN * 4, us), call="qgemv_q2",
                                        l2="weights rotate over 24 copies (0.6 GB)")
    gq, uq = q2w(0, I.TID_GATE, FFN, HIDDEN), q2w(0, I.TID_UP, FFN, HIDDEN)
    gqs, uqs = copies(gq, 12), copies(uq, 12)
    x = qg.to_device(I.bf16_normal(0, I.TID_X, HIDDEN), dev)
    hq = torch.empty(FFN, dtype=torch.float32, device=dev)
    qargs = [((qg.qg_int4_weight * 2)(a_.struct, b_.struct), (P * 2)(hq.data_ptr(), None)) for a_, b_ in zip(gqs, uqs)]
    us = tl(lambda i: lib.qgemv_q2_multi(2, qargs[i % 12][0], P(x.data_ptr()), qg.QG_X_BF16, qargs[i % 12][1],
                                         qg.QG_EPI_SWIGLU, s), 100)
    res["n4_q2_gateup_swiglu_17408x5120"] = dict(gb(2 * q2bytes(FFN, HIDDEN) + HIDDEN * 2 + FFN * 4, us),
                                                call="qgemv_q2_multi (SwiGLU)", l2="weights rotate over 12 copies")
    del dq, dqs, gq, uq, gqs, uqs
    # ... and the 2-bit MoE layer on the MoE config's shapes (router inside the gate/up kernel)
    E2, H2, I2, K2 = 128, 2048, 768, 8
    def q2stack(tid, out, in_dim):
        d = I.int2_weight(0, tid, out, in_dim, n_mat=E2)
        t = lambda a: qg.to_device(a, dev)
        return qg.Int4Weight(t(d["packed"]), t(d["scales"]), t(d["biases"]), out, in_dim, n_mat=E2, bits=2)
    g2, u2, d2 = q2stack(I.TID_GATE, I2, H2), q2stack(I.TID_UP, I2, H2), q2stack(I.TID_DOWN, H2, I2)
    lg2 = [qg.to_device(I.f32_normal(i, I.TID_LOGITS, E2), dev) for i in range(16)]
    x2 = qg.to_device(I.bf16_normal(0, I.TID_X, H2), dev)
    r2 = qg.to_device(I.bf16_normal(0, I.TID_RESID, H2), dev)
    i2 = torch.empty(K2, dtype=torch.int32, device=dev)
    p2 = torch.empty(K2, dtype=torch.float32, device=dev)
    y2 = torch.empty(H2, dtype=torch.float32, device=dev)
    w2 = torch.empty(qg.qg_workspace_bytes(qg.QG_OP_MOE, d2, K2), dtype=torch.uint8, device=dev)
    us = tl(lambda i: lib.moe_layer_q2(P(lg2[i % 16].data_ptr()), 1, byref(g2.struct), byref(u2.struct),
                                       byref(d2.struct), K2, P(x2.data_ptr()), P(r2.data_ptr()), P(y2.data_ptr()),
                                       P(i2.data_ptr()), P(p2.data_ptr()), P(w2.data_ptr()), w2.numel(), s), 100)
    nb2 = K2 * (2 * q2bytes(I2, H2) + q2bytes(H2, I2)) + 2 * H2 * 2 + E2 * 4 + H2 * 4
    res["n4_q2_moe_layer_T1"] = dict(gb(nb2, us), call="moe_layer_q2", kernels=2,
                                     l2="128-expert 2-bit pool, router logits rotate over 16 vectors")
    del g2, u2, d2

    # config 4: dequant-GEMM, W 17408 x 5120, X T x 5120
    w = qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_W, FFN, HIDDEN), dev)
    ws_ = copies(w, 12)
    for T, tc_min, label in ((8, 9, "gemv_path"), (8, 0, "tensor_core_path"), (32, 0, "tensor_core_path"),
                             (256, 0, "tensor_core_path")):
        qg.qg_tune_qgemm(tc_min)
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, HIDDEN)), dev)
        Y = torch.empty((T, FFN), dtype=torch.float32, device=dev)
        need = qg.qg_workspace_bytes(qg.QG_OP_QGEMM, w, T)
        wsb = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        args = [(byref(c.struct), P(X.data_ptr()), T, P(Y.data_ptr()), P(wsb.data_ptr()), wsb.numel(), s) for c in ws_]
        gemv_path = T < (tc_min or 3)
        us = tl(lambda i: lib.qgemm_int4(*args[i % 12]), 30 if gemv_path else 60)
        nbytes = weight_bytes(FFN, HIDDEN) + T * HIDDEN * 2 + T * FFN * 4
        tf = 2.0 * T * FFN * HIDDEN / us / 1e6
        e = dict(gb(nbytes, us), path=label, TFLOPs=round(tf, 1), frac_of_tensor_peak=round(tf / peak_tf, 4),
                 launches=(T if gemv_path else 2))
        res[f"c4_qgemm_T{T}_{label}"] = e
    qg.qg_tune_qgemm(0)

    # next row N2: the prefill form of the shared-input quartet (in 2048), one launch for all four
    # projections against one qgemm_int4 call each
    outs = (8192, 4096, 32, 32)
    mats = [qg.Int4Weight.from_numpy(I.int4_weight(0, I.TID_MULTI + j, o, 2048), dev) for j, o in enumerate(outs)]
    sets = [mats] + [[copies(m, 2)[1] for m in mats] for _ in range(11)]
    for T in (32, 256):
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, 2048)), dev)
        Ys = [torch.empty((T, o), dtype=torch.float32, device=dev) for o in outs]
        need = qg.qg_workspace_bytes(qg.QG_OP_QGEMM, mats[0], T)
        wsb = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        margs = [((qg.qg_int4_weight * 4)(*[m.struct for m in st]), (P * 4)(*[t.data_ptr() for t in Ys])) for st in sets]
        us = tl(lambda i: lib.qgemm_int4_multi(4, margs[i % 12][0], P(X.data_ptr()), T, margs[i % 12][1],
                                               P(wsb.data_ptr()), wsb.numel(), s), 60)

        def separate(i):
            rc = 0
            for j in range(4):
                rc |= lib.qgemm_int4(byref(sets[i % 12][j].struct), P(X.data_ptr()), T, P(Ys[j].data_ptr()),
                                     P(wsb.data_ptr()), wsb.numel(), s)
            return rc
        us_sep = tl(separate, 30)
        nbytes = sum(weight_bytes(o, 2048) for o in outs) + T * 2048 * 2 + T * 4 * sum(outs)
        tf = 2.0 * T * sum(outs) * 2048 / us / 1e6
        res[f"n2_qgemm_multi_quartet_T{T}"] = dict(gb(nbytes, us), call="qgemm_int4_multi", TFLOPs=round(tf, 1),
                                                   us_separate_calls=round(us_sep, 3), launches=2,
                                                   l2="weights rotate over 12 copies")
    assert qg.qg_device_status() == 0
    return res


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


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


def oracle_config_times(threads: int, rows_per_sample: int = 192):
    """The fp64 oracle timed per configuration, single-threaded and on `threads` host threads: a
    sample of rows of each matrix (the oracle's cost per row depends only on the row length), scaled
    to the call's rows; the MoE step (8 of 128 experts) in full, single-threaded (the oracle's MoE
    routine is single-threaded).  Returns {config: {"ms_1": .., "ms_n": .., "threads": n, ...}}."""
    import oracle
    from moe_int4_affine_gb300 import inputs as I

    rows_n = max(rows_per_sample, 64 * threads)  # (enough rows per thread for the split to pay)

    def per_row(in_dim, T=1):
        w = I.int4_weight(7, I.TID_W, rows_n, in_dim)
        X = I.bf16_normal(7, I.TID_X, (T, in_dim))
        out = {}
        for n, rows in ((1, rows_per_sample), (threads, rows_n)):
            t0 = time.perf_counter()
            if T == 1:
                oracle.qgemv(w["packed"], w["scales"], w["biases"], X[0], rows=(0, rows), threads=n)
            else:
                oracle.qgemm(w["packed"], w["scales"], w["biases"], X, rows=(0, rows), threads=n)
            out[n] = (time.perf_counter() - t0) / rows
        return out

    res = {}
    cache = {}

    def call(name, mats, T=1):  # mats: [(out, in)]
        ms = {1: 0.0, threads: 0.0}
        for o, i in mats:
            key = (i, T)
            if key not in cache:
                cache[key] = per_row(i, T)
            for n in ms:
                ms[n] += cache[key][n] * o * 1e3
        res[name] = {"ms_1": round(ms[1], 3), "ms_n": round(ms[threads], 3), "threads": threads,
                     "sample": f"{rows_per_sample} (one thread) or {rows_n} ({threads} threads) rows of each "
                               f"row length, scaled to the call's rows"}

    call("c0_gemv_256x1024", [(256, 1024)])
    call("c1_gemv_gate_up_17408x5120", [(17408, 5120), (17408, 5120)])
    call("c1_gemv_down_5120x17408", [(5120, 17408)])
    call("c1_decode_layer", [(17408, 5120), (17408, 5120), (5120, 17408)])
    call("c2_quartet_8192_4096_32_32", [(8192, 2048), (4096, 2048), (32, 2048), (32, 2048)])
    call("c2_triple_4096_512_512", [(4096, 2048), (512, 2048), (512, 2048)])
    for T in (8, 32, 256):
        call(f"c4_qgemm_T{T}", [(17408, 5120)], T)
    # MoE T = 1: router + 8 experts' gate/up and down (hidden 2048, intermediate 768), in full
    E, HID, INTER = 8, 2048, 768  # the 8 selected of the 128: the oracle reads only those
    g = I.int4_weight(0, I.TID_GATE, INTER, HID, n_mat=E)
    u = I.int4_weight(0, I.TID_UP, INTER, HID, n_mat=E)
    d = I.int4_weight(0, I.TID_DOWN, HID, INTER, n_mat=E)
    x = I.bf16_normal(0, I.TID_X, HID)
    r = I.bf16_normal(0, I.TID_RESID, HID)
    logits = I.f32_normal(0, I.TID_LOGITS, 128)
    t0 = time.perf_counter()
    idx, pr = oracle.router_topk(logits, 8)
    oracle.moe(tuple(g[k] for k in ("packed", "scales", "biases")), tuple(u[k] for k in ("packed", "scales", "biases")),
               tuple(d[k] for k in ("packed", "scales", "biases")), np.arange(8, dtype=np.uint32), pr, x, r)
    res["c3_moe_layer_T1"] = {"ms_1": round((time.perf_counter() - t0) * 1e3, 3), "threads": 1,
                              "sample": "the full step (router + 8 experts), single-threaded"}
    return res


def cpu_baseline(target_s: float = 12.0):
    """The oracle on whole-layer row samples, repeated until about target_s seconds of CPU work."""
    threads = os.cpu_count() or 1
    dt, nb = oracle_layer_sample(0.002, threads)  # calibration
    frac = min(1.0, 0.002 * target_s / max(dt, 1e-3))
    reps = 1
    if frac >= 1.0:
        dt1, _ = oracle_layer_sample(1.0, threads)
        reps = max(1, int(target_s / max(dt1, 1e-3)))
    tot_t, tot_b = 0.0, 0
    for _ in range(reps):
        dt, nb = oracle_layer_sample(frac, threads)
        tot_t += dt
        tot_b += nb
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} x the first {frac:.4f} of the rows of gate, up and down ({tot_b / 1e6:.1f} MB), "
                      f"fp64 C oracle, {threads} host threads, {tot_t:.1f} s"}


def run_reference(args, world=1):
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
            "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "dense decode layer M=1: gate+up 17408x5120 -> down 5120x17408 (row sample)",
                       "sample_fraction": round(frac, 5)},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {frac:.4f} of each matrix's rows per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(case: str, T: int, bits: int, kind: str) -> int:
    """Small fixed invocations of the library's kernels for profilers (ncu): a case builds its seeded
    synthetic inputs (a few hundred MB at most on the device), runs its calls three times and prints
    "ok <device status>".  Nothing is timed.  Cases: layer (gate/up SwiGLU pair + down, 17408 x
    5120), down_bf16 (the M = 1 GEMV 5120 x 17408, bf16 x), moe (router + MoE gather, 128 experts,
    top 8), moe_layer (the same through moe_layer_int4), qgemm (17408 x 5120, T tokens), quant
    (encode 17408 x 5120 weights of `kind` to `bits`), moe_prefill (128 experts, top 8, T tokens)."""
    import torch

    from moe_int4_affine_gb300 import build

    build.build()
    from moe_int4_affine_gb300 import inputs as I
    from moe_int4_affine_gb300 import qg

    qg.qg_set_pdl(True)
    reps = 3
    W = lambda seed, tid, out, in_dim, n_mat=None: qg.Int4Weight.from_numpy(  # noqa: E731
        I.int4_weight(seed, tid, out, in_dim, n_mat=n_mat))
    if case == "layer":
        g, u, d = W(0, I.TID_GATE, 17408, 5120), W(0, I.TID_UP, 17408, 5120), W(0, I.TID_DOWN, 5120, 17408)
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 5120))
        for _ in range(reps):
            qg.dense_layer_int4(g, u, d, x)
    elif case == "down_bf16":
        d = W(0, I.TID_DOWN, 5120, 17408)
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 17408))
        y = torch.empty(5120, device="cuda")
        for _ in range(reps):
            qg.qgemv_int4(d, x, y)
    elif case in ("moe", "moe_layer"):
        g, u = W(0, I.TID_GATE, 768, 2048, 128), W(0, I.TID_UP, 768, 2048, 128)
        d = W(0, I.TID_DOWN, 2048, 768, 128)
        x = qg.to_device(I.bf16_normal(0, I.TID_X, 2048))
        r = qg.to_device(I.bf16_normal(0, I.TID_RESID, 2048))
        for i in range(reps):
            logits = qg.to_device(I.f32_normal(i, I.TID_LOGITS, 128))
            if case == "moe":
                idx, p = qg.moe_router_topk(logits, k=8)
                qg.moe_gather_qgemv_int4(g, u, d, idx, p, x, r)
            else:
                qg.moe_layer_int4(logits, g, u, d, x, r, k=8)
    elif case == "qgemm":
        w = W(0, I.TID_W, 17408, 5120)
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, 5120)))
        for _ in range(reps):
            qg.qgemm_int4(w, X)
    elif case == "quant":
        shape = (17408, 5120)
        w = qg.to_device(I.bf16_normal(0, I.TID_W, shape) if kind == "bf16" else I.f32_normal(0, I.TID_W, shape))
        for _ in range(reps):
            qg.quantize_affine_q64a(w, bits)
    elif case == "moe_prefill":
        g, u = W(0, I.TID_GATE, 768, 2048, 128), W(0, I.TID_UP, 768, 2048, 128)
        d = W(0, I.TID_DOWN, 2048, 768, 128)
        X = qg.to_device(I.bf16_normal(0, I.TID_X, (T, 2048)))
        r = qg.to_device(I.bf16_normal(0, I.TID_RESID, (T, 2048)))
        for i in range(reps):
            qg.moe_prefill_int4(qg.to_device(I.f32_normal(i, I.TID_LOGITS, (T, 128))), g, u, d, X, r, k=8)
    else:
        print(f"unknown case {case!r}", file=sys.stderr)
        return 2
    torch.cuda.synchronize()
    status = qg.qg_device_status()
    print("ok", status)
    return 0 if status == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qg", choices=["qg", "reference"])
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed steps under the clock sampler")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration section")
    ap.add_argument("--case", default=None, help="run one fixed, untimed invocation for a profiler (see run_case)")
    ap.add_argument("--T", type=int, default=256, help="--case qgemm / moe_prefill: tokens")
    ap.add_argument("--bits", type=int, default=4, help="--case quant: code width")
    ap.add_argument("--kind", default="bf16", choices=["bf16", "f32"], help="--case quant: weight type")
    args = ap.parse_args(argv)
    if args.case:
        return run_case(args.case, args.T, args.bits, args.kind)
    args.warmup = max(3, args.warmup)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist

        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(run_reference(args, world)), flush=True)
            return 0
        line = run_qg(args, rank, world, local_rank)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
                try:  # (a reported baseline: a failure here must not drop the line)
                    line["cpu_baseline"]["per_config"] = oracle_config_times(os.cpu_count() or 1)
                except Exception as e:  # noqa: BLE001
                    line["cpu_baseline"]["per_config"] = {"error": f"{type(e).__name__}: {e}"}
            print(json.dumps(line), flush=True)
        return 0
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
