"""Benchmark: one Qwen3-32B-shaped decoder layer, forward + backward, bf16,
on one GB300 (batch 1 x seq 2048, hidden 5120, 64 query / 8 KV heads of dim
128, SwiGLU intermediate 25600, RoPE base 1e6, causal). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one kl_layer_forward + kl_layer_backward over the whole batch.
`value` is whole-job tokens/s with inputs resident in HBM; `e2e` is the same
metric through the C ABI with pinned host buffers (H2D of X and dY and D2H of
dX inside the timed region). The weights (975 MB) exceed L2 (129 MB), so no
flush is needed between steps. N > 1 runs N independent replicas (weak
scaling; the path needs no collective). `--impl reference` times the fp64
CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(B=1, S=2048, H=5120, Hq=64, Hkv=8, d=128, I=25600, eps=1e-6, rope_base=1e6)
METRIC = "layer fwd+bwd tokens/s (Qwen3-32B dims, bf16, 1 GB300); % of tensor-core peak"
CONFIG = {"workload": "qwen3_32b_layer_fwd_bwd", "batch": 1, "seq_len": 2048, "hidden": 5120,
          "heads_q": 64, "heads_kv": 8, "head_dim": 128, "intermediate": 25600, "rope_base": 1e6,
          "causal": True, "l2": "inputs larger than L2 (975 MB of weights per step)"}
CPU_SAMPLE_S = 1024  # tokens per oracle step (full layer dims)


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


class Clocks:
    """nvidia-smi sampler for the timed region (every 200 ms)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def build_inputs(torch, K, L, synth, device, seed=0):
    cfg = L.make_cfg(**WORKLOAD, dtype=K.KL_BF16)
    w = {}
    for n, shp in L.weight_shapes(cfg).items():
        if n.startswith("gamma"):
            w[n] = synth.device_normal(shp, 0.02, 1.0, seed, f"layer0.{n}", torch.bfloat16, device)
        else:
            w[n] = synth.device_normal(shp, 0.02, 0.0, seed, f"layer0.{n}", torch.bfloat16, device)
    T = WORKLOAD["B"] * WORKLOAD["S"]
    X = synth.device_normal((T, WORKLOAD["H"]), 1.0, 0.0, seed, "X", torch.bfloat16, device)
    dY = synth.device_normal((T, WORKLOAD["H"]), 1.0, 0.0, seed, "dY", torch.bfloat16, device)
    return cfg, w, X, dY


def read_profile(K):
    lib = K.load()

    class Entry(ctypes.Structure):
        _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("ms", ctypes.c_double),
                    ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]

    arr = (Entry * 64)()
    lib.kl_profile_read.restype = ctypes.c_int32
    lib.kl_profile_read.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    n = lib.kl_profile_read(ctypes.cast(arr, ctypes.c_void_p), 64)
    out = {}
    for i in range(max(n, 0)):
        e = arr[i]
        out[e.name.decode()] = {"launches": e.launches, "ms": e.ms, "flops": e.flops, "bytes": e.bytes}
    return out


def bench_ours(args, rank, world, local_rank, dist):
    import torch

    import bwd_qwen3_layer_gb300 as K
    from bwd_qwen3_layer_gb300 import layer as L
    from bwd_qwen3_layer_gb300 import synth

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    lib = K.load()
    lib.kl_profile_enable.argtypes = [ctypes.c_int32]
    lib.kl_launch_count.restype = ctypes.c_uint64
    cfg, w, X, dY = build_inputs(torch, K, L, synth, device, seed=rank)
    T = WORKLOAD["B"] * WORKLOAD["S"]
    buf = L.LayerBuffers(cfg, device)
    ws = L.weights_struct(w)
    grads, gst = L.alloc_grads(cfg, device, K.KL_BF16)
    Y = torch.empty_like(X)
    dX = torch.empty_like(X)
    stream = torch.cuda.current_stream(device)

    def step(x_ptr, dy_ptr, dx_ptr):
        K.kl_layer_forward(cfg, ws, x_ptr, Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(), buf.fwd_ws.numel(),
                           stream)
        K.kl_layer_backward(cfg, ws, buf.saved, dy_ptr, dx_ptr, gst, buf.bwd_ws.data_ptr(), buf.bwd_ws.numel(),
                            stream)

    for _ in range(args.warmup):
        step(X.data_ptr(), dY.data_ptr(), dX.data_ptr())
    torch.cuda.synchronize()
    K.kl_device_status(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timed region (profiler on: per-kernel events) ----
    clocks = Clocks(local_rank)
    barrier()
    clocks.start()
    time.sleep(0.25)
    lib.kl_profile_enable(1)
    n0 = lib.kl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(X.data_ptr(), dY.data_ptr(), dX.data_ptr())
    e1.record(stream)
    barrier()
    launches = lib.kl_launch_count() - n0
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    prof = read_profile(K)
    lib.kl_profile_enable(0)

    # ---- end-to-end through the C ABI with pinned host buffers ----
    hX = X.cpu().pin_memory()
    hdY = dY.cpu().pin_memory()
    hdX = torch.empty_like(hX).pin_memory()
    dX2, X2, dY2 = torch.empty_like(X), torch.empty_like(X), torch.empty_like(X)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        X2.copy_(hX, non_blocking=True)
        dY2.copy_(hdY, non_blocking=True)
        step(X2.data_ptr(), dY2.data_ptr(), dX2.data_ptr())
        hdX.copy_(dX2, non_blocking=True)
    f1.record(stream)
    barrier()
    ms_e2e = f0.elapsed_time(f1)
    K.kl_device_status(stream)

    if dist is not None:
        t = torch.tensor([ms, ms_e2e], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, ms_e2e = float(t[0]), float(t[1])
    return dict(ms=ms, ms_e2e=ms_e2e, prof=prof, clocks=clk, launches=int(launches), T=T,
                h2d=2 * X.numel() * X.element_size(), d2h=dX.numel() * dX.element_size())


def oracle_sample(steps: int):
    """Times the fp64 oracle's layer forward+backward at full layer dims on a
    bounded token sample. Returns (tokens_per_s, seconds, cores, description)."""
    import numpy as np

    import oracle as O

    S = CPU_SAMPLE_S
    W = WORKLOAD
    cfg = O.LayerConfig(B=1, S=S, H=W["H"], Hq=W["Hq"], Hkv=W["Hkv"], d=W["d"], I=W["I"],
                        eps=W["eps"], rope_base=W["rope_base"])
    rng = np.random.default_rng(0)
    Dq, Dkv = W["Hq"] * W["d"], W["Hkv"] * W["d"]
    w = {"gamma1": 1 + 0.02 * rng.standard_normal(W["H"]), "Wq": 0.02 * rng.standard_normal((Dq, W["H"])),
         "Wk": 0.02 * rng.standard_normal((Dkv, W["H"])), "Wv": 0.02 * rng.standard_normal((Dkv, W["H"])),
         "Wo": 0.02 * rng.standard_normal((W["H"], Dq)), "gamma2": 1 + 0.02 * rng.standard_normal(W["H"]),
         "Wg": 0.02 * rng.standard_normal((W["I"], W["H"])), "Wu": 0.02 * rng.standard_normal((W["I"], W["H"])),
         "Wd": 0.02 * rng.standard_normal((W["H"], W["I"]))}
    X = rng.standard_normal((S, W["H"]))
    dY = rng.standard_normal((S, W["H"]))
    times = []
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        Y, saved = O.layer_forward(cfg, w, X)
        O.layer_backward(cfg, w, saved, dY)
        times.append(time.perf_counter() - t0)
    sec = statistics.median(times)
    cores = os.cpu_count()
    desc = (f"fp64 numpy oracle, one full-dims layer fwd+bwd on {S} tokens (batch 1, seq {S}) per step, "
            f"median of {len(times)}; BLAS threads default to all {cores} host cores")
    return S / sec, sec, cores, desc


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        if rank != 0:
            return
        steps = max(1, min(args.steps, 3))
        for _ in range(min(args.warmup, 1)):
            pass
        tps, sec, cores, desc = oracle_sample(steps)
        line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
                "warmup": 0, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": CONFIG, "impl": "reference",
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod
    r = bench_ours(args, rank, world, local_rank, dist)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    pk = peaks()
    tokens = r["T"] * args.steps * world
    value = tokens / (r["ms"] / 1e3)
    e2e = tokens / (r["ms_e2e"] / 1e3)
    kernels = {}
    for name, e in sorted(r["prof"].items(), key=lambda kv: -kv[1]["ms"]):
        per = e["ms"] / e["launches"] / 1e3
        ent = {"launches": e["launches"], "ms_per_launch": round(e["ms"] / e["launches"], 4),
               "share": round(e["ms"] / sum(v["ms"] for v in r["prof"].values()), 4)}
        if e["flops"] > 0:
            a = e["flops"] / e["launches"] / per / 1e12
            ent.update(achieved=round(a, 2), unit="TFLOP/s", frac=round(a / pk["bf16_tflops_sustained"], 4))
        else:
            a = e["bytes"] / e["launches"] / per / 1e9
            ent.update(achieved=round(a, 1), unit="GB/s", frac=round(a / pk["hbm_gbs"], 4))
        kernels[name] = ent
    dom = max(r["prof"].items(), key=lambda kv: kv[1]["ms"])
    dname, d = dom
    per = d["ms"] / d["launches"] / 1e3
    if d["flops"] > 0:
        ach = d["flops"] / d["launches"] / per / 1e12
        roof = {"kernel": dname, "bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops_sustained"], 4), "traffic": None,
                "peak_src": f"{pk['src']} bf16_tflops_sustained"}
    else:
        ach = d["bytes"] / d["launches"] / per / 1e9
        roof = {"kernel": dname, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": None,
                "peak_src": f"{pk['src']} hbm_gbs"}
    total_flops = sum(e["flops"] for e in r["prof"].values()) / args.steps
    agg_tflops = total_flops / (r["ms"] / args.steps / 1e3) / 1e12
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["ms"] / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": CONFIG | {"parallelism": f"replicas x{world}"},
            "tensor_frac_aggregate": round(agg_tflops / pk["bf16_tflops_sustained"], 4),
            "aggregate_tflops": round(agg_tflops, 2),
            "roofline": roof, "kernels": kernels, "gpu_launches": r["launches"], "clocks": r["clocks"],
            "e2e": {"value": round(e2e, 1), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]}}
    if world == 1 and not args.no_cpu_baseline:
        tps, sec, cores, desc = oracle_sample(1)
        line["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
