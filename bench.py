"""Benchmark of the GB300 Qwen3 layer path. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload layer|attention|lmhead|stream|stream_recompute|stream_fwd64|decode]

Workloads (Qwen3-32B dims: hidden 5120, 64 query / 8 KV heads of dim 128,
SwiGLU intermediate 25600, RoPE base 1e6, causal; bf16):
  layer      (default) one decoder layer forward + backward, batch 1 x seq 2048;
             a step is kl_layer_forward + kl_layer_backward
  attention  causal GQA attention forward + backward, batch 1 x seq 32768
  lmhead     lm-head logits + single-launch CE/argmax + dX/dW, 4096 tokens,
             vocab 151936
  stream     8 layers streamed from pinned host memory, batch 2 x seq 4096,
             lm-head CE, backward, global-norm clip at 1.0, gradients to
             device memory (one kl_stream_run per step)
  stream_recompute
             the same step keeping only each layer's input between forward
             and backward (the layer's forward runs again before its backward)
  stream_fwd64
             64 layers forward only (kl_stream_forward), batch 1 x seq 2048,
             weights streamed from pinned host memory; reports the driver's
             device memory (independent of depth)
  decode     one layer's forward for one new token of each of 64 sequences
             whose keys and values (context 4096) sit in a paged cache
             (kl_layer_forward_paged, block size 16, blocks shuffled over
             the pool); bound by HBM: the layer's weights and the context's
             keys and values are read once per step
The stream workloads also time the same call with every layer's weights
already in device memory ("bulk": no uploads) to show how much of the host
link the compute hides.

`value` is whole-job tokens/s with inputs resident in HBM; `e2e` is the same
metric through the C ABI with each step's inputs copied from pinned host
memory and its result read back inside the timed region, the copies of step
k+1 (in) and k-1 (out) running on a copy stream while step k computes, as a
training or serving loop feeds the GPU (the stream workloads' driver reads its
results back inside the step, so there the copies stay in line). The per-kernel
region and the e2e region each start after 2 s of idle, so all three short
regions are timed from the same (burst) state of the board's power average.
The default layer run adds `later_region`: the same step timed over one second
after the other regions, when the board has reached its power limit. Every workload's
inputs exceed L2 (129 MB), so no flush is needed between steps. N > 1 runs N
independent replicas (weak scaling; the path needs no collective).
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

QWEN = dict(H=5120, Hq=64, Hkv=8, d=128, I=25600, eps=1e-6, rope_base=1e6)
METRIC = "layer fwd+bwd tokens/s (Qwen3-32B dims, bf16, 1 GB300); % of tensor-core peak"
WORKLOADS = {
    "layer": dict(B=1, S=2048, desc="qwen3_32b_layer_fwd_bwd"),
    "attention": dict(B=1, S=32768, desc="gqa_attention_fwd_bwd_S32768"),
    "lmhead": dict(N=4096, V=151936, desc="lmhead_ce_argmax_fwd_bwd_N4096_V151936"),
    "stream": dict(B=2, S=4096, L=8, V=151936, clip=1.0, mode=0, desc="stream_8_layers_T8192_ce_clip"),
    "stream_recompute": dict(B=2, S=4096, L=8, V=151936, clip=1.0, mode=1,
                             desc="stream_8_layers_T8192_ce_clip_recompute"),
    "stream_fwd64": dict(B=1, S=2048, L=64, distinct=4, mode=2, desc="stream_forward_64_layers_T2048"),
    "decode": dict(B=64, ctx=4096, block=16, desc="decode_layer_B64_ctx4096_paged"),
}
METRICS = {
    "layer": METRIC,
    "attention": "causal GQA attention fwd+bwd tokens/s (seq 32768, 64/8 heads, d 128, bf16, 1 GB300)",
    "lmhead": "lm-head CE+argmax fwd+bwd tokens/s (4096 tokens, vocab 151936, bf16, 1 GB300)",
    "stream": "8-layer streamed training step tokens/s (batch 2 x 4096, bf16, 1 GB300)",
    "stream_recompute": "8-layer streamed training step with activation recompute tokens/s (batch 2 x 4096, bf16, "
                        "1 GB300)",
    "stream_fwd64": "64-layer streamed forward tokens/s (batch 1 x 2048, bf16, 1 GB300)",
    "decode": "one-layer decode tokens/s, paged KV cache (64 sequences x context 4096, Qwen3-32B dims, bf16, 1 GB300)",
}


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


def traffic_record(workload, group):
    """DRAM bytes per launch of a kernel group on a workload, from a committed
    ncu capture (profiles/traffic.json), or None when there is no record or the
    source file of the kernel has changed since the counters were taken."""
    try:
        import hashlib

        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)["records"]
        for rec in recs:
            if rec["workload"] != workload or rec["group"] != group:
                continue
            with open(os.path.join(ROOT, rec["source"]), "rb") as f:
                digest = hashlib.sha256(f.read()).hexdigest()
            return rec["bytes_per_launch"] if digest == rec["source_sha256"] else None
    except Exception:
        return None
    return None


class Clocks:
    """nvidia-smi sampler (every 20 ms, read-only query). mark() brackets the
    timed region by wall clock; stop() reports the samples taken inside it."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.f = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    @staticmethod
    def _stamp(text):
        """nvidia-smi's local-time stamp 'YYYY/MM/DD HH:MM:SS.mmm' as epoch seconds."""
        try:
            whole, _, frac = text.strip().partition(".")
            return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
        except ValueError:
            return None

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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 10:
                continue
            try:
                parsed.append((self._stamp(r[0]), float(r[2]), float(r[3]),
                               [n for n, v in zip(names, r[6:10]) if v.lower().startswith("active")]))
            except ValueError:
                continue
        inside = [p for p in parsed if p[0] is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.01 <= p[0] <= self.t1 + 0.01]
        use = inside or parsed            # a region shorter than one period: every sample
        sm = [p[1] for p in use]
        reasons = sorted({n for p in use for n in p[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": use[-1][2] if use else None,
                "reasons": reasons, "samples": len(sm), "samples_in_timed_region": len(inside),
                "period_ms": self.PERIOD_MS}


def read_profile(K):
    lib = K.load()

    class Entry(ctypes.Structure):
        _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("ms", ctypes.c_double),
                    ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]

    arr = (Entry * 64)()
    n = lib.kl_profile_read(ctypes.cast(arr, ctypes.c_void_p), 64)
    out = {}
    for i in range(max(n, 0)):
        e = arr[i]
        out[e.name.decode()] = {"launches": e.launches, "ms": e.ms, "flops": e.flops, "bytes": e.bytes}
    return out


# ----------------------------------------------------------------------------
# workloads: each returns (units_per_step, step(), e2e_step(), h2d, d2h, config)
# ----------------------------------------------------------------------------

class PipelinedIO:
    """The end-to-end step as a training or serving loop runs it: step k's
    inputs go up from pinned host memory on a copy stream while step k-1
    computes, and step k's result comes down while step k+1 computes (two
    device copies of every buffer the copies touch). begin() issues the first
    upload and end() joins the copy stream, so every copy of the timed steps
    lies inside the timed region; the bytes moved per step are unchanged."""

    def __init__(self, torch, device, stream, ins, outs, run):
        self.torch, self.main = torch, stream
        self.cs = torch.cuda.Stream(device)
        self.hin = [h for h, _ in ins]
        self.hout = [h for _, h in outs]
        self.din = [[torch.empty_like(d) for _, d in ins] for _ in range(2)]
        self.dout = [[torch.empty_like(d) for d, _ in outs] for _ in range(2)]
        self.run = run
        mk = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_done, self.ev_out = mk(), mk(), mk()
        self.k = self.steps = 0

    def _upload(self, k):
        b = k % 2
        with self.torch.cuda.stream(self.cs):
            if k >= 2:
                self.cs.wait_event(self.ev_done[b])      # step k-2 has finished reading these buffers
            for d, h in zip(self.din[b], self.hin):
                d.copy_(h, non_blocking=True)
            self.ev_in[b].record(self.cs)

    def begin(self, steps):
        self.k, self.steps = 0, steps
        self.cs.wait_stream(self.main)
        self._upload(0)

    def __call__(self):
        k, b = self.k, self.k % 2
        self.main.wait_event(self.ev_in[b])
        if k >= 2:
            self.main.wait_event(self.ev_out[b])          # step k-2's result has left these buffers
        self.run(self.din[b], self.dout[b])
        self.ev_done[b].record(self.main)
        if k + 1 < self.steps:
            self._upload(k + 1)
        with self.torch.cuda.stream(self.cs):
            self.cs.wait_event(self.ev_done[b])
            for h, d in zip(self.hout, self.dout[b]):
                h.copy_(d, non_blocking=True)
            self.ev_out[b].record(self.cs)
        self.k += 1

    def end(self):
        self.main.wait_stream(self.cs)


def setup_layer(torch, K, L, synth, device, seed):
    wl = WORKLOADS["layer"]
    cfg = L.make_cfg(wl["B"], wl["S"], **QWEN, dtype=K.KL_BF16)
    w = {}
    for n, shp in L.weight_shapes(cfg).items():
        w[n] = synth.device_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, seed, f"layer0.{n}",
                                   torch.bfloat16, device)
    T = wl["B"] * wl["S"]
    X = synth.device_normal((T, QWEN["H"]), 1.0, 0.0, seed, "X", torch.bfloat16, device)
    dY = synth.device_normal((T, QWEN["H"]), 1.0, 0.0, seed, "dY", torch.bfloat16, device)
    buf = L.LayerBuffers(cfg, device)
    ws = L.weights_struct(w)
    grads, gst = L.alloc_grads(cfg, device, K.KL_BF16)
    Y, dX = torch.empty_like(X), torch.empty_like(X)
    stream = torch.cuda.current_stream(device)

    def run(x, dy, dx):
        K.kl_layer_forward(cfg, ws, x.data_ptr(), Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(),
                           buf.fwd_ws.numel(), stream)
        K.kl_layer_backward(cfg, ws, buf.saved, dy.data_ptr(), dx.data_ptr(), gst, buf.bwd_ws.data_ptr(),
                            buf.bwd_ws.numel(), stream)

    hX, hdY = X.cpu().pin_memory(), dY.cpu().pin_memory()
    hdX = torch.empty_like(hX).pin_memory()
    e2e = PipelinedIO(torch, device, stream, [(hX, X), (hdY, dY)], [(dX, hdX)],
                      lambda i, o: run(i[0], i[1], o[0]))
    keep = (w, buf, grads, X, dY, Y, dX, hX, hdY, hdX)
    cfgd = {"workload": wl["desc"], "batch": wl["B"], "seq_len": wl["S"], "hidden": QWEN["H"],
            "heads_q": QWEN["Hq"], "heads_kv": QWEN["Hkv"], "head_dim": QWEN["d"], "intermediate": QWEN["I"],
            "rope_base": QWEN["rope_base"], "causal": True,
            "l2": "inputs larger than L2 (975 MB of weights per step)"}
    return T, (lambda: run(X, dY, dX)), e2e, 2 * X.numel() * 2, X.numel() * 2, cfgd, keep


def setup_attention(torch, K, L, synth, device, seed):
    wl = WORKLOADS["attention"]
    B, S, Hq, Hkv, d = wl["B"], wl["S"], QWEN["Hq"], QWEN["Hkv"], QWEN["d"]
    T = B * S
    bf = torch.bfloat16
    q = synth.device_normal((T, Hq * d), 1.0, 0.0, seed, "att.q", bf, device)
    k = synth.device_normal((T, Hkv * d), 1.0, 0.0, seed, "att.k", bf, device)
    v = synth.device_normal((T, Hkv * d), 1.0, 0.0, seed, "att.v", bf, device)
    do = synth.device_normal((T, Hq * d), 1.0, 0.0, seed, "att.do", bf, device)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(K.kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def run(qq, kk, vv, dd, dqo=dq):
        K.kl_attention_fwd(B, S, Hq, Hkv, d, K.KL_BF16, qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), stream)
        K.kl_attention_bwd(B, S, Hq, Hkv, d, K.KL_BF16, qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), dd.data_ptr(), dqo.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                           ws.numel(), stream)

    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, do))
    hdq = torch.empty_like(hq).pin_memory()
    e2e = PipelinedIO(torch, device, stream, [(hq, q), (hk, k), (hv, v), (hdo, do)], [(dq, hdq)],
                      lambda i, o_: run(*i, dqo=o_[0]))
    keep = (q, k, v, do, o, lse, dq, dk, dv, ws, hq, hk, hv, hdo, hdq)
    cfgd = {"workload": wl["desc"], "batch": B, "seq_len": S, "heads_q": Hq, "heads_kv": Hkv, "head_dim": d,
            "causal": True, "l2": "inputs larger than L2 (Q/K/V/dO 1.2 GB)"}
    h2d = sum(t.numel() * 2 for t in (q, k, v, do))
    return T, (lambda: run(q, k, v, do)), e2e, h2d, dq.numel() * 2, cfgd, keep


def setup_lmhead(torch, K, L, synth, device, seed):
    wl = WORKLOADS["lmhead"]
    N, V, H = wl["N"], wl["V"], QWEN["H"]
    bf = torch.bfloat16
    X = synth.device_normal((N, H), 1.0, 0.0, seed, "lm.X", bf, device)
    W = synth.device_normal((V, H), 0.02, 0.0, seed, "lm.W", bf, device)
    tgt = synth.device_randint((N,), V, seed, "lm.targets", device)
    cfg = L.lmhead_cfg(N, H, V, K.KL_BF16)
    loss = torch.zeros(1, dtype=torch.float32, device=device)
    arg = torch.empty(N, dtype=torch.int32, device=device)
    dX = torch.empty_like(X)
    dW = torch.empty_like(W)
    ws = L.lmhead_ws(cfg, device)
    stream = torch.cuda.current_stream(device)

    def run(x, t, lo=loss):
        K.kl_lmhead_ce_argmax(cfg, x.data_ptr(), W.data_ptr(), t.data_ptr(), lo.data_ptr(), arg.data_ptr(), 0,
                              dX.data_ptr(), dW.data_ptr(), ws.data_ptr(), ws.numel(), stream)

    hX, ht = X.cpu().pin_memory(), tgt.cpu().pin_memory()
    hloss = torch.empty(1, dtype=torch.float32).pin_memory()
    e2e = PipelinedIO(torch, device, stream, [(hX, X), (ht, tgt)], [(loss, hloss)],
                      lambda i, o: run(i[0], i[1], lo=o[0]))
    keep = (X, W, tgt, loss, arg, dX, dW, ws, hX, ht, hloss)
    cfgd = {"workload": wl["desc"], "tokens": N, "hidden": H, "vocab": V,
            "l2": "inputs larger than L2 (W 1.56 GB, fp32 logits 2.49 GB)"}
    return N, (lambda: run(X, tgt)), e2e, X.numel() * 2 + N * 4, 4, cfgd, keep


def setup_stream(torch, K, L, synth, device, seed, name="stream"):
    wl = WORKLOADS[name]
    B, S, nl, mode = wl["B"], wl["S"], wl["L"], wl["mode"]
    train = mode != K.KL_STREAM_FORWARD
    V = wl.get("V", 0)
    T, H = B * S, QWEN["H"]
    cfg = L.make_cfg(B, S, **QWEN, dtype=K.KL_BF16)
    bf = torch.bfloat16
    distinct = wl.get("distinct", nl)   # host weight sets; layer l uses set l % distinct
    hosts = []
    for li in range(distinct):
        w = {}
        for n, shp in L.weight_shapes(cfg).items():
            t = synth.device_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, seed, f"l{li}.{n}", bf, device)
            w[n] = t.cpu().pin_memory()
        hosts.append(w)
    structs = [L.weights_struct(hosts[li % distinct]) for li in range(nl)]
    W = synth.device_normal((V, H), 0.02, 0.0, seed, "lm.W", bf, device).cpu().pin_memory() if train else None
    X = synth.device_normal((T, H), 1.0, 0.0, seed, "X", bf, device)
    tgt = synth.device_randint((T,), V, seed, "lm.targets", device) if train else None
    Y = torch.empty_like(X)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(device)[0]
    h = K.kl_stream_create(K.StreamCfg(cfg, nl, V, mode), structs, W.data_ptr() if train else None)
    free1 = torch.cuda.mem_get_info(device)[0]
    grads, gs = [], []
    if train:
        for _ in range(nl):
            g = {n: torch.empty(shp, dtype=torch.float32, device=device) for n, shp in L.weight_shapes(cfg).items()}
            grads.append(g)
            gs.append(K.LayerGrads(*[g[n].data_ptr() for n in K.WEIGHT_FIELDS], K.KL_F32))
    dW = torch.empty(V, H, dtype=torch.float32, device=device) if train else None
    stream = torch.cuda.current_stream(device)

    def run(handle, x, t):
        if train:
            K.kl_stream_run(handle, x.data_ptr(), t.data_ptr(), wl["clip"], gs, dW.data_ptr(), stream)
        else:
            K.kl_stream_forward(handle, x.data_ptr(), Y.data_ptr(), stream)

    hX = X.cpu().pin_memory()
    ht = tgt.cpu().pin_memory() if train else None
    hY = torch.empty_like(hX).pin_memory()
    X2 = torch.empty_like(X)
    t2 = torch.empty_like(tgt) if train else None

    def e2e():
        X2.copy_(hX, non_blocking=True)
        if train:
            t2.copy_(ht, non_blocking=True)
        run(h, X2, t2)       # returns after the step (training: loss, norm, coef read back)
        if not train:
            hY.copy_(Y, non_blocking=True)

    layer_bytes = sum(t.numel() * t.element_size() for t in hosts[0].values())
    weight_h2d = nl * layer_bytes * (2 if train else 1) + (V * H * 2 if train else 0)

    def after(args):
        """Destroys the streamed driver, then times the same call with every
        layer's weights already in device memory (bulk: no uploads), and the
        plain host-to-device copy rate of the same pinned weight sets (the
        host link this box gives the stream)."""
        dev_bytes = K.kl_stream_device_bytes(h)
        K.kl_stream_destroy(h)
        dev_sets = [{n: t.to(device) for n, t in w.items()} for w in hosts]
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for w, dw in zip(hosts, dev_sets):
            for n in w:
                dw[n].copy_(w[n], non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        copy_bytes = sum(t.numel() * t.element_size() for w in hosts for t in w.values())
        link_gbs = copy_bytes / (c0.elapsed_time(c1) / 1e3) / 1e9
        dstructs = [L.weights_struct(dev_sets[li % distinct]) for li in range(nl)]
        Wd = W.to(device) if train else None
        hb = K.kl_stream_create(K.StreamCfg(cfg, nl, V, mode), dstructs, Wd.data_ptr() if train else None)
        try:
            for _ in range(args.warmup):
                run(hb, X, tgt)
            torch.cuda.synchronize()
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(args.steps):
                run(hb, X, tgt)
            b1.record(stream)
            torch.cuda.synchronize()
            ms_bulk = b0.elapsed_time(b1) / args.steps
        finally:
            K.kl_stream_destroy(hb)
        del dev_sets, Wd
        return {"driver_device_bytes": dev_bytes, "device_bytes_at_create": free0 - free1,
                "weight_h2d_bytes_per_step": weight_h2d, "ms_per_step_bulk": round(ms_bulk, 3),
                "host_link_copy_gbs": round(link_gbs, 1)}

    keep = {"objs": (hosts, W, X, tgt, grads, dW, Y, hX, ht, hY, X2, t2), "after": after}
    cfgd = {"workload": wl["desc"], "layers": nl, "batch": B, "seq_len": S, "hidden": H,
            "weights": "pinned host, two device slots", "l2": "inputs larger than L2"}
    if distinct < nl:
        cfgd["host_weight_sets"] = f"{distinct} distinct sets, layer l uses set l mod {distinct}; every layer " \
                                   "is uploaded on its own"
    if train:
        cfgd.update(vocab=V, clip_max_norm=wl["clip"], grads="fp32, device",
                    activations="inputs only, layer forward recomputed" if mode == K.KL_STREAM_RECOMPUTE
                    else "every layer's saved set")
        return T, (lambda: run(h, X, tgt)), e2e, X.numel() * 2 + T * 4, 12, cfgd, keep
    cfgd.update(activations="one layer's working set")
    return T, (lambda: run(h, X, tgt)), e2e, X.numel() * 2, Y.numel() * 2, cfgd, keep


def setup_decode(torch, K, L, synth, device, seed):
    wl = WORKLOADS["decode"]
    B, ctx, bs = wl["B"], wl["ctx"], wl["block"]
    H = QWEN["H"]
    cfg = L.make_cfg(B, 1, **QWEN, dtype=K.KL_BF16)
    w = {}
    for n, shp in L.weight_shapes(cfg).items():
        w[n] = synth.device_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, seed, f"dec.{n}", torch.bfloat16,
                                   device)
    max_blocks = (ctx + 1 + bs - 1) // bs
    n_blocks = B * max_blocks
    kv_w = QWEN["Hkv"] * QWEN["d"]
    kp = synth.device_normal((n_blocks, bs, kv_w), 1.0, 0.0, seed, "dec.kpool", torch.bfloat16, device)
    vp = synth.device_normal((n_blocks, bs, kv_w), 1.0, 0.0, seed, "dec.vpool", torch.bfloat16, device)
    gen = torch.Generator(device="cpu").manual_seed(seed)
    table = torch.randperm(n_blocks, generator=gen).to(torch.int32).reshape(B, max_blocks).to(device)
    ctx_t = torch.full((B,), ctx, dtype=torch.int32, device=device)
    X = synth.device_normal((B, H), 1.0, 0.0, seed, "dec.X", torch.bfloat16, device)
    Y = torch.empty_like(X)
    pc = K.PagedCfg(B, 1, bs, max_blocks, n_blocks)
    ws = torch.empty(K.kl_layer_forward_paged_ws_bytes(cfg, pc), dtype=torch.uint8, device=device)
    wst = L.weights_struct(w)
    stream = torch.cuda.current_stream(device)

    def run(x, y):
        K.kl_layer_forward_paged(cfg, pc, wst, x.data_ptr(), y.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                 table.data_ptr(), ctx_t.data_ptr(), ws.data_ptr(), ws.numel(), stream)

    hX = X.cpu().pin_memory()
    hY = torch.empty_like(hX).pin_memory()
    e2e = PipelinedIO(torch, device, stream, [(hX, X)], [(Y, hY)], lambda i, o: run(i[0], o[0]))

    weight_bytes = sum(t.numel() * t.element_size() for t in w.values())
    kv_bytes = 2 * B * (ctx + 1) * kv_w * 2
    keep = (w, kp, vp, table, ctx_t, X, Y, ws, hX, hY)
    cfgd = {"workload": wl["desc"], "sequences": B, "context": ctx, "new_tokens_per_sequence": 1,
            "block_size": bs, "hidden": H, "heads_q": QWEN["Hq"], "heads_kv": QWEN["Hkv"], "head_dim": QWEN["d"],
            "intermediate": QWEN["I"], "l2": "inputs larger than L2 (975 MB weights + 1.07 GB cache per step)",
            "hbm_bytes_per_step": weight_bytes + kv_bytes + 4 * B * H * 2, "roofline_bytes": True}
    return B, (lambda: run(X, Y)), e2e, X.numel() * 2, Y.numel() * 2, cfgd, keep


SETUP = {"layer": setup_layer, "attention": setup_attention, "lmhead": setup_lmhead,
         "stream": lambda *a, **k: setup_stream(*a, **k, name="stream"),
         "stream_recompute": lambda *a, **k: setup_stream(*a, **k, name="stream_recompute"),
         "stream_fwd64": lambda *a, **k: setup_stream(*a, **k, name="stream_fwd64"),
         "decode": setup_decode}


def max_over_ranks(vals, dist, device):
    """Each rank's timings, reduced to the maximum over ranks: the slowest
    rank sets the job's time. Without a process group, the values as given."""
    if dist is None:
        return [float(v) for v in vals]
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(units_per_rank_step, steps, world, ms):
    """Units that all ranks processed per second of the job's time (weak
    scaling: every rank handles its own units_per_rank_step each step)."""
    return units_per_rank_step * steps * world / (ms / 1e3)


IDLE_S = 2.0   # idle seconds before each timed region after the first


def bench_ours(args, rank, world, local_rank, dist, later_s=0.0):
    """Timed regions of one workload: device-resident (value), per-launch
    events (kernels), end to end (e2e) and, with later_s > 0, a region of at
    least later_s seconds after those (the board then at its power limit)."""
    import torch

    import bwd_qwen3_layer_gb300 as K
    from bwd_qwen3_layer_gb300 import layer as L
    from bwd_qwen3_layer_gb300 import synth

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    lib = K.load()
    units, step, e2e, h2d, d2h, cfgd, keep = SETUP[args.workload](torch, K, L, synth, device, seed=rank)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K.kl_device_status(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timed region (no per-launch events: consecutive
    # kernels may overlap their prologue with the predecessor's tail) ----
    clocks = Clocks(local_rank)
    barrier()
    clocks.start()
    time.sleep(0.25)
    n0 = lib.kl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    clocks.mark(False)
    launches = lib.kl_launch_count() - n0
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)

    # ---- the same steps again with the launch profiler on (CUDA events
    # around every launch): per-kernel times and roofline fractions. Each
    # region starts after the same idle time, so the board's power average
    # is where it was before the first one and every short region is timed
    # under the same (burst) conditions ----
    barrier()
    time.sleep(IDLE_S)
    lib.kl_profile_enable(1)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    barrier()
    ms_prof = p0.elapsed_time(p1)
    prof = read_profile(K)
    lib.kl_profile_enable(0)

    # ---- end to end through the C ABI with pinned host buffers ----
    pipelined = hasattr(e2e, "begin")
    if pipelined:                                     # the copy stream's first steps, untimed
        e2e.begin(2)
        e2e()
        e2e()
        e2e.end()
    barrier()
    time.sleep(IDLE_S)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    if pipelined:
        e2e.begin(args.steps)
    for _ in range(args.steps):
        e2e()
    if pipelined:
        e2e.end()
    f1.record(stream)
    barrier()
    ms_e2e = f0.elapsed_time(f1)

    # ---- a later, longer region of the same steps (clocks sampled again) ----
    later = None
    if later_s > 0:
        n_later = max(args.steps, int(math.ceil(later_s * 1e3 / (ms / args.steps))))
        lclk = Clocks(local_rank)
        barrier()
        lclk.start()
        time.sleep(0.25)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lclk.mark(True)
        g0.record(stream)
        for _ in range(n_later):
            step()
        g1.record(stream)
        barrier()
        lclk.mark(False)
        (ms_later,) = max_over_ranks([g0.elapsed_time(g1)], dist, device)
        later = {"steps": n_later, "ms_per_step": round(ms_later / n_later, 4),
                 "value": round(job_throughput(units, n_later, world, ms_later), 1), "clocks": lclk.stop()}
    K.kl_device_status(stream)
    extra = None
    if isinstance(keep, dict) and "after" in keep:
        extra = keep["after"](args)
        extra["link_hidden"] = round(extra["ms_per_step_bulk"] / (ms / args.steps), 4)
        extra["weight_h2d_gbs"] = round(extra["weight_h2d_bytes_per_step"] / (ms / args.steps) / 1e6, 1)
    ms, ms_e2e = max_over_ranks([ms, ms_e2e], dist, device)
    return dict(ms=ms, ms_e2e=ms_e2e, ms_prof=ms_prof, prof=prof, clocks=clk, launches=int(launches), units=units,
                h2d=h2d, d2h=d2h, config=cfgd, extra=extra, later=later)


# ----------------------------------------------------------------------------
# the oracle on a bounded sample of the workload (cpu_baseline, --impl reference)
# ----------------------------------------------------------------------------

def _oracle_weights(rng, H, Hq, Hkv, d, I):
    Dq, Dkv = Hq * d, Hkv * d
    n = lambda *s: 0.02 * rng.standard_normal(s)  # noqa: E731
    return {"gamma1": 1 + n(H), "Wq": n(Dq, H), "Wk": n(Dkv, H), "Wv": n(Dkv, H), "Wo": n(H, Dq),
            "gamma2": 1 + n(H), "Wg": n(I, H), "Wu": n(I, H), "Wd": n(H, I)}


def oracle_sample(workload: str, steps: int):
    """Times the fp64 oracle on a bounded sample of `workload`.
    Returns (tokens_per_s, seconds_per_step, cores, description)."""
    import numpy as np

    import oracle as O

    rng = np.random.default_rng(0)
    Q = QWEN
    cores = os.cpu_count()
    times = []
    if workload == "layer":
        S = 1024
        cfg = O.LayerConfig(B=1, S=S, H=Q["H"], Hq=Q["Hq"], Hkv=Q["Hkv"], d=Q["d"], I=Q["I"])
        w = _oracle_weights(rng, Q["H"], Q["Hq"], Q["Hkv"], Q["d"], Q["I"])
        X, dY = rng.standard_normal((S, Q["H"])), rng.standard_normal((S, Q["H"]))

        def one():
            Y, saved = O.layer_forward(cfg, w, X)
            O.layer_backward(cfg, w, saved, dY)
        units = S
        desc = f"one full-dims layer fwd+bwd on {S} tokens (batch 1, seq {S})"
    elif workload == "attention":
        S = 2048
        q = rng.standard_normal((S, Q["Hq"], Q["d"]))
        k = rng.standard_normal((S, Q["Hkv"], Q["d"]))
        v = rng.standard_normal((S, Q["Hkv"], Q["d"]))
        do = rng.standard_normal((S, Q["Hq"], Q["d"]))

        def one():
            O.attention_fwd(q, k, v, 1, S)
            O.attention_bwd(q, k, v, do, 1, S)
        units = S
        desc = (f"causal GQA attention fwd+bwd at seq {S} (64/8 heads, d 128); tokens/s at seq 32768 is "
                f"this figure x {S}/32768 (quadratic cost)")
    elif workload == "lmhead":
        N, V = 256, WORKLOADS["lmhead"]["V"]
        X = rng.standard_normal((N, Q["H"]))
        W = 0.02 * rng.standard_normal((V, Q["H"]))
        t = rng.integers(0, V, N)

        def one():
            O.lmhead_ce(X, W, t)
        units = N
        desc = f"lm-head CE+argmax fwd+bwd on {N} tokens, hidden 5120, vocab {V}"
    elif workload == "decode":
        Bs, ctx, bs = 8, WORKLOADS["decode"]["ctx"], WORKLOADS["decode"]["block"]
        cfg = O.LayerConfig(B=Bs, S=1, H=Q["H"], Hq=Q["Hq"], Hkv=Q["Hkv"], d=Q["d"], I=Q["I"])
        w = _oracle_weights(rng, Q["H"], Q["Hq"], Q["Hkv"], Q["d"], Q["I"])
        maxb = (ctx + 1 + bs - 1) // bs
        table = rng.permutation(Bs * maxb).reshape(Bs, maxb)
        kp = rng.standard_normal((Bs * maxb, bs, Q["Hkv"], Q["d"]))
        vp = rng.standard_normal((Bs * maxb, bs, Q["Hkv"], Q["d"]))
        X = rng.standard_normal((Bs, Q["H"]))
        ctxa = np.full(Bs, ctx)

        def one():
            O.layer_forward_paged(cfg, w, X, kp, vp, table, ctxa, 1)
        units = Bs
        desc = f"one full-dims layer's paged decode step for {Bs} sequences at context {ctx}"
    elif workload == "stream_fwd64":   # one layer forward on a token sample, scaled to 64 layers
        S = 512
        cfg = O.LayerConfig(B=1, S=S, H=Q["H"], Hq=Q["Hq"], Hkv=Q["Hkv"], d=Q["d"], I=Q["I"])
        w = _oracle_weights(rng, Q["H"], Q["Hq"], Q["Hkv"], Q["d"], Q["I"])
        X = rng.standard_normal((S, Q["H"]))
        nl = WORKLOADS["stream_fwd64"]["L"]

        def one():
            O.layer_forward(cfg, w, X)
            return 0.0
        units = S
        desc = (f"one full-dims layer forward on {S} tokens (batch 1, seq {S}); step time = {nl} x layer; "
                f"tokens/s at seq 2048 is below this (attention grows with the sequence)")
    else:   # stream, stream_recompute: one layer + the head on a token sample, scaled to 8 layers
        # (recompute changes where activations live, not what is computed)
        S = 256
        cfg = O.LayerConfig(B=1, S=S, H=Q["H"], Hq=Q["Hq"], Hkv=Q["Hkv"], d=Q["d"], I=Q["I"])
        w = _oracle_weights(rng, Q["H"], Q["Hq"], Q["Hkv"], Q["d"], Q["I"])
        V = WORKLOADS["stream"]["V"]
        X = rng.standard_normal((S, Q["H"]))
        W = 0.02 * rng.standard_normal((V, Q["H"]))
        t = rng.integers(0, V, S)
        nl = WORKLOADS["stream"]["L"]

        def one():
            Y, saved = O.layer_forward(cfg, w, X)
            t0 = time.perf_counter()
            head = O.lmhead_ce(Y, W, t)
            th = time.perf_counter() - t0
            O.layer_backward(cfg, w, saved, head["dX"])
            return th
        units = S
        desc = (f"one full-dims layer fwd+bwd plus the lm-head CE on {S} tokens; step time = "
                f"{nl} x layer + head")
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        th = one()
        dt = time.perf_counter() - t0
        if workload.startswith("stream"):
            dt = nl * (dt - th) + th
        times.append(dt)
    sec = statistics.median(times)
    desc = f"fp64 numpy oracle: {desc}; median of {len(times)}; BLAS threads default to all {cores} host cores"
    return units / sec, sec, cores, desc


def pick_tensor_peak(pk, region_ms, clocks=None):
    """The tensor-core denominator for kernels timed in a region of region_ms:
    the burst GEMM figure for a short region (the board has not yet reached its
    power cap), the sustained one for a region of half a second or more, unless
    the region's clock record shows the SMs at (within 3 % of) their maximum
    clock throughout the median, i.e. the board was not held at its power cap
    (a stream step waiting on a slow host link): then the burst figure."""
    if region_ms < 500.0:
        return pk["bf16_tflops"], f"{pk['src']} bf16_tflops (burst: timed region {region_ms / 1e3:.2f} s < 0.5 s)"
    sm, smax = (clocks or {}).get("sm_mhz"), (clocks or {}).get("sm_max_mhz")
    if sm and smax and sm >= 0.97 * smax:
        return (pk["bf16_tflops"], f"{pk['src']} bf16_tflops (burst: timed region {region_ms / 1e3:.2f} s at a median "
                                   f"SM clock of {sm:.0f} of {smax:.0f} MHz, not power-capped)")
    return (pk["bf16_tflops_sustained"],
            f"{pk['src']} bf16_tflops_sustained (timed region {region_ms / 1e3:.2f} s >= 0.5 s)")


def summarize(r, workload, steps, world, pk):
    """Throughput, per-kernel roofline figures and the dominant kernel's
    roofline of one bench_ours result."""
    value = job_throughput(r["units"], steps, world, r["ms"])
    e2e = job_throughput(r["units"], steps, world, r["ms_e2e"])
    tpk, tsrc = pick_tensor_peak(pk, r["ms_prof"], r["clocks"])
    prof = r["prof"]
    total_ms = sum(v["ms"] for v in prof.values()) or 1.0
    kernels, above = {}, []
    for name, e in sorted(prof.items(), key=lambda kv: -kv[1]["ms"]):
        per = e["ms"] / e["launches"] / 1e3
        ent = {"launches": e["launches"], "ms_per_launch": round(e["ms"] / e["launches"], 4),
               "share": round(e["ms"] / total_ms, 4)}
        if e["flops"] > 0:
            a = e["flops"] / e["launches"] / per / 1e12
            ent.update(achieved=round(a, 2), unit="TFLOP/s", frac=round(a / tpk, 4))
        elif e["bytes"] > 0:
            a = e["bytes"] / e["launches"] / per / 1e9
            ent.update(achieved=round(a, 1), unit="GB/s", frac=round(a / pk["hbm_gbs"], 4))
        if ent.get("frac", 0.0) > 1.0:
            above.append(name)
        kernels[name] = ent
    # roofline of the dominant kernel: labelled launches of one kernel are
    # grouped (every "gemm.*" call site runs gemm_bf16_tc_kernel)
    groups = {}
    for name, e in prof.items():
        key = "gemm_bf16_tc" if name.startswith("gemm.") or name == "gemm" else name
        g = groups.setdefault(key, {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0})
        for f in g:
            g[f] += e[f]
    dname, d = max(groups.items(), key=lambda kv: kv[1]["ms"])
    per = d["ms"] / d["launches"] / 1e3
    traffic = traffic_record(workload, dname)
    if r["config"].get("roofline_bytes"):
        # bandwidth-bound workload: the dominant kernel group against HBM, plus the whole step
        ach = d["bytes"] / d["launches"] / per / 1e9
        step_gbs = r["config"]["hbm_bytes_per_step"] / (r["ms"] / steps / 1e3) / 1e9
        roof = {"kernel": dname, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": traffic,
                "peak_src": f"{pk['src']} hbm_gbs",
                "step": {"bytes": r["config"]["hbm_bytes_per_step"], "achieved": round(step_gbs, 1),
                         "frac": round(step_gbs / pk["hbm_gbs"], 4)}}
    elif d["flops"] > 0:
        ach = d["flops"] / d["launches"] / per / 1e12
        roof = {"kernel": dname, "bound": "tensor", "achieved": round(ach, 2), "peak": tpk,
                "unit": "TFLOP/s", "frac": round(ach / tpk, 4), "traffic": traffic, "peak_src": tsrc,
                "frac_burst": round(ach / pk["bf16_tflops"], 4),
                "frac_sustained": round(ach / pk["bf16_tflops_sustained"], 4)}
    else:
        ach = d["bytes"] / d["launches"] / per / 1e9
        roof = {"kernel": dname, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": traffic,
                "peak_src": f"{pk['src']} hbm_gbs"}
    roof["timed"] = (f"per-launch CUDA events over a second timed region of the same {steps} steps "
                     f"({r['ms_prof'] / steps:.4f} ms per step with the events)")
    total_flops = sum(e["flops"] for e in prof.values()) / steps
    agg_tflops = total_flops / (r["ms"] / steps / 1e3) / 1e12
    out = {"value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(r["ms"] / steps, 4)}
    if total_flops > 0:
        bpk, bsrc = pick_tensor_peak(pk, r["ms"], r["clocks"])
        out.update(tensor_frac_aggregate=round(agg_tflops / bpk, 4), aggregate_tflops=round(agg_tflops, 2),
                   aggregate_peak_src=bsrc)
    out.update(roofline=roof, kernels=kernels, kernels_frac_above_1=above, gpu_launches=r["launches"],
               clocks=r["clocks"],
               e2e={"value": round(e2e, 1), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]})
    if r["extra"] is not None:
        out["stream"] = r["extra"]
    return out


EXTRAS = {"attention": (5, 3), "lmhead": (10, 3), "stream": (3, 3), "stream_recompute": (3, 3),
          "stream_fwd64": (3, 3), "decode": (20, 3)}


def measure_extras(args, pk):
    """Short runs of the long-context attention, lm-head, 8-layer stream (and
    its recompute mode), 64-layer streamed forward and paged decode workloads
    in the same process, each with its own timed region, per-kernel figures
    and clock record (steps, warm-up per EXTRAS)."""
    out = {}
    for wl, (steps, warm) in EXTRAS.items():
        a = argparse.Namespace(**vars(args))
        a.workload, a.steps, a.warmup = wl, steps, warm
        t0 = time.time()
        r = bench_ours(a, 0, 1, 0, None)
        ent = {"metric": METRICS[wl], "steps": steps, "warmup": warm} | summarize(r, wl, steps, 1, pk)
        ent["config"] = r["config"]
        ent["wall_s"] = round(time.time() - t0, 1)
        out[wl] = ent
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="layer", choices=list(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="layer workload: skip the short runs of the other workloads")
    ap.add_argument("--no-later", action="store_true",
                    help="layer workload: skip the one-second later region")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.workload.startswith("stream") and "--steps" not in sys.argv:
        args.steps = 5
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)
    metric = METRICS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        steps = max(1, min(args.steps, 3))
        tps, sec, cores, desc = oracle_sample(args.workload, steps)
        line = {"metric": metric, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
                "warmup": 0, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOADS[args.workload]["desc"]}, "impl": "reference",
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
    # the headline layer step also runs a one-second region after the others
    r = bench_ours(args, rank, world, local_rank, dist,
                   later_s=1.0 if args.workload == "layer" and not args.no_later else 0.0)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    pk = peaks()
    line = {"metric": metric} | summarize(r, args.workload, args.steps, world, pk)
    line.update({"n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                 "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"})
    line["config"] = r["config"] | {"parallelism": f"replicas x{world}"}
    if r["later"] is not None:
        line["later_region"] = r["later"]
    if world == 1 and args.workload == "layer" and not args.no_extra:
        line["workloads"] = measure_extras(args, pk)
    if world == 1 and not args.no_cpu_baseline:
        tps, sec, cores, desc = oracle_sample(args.workload, 3)
        line["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
