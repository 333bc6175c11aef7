"""torch-side helpers around the C structs: device buffers for saved
activations, workspace and gradients, allocated with torch (plumbing only;
no arithmetic of the layer happens here)."""
from __future__ import annotations

import torch

from . import (KL_BF16, KL_F32, LayerCfg, LayerGrads, LayerWeights, LmheadCfg, QK_WEIGHT_FIELDS, WEIGHT_FIELDS,
               kl_layer_bwd_workspace_bytes, kl_layer_fwd_workspace_bytes, kl_layer_saved_bytes, kl_layer_saved_carve,
               kl_lmhead_workspace_bytes)

TORCH_DTYPE = {KL_F32: torch.float32, KL_BF16: torch.bfloat16}
SYNTH_NAMES = {"gamma1": "gamma1", "wq": "Wq", "wk": "Wk", "wv": "Wv", "wo": "Wo",
               "gamma2": "gamma2", "wg": "Wg", "wu": "Wu", "wd": "Wd",
               "gamma_q": "gamma_q", "gamma_k": "gamma_k"}


def make_cfg(B, S, H, Hq, Hkv, d, I, eps=1e-6, rope_base=1e6, dtype=KL_BF16, qk_norm=False,
             rope_interleaved=False) -> LayerCfg:
    return LayerCfg(B, S, H, Hq, Hkv, d, I, eps, rope_base, dtype, int(qk_norm), int(rope_interleaved))


def weight_fields(cfg: LayerCfg) -> tuple:
    return WEIGHT_FIELDS + (QK_WEIGHT_FIELDS if cfg.qk_norm else ())


def weight_shapes(cfg: LayerCfg) -> dict:
    H, Dq, Dkv, I = cfg.H, cfg.Hq * cfg.d, cfg.Hkv * cfg.d, cfg.I
    shapes = {"gamma1": (H,), "wq": (Dq, H), "wk": (Dkv, H), "wv": (Dkv, H), "wo": (H, Dq),
              "gamma2": (H,), "wg": (I, H), "wu": (I, H), "wd": (H, I)}
    if cfg.qk_norm:
        shapes.update(gamma_q=(cfg.d,), gamma_k=(cfg.d,))
    return shapes


def weights_struct(w: dict) -> LayerWeights:
    return LayerWeights(*[w[n].data_ptr() if n in w else None for n in WEIGHT_FIELDS + QK_WEIGHT_FIELDS])


def alloc_grads(cfg: LayerCfg, device, dtype: int) -> tuple:
    g = {}
    for n, shp in weight_shapes(cfg).items():
        dt = torch.float32 if n.startswith("gamma") else TORCH_DTYPE[dtype]
        g[n] = torch.empty(shp, dtype=dt, device=device)
    st = LayerGrads(*[g[n].data_ptr() for n in WEIGHT_FIELDS], dtype,
                    *[g[n].data_ptr() if n in g else None for n in QK_WEIGHT_FIELDS])
    return g, st


class LayerBuffers:
    """Saved-activation buffer (carved by the library) and backward workspace."""

    def __init__(self, cfg: LayerCfg, device):
        self.cfg = cfg
        nb = kl_layer_saved_bytes(cfg)
        self.saved_mem = torch.empty(nb, dtype=torch.uint8, device=device)
        self.saved = kl_layer_saved_carve(cfg, self.saved_mem.data_ptr(), nb)
        self.fwd_ws = torch.empty(max(256, kl_layer_fwd_workspace_bytes(cfg)), dtype=torch.uint8, device=device)
        nb = kl_layer_bwd_workspace_bytes(cfg)
        self.bwd_ws = torch.empty(nb, dtype=torch.uint8, device=device)

    def view(self, name: str, shape, dtype) -> torch.Tensor:
        """A tensor view of one saved buffer (for checks)."""
        p = getattr(self.saved, name)
        off = p - self.saved_mem.data_ptr()
        n = 1
        for s in shape:
            n *= s
        es = torch.tensor([], dtype=dtype).element_size()
        return self.saved_mem[off: off + n * es].view(dtype).view(*shape)


def lmhead_cfg(N, H, V, dtype=KL_BF16, dw_dtype=None) -> LmheadCfg:
    return LmheadCfg(N, H, V, dtype, dtype if dw_dtype is None else dw_dtype)


def lmhead_ws(cfg: LmheadCfg, device) -> torch.Tensor:
    return torch.empty(kl_lmhead_workspace_bytes(cfg), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------
# one-call runners on host arrays (upload, call the C ABI, download)
# --------------------------------------------------------------------------

def to_device(a, dtype: int, device) -> torch.Tensor:
    return torch.as_tensor(a, dtype=torch.float64).to(TORCH_DTYPE[dtype]).to(device).contiguous()


def run_layer(cfg: LayerCfg, w_host: dict, X_host, dY_host, device="cuda", grad_dtype=None,
              keep=False):
    """Forward and backward of one layer on host arrays (synth names for the
    weights: gamma1, Wq, ...). Returns a dict of fp64 numpy arrays: Y, dX, the
    nine gradients (synth names) and the saved activations."""
    from . import kl_layer_backward, kl_layer_forward

    dt = cfg.dtype
    gdt = dt if grad_dtype is None else grad_dtype
    w = {n: to_device(w_host[SYNTH_NAMES[n]], dt, device) for n in weight_fields(cfg)}
    T = cfg.B * cfg.S
    X = to_device(X_host, dt, device)
    dY = to_device(dY_host, dt, device)
    Y = torch.empty(T, cfg.H, dtype=TORCH_DTYPE[dt], device=device)
    dX = torch.empty_like(Y)
    buf = LayerBuffers(cfg, device)
    ws = weights_struct(w)
    kl_layer_forward(cfg, ws, X.data_ptr(), Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(),
                     buf.fwd_ws.numel())
    grads, gst = alloc_grads(cfg, device, gdt)
    kl_layer_backward(cfg, ws, buf.saved, dY.data_ptr(), dX.data_ptr(), gst, buf.bwd_ws.data_ptr(),
                      buf.bwd_ws.numel())
    torch.cuda.synchronize()
    out = {"Y": Y.double().cpu().numpy(), "dX": dX.double().cpu().numpy()}
    for n in weight_fields(cfg):
        out["d" + SYNTH_NAMES[n]] = grads[n].double().cpu().numpy()
    Dq, Dkv = cfg.Hq * cfg.d, cfg.Hkv * cfg.d
    sdt = TORCH_DTYPE[dt]
    shapes = {"h1": ((T, cfg.H), sdt), "rstd1": ((T,), torch.float32), "q": ((T, Dq), sdt),
              "k": ((T, Dkv), sdt), "v": ((T, Dkv), sdt), "o": ((T, Dq), sdt),
              "lse": ((cfg.B, cfg.Hq, cfg.S), torch.float32), "x2": ((T, cfg.H), sdt),
              "h2": ((T, cfg.H), sdt), "rstd2": ((T,), torch.float32), "g": ((T, cfg.I), sdt),
              "u": ((T, cfg.I), sdt), "m": ((T, cfg.I), sdt)}
    if cfg.qk_norm:
        shapes.update(q_pre=((T, Dq), sdt), k_pre=((T, Dkv), sdt), rstd_q=((T, cfg.Hq), torch.float32),
                      rstd_k=((T, cfg.Hkv), torch.float32))
    out["saved"] = {k: buf.view(k, s, d).double().cpu().numpy() for k, (s, d) in shapes.items()}
    if keep:
        out["_keep"] = (w, X, dY, Y, dX, buf, grads)
    return out


def run_lmhead(N, H, V, X_host, W_host, targets_host, dtype=KL_BF16, dw_dtype=None, device="cuda"):
    """lm-head CE + argmax + dX/dW on host arrays; returns fp64 numpy results."""
    from . import kl_lmhead_ce_argmax

    cfg = lmhead_cfg(N, H, V, dtype, dw_dtype)
    X = to_device(X_host, dtype, device)
    W = to_device(W_host, dtype, device)
    tgt = torch.as_tensor(targets_host, dtype=torch.int32).to(device)
    loss = torch.zeros(1, dtype=torch.float32, device=device)
    arg = torch.empty(N, dtype=torch.int32, device=device)
    dz = torch.empty(N, V, dtype=TORCH_DTYPE[dtype], device=device)
    dX = torch.empty(N, H, dtype=TORCH_DTYPE[dtype], device=device)
    dW = torch.empty(V, H, dtype=TORCH_DTYPE[cfg.dw_dtype], device=device)
    ws = lmhead_ws(cfg, device)
    kl_lmhead_ce_argmax(cfg, X.data_ptr(), W.data_ptr(), tgt.data_ptr(), loss.data_ptr(), arg.data_ptr(),
                        dz.data_ptr(), dX.data_ptr(), dW.data_ptr(), ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    z = ws[: N * V * 4].view(torch.float32).view(N, V)
    return {"loss": float(loss.item()), "argmax": arg.cpu().numpy().astype("int64"),
            "z": z.double().cpu().numpy(), "dz": dz.double().cpu().numpy(),
            "dX": dX.double().cpu().numpy(), "dW": dW.double().cpu().numpy()}


def _stream_weights(cfg: LayerCfg, layers_host: list, weights_on_device: bool, device, keep: list) -> list:
    """LayerWeights structs over pinned host (streamed) or device (bulk) copies
    of each layer's host arrays (synth names); the tensors are kept in `keep`."""
    dt = TORCH_DTYPE[cfg.dtype]
    hl = []
    for lw in layers_host:
        w = {}
        for n in weight_fields(cfg):
            t = torch.as_tensor(lw[SYNTH_NAMES[n]], dtype=torch.float64).to(dt).contiguous()
            w[n] = t.to(device) if weights_on_device else t.pin_memory()
        keep.append(w)
        hl.append(weights_struct(w))
    return hl


def run_stream(cfg: LayerCfg, n_layers: int, V: int, layers_host: list, W_lm_host, X_host, targets_host,
               clip: float, weights_on_device=False, grads_on_host=False, device="cuda", repeat=1, mode=0):
    """One (or `repeat`) layer-streaming training step(s) through kl_stream_*.

    layers_host: per layer a dict of host arrays (synth names). Weights are
    handed over as pinned host memory (streamed) or device memory (bulk).
    mode: KL_STREAM_SAVE_ALL (0) or KL_STREAM_RECOMPUTE (1).
    Returns dict(result=(loss, norm, coef), grads=[{name: fp64 array}], dW_lm=array, device_bytes)."""
    from . import (StreamCfg, kl_stream_create, kl_stream_destroy, kl_stream_device_bytes,
                   kl_stream_run)

    dt = cfg.dtype
    keep = []
    hl = _stream_weights(cfg, layers_host, weights_on_device, device, keep)
    W = torch.as_tensor(W_lm_host, dtype=torch.float64).to(TORCH_DTYPE[dt]).contiguous()
    W = W.to(device) if weights_on_device else W.pin_memory()
    scfg = StreamCfg(cfg, n_layers, V, mode)
    h = kl_stream_create(scfg, hl, W.data_ptr())
    try:
        X = to_device(X_host, dt, device)
        tgt = torch.as_tensor(targets_host, dtype=torch.int32).to(device)
        gl, gs = [], []
        for _ in range(n_layers):
            g = {n: torch.empty(shp, dtype=torch.float32, device="cpu" if grads_on_host else device)
                 for n, shp in weight_shapes(cfg).items()}
            if grads_on_host:
                g = {n: t.pin_memory() for n, t in g.items()}
            gl.append(g)
            gs.append(LayerGrads(*[g[n].data_ptr() for n in WEIGHT_FIELDS], KL_F32,
                                 *[g[n].data_ptr() if n in g else None for n in QK_WEIGHT_FIELDS]))
        dW = torch.empty(V, cfg.H, dtype=torch.float32, device="cpu" if grads_on_host else device)
        if grads_on_host:
            dW = dW.pin_memory()
        for _ in range(repeat):
            res = kl_stream_run(h, X.data_ptr(), tgt.data_ptr(), clip, gs, dW.data_ptr())
        torch.cuda.synchronize()
        out = {"result": (res.loss, res.total_norm, res.clip_coef), "device_bytes": kl_stream_device_bytes(h),
               "grads": [{SYNTH_NAMES[n]: g[n].double().cpu().numpy() for n in weight_fields(cfg)} for g in gl],
               "dW_lm": dW.double().cpu().numpy()}
    finally:
        kl_stream_destroy(h)
    return out


def run_stream_forward(cfg: LayerCfg, layers_host: list, X_host, weights_on_device=False, device="cuda",
                       mode=2, repeat=1, W_lm_host=None, V=0):
    """Forward only through every layer with kl_stream_forward (weights
    streamed from pinned host memory, or bulk from device memory). A training
    mode (SAVE_ALL, RECOMPUTE) also needs the lm-head weight W_lm_host [V, H].
    Returns dict(Y=fp64 array [T, H], device_bytes)."""
    from . import StreamCfg, kl_stream_create, kl_stream_destroy, kl_stream_device_bytes, kl_stream_forward

    keep = []
    hl = _stream_weights(cfg, layers_host, weights_on_device, device, keep)
    W = None
    if W_lm_host is not None:
        W = torch.as_tensor(W_lm_host, dtype=torch.float64).to(TORCH_DTYPE[cfg.dtype]).contiguous()
        W = W.to(device) if weights_on_device else W.pin_memory()
    h = kl_stream_create(StreamCfg(cfg, len(layers_host), V, mode), hl, None if W is None else W.data_ptr())
    try:
        X = to_device(X_host, cfg.dtype, device)
        Y = torch.empty_like(X)
        for _ in range(repeat):
            kl_stream_forward(h, X.data_ptr(), Y.data_ptr())
        out = {"Y": Y.double().cpu().numpy(), "device_bytes": kl_stream_device_bytes(h)}
    finally:
        kl_stream_destroy(h)
    return out
