"""Layer streaming (kl_stream_*): a reduced-size stack against the oracle's
stack (forward through every layer, lm-head CE, backward in reverse, global
grad-norm clip), streamed weights against device-resident ("bulk") weights,
and pinned-host gradient destinations against device ones."""
import math

import numpy as np
import pytest

import oracle as O
from bwd_qwen3_layer_gb300 import layer as L
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, TOL_F32, assert_rel

pytestmark = pytest.mark.gpu


def _inputs(n_layers, B, S, H, Hq, Hkv, d, I, V, seed, bf16, qk_norm=False):
    layers = [synth.layer_weights(seed, H, Hq, Hkv, d, I, bf16=bf16, prefix=f"l{i}", qk_norm=qk_norm)
              for i in range(n_layers)]
    X = synth.normal(seed, "X", (B * S, H))
    W = synth.normal(seed, "lm.W", (V, H), std=0.02)
    if bf16:
        X, W = synth.round_bf16(X), synth.round_bf16(W)
    else:
        layers = [{k: v.astype(np.float32).astype(np.float64) for k, v in lw.items()} for lw in layers]
        X, W = X.astype(np.float32).astype(np.float64), W.astype(np.float32).astype(np.float64)
    tgt = synth.randint(seed, "lm.targets", (B * S,), V)
    return layers, X, W, tgt


def _compare(got, ref, tol, loss_tol):
    loss, norm, coef = got["result"]
    assert abs(loss - ref["loss"]) <= loss_tol
    assert math.isclose(norm, ref["total_norm"], rel_tol=tol)
    assert math.isclose(coef, ref["clip_coef"], rel_tol=tol)
    for li, g in enumerate(ref["grads"]):
        for name, want in g.items():
            assert_rel(got["grads"][li][name], want, tol, f"layer {li} d{name}")
    assert_rel(got["dW_lm"], ref["dW_lm"], tol, "dW_lm")


@pytest.mark.parametrize("dt", [1, 0])
def test_stream_matches_oracle_with_active_clip(kl, dt):
    if dt == 1:
        dims = dict(B=2, S=64, H=256, Hq=4, Hkv=2, d=128, I=512)
        V, tol, ltol = 1024, TOL_BF16, 1e-3
    else:   # the tiny fp32 layer's dims
        dims = dict(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172)
        V, tol, ltol = 256, TOL_F32, 1e-5
    nl = 2
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=3, bf16=dt == 1)
    ocfg = O.LayerConfig(**dims)
    free = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=1e9)
    clip = 0.5 * free["total_norm"]                  # make the clip bite
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=clip)
    cfg = L.make_cfg(**dims, dtype=dt)
    got = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip)
    _compare(got, ref, tol, ltol)
    assert got["result"][2] < 0.51


def test_stream_with_layer_options(kl):
    """Per-head q/k norms (their gains streamed with the layer, their gradients
    in the global norm) and interleaved rotary planes, bf16, clip active."""
    dims = dict(B=2, S=64, H=256, Hq=4, Hkv=2, d=128, I=512)
    V, nl = 1024, 2
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=4, bf16=True, qk_norm=True)
    ocfg = O.LayerConfig(**dims, qk_norm=True, rope_interleaved=True)
    free = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=1e9)
    clip = 0.5 * free["total_norm"]
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=clip)
    assert "gamma_q" in ref["grads"][0]
    cfg = L.make_cfg(**dims, dtype=1, qk_norm=True, rope_interleaved=True)
    got = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip)
    _compare(got, ref, TOL_BF16, 1e-3)


def test_streamed_equals_bulk(kl):
    """Streaming changes where weights live, not the arithmetic: the loss, the
    global norm and every gradient are bit-identical (no kernel on the path
    accumulates in a run-dependent order)."""
    dims = dict(B=1, S=128, H=256, Hq=4, Hkv=2, d=128, I=512)
    nl, V = 3, 1024
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=4, bf16=True)
    cfg = L.make_cfg(**dims, dtype=1)
    streamed = L.run_stream(cfg, nl, V, layers, W, X, tgt, 1.0, repeat=2)
    bulk = L.run_stream(cfg, nl, V, layers, W, X, tgt, 1.0, weights_on_device=True)
    assert streamed["result"][0] == bulk["result"][0]
    assert streamed["result"][1] == bulk["result"][1]
    for li in range(nl):
        for name in streamed["grads"][li]:
            assert np.array_equal(streamed["grads"][li][name], bulk["grads"][li][name]), f"{li} {name}"
    assert np.array_equal(streamed["dW_lm"], bulk["dW_lm"])
    # the streamed driver holds two weight slots, not every layer
    per_layer = 2 * sum(int(np.prod(v.shape)) for v in layers[0].values())
    assert streamed["device_bytes"] < bulk["device_bytes"] + 3 * per_layer


def test_host_gradient_destinations(kl):
    dims = dict(B=1, S=64, H=256, Hq=4, Hkv=2, d=128, I=512)
    nl, V = 3, 512
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=6, bf16=True)
    cfg = L.make_cfg(**dims, dtype=1)
    ocfg = O.LayerConfig(**dims)
    free = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=1e9)
    clip = 0.25 * free["total_norm"]
    a = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip, grads_on_host=True)
    b = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip)
    assert a["result"][0] == b["result"][0]
    for li in range(nl):
        for name in a["grads"][li]:
            assert np.array_equal(a["grads"][li][name], b["grads"][li][name]), f"{li} {name}"
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=clip)
    _compare(a, ref, TOL_BF16, 1e-3)


@pytest.mark.parametrize("dt", [1, 0])
def test_recompute_matches_oracle_and_save_all(kl, dt):
    """Activation recompute: only each layer's input is kept; the layer's forward
    runs again before its backward. Same loss and gradients bit for bit (the
    rerun forward repeats every bit), far less device memory."""
    if dt == 1:
        dims = dict(B=2, S=64, H=256, Hq=4, Hkv=2, d=128, I=512)
        V, tol, ltol = 1024, TOL_BF16, 1e-3
    else:
        dims = dict(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172)
        V, tol, ltol = 256, TOL_F32, 1e-5
    nl = 3
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=8, bf16=dt == 1)
    ocfg = O.LayerConfig(**dims)
    free = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=1e9)
    clip = 0.5 * free["total_norm"]
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=clip)
    cfg = L.make_cfg(**dims, dtype=dt)
    rec = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip, mode=kl.KL_STREAM_RECOMPUTE)
    _compare(rec, ref, tol, ltol)
    full = L.run_stream(cfg, nl, V, layers, W, X, tgt, clip, mode=kl.KL_STREAM_SAVE_ALL)
    assert rec["result"][0] == full["result"][0]
    for li in range(nl):
        for name in rec["grads"][li]:
            assert np.array_equal(rec["grads"][li][name], full["grads"][li][name]), f"{li} {name}"
    saved = kl.kl_layer_saved_bytes(cfg)
    assert rec["device_bytes"] <= full["device_bytes"] - (nl - 1) * saved


def test_recompute_bulk_with_layer_options(kl):
    dims = dict(B=1, S=96, H=256, Hq=4, Hkv=2, d=128, I=384)
    V, nl = 512, 2
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=9, bf16=True, qk_norm=True)
    ocfg = O.LayerConfig(**dims, qk_norm=True, rope_interleaved=True)
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=1.0)
    cfg = L.make_cfg(**dims, dtype=1, qk_norm=True, rope_interleaved=True)
    got = L.run_stream(cfg, nl, V, layers, W, X, tgt, 1.0, weights_on_device=True,
                       mode=kl.KL_STREAM_RECOMPUTE)
    _compare(got, ref, TOL_BF16, 1e-3)


def _oracle_forward(ocfg, layers, X):
    h = X
    for lw in layers:
        h, _ = O.layer_forward(ocfg, lw, h)
    return h


@pytest.mark.parametrize("dt", [1, 0])
def test_stream_forward_is_lossless_and_depth_independent(kl, dt):
    """Forward-only streaming: the streamed result equals the bulk one bit for
    bit and the oracle's chain within tolerance; the driver's device memory does
    not depend on the depth."""
    if dt == 1:
        dims = dict(B=1, S=160, H=256, Hq=4, Hkv=2, d=128, I=512)
        tol = TOL_BF16
    else:
        dims = dict(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172)
        tol = TOL_F32
    nl = 5
    layers, X, W, _ = _inputs(nl, **dims, V=64, seed=10, bf16=dt == 1)
    cfg = L.make_cfg(**dims, dtype=dt)
    streamed = L.run_stream_forward(cfg, layers, X, repeat=2)
    bulk = L.run_stream_forward(cfg, layers, X, weights_on_device=True)
    assert np.array_equal(streamed["Y"], bulk["Y"])
    # the training driver's forward (every layer's activations kept) agrees too
    full = L.run_stream_forward(cfg, layers, X, mode=kl.KL_STREAM_SAVE_ALL, W_lm_host=W, V=64)
    assert np.array_equal(streamed["Y"], full["Y"])
    assert_rel(streamed["Y"], _oracle_forward(O.LayerConfig(**dims), layers, X), tol, "Y")
    shallow = L.run_stream_forward(cfg, layers[:2], X)
    assert shallow["device_bytes"] == streamed["device_bytes"]
    assert full["device_bytes"] > streamed["device_bytes"] + (nl - 2) * kl.kl_layer_saved_bytes(cfg)


def test_stream_forward_only_refuses_training(kl):
    dims = dict(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172)
    layers, X, W, tgt = _inputs(1, **dims, V=64, seed=11, bf16=False)
    cfg = L.make_cfg(**dims, dtype=0)
    import torch
    keep = []
    hl = L._stream_weights(cfg, layers, False, "cuda", keep)
    h = kl.kl_stream_create(kl.StreamCfg(cfg, 1, 0, kl.KL_STREAM_FORWARD), hl, None)
    try:
        Xd = torch.zeros(32, 64, device="cuda")
        tg = torch.zeros(32, dtype=torch.int32, device="cuda")
        g = {n: torch.empty(s, device="cuda") for n, s in L.weight_shapes(cfg).items()}
        gs = kl.LayerGrads(*[g[n].data_ptr() for n in kl.WEIGHT_FIELDS], kl.KL_F32, None, None)
        dW = torch.empty(64, 64, device="cuda")
        with pytest.raises(kl.KLError):
            kl.kl_stream_run(h, Xd.data_ptr(), tg.data_ptr(), 1.0, [gs], dW.data_ptr())
    finally:
        kl.kl_stream_destroy(h)
