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
    """Streaming changes where weights live, not the arithmetic: the loss is
    bit-identical, gradients agree up to the order of fp32 atomic additions
    in the attention backward."""
    dims = dict(B=1, S=128, H=256, Hq=4, Hkv=2, d=128, I=512)
    nl, V = 3, 1024
    layers, X, W, tgt = _inputs(nl, **dims, V=V, seed=4, bf16=True)
    cfg = L.make_cfg(**dims, dtype=1)
    streamed = L.run_stream(cfg, nl, V, layers, W, X, tgt, 1.0, repeat=2)
    bulk = L.run_stream(cfg, nl, V, layers, W, X, tgt, 1.0, weights_on_device=True)
    assert streamed["result"][0] == bulk["result"][0]
    assert math.isclose(streamed["result"][1], bulk["result"][1], rel_tol=1e-5)
    for li in range(nl):
        for name in streamed["grads"][li]:
            assert_rel(streamed["grads"][li][name], bulk["grads"][li][name], 1e-4, f"{li} {name}")
    assert_rel(streamed["dW_lm"], bulk["dW_lm"], 1e-6, "dW_lm")
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
            assert_rel(a["grads"][li][name], b["grads"][li][name], 1e-4, f"{li} {name}")
    ref = O.stack_fwd_bwd(ocfg, layers, W, X, tgt, max_norm=clip)
    _compare(a, ref, TOL_BF16, 1e-3)
