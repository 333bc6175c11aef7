"""The whole decoder layer (forward with saved activations, backward to dX
and all nine parameter gradients) through the C ABI against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import layer as L
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, TOL_F32, assert_rel

pytestmark = pytest.mark.gpu

GRAD_NAMES = ("gamma1", "Wq", "Wk", "Wv", "Wo", "gamma2", "Wg", "Wu", "Wd")


def _run_both(kl, B, S, H, Hq, Hkv, d, I, dt, seed, grad_dtype=None, w=None, qk_norm=False, inter=False):
    bf = dt == kl.KL_BF16
    cfg = L.make_cfg(B, S, H, Hq, Hkv, d, I, dtype=dt, qk_norm=qk_norm, rope_interleaved=inter)
    ocfg = O.LayerConfig(B=B, S=S, H=H, Hq=Hq, Hkv=Hkv, d=d, I=I, qk_norm=qk_norm, rope_interleaved=inter)
    if w is None:
        w = synth.layer_weights(seed, H, Hq, Hkv, d, I, bf16=bf, qk_norm=qk_norm)
    inp = synth.layer_inputs(seed, B * S, H, bf16=bf)
    if not bf:   # fp32 mode: both sides see the fp32-representable values
        w = {k: v.astype(np.float32).astype(np.float64) for k, v in w.items()}
        inp = {k: v.astype(np.float32).astype(np.float64) for k, v in inp.items()}
    got = L.run_layer(cfg, w, inp["X"], inp["dY"], grad_dtype=grad_dtype)
    Y, saved = O.layer_forward(ocfg, w, inp["X"])
    dX, grads, _ = O.layer_backward(ocfg, w, saved, inp["dY"])
    return got, Y, dX, grads, saved, w, inp


def test_tiny_fp32_layer(kl):
    """The tiny fp32 workload: B1 S32 H64 Hq4 Hkv2 d16 I172, eps 1e-6, base 1e6, seed 0."""
    got, Y, dX, grads, saved, _, _ = _run_both(kl, 1, 32, 64, 4, 2, 16, 172, kl.KL_F32, 0)
    assert_rel(got["Y"], Y, TOL_F32, "Y")
    assert_rel(got["dX"], dX, TOL_F32, "dX")
    for n in GRAD_NAMES:
        assert_rel(got["d" + n], grads[n], TOL_F32, "d" + n)
    assert_rel(got["saved"]["lse"], saved["lse"], TOL_F32, "lse")


@pytest.mark.parametrize("B,S,H,Hq,Hkv,I", [(2, 200, 512, 8, 2, 1376), (1, 128, 256, 2, 2, 512),
                                           (1, 333, 640, 8, 1, 1000)])
def test_bf16_layer(kl, B, S, H, Hq, Hkv, I):
    got, Y, dX, grads, saved, _, _ = _run_both(kl, B, S, H, Hq, Hkv, 128, I, kl.KL_BF16, 5)
    assert_rel(got["Y"], Y, TOL_BF16, "Y")
    assert_rel(got["dX"], dX, TOL_BF16, "dX")
    for n in GRAD_NAMES:
        assert_rel(got["d" + n], grads[n], TOL_BF16, "d" + n)
    for k in ("q", "k", "v", "o", "x2", "g", "u", "m"):
        assert_rel(got["saved"][k], saved[k].reshape(got["saved"][k].shape), TOL_BF16, k)


OPTION_CASES = [(True, False), (False, True), (True, True)]


@pytest.mark.parametrize("qk_norm,inter", OPTION_CASES)
def test_tiny_fp32_layer_options(kl, qk_norm, inter):
    """Per-head q/k RMSNorm and/or interleaved rotary planes, fp32, tiny workload."""
    got, Y, dX, grads, saved, _, _ = _run_both(kl, 1, 32, 64, 4, 2, 16, 172, kl.KL_F32, 1, qk_norm=qk_norm,
                                               inter=inter)
    assert_rel(got["Y"], Y, TOL_F32, "Y")
    assert_rel(got["dX"], dX, TOL_F32, "dX")
    names = GRAD_NAMES + (("gamma_q", "gamma_k") if qk_norm else ())
    for n in names:
        assert_rel(got["d" + n], grads[n], TOL_F32, "d" + n)
    keys = ("q", "k") + (("q_pre", "k_pre", "rstd_q", "rstd_k") if qk_norm else ())
    for k in keys:
        assert_rel(got["saved"][k], saved[k].reshape(got["saved"][k].shape), TOL_F32, k)


@pytest.mark.parametrize("qk_norm,inter", OPTION_CASES)
@pytest.mark.parametrize("B,S,H,Hq,Hkv,I", [(2, 200, 512, 8, 2, 1376), (1, 333, 640, 8, 1, 1000)])
def test_bf16_layer_options(kl, qk_norm, inter, B, S, H, Hq, Hkv, I):
    got, Y, dX, grads, saved, _, _ = _run_both(kl, B, S, H, Hq, Hkv, 128, I, kl.KL_BF16, 7, qk_norm=qk_norm,
                                               inter=inter)
    assert_rel(got["Y"], Y, TOL_BF16, "Y")
    assert_rel(got["dX"], dX, TOL_BF16, "dX")
    names = GRAD_NAMES + (("gamma_q", "gamma_k") if qk_norm else ())
    for n in names:
        assert_rel(got["d" + n], grads[n], TOL_BF16, "d" + n)
    keys = ("q", "k", "v", "o") + (("q_pre", "k_pre", "rstd_q", "rstd_k") if qk_norm else ())
    for k in keys:
        assert_rel(got["saved"][k], saved[k].reshape(got["saved"][k].shape), TOL_BF16, k)


def test_bf16_layer_fp32_grads(kl):
    got, Y, dX, grads, _, _, _ = _run_both(kl, 1, 160, 256, 4, 2, 128, 512, kl.KL_BF16, 6, grad_dtype=kl.KL_F32)
    for n in GRAD_NAMES:
        assert_rel(got["d" + n], grads[n], TOL_BF16, "d" + n)


@pytest.mark.parametrize("dt", [0, 1])
def test_zero_output_projections(kl, dt):
    """Wo = Wd = 0: Y = X and dX = dY bit-exactly; only dWo and dWd are non-zero."""
    d = 128 if dt == 1 else 16
    H, Hq, Hkv, I, B, S = 256, 4, 2, 384, 1, 96
    w = synth.layer_weights(9, H, Hq, Hkv, d, I, bf16=dt == 1)
    w["Wo"] = np.zeros_like(w["Wo"])
    w["Wd"] = np.zeros_like(w["Wd"])
    got, Y, dX, grads, _, w, inp = _run_both(kl, B, S, H, Hq, Hkv, d, I, dt, 9, w=w)
    assert np.array_equal(got["Y"], inp["X"])
    assert np.array_equal(got["dX"], inp["dY"])
    for n in ("gamma1", "Wq", "Wk", "Wv", "gamma2", "Wg", "Wu"):
        assert np.all(got["d" + n] == 0.0), n
    assert np.any(got["dWo"] != 0.0) and np.any(got["dWd"] != 0.0)


@pytest.mark.parametrize("S,Hq,Hkv", [(128, 4, 2), (640, 16, 2)])
def test_repeat_is_deterministic(kl, S, Hq, Hkv):
    """A layer step repeats bit for bit: forward output, dX and every gradient
    (the attention's dK/dV partials and every GEMM sum in a fixed order)."""
    cfg = L.make_cfg(1, S, 256, Hq, Hkv, 128, 512, dtype=kl.KL_BF16)
    w = synth.layer_weights(3, 256, Hq, Hkv, 128, 512, bf16=True)
    inp = synth.layer_inputs(3, S, 256, bf16=True)
    a = L.run_layer(cfg, w, inp["X"], inp["dY"])
    b = L.run_layer(cfg, w, inp["X"], inp["dY"])
    assert set(a) == set(b)
    for n in a:
        if isinstance(a[n], dict):           # the saved activations
            for k in a[n]:
                assert np.array_equal(a[n][k], b[n][k]), f"{n}.{k}"
        else:
            assert np.array_equal(a[n], b[n]), n
    kl.kl_device_status()
