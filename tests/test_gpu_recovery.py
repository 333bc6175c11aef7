"""Recovery after a kernel gave up on a wait. Such a launch sets the timeout bit
of the device error word and can leave arrival counts behind in the few-rows
GEMM's shared-tile counters and in the fused RMSNorm backward's grid barrier.
The library's test hook leaves both in that state without any kernel waiting;
kl_device_status must then report the timeout and zero the counters, and the
next launches of both kernels must give the same bits as before."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, assert_rel, dev, host

pytestmark = pytest.mark.gpu


def _few_rows(kl):
    """A 64-row product whose 128-column tiles are shared out between CTAs along
    K, so every launch counts pieces in the arrival counters."""
    M, N, K = 64, 1344, 2560
    A = synth.round_bf16(synth.normal(11, "rec.A", (M, K)))
    B = synth.round_bf16(synth.normal(11, "rec.B", (N, K)))
    a, b = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    nb = kl.kl_gemm_scratch_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

    def run():
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, kl.KL_F32,
                      ws=ws.data_ptr(), ws_bytes=nb)
        return C

    return run, O.linear(A, B)


def _rms_bwd(kl):
    """The bf16 RMSNorm backward with its gain gradient: one cooperative launch
    whose CTAs meet at the grid barrier before the column sums."""
    rows, width, eps = 300, 5120, 1e-6
    x = synth.round_bf16(synth.normal(12, "rec.x", (rows, width)))
    g = synth.round_bf16(synth.normal(12, "rec.g", (width,), std=0.02, mean=1.0))
    dh = synth.normal(12, "rec.dh", (rows, width)).astype(np.float32).astype(np.float64)
    X, G, DH = dev(x, torch.bfloat16), dev(g, torch.bfloat16), dev(dh, torch.float32)
    H = torch.empty_like(X)
    r = torch.empty(rows, dtype=torch.float32, device="cuda")
    kl.kl_rmsnorm_fwd(rows, width, kl.KL_BF16, X.data_ptr(), G.data_ptr(), eps, H.data_ptr(), r.data_ptr())
    ws = torch.empty(kl.kl_rmsnorm_bwd_ws_bytes(rows, width), dtype=torch.uint8, device="cuda")

    def run():
        DX = torch.empty_like(X)
        dg = torch.full((width,), float("nan"), dtype=torch.float32, device="cuda")
        kl.kl_rmsnorm_bwd(rows, width, kl.KL_BF16, DH.data_ptr(), kl.KL_F32, X.data_ptr(), G.data_ptr(),
                          r.data_ptr(), 0, DX.data_ptr(), dg.data_ptr(), ws.data_ptr(), ws.numel())
        return DX, dg

    _, r_ref = O.rmsnorm_fwd(x, g, eps)
    return run, O.rmsnorm_bwd(dh, x, g, r_ref)


def test_counters_left_by_a_timed_out_launch_are_cleared(kl):
    gemm, c_ref = _few_rows(kl)
    rms, (dx_ref, dg_ref) = _rms_bwd(kl)
    C0 = gemm()
    DX0, dg0 = rms()
    torch.cuda.synchronize()
    assert kl.kl_device_status() == 0
    assert_rel(host(C0), c_ref, 1e-5, "C before")
    assert_rel(host(DX0), dx_ref, TOL_BF16, "dx before")
    assert_rel(host(dg0), dg_ref, 1e-5, "dgamma before")

    kl.kl_test_abandon_counters()
    with pytest.raises(kl.KLError) as err:
        kl.kl_device_status()
    assert err.value.status == kl.KL_ERR_TIMEOUT
    assert kl.kl_device_status() == 0          # the word was cleared by the read

    C1 = gemm()
    DX1, dg1 = rms()
    torch.cuda.synchronize()
    assert kl.kl_device_status() == 0
    assert torch.equal(C1, C0)
    assert torch.equal(DX1, DX0)
    assert torch.equal(dg1, dg0)
