"""lm-head: logits GEMM, single-launch CE + argmax + dlogits, dX and dW,
against the oracle; and the CE kernel alone on fp32 logits."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import layer as L
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, TOL_LOSS, argmax_ok, assert_rel, dev, host

pytestmark = pytest.mark.gpu


def test_tiny_fp32_lmhead(kl):
    """Tiny fp32 workload's head: 32 tokens, hidden 64, vocab 256, seed 0."""
    lm = synth.lmhead_inputs(0, 32, 64, 256)
    lm = {k: (v.astype(np.float32).astype(np.float64) if k != "targets" else v) for k, v in lm.items()}
    r = L.run_lmhead(32, 64, 256, lm["X"], lm["W"], lm["targets"], dtype=kl.KL_F32)
    ref = O.lmhead_ce(lm["X"], lm["W"], lm["targets"])
    assert abs(r["loss"] - ref["loss"]) <= 1e-5
    bad, _ = argmax_ok(ref["z"], r["argmax"], gap=1e-5)
    assert len(bad) == 0
    for k in ("dz", "dX", "dW"):
        assert_rel(r[k], ref[k], 1e-5, k)


@pytest.mark.parametrize("N,H,V", [(300, 512, 4104), (64, 256, 1024), (1000, 256, 32000)])
def test_bf16_lmhead(kl, N, H, V):
    lm = synth.lmhead_inputs(1, N, H, V, bf16=True)
    r = L.run_lmhead(N, H, V, lm["X"], lm["W"], lm["targets"])
    ref = O.lmhead_ce(lm["X"], lm["W"], lm["targets"])
    assert abs(r["loss"] - ref["loss"]) <= TOL_LOSS
    bad, decided = argmax_ok(ref["z"], r["argmax"])
    assert len(bad) == 0 and decided > 0
    assert_rel(r["z"], ref["z"], 1e-5, "z")
    for k in ("dz", "dX", "dW"):
        assert_rel(r[k], ref[k], TOL_BF16, k)


@pytest.mark.parametrize("N,V,dz_dt", [(129, 151936, 1), (7, 1000, 0), (3, 6, 0), (64, 4100, 1)])
def test_ce_kernel_on_fp32_logits(kl, N, V, dz_dt):
    """Same precision on both sides: the oracle reads the very fp32 logits the
    kernel reads, so argmax must match on every row."""
    z = (4 * synth.normal(2, "ce.z", (N, V))).astype(np.float32).astype(np.float64)
    tgt = synth.randint(2, "ce.t", (N,), V)
    Z = dev(z, torch.float32)
    T = torch.as_tensor(tgt, dtype=torch.int32).cuda()
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    arg = torch.empty(N, dtype=torch.int32, device="cuda")
    dz = torch.empty(N, V, dtype=torch.float32 if dz_dt == 0 else torch.bfloat16, device="cuda")
    ws = torch.empty(kl.kl_ce_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # twice: the kernel resets its own completion counter
        kl.kl_ce_argmax(N, V, Z.data_ptr(), T.data_ptr(), loss.data_ptr(), arg.data_ptr(), dz.data_ptr(),
                        dz_dt, ws.data_ptr(), ws.numel())
        torch.cuda.synchronize()
        l_ref, a_ref, dz_ref, _ = O.ce_argmax(z, tgt)
        assert abs(loss.item() - l_ref) <= 1e-4 * max(1.0, abs(l_ref))
        assert np.array_equal(arg.cpu().numpy(), a_ref)
        assert_rel(host(dz), dz_ref, 1e-5 if dz_dt == 0 else 4e-3, "dz")
    assert kl.kl_device_status() == 0


def test_ce_target_out_of_range_sets_device_error(kl):
    N, V = 4, 64
    Z = torch.zeros(N, V, dtype=torch.float32, device="cuda")
    T = torch.tensor([0, 1, V + 5, 2], dtype=torch.int32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    arg = torch.empty(N, dtype=torch.int32, device="cuda")
    dz = torch.empty(N, V, dtype=torch.float32, device="cuda")
    ws = torch.empty(kl.kl_ce_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    kl.kl_ce_argmax(N, V, Z.data_ptr(), T.data_ptr(), loss.data_ptr(), arg.data_ptr(), dz.data_ptr(), 0,
                    ws.data_ptr(), ws.numel())
    with pytest.raises(kl.KLError) as e:
        kl.kl_device_status()
    assert e.value.status == kl.KL_ERR_DEVICE
    assert kl.kl_device_status() == 0     # the word was cleared
