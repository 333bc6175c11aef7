"""The allocation-free cross-entropy entry point.

kl_ce_argmax_noalloc serves callers that cannot pass the library a device
workspace (an application that owns all device memory through its own pool,
a plugin without an allocator hook, a loop that cannot take cudaMalloc's
implicit synchronisation). It must give the same results as kl_ce_argmax,
which takes a caller-allocated workspace, and keep giving them on back-to-back
calls even though every call reuses the same static scratch array.

Collected last on purpose (file name), so that a run stopping at its first
failure has run every other test already. It passes alone in a fresh process
too: the first call on the device performs the scratch address lookup.
"""
import numpy as np
import pytest
import torch

from bwd_qwen3_layer_gb300 import synth
from _parity import assert_rel, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,V,dz_dt", [(257, 151936, 1), (33, 1000, 0)])
def test_noalloc_matches_workspace_entry_point(kl, N, V, dz_dt):
    z = (4 * synth.normal(7, "noalloc.z", (N, V))).astype(np.float32).astype(np.float64)
    tgt = synth.randint(7, "noalloc.t", (N,), V)
    Z = dev(z, torch.float32)
    T = torch.as_tensor(tgt, dtype=torch.int32).cuda()
    dzt = torch.float32 if dz_dt == 0 else torch.bfloat16

    # the existing entry point, with its own workspace
    loss_ref = torch.zeros(1, dtype=torch.float32, device="cuda")
    arg_ref = torch.empty(N, dtype=torch.int32, device="cuda")
    dz_ref = torch.empty(N, V, dtype=dzt, device="cuda")
    ws = torch.empty(kl.kl_ce_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    kl.kl_ce_argmax(N, V, Z.data_ptr(), T.data_ptr(), loss_ref.data_ptr(), arg_ref.data_ptr(),
                    dz_ref.data_ptr(), dz_dt, ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()

    for call in range(2):      # two calls in a row share the static scratch
        loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        arg = torch.full((N,), -1, dtype=torch.int32, device="cuda")
        dz = torch.full((N, V), float("nan"), dtype=dzt, device="cuda")
        kl.kl_ce_argmax_noalloc(N, V, Z.data_ptr(), T.data_ptr(), loss.data_ptr(), arg.data_ptr(),
                                dz.data_ptr(), dz_dt)
        torch.cuda.synchronize()
        assert abs(loss.item() - loss_ref.item()) <= 1e-6 * max(1.0, abs(loss_ref.item())), call
        assert torch.equal(arg, arg_ref), call
        assert_rel(host(dz), host(dz_ref), 1e-6, f"dlogits call {call}")
    assert kl.kl_device_status() == 0


def test_noalloc_rejects_rows_beyond_static_scratch(kl):
    N = kl.KL_CE_NOALLOC_MAX_ROWS + 1
    with pytest.raises(kl.KLError) as e:
        kl.kl_ce_argmax_noalloc(N, 8, 0, 0, 0, 0, 0, 0)
    assert e.value.status == kl.KL_ERR_UNSUPPORTED
    assert "static scratch" in str(e.value)
