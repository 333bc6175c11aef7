"""Shared helpers of the parity tests (comparison only)."""
import numpy as np
import torch

TOL_F32 = 1e-5      # fp32 mode, per-tensor rel-L2
TOL_BF16 = 1.5e-2   # bf16 tensor-core mode, per-tensor rel-L2
TOL_LOSS = 1e-3     # absolute, mean CE loss
ARGMAX_GAP = 1e-2   # argmax must match wherever the oracle's top-2 gap exceeds this


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    if den == 0.0:
        return float(np.linalg.norm(got))
    return float(np.linalg.norm(got - want) / den)


def assert_rel(got, want, tol, name=""):
    r = rel_l2(got, want)
    assert r <= tol, f"{name}: rel-L2 {r:.3e} > {tol:.1e}"
    return r


def dev(a, dtype, device="cuda"):
    return torch.as_tensor(np.asarray(a, np.float64)).to(dtype).to(device).contiguous()


def host(t):
    return t.double().cpu().numpy()


def argmax_ok(z_oracle, arg_gpu, gap=ARGMAX_GAP):
    """Indices of rows whose top-2 gap exceeds `gap` and whose argmax differs."""
    z = np.asarray(z_oracle, np.float64)
    top2 = np.sort(z, axis=1)[:, -2:]
    decided = (top2[:, 1] - top2[:, 0]) > gap
    want = np.argmax(z, axis=1)
    bad = np.nonzero(decided & (want != np.asarray(arg_gpu)))[0]
    return bad, int(decided.sum())
