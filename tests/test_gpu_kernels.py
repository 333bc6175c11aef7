"""Each of the layer's kernels alone against the oracle: RMSNorm forward and
backward, RoPE both directions, SwiGLU forward and backward, causal GQA
attention forward and backward (bf16 tensor cores at head dim 128; fp32 at
small head dims), on ragged sizes."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, assert_rel, dev, host

pytestmark = pytest.mark.gpu

DT = {0: torch.float32, 1: torch.bfloat16}


def _maybe_round(a, dt):
    return synth.round_bf16(a) if dt == 1 else a.astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("dt,rows,width", [(1, 300, 5120), (1, 1500, 5120), (1, 700, 8192), (1, 37, 200),
                                           (0, 1000, 1024), (0, 33, 64), (0, 5, 70)])
def test_rmsnorm(kl, dt, rows, width):
    tol = TOL_BF16 if dt == 1 else 1e-6
    x = _maybe_round(synth.normal(0, "rms.x", (rows, width)), dt)
    g = _maybe_round(synth.normal(0, "rms.g", (width,), std=0.02, mean=1.0), dt)
    dh = synth.normal(0, "rms.dh", (rows, width)).astype(np.float32).astype(np.float64)
    res = _maybe_round(synth.normal(0, "rms.res", (rows, width)), dt)
    eps = 1e-6
    X, G = dev(x, DT[dt]), dev(g, DT[dt])
    H = torch.empty_like(X)
    r = torch.empty(rows, dtype=torch.float32, device="cuda")
    kl.kl_rmsnorm_fwd(rows, width, dt, X.data_ptr(), G.data_ptr(), eps, H.data_ptr(), r.data_ptr())
    h_ref, r_ref = O.rmsnorm_fwd(x, g, eps)
    torch.cuda.synchronize()
    assert_rel(host(H), h_ref, tol, "h")
    assert_rel(host(r), r_ref, 1e-6, "rstd")
    DH = dev(dh, torch.float32)
    RES = dev(res, DT[dt])
    DX = torch.empty_like(X)
    dg = torch.empty(width, dtype=torch.float32, device="cuda")
    ws = torch.empty(kl.kl_rmsnorm_bwd_ws_bytes(rows, width), dtype=torch.uint8, device="cuda")
    kl.kl_rmsnorm_bwd(rows, width, dt, DH.data_ptr(), 0, X.data_ptr(), G.data_ptr(), r.data_ptr(),
                      RES.data_ptr(), DX.data_ptr(), dg.data_ptr(), ws.data_ptr(), ws.numel())
    dx_ref, dg_ref = O.rmsnorm_bwd(dh, x, g, r_ref)
    torch.cuda.synchronize()
    assert_rel(host(DX), dx_ref + res, tol, "dx")
    assert_rel(host(dg), dg_ref, 1e-5, "dgamma")


@pytest.mark.parametrize("dt,B,S,heads,d", [(1, 2, 77, 9, 128), (0, 1, 32, 4, 16), (1, 1, 4096, 2, 128),
                                            (0, 1, 40000, 1, 128)])
def test_rope(kl, dt, B, S, heads, d):
    """Both directions against the oracle; the fp32 case at 40000 positions holds
    the angle reduction (fixed-point turns) to fp32 accuracy far along a sequence."""
    base = 1e6
    x = _maybe_round(synth.normal(0, "rope.x", (B * S, heads, d)), dt)
    X = dev(x.reshape(B * S, heads * d), DT[dt])
    kl.kl_rope(B, S, heads, d, base, dt, X.data_ptr(), 1)
    torch.cuda.synchronize()
    tol = 4e-3 if dt == 1 else 1e-6
    want = O.rope_fwd(x, B, S, base).reshape(B * S, heads * d)
    assert_rel(host(X), want, tol, "rope fwd")
    Y = dev(want, DT[dt])
    kl.kl_rope(B, S, heads, d, base, dt, Y.data_ptr(), -1)
    torch.cuda.synchronize()
    assert_rel(host(Y), O.rope_bwd(want.reshape(B * S, heads, d), B, S, base).reshape(B * S, -1), tol,
               "rope bwd")


@pytest.mark.parametrize("dt,n", [(1, 4096 * 8 + 8), (1, 1001), (0, 5000), (0, 999)])
def test_swiglu(kl, dt, n):
    g = _maybe_round(3 * synth.normal(0, "sw.g", (n,)), dt)
    u = _maybe_round(synth.normal(0, "sw.u", (n,)), dt)
    dm = _maybe_round(synth.normal(0, "sw.dm", (n,)), dt)
    G, U, DM = dev(g, DT[dt]), dev(u, DT[dt]), dev(dm, DT[dt])
    M, DG, DU = torch.empty_like(G), torch.empty_like(G), torch.empty_like(G)
    kl.kl_swiglu_fwd(n, dt, G.data_ptr(), U.data_ptr(), M.data_ptr())
    kl.kl_swiglu_bwd(n, dt, DM.data_ptr(), G.data_ptr(), U.data_ptr(), DG.data_ptr(), DU.data_ptr())
    torch.cuda.synchronize()
    tol = 4e-3 if dt == 1 else 1e-6
    assert_rel(host(M), O.swiglu_fwd(g, u), tol, "m")
    dg_ref, du_ref = O.swiglu_bwd(dm, g, u)
    assert_rel(host(DG), dg_ref, tol, "dg")
    assert_rel(host(DU), du_ref, tol, "du")


ATT_CASES = [
    (1, 2, 200, 8, 2, 128),     # two sequences, ragged vs 64-row tiles, GQA 4:1
    (1, 1, 64, 2, 2, 128),      # exactly one tile, MHA
    (1, 1, 1, 4, 1, 128),       # a single token: O = v0
    (1, 1, 1000, 16, 2, 128),   # longer, GQA 8:1
    (1, 1, 331, 8, 1, 128),     # length not a multiple of 4: lse / D read from global memory
    (0, 1, 32, 4, 2, 16),       # tiny fp32 workload
    (0, 2, 19, 6, 3, 40),
    (1, 2, 700, 64, 8, 128),    # more (head, query-tile) items than SMs: the persistent forward, ragged, B = 2
    (1, 3, 130, 64, 8, 128),    # persistent forward with three sequences of two query tiles each
]


@pytest.mark.parametrize("dt,B,S,Hq,Hkv,d", ATT_CASES)
def test_attention(kl, dt, B, S, Hq, Hkv, d):
    T = B * S
    q = _maybe_round(synth.normal(0, "att.q", (T, Hq, d)), dt)
    k = _maybe_round(synth.normal(0, "att.k", (T, Hkv, d)), dt)
    v = _maybe_round(synth.normal(0, "att.v", (T, Hkv, d)), dt)
    do = _maybe_round(synth.normal(0, "att.do", (T, Hq, d)), dt)
    Q, Kt, Vt, DO = (dev(a.reshape(T, -1), DT[dt]) for a in (q, k, v, do))
    Ot = torch.empty_like(Q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")
    kl.kl_attention_fwd(B, S, Hq, Hkv, d, dt, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                        lse.data_ptr())
    o_ref, lse_ref = O.attention_fwd(q, k, v, B, S)
    torch.cuda.synchronize()
    tol = TOL_BF16 if dt == 1 else 1e-5
    assert_rel(host(Ot), o_ref.reshape(T, -1), tol, "O")
    assert np.max(np.abs(host(lse) - lse_ref)) < (2e-3 if dt == 1 else 1e-5)
    # backward from the GPU's own O (as the layer does)
    o_used = host(Ot).reshape(T, Hq, d)
    dq = torch.empty_like(Q)
    dk = torch.empty_like(Kt)
    dv = torch.empty_like(Vt)
    ws = torch.empty(kl.kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d), dtype=torch.uint8, device="cuda")
    kl.kl_attention_bwd(B, S, Hq, Hkv, d, dt, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                        lse.data_ptr(), DO.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        ws.data_ptr(), ws.numel())
    dq_ref, dk_ref, dv_ref = O.attention_bwd(q, k, v, do, B, S)
    torch.cuda.synchronize()
    del o_used
    assert_rel(host(dq), dq_ref.reshape(T, -1), tol, "dq")
    assert_rel(host(dk), dk_ref.reshape(T, -1), tol, "dk")
    assert_rel(host(dv), dv_ref.reshape(T, -1), tol, "dv")
    if S == 1:
        np.testing.assert_allclose(host(Ot).reshape(T, Hq, d), np.repeat(v, Hq // Hkv, axis=1), rtol=1e-2,
                                   atol=1e-2)


def _att_bwd(kl, B, S, Hq, Hkv, d, Q, Kt, Vt, Ot, lse, DO):
    dq, dk, dv = torch.empty_like(Q), torch.empty_like(Kt), torch.empty_like(Vt)
    ws = torch.empty(kl.kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d), dtype=torch.uint8, device="cuda")
    kl.kl_attention_bwd(B, S, Hq, Hkv, d, 1, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                        lse.data_ptr(), DO.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("B,S,Hq,Hkv", [(1, 300, 8, 1), (2, 130, 16, 2)])
def test_attention_dkdv_group_split(kl, monkeypatch, B, S, Hq, Hkv):
    """dK/dV walk a kv head's whole query-head group in one CTA or split it over
    a cluster of 2 or 4 CTAs (partials summed in rank order through distributed
    shared memory): every split matches the oracle, and each repeats bit for bit."""
    d, T = 128, B * S
    q = synth.round_bf16(synth.normal(5, "att.q", (T, Hq, d)))
    k = synth.round_bf16(synth.normal(5, "att.k", (T, Hkv, d)))
    v = synth.round_bf16(synth.normal(5, "att.v", (T, Hkv, d)))
    do = synth.round_bf16(synth.normal(5, "att.do", (T, Hq, d)))
    Q, Kt, Vt, DO = (dev(a.reshape(T, -1), torch.bfloat16) for a in (q, k, v, do))
    Ot = torch.empty_like(Q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")
    kl.kl_attention_fwd(B, S, Hq, Hkv, d, 1, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                        lse.data_ptr())
    _, dk_ref, dv_ref = O.attention_bwd(q, k, v, do, B, S)
    for split in ("1", "2", "4"):
        monkeypatch.setenv("KL_ATTN_DKDV_SPLIT", split)
        _, dk, dv = _att_bwd(kl, B, S, Hq, Hkv, d, Q, Kt, Vt, Ot, lse, DO)
        assert_rel(host(dk), dk_ref.reshape(T, -1), TOL_BF16, f"dk split {split}")
        assert_rel(host(dv), dv_ref.reshape(T, -1), TOL_BF16, f"dv split {split}")
        _, dk2, dv2 = _att_bwd(kl, B, S, Hq, Hkv, d, Q, Kt, Vt, Ot, lse, DO)
        assert torch.equal(dk, dk2) and torch.equal(dv, dv2), split
    kl.kl_device_status()


def test_attention_bwd_overlap_matches_serial_and_joins(kl):
    """At long sequences the dK/dV kernel runs on a second stream beside the dQ
    kernel (fork and join events). The overlapped backward gives the same bits
    as the one-after-the-other backward (which the launch profiler forces), and
    a library kernel launched on the caller's stream right behind it, with no
    host synchronisation (programmatic dependent launch), reads the finished dK."""
    B, S, Hq, Hkv, d = 1, 16384, 64, 8, 128
    T = B * S
    dn = lambda shp, name: synth.device_normal(shp, 1.0, 0.0, 5, name, torch.bfloat16, "cuda")  # noqa: E731
    Q, DO = dn((T, Hq * d), "ov.q"), dn((T, Hq * d), "ov.do")
    Kt, Vt = dn((T, Hkv * d), "ov.k"), dn((T, Hkv * d), "ov.v")
    Ot = torch.empty_like(Q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")
    kl.kl_attention_fwd(B, S, Hq, Hkv, d, 1, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                        lse.data_ptr())
    ws = torch.empty(kl.kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d), dtype=torch.uint8, device="cuda")

    def bwd():
        dq, dk, dv = torch.empty_like(Q), torch.empty_like(Kt), torch.empty_like(Vt)
        kl.kl_attention_bwd(B, S, Hq, Hkv, d, 1, Q.data_ptr(), Kt.data_ptr(), Vt.data_ptr(), Ot.data_ptr(),
                            lse.data_ptr(), DO.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            ws.data_ptr(), ws.numel())
        return dq, dk, dv

    lib = kl.load()
    lib.kl_profile_enable(1)
    serial = bwd()
    torch.cuda.synchronize()
    lib.kl_profile_enable(0)
    ones = torch.ones(Hkv * d, dtype=torch.bfloat16, device="cuda")
    h_next, r_next = torch.empty_like(Kt), torch.empty(T, dtype=torch.float32, device="cuda")
    overlapped = bwd()
    kl.kl_rmsnorm_fwd(T, Hkv * d, 1, overlapped[1].data_ptr(), ones.data_ptr(), 1e-6, h_next.data_ptr(),
                      r_next.data_ptr())
    torch.cuda.synchronize()
    for a, b, name in zip(serial, overlapped, ("dq", "dk", "dv")):
        assert torch.equal(a, b), name
    h_ref, r_ref = torch.empty_like(Kt), torch.empty(T, dtype=torch.float32, device="cuda")
    kl.kl_rmsnorm_fwd(T, Hkv * d, 1, overlapped[1].data_ptr(), ones.data_ptr(), 1e-6, h_ref.data_ptr(),
                      r_ref.data_ptr())
    torch.cuda.synchronize()
    assert torch.equal(h_next, h_ref) and torch.equal(r_next, r_ref)
    assert float(overlapped[1].float().abs().sum()) > 0.0
    kl.kl_device_status()
