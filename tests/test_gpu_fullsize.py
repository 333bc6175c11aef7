"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times.

* One Qwen3-32B-shaped layer, bf16, batch 1 x seq 2048: the whole forward and
  backward against the fp64 oracle on every tensor (the oracle needs ~20 s of
  host fp64 here).
* Long-context GQA attention, seq 32768, 64/8 heads: sampled (token, head)
  rows of O, lse and dQ against the oracle's one-row evaluation; dK/dV on key
  rows near the end of the sequence (their query columns are short); and two
  whole-sequence identities: the sum over keys of dK is zero for every
  key/value head, and the sum over keys of dV equals the sum of dO over the
  head group's query rows.
* lm-head, 4096 tokens x vocab 151936: sampled logit rows against X W^T, the
  CE step on the kernel's own fp32 logits (every row), sampled dX rows and dW
  rows against their definitions.

Inputs are drawn on the device (seeded) and read back for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import layer as L
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, TOL_LOSS, argmax_ok, assert_rel, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

QWEN = dict(H=5120, Hq=64, Hkv=8, d=128, I=25600)


def _dev_normal(shape, std, mean, name, seed=11):
    return synth.device_normal(shape, std, mean, seed, name, torch.bfloat16, "cuda")


def test_qwen3_layer_T2048_full_parity(kl):
    B, S = 1, 2048
    cfg = L.make_cfg(B, S, **QWEN, dtype=kl.KL_BF16)
    w = {}
    for n, shp in L.weight_shapes(cfg).items():
        w[n] = _dev_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, f"full.{n}")
    T = B * S
    X = _dev_normal((T, QWEN["H"]), 1.0, 0.0, "full.X")
    dY = _dev_normal((T, QWEN["H"]), 1.0, 0.0, "full.dY")
    w_host = {L.SYNTH_NAMES[n]: host(t) for n, t in w.items()}
    got = L.run_layer(cfg, w_host, host(X), host(dY))
    ocfg = O.LayerConfig(B=B, S=S, **QWEN)
    Y, saved = O.layer_forward(ocfg, w_host, host(X))
    assert_rel(got["Y"], Y, TOL_BF16, "Y")
    for k in ("h1", "q", "k", "v", "o", "x2", "h2", "g", "u", "m"):
        assert_rel(got["saved"][k], saved[k].reshape(got["saved"][k].shape), TOL_BF16, k)
    assert_rel(got["saved"]["lse"], saved["lse"], TOL_BF16, "lse")
    dX, grads, _ = O.layer_backward(ocfg, w_host, saved, host(dY))
    assert_rel(got["dX"], dX, TOL_BF16, "dX")
    for n, g in grads.items():
        assert_rel(got["d" + n], g, TOL_BF16, "d" + n)


def test_qwen3_layer_T2048_forward_bit_reproducible(kl):
    """At full size the q/k/v, O and down projections split their last round of
    tiles along K; the pieces are summed in a fixed order whichever CTA lands
    last, so the whole forward (every saved tensor and Y) repeats bit for bit."""
    B, S = 1, 2048
    cfg = L.make_cfg(B, S, **QWEN, dtype=kl.KL_BF16)
    w = {n: _dev_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, f"rep.{n}")
         for n, shp in L.weight_shapes(cfg).items()}
    X = _dev_normal((B * S, QWEN["H"]), 1.0, 0.0, "rep.X")
    ws = L.weights_struct(w)
    buf = L.LayerBuffers(cfg, "cuda")
    outs = []
    for _ in range(2):
        Y = torch.empty_like(X)
        kl.kl_layer_forward(cfg, ws, X.data_ptr(), Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(),
                            buf.fwd_ws.numel())
        torch.cuda.synchronize()
        outs.append((Y.clone(), buf.saved_mem.clone()))
    kl.kl_device_status()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


def test_qwen3_layer_T2048_backward_bit_reproducible(kl):
    """The full-size backward in the bench's launch configuration repeats bit
    for bit: dX and every weight gradient (the attention's dK/dV partials meet
    in rank order, every GEMM output element is summed in one fixed order)."""
    B, S = 1, 2048
    cfg = L.make_cfg(B, S, **QWEN, dtype=kl.KL_BF16)
    w = {n: _dev_normal(shp, 0.02, 1.0 if n.startswith("gamma") else 0.0, f"repb.{n}")
         for n, shp in L.weight_shapes(cfg).items()}
    X = _dev_normal((B * S, QWEN["H"]), 1.0, 0.0, "repb.X")
    dY = _dev_normal((B * S, QWEN["H"]), 1.0, 0.0, "repb.dY")
    ws = L.weights_struct(w)
    buf = L.LayerBuffers(cfg, "cuda")
    grads, gst = L.alloc_grads(cfg, "cuda", kl.KL_BF16)
    Y = torch.empty_like(X)
    kl.kl_layer_forward(cfg, ws, X.data_ptr(), Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(), buf.fwd_ws.numel())
    outs = []
    for _ in range(2):
        dX = torch.empty_like(X)
        kl.kl_layer_backward(cfg, ws, buf.saved, dY.data_ptr(), dX.data_ptr(), gst, buf.bwd_ws.data_ptr(),
                             buf.bwd_ws.numel())
        torch.cuda.synchronize()
        outs.append([dX.clone()] + [grads[n].clone() for n in sorted(grads)])
    kl.kl_device_status()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


def test_attention_S32768_sampled_and_invariants(kl):
    B, S, Hq, Hkv, d = 1, 32768, 64, 8, 128
    T = B * S
    q = _dev_normal((T, Hq * d), 1.0, 0.0, "att32k.q")
    k = _dev_normal((T, Hkv * d), 1.0, 0.0, "att32k.k")
    v = _dev_normal((T, Hkv * d), 1.0, 0.0, "att32k.v")
    do = _dev_normal((T, Hq * d), 1.0, 0.0, "att32k.do")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")
    kl.kl_attention_fwd(B, S, Hq, Hkv, d, kl.KL_BF16, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr())
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(kl.kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d), dtype=torch.uint8, device="cuda")
    kl.kl_attention_bwd(B, S, Hq, Hkv, d, kl.KL_BF16, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                        ws.numel())
    torch.cuda.synchronize()
    qh, kh, vh, doh = (host(t) for t in (q, k, v, do))
    qh, doh = qh.reshape(T, Hq, d), doh.reshape(T, Hq, d)
    kh, vh = kh.reshape(T, Hkv, d), vh.reshape(T, Hkv, d)
    oh, lseh = host(o).reshape(T, Hq, d), host(lse)
    rng = np.random.default_rng(0)
    toks = np.concatenate([[0, 1, 63, 64, 4095, S - 1], rng.integers(0, S, 26)])
    heads = rng.integers(0, Hq, len(toks))
    o_ref, lse_ref = O.attention_fwd_rows(qh, kh, vh, B, S, toks, heads)
    assert_rel(np.array([oh[t, h] for t, h in zip(toks, heads)]), o_ref, TOL_BF16, "O rows")
    assert_rel(np.array([lseh[0, h, t] for t, h in zip(toks, heads)]), lse_ref, TOL_BF16, "lse rows")
    # dQ rows: dS_row = P_row * (dP_row - D_row), dq = dS_row K / sqrt(d)
    grp = Hq // Hkv
    dqh = host(dq).reshape(T, Hq, d)
    want, gotr = [], []
    for t, h in zip(toks, heads):
        j = h // grp
        s = kh[: t + 1, j] @ qh[t, h] / np.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        dp = vh[: t + 1, j] @ doh[t, h]
        ds = p * (dp - np.dot(p, dp))
        want.append(ds @ kh[: t + 1, j] / np.sqrt(d))
        gotr.append(dqh[t, h])
    assert_rel(np.array(gotr), np.array(want), TOL_BF16, "dQ rows")
    # dK, dV on the last keys of the sequence: only queries i >= key contribute
    dkh, dvh = host(dk).reshape(T, Hkv, d), host(dv).reshape(T, Hkv, d)
    keys = np.array([S - 1, S - 2, S - 17, S - 100, S - 511])
    tail = S - 512
    for j in (0, Hkv - 1):
        dk_want = np.zeros((len(keys), d))
        dv_want = np.zeros((len(keys), d))
        for h in range(j * grp, (j + 1) * grp):
            sc = qh[tail:, h] @ kh[:, j].T / np.sqrt(d)          # [512, S]
            mask = np.arange(S)[None, :] <= np.arange(tail, S)[:, None]
            sc = np.where(mask, sc, -np.inf)
            P = np.exp(sc - sc.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            dP = doh[tail:, h] @ vh[:, j].T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            for n, key in enumerate(keys):
                dk_want[n] += dS[:, key] @ qh[tail:, h] / np.sqrt(d)
                dv_want[n] += P[:, key] @ doh[tail:, h]
        assert_rel(dkh[keys, j], dk_want, TOL_BF16, f"dK tail rows head {j}")
        assert_rel(dvh[keys, j], dv_want, TOL_BF16, f"dV tail rows head {j}")
    # whole-sequence identities over every key
    for j in range(Hkv):
        scale = np.linalg.norm(dkh[:, j], axis=1).sum()
        assert np.linalg.norm(dkh[:, j].sum(axis=0)) < 1e-2 * scale
        dv_sum_want = doh[:, j * grp:(j + 1) * grp].sum(axis=(0, 1))
        assert_rel(dvh[:, j].sum(axis=0), dv_sum_want, TOL_BF16, f"sum dV head {j}")


def test_lmhead_N4096_V151936_sampled(kl):
    N, H, V = 4096, 5120, 151936
    X = _dev_normal((N, H), 1.0, 0.0, "lm.X")
    W = _dev_normal((V, H), 0.02, 0.0, "lm.W")
    tgt = synth.device_randint((N,), V, 11, "lm.targets", "cuda")
    cfg = L.lmhead_cfg(N, H, V, kl.KL_BF16)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    arg = torch.empty(N, dtype=torch.int32, device="cuda")
    dz = torch.empty(N, V, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, H, dtype=torch.bfloat16, device="cuda")
    ws = L.lmhead_ws(cfg, "cuda")
    kl.kl_lmhead_ce_argmax(cfg, X.data_ptr(), W.data_ptr(), tgt.data_ptr(), loss.data_ptr(), arg.data_ptr(),
                           dz.data_ptr(), dX.data_ptr(), dW.data_ptr(), ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    Xh, Wh = host(X), host(W)
    t = tgt.cpu().numpy().astype(np.int64)
    zt = ws[: N * V * 4].view(torch.float32).view(N, V)
    rng = np.random.default_rng(1)
    rows = np.concatenate([[0, N - 1], rng.integers(0, N, 14)])
    cols = np.concatenate([t[:4], rng.integers(0, V, 12)])
    z_ref = Xh[rows] @ Wh.T
    assert_rel(zt[torch.as_tensor(rows, device="cuda")].double().cpu().numpy(), z_ref, 1e-5, "logit rows")
    bad, decided = argmax_ok(z_ref, arg.cpu().numpy()[rows])
    assert len(bad) == 0 and decided > 0
    # the CE step on the kernel's own fp32 logits, every row (blocks of rows)
    loss_ref, arg_ref = 0.0, []
    dz_rows = {}
    dz_cols = np.zeros((N, len(cols)))
    for r0 in range(0, N, 256):
        zb = zt[r0:r0 + 256].double().cpu().numpy()
        lb, ab, dzb, _ = O.ce_argmax(zb, t[r0:r0 + 256])
        nb = zb.shape[0]
        loss_ref += lb * nb / N
        dzb *= nb / N                      # the oracle scaled by 1/nb; the batch is N
        arg_ref.append(ab)
        dz_cols[r0:r0 + nb] = dzb[:, cols]
        for r in rows:
            if r0 <= r < r0 + nb:
                dz_rows[int(r)] = dzb[r - r0]
    assert abs(loss.item() - loss_ref) <= TOL_LOSS
    assert np.array_equal(arg.cpu().numpy(), np.concatenate(arg_ref))
    dzr = np.array([dz_rows[int(r)] for r in rows])
    assert_rel(host(dz[torch.as_tensor(rows, device="cuda")]), dzr, 4e-3, "dlogit rows")
    # dX rows = dz W, dW rows = dz[:, v]^T X
    assert_rel(host(dX)[rows], dzr @ Wh, TOL_BF16, "dX rows")
    assert_rel(host(dW[torch.as_tensor(cols, device="cuda")]), dz_cols.T @ Xh, TOL_BF16, "dW rows")
