"""Runs one kernel of the layer at its Qwen3-32B workload shape through the C
ABI, a few times, with a small device footprint: the target for Nsight
Compute captures of a single kernel.

  python -m bwd_qwen3_layer_gb300.profile_case CASE [--iters N]

Cases (T = 2048 tokens, hidden 5120, 64/8 heads of 128, intermediate 25600):
  gemm_gateup   [g|u] = h2 [Wg;Wu]^T  as one 2048 x 51200 x 5120 product (K-major)
  gemm_qkv      q,k,v projections, 2048 x 10240 x 5120
  gemm_dgrad    dm = dY Wd, 2048 x 25600 x 5120 (B MN-major)
  gemm_wgrad    dWd = dY^T m, 5120 x 25600 x 2048 (both MN-major)
  attn_fwd      causal GQA attention forward, S = 2048 (--seq to change)
  attn_bwd      its backward
  ce            CE + argmax + dlogits on 4096 x 151936 fp32 logits (--rows to change)
  rmsnorm_fwd   RMSNorm forward, 2048 x 5120
  rmsnorm_bwd   RMSNorm backward with fp32 dh and a residual gradient, 2048 x 5120
  rope          in-place rotation of q [2048, 64, 128]
  swiglu_fwd    m = silu(g) u over 2048 x 25600
  swiglu_bwd    dg, du over 2048 x 25600
  layer         one whole layer forward + backward (for the layer-internal
                kernels; ~4 GB on the device)
  paged_attn    decode attention over a paged cache: 64 sequences x context
                4096, one new token each, block size 16 (~1.1 GB of cache)
  down_few_rows the decode step's down projection: 64 rows x 25600 against
                5120 x 25600 weights (262 MB) plus the residual, through
                kl_gemm_ex with its scratch (the few-rows kernel)
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bwd_qwen3_layer_gb300 as K  # noqa: E402

T, H, I, HQ, HKV, D = 2048, 5120, 25600, 64, 8, 128


def _rand(shape, std=1.0, dtype=torch.bfloat16):
    return (torch.randn(shape, device="cuda") * std).to(dtype)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seq", type=int, default=T, help="attention cases: sequence length (batch 1)")
    ap.add_argument("--rows", type=int, default=4096, help="ce: rows of logits")
    a = ap.parse_args()
    torch.manual_seed(0)
    K.load()
    bf = K.KL_BF16
    if a.case.startswith("gemm"):
        if a.case == "gemm_gateup":
            M, N, Kd, amn, bmn = T, 2 * I, H, 0, 0
        elif a.case == "gemm_qkv":
            M, N, Kd, amn, bmn = T, HQ * D + 2 * HKV * D, H, 0, 0
        elif a.case == "gemm_dgrad":
            M, N, Kd, amn, bmn = T, I, H, 0, 1
        elif a.case == "gemm_wgrad":
            M, N, Kd, amn, bmn = H, I, T, 1, 1
        else:
            raise SystemExit(f"unknown case {a.case}")
        A = _rand((Kd, M) if amn else (M, Kd))
        B = _rand((Kd, N) if bmn else (N, Kd), 0.02)
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        lda, ldb = (M if amn else Kd), (N if bmn else Kd)

        def run():
            K.kl_gemm(M, N, Kd, bf, A.data_ptr(), lda, amn, B.data_ptr(), ldb, bmn, C.data_ptr(), N, bf)
    elif a.case in ("attn_fwd", "attn_bwd"):
        S = a.seq
        q, k, v = _rand((S, HQ * D)), _rand((S, HKV * D)), _rand((S, HKV * D))
        o = torch.empty_like(q)
        lse = torch.empty(HQ, S, dtype=torch.float32, device="cuda")
        K.kl_attention_fwd(1, S, HQ, HKV, D, bf, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr())
        do = _rand((S, HQ * D))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(K.kl_attention_bwd_ws_bytes(1, S, HQ, HKV, D), dtype=torch.uint8, device="cuda")

        def run():
            if a.case == "attn_fwd":
                K.kl_attention_fwd(1, S, HQ, HKV, D, bf, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr())
            else:
                K.kl_attention_bwd(1, S, HQ, HKV, D, bf, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                   ws.data_ptr(), ws.numel())
    elif a.case == "ce":
        N, V = a.rows, 151936
        z = torch.randn(N, V, device="cuda") * 4
        tgt = torch.randint(0, V, (N,), device="cuda", dtype=torch.int32)
        loss = torch.zeros(1, device="cuda")
        arg = torch.empty(N, dtype=torch.int32, device="cuda")
        dz = torch.empty(N, V, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(K.kl_ce_workspace_bytes(N), dtype=torch.uint8, device="cuda")

        def run():
            K.kl_ce_argmax(N, V, z.data_ptr(), tgt.data_ptr(), loss.data_ptr(), arg.data_ptr(), dz.data_ptr(), bf,
                           ws.data_ptr(), ws.numel())
    elif a.case in ("rmsnorm_fwd", "rmsnorm_bwd"):
        x, gamma = _rand((T, H)), 1.0 + _rand((H,), 0.02)
        h = torch.empty_like(x)
        rstd = torch.empty(T, dtype=torch.float32, device="cuda")
        K.kl_rmsnorm_fwd(T, H, bf, x.data_ptr(), gamma.data_ptr(), 1e-6, h.data_ptr(), rstd.data_ptr())
        dh = torch.randn(T, H, device="cuda")
        resid = _rand((T, H))
        dx = torch.empty_like(x)
        dgamma = torch.empty(H, dtype=torch.float32, device="cuda")
        ws = torch.empty(K.kl_rmsnorm_bwd_ws_bytes(T, H), dtype=torch.uint8, device="cuda")

        def run():
            if a.case == "rmsnorm_fwd":
                K.kl_rmsnorm_fwd(T, H, bf, x.data_ptr(), gamma.data_ptr(), 1e-6, h.data_ptr(), rstd.data_ptr())
            else:
                K.kl_rmsnorm_bwd(T, H, bf, dh.data_ptr(), K.KL_F32, x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(),
                                 resid.data_ptr(), dx.data_ptr(), dgamma.data_ptr(), ws.data_ptr(), ws.numel())
    elif a.case == "rope":
        q = _rand((T, HQ * D))

        def run():
            K.kl_rope(1, T, HQ, D, 1e6, bf, q.data_ptr(), 1)
    elif a.case in ("swiglu_fwd", "swiglu_bwd"):
        g, u, dm = _rand((T, I)), _rand((T, I)), _rand((T, I))
        m, dg, du = torch.empty_like(g), torch.empty_like(g), torch.empty_like(g)

        def run():
            if a.case == "swiglu_fwd":
                K.kl_swiglu_fwd(T * I, bf, g.data_ptr(), u.data_ptr(), m.data_ptr())
            else:
                K.kl_swiglu_bwd(T * I, bf, dm.data_ptr(), g.data_ptr(), u.data_ptr(), dg.data_ptr(), du.data_ptr())
    elif a.case == "paged_attn":
        B, ctx, bs = 64, 4096, 16
        max_blocks = (ctx + 1 + bs - 1) // bs
        n_blocks = B * max_blocks
        kp = _rand((n_blocks, bs, HKV * D))
        vp = _rand((n_blocks, bs, HKV * D))
        table = torch.randperm(n_blocks, device="cuda").to(torch.int32).reshape(B, max_blocks)
        ctx_t = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
        q = _rand((B, HQ * D))
        o = torch.empty_like(q)
        pc = K.PagedCfg(B, 1, bs, max_blocks, n_blocks)
        nb = K.kl_paged_attention_ws_bytes(pc, HQ, HKV, D)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")

        def run():
            K.kl_paged_attention(pc, HQ, HKV, D, bf, q.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(),
                                 ctx_t.data_ptr(), o.data_ptr(), 0, ws.data_ptr(), nb)
    elif a.case == "down_few_rows":
        M, N, Kd = 64, H, I
        A = _rand((M, Kd))
        Bw = _rand((N, Kd), 0.02)
        R = _rand((M, N))
        C = torch.empty_like(R)
        nb = K.kl_gemm_scratch_bytes()
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

        def run():
            K.kl_gemm_ex(M, N, Kd, bf, A.data_ptr(), Kd, 0, Bw.data_ptr(), Kd, 0, C.data_ptr(), N, bf, R.data_ptr(),
                         N, bf, ws=ws.data_ptr(), ws_bytes=nb)
    elif a.case == "layer":
        from . import layer as L
        cfg = L.make_cfg(1, T, H, HQ, HKV, D, I, dtype=bf)
        w = {n: (1.0 + _rand(shp, 0.02)) if n.startswith("gamma") else _rand(shp, 0.02)
             for n, shp in L.weight_shapes(cfg).items()}
        wst = L.weights_struct(w)
        X, dY = _rand((T, H)), _rand((T, H))
        Y, dX = torch.empty_like(X), torch.empty_like(X)
        buf = L.LayerBuffers(cfg, "cuda")
        grads, gst = L.alloc_grads(cfg, "cuda", bf)

        def run():
            K.kl_layer_forward(cfg, wst, X.data_ptr(), Y.data_ptr(), buf.saved, buf.fwd_ws.data_ptr(),
                               buf.fwd_ws.numel())
            K.kl_layer_backward(cfg, wst, buf.saved, dY.data_ptr(), dX.data_ptr(), gst, buf.bwd_ws.data_ptr(),
                                buf.bwd_ws.numel())
    else:
        raise SystemExit(f"unknown case {a.case}")
    for _ in range(a.iters):
        run()
    torch.cuda.synchronize()
    K.kl_device_status()
    print(f"{a.case}: {a.iters} launches ok")


if __name__ == "__main__":
    main()
