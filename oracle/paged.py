"""fp64 oracle: the forward path with a paged key/value cache.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain definitions with
numpy fp64, no blocking or fusion.

Sources: "From-scratch GPU LLM training" ("What is built": a GPU forward path
with a paged key-value cache) and "KYNETRA FOUNDRY" (paged-KV paragraph: each
sequence's cache is cut into fixed-size token blocks that live anywhere in a
global block pool; a per-sequence block table maps logical token positions to
physical blocks, and attention gathers keys and values through it).

Readings (the pages fix no layout or interface):
* a pool holds [n_blocks, block_size, heads, d]; token position p of sequence
  b lives in physical block table[b, p // block_size], slot p % block_size;
* a step feeds n_new new tokens to each of B sequences; sequence b already
  holds ctx[b] tokens, so new token i sits at absolute position ctx[b] + i;
  the rotary angle and the causal limit use that absolute position;
* the new tokens' keys and values (after the rotation) are written to the
  cache before attention, so a new query attends to its own key.
"""
from __future__ import annotations

import numpy as np

from .qwen3_layer import LayerConfig, _kv_head, linear, rmsnorm_fwd, swiglu_fwd


def rope_at(x: np.ndarray, pos: np.ndarray, base: float, interleaved: bool = False) -> np.ndarray:
    """Rotate row n of x [n, heads, d] by the angles pos[n] * base^(-2i/d)
    (the rotary definition at an arbitrary absolute position)."""
    x = np.asarray(x, np.float64)
    n, nh, d = x.shape
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[:, None] * (base ** (-2.0 * i / d))[None, :]   # [n, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = a * c - b * s
        y[..., 1::2] = a * s + b * c
        return y
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def positions(ctx, n_new: int) -> np.ndarray:
    """Absolute position of each new token, rows ordered b * n_new + i."""
    ctx = np.asarray(ctx, np.int64)
    return (ctx[:, None] + np.arange(n_new)[None, :]).reshape(-1)


def paged_write(k_pool, v_pool, table, ctx, k_new, v_new, n_new: int):
    """Copies of the pools with the new tokens' rows (k_new, v_new [B*n_new,
    heads, d]) placed at their absolute positions through the block table."""
    kp = np.array(k_pool, np.float64, copy=True)
    vp = np.array(v_pool, np.float64, copy=True)
    bs = kp.shape[1]
    B = len(ctx)
    for b in range(B):
        for i in range(n_new):
            p = int(ctx[b]) + i
            blk = int(table[b][p // bs])
            kp[blk, p % bs] = k_new[b * n_new + i]
            vp[blk, p % bs] = v_new[b * n_new + i]
    return kp, vp


def gather(pool, table_row, length: int) -> np.ndarray:
    """The first `length` token rows of one sequence, in position order."""
    bs = pool.shape[1]
    return np.stack([pool[int(table_row[p // bs]), p % bs] for p in range(length)]) if length else \
        np.zeros((0,) + pool.shape[2:])


def paged_attention(q, k_pool, v_pool, table, ctx, n_new: int):
    """Causal GQA attention of the new queries q [B*n_new, Hq, d] over each
    sequence's cached keys and values (positions 0 .. ctx[b] + n_new - 1, the
    new ones included): query i of sequence b sees keys at positions
    <= ctx[b] + i. Scale 1/sqrt(d), query head h reads key/value head
    floor(h * Hkv / Hq). Returns (O [B*n_new, Hq, d], lse [B, Hq, n_new])."""
    q = np.asarray(q, np.float64)
    _, Hq, d = q.shape
    Hkv = k_pool.shape[2]
    B = len(ctx)
    O = np.zeros_like(q)
    lse = np.zeros((B, Hq, n_new))
    for b in range(B):
        L = int(ctx[b]) + n_new
        K = gather(np.asarray(k_pool, np.float64), table[b], L)     # [L, Hkv, d]
        V = gather(np.asarray(v_pool, np.float64), table[b], L)
        for i in range(n_new):
            pos = int(ctx[b]) + i
            for h in range(Hq):
                j = _kv_head(h, Hq, Hkv)
                s = K[: pos + 1, j, :] @ q[b * n_new + i, h, :] / np.sqrt(d)
                mx = np.max(s)
                e = np.exp(s - mx)
                den = np.sum(e)
                O[b * n_new + i, h, :] = (e / den) @ V[: pos + 1, j, :]
                lse[b, h, i] = mx + np.log(den)
    return O, lse


def layer_forward_paged(cfg: LayerConfig, w: dict, X, k_pool, v_pool, table, ctx, n_new: int):
    """The layer forward of layer_forward for n_new new tokens per sequence
    (X [B*n_new, H]) against a paged cache: q, k at their absolute positions,
    the new keys and values written to the cache, then attention over it.
    Returns (Y, k_pool', v_pool', extra) with the updated pool copies."""
    Hq, Hkv, d = cfg.Hq, cfg.Hkv, cfg.d
    X = np.asarray(X, np.float64)
    T = X.shape[0]
    h1, _ = rmsnorm_fwd(X, w["gamma1"], cfg.eps)
    q = linear(h1, w["Wq"]).reshape(T, Hq, d)
    k = linear(h1, w["Wk"]).reshape(T, Hkv, d)
    v = linear(h1, w["Wv"]).reshape(T, Hkv, d)
    if cfg.qk_norm:
        q, _ = rmsnorm_fwd(q, w["gamma_q"], cfg.eps)
        k, _ = rmsnorm_fwd(k, w["gamma_k"], cfg.eps)
    pos = positions(ctx, n_new)
    qr = rope_at(q, pos, cfg.rope_base, cfg.rope_interleaved)
    kr = rope_at(k, pos, cfg.rope_base, cfg.rope_interleaved)
    kp, vp = paged_write(k_pool, v_pool, table, ctx, kr, v, n_new)
    O, lse = paged_attention(qr, kp, vp, table, ctx, n_new)
    x2 = X + linear(O.reshape(T, Hq * d), w["Wo"])
    h2, _ = rmsnorm_fwd(x2, w["gamma2"], cfg.eps)
    m = swiglu_fwd(linear(h2, w["Wg"]), linear(h2, w["Wu"]))
    Y = x2 + linear(m, w["Wd"])
    return Y, kp, vp, dict(q=qr, k=kr, v=v, o=O.reshape(T, Hq * d), lse=lse)
