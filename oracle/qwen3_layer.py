"""fp64 oracle: one pre-norm Qwen3-style decoder layer, forward and backward,
and the lm-head softmax cross-entropy with argmax.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain definitions,
written out with numpy fp64; a matrix product is the only library primitive
used as a step. No blocking, fusion or reordering.

Layout conventions (a choice; the pages do not fix them): tokens are
flattened t = b*S + s, position of token t is s; weights are stored
[out, in] and applied as y = x @ W.T; q is [T, Hq, d], k and v [T, Hkv, d];
lse is [B, Hq, S].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class LayerConfig:
    B: int
    S: int
    H: int
    Hq: int
    Hkv: int
    d: int
    I: int
    eps: float = 1e-6
    rope_base: float = 1e6
    # Options beyond the pages' layer (whose "10 of 10 tensors" count implies
    # neither): Qwen3's per-head RMSNorm of q and k before the rotation (gains
    # gamma_q, gamma_k of length d shared by all heads), and rotary planes of
    # adjacent pairs (2i, 2i+1) instead of (i, i + d/2).
    qk_norm: bool = False
    rope_interleaved: bool = False

    @property
    def T(self) -> int:
        return self.B * self.S


# ----------------------------------------------------------------------------
# Matrix multiply (capability list: "matrix-multiply" gradient kernel)
# ----------------------------------------------------------------------------

def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T with W stored [out, in]."""
    return np.asarray(x, np.float64) @ np.asarray(W, np.float64).T


# ----------------------------------------------------------------------------
# RMSNorm (capability list: "RMSNorm"; KYNETRA FOUNDRY pre-norm paragraph)
# Reading: epsilon inside the square root, mean over the hidden dimension,
# gain multiplies after normalisation.
# ----------------------------------------------------------------------------

def rmsnorm_fwd(x: np.ndarray, gamma: np.ndarray, eps: float):
    """h = gamma * x / sqrt(mean(x^2) + eps).  Returns (h, rstd[T])."""
    x = np.asarray(x, np.float64)
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    h = np.asarray(gamma, np.float64) * x * rstd[..., None]
    return h, rstd


def rmsnorm_bwd(dh: np.ndarray, x: np.ndarray, gamma: np.ndarray, rstd: np.ndarray):
    """Gradient of rmsnorm_fwd.

    With n = x * rstd and dn = dh * gamma:
      dx = rstd * (dn - n * mean(dn * n))   (mean over the hidden dimension)
      dgamma = sum over tokens of dh * n
    Returns (dx, dgamma).
    """
    dh = np.asarray(dh, np.float64)
    x = np.asarray(x, np.float64)
    n = x * rstd[..., None]
    dn = dh * np.asarray(gamma, np.float64)
    dx = rstd[..., None] * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))
    dgamma = np.sum((dh * n).reshape(-1, x.shape[-1]), axis=0)
    return dx, dgamma


# ----------------------------------------------------------------------------
# Rotary position embedding (capability list: "RoPE"; KYNETRA FOUNDRY rotary
# paragraph: each query/key vector is cut into 2-D planes, each plane turned by
# absolute position times a frequency that falls geometrically across the
# dimensions).
# Readings: plane i pairs element i with element i + d/2 ("rotate half");
# frequency_i = base^(-2i/d), i = 0 .. d/2-1; positions restart at 0 in each
# sequence of the batch.
# ----------------------------------------------------------------------------

def rope_angles(S: int, d: int, base: float) -> np.ndarray:
    """angle[s, i] = s * base^(-2i/d), fp64, shape [S, d/2]."""
    i = np.arange(d // 2, dtype=np.float64)
    freq = base ** (-2.0 * i / d)
    return np.arange(S, dtype=np.float64)[:, None] * freq[None, :]


def _rope_rotate(x: np.ndarray, B: int, S: int, base: float, sign: float,
                 interleaved: bool = False) -> np.ndarray:
    x = np.asarray(x, np.float64)
    T, nh, d = x.shape
    assert T == B * S
    ang = sign * rope_angles(S, d, base)                      # [S, d/2]
    c = np.tile(np.cos(ang), (B, 1))[:, None, :]              # [T, 1, d/2]
    s = np.tile(np.sin(ang), (B, 1))[:, None, :]
    if interleaved:                                           # plane i = (x_2i, x_2i+1)
        a, b = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = a * c - b * s
        y[..., 1::2] = a * s + b * c
        return y
    a, b = x[..., : d // 2], x[..., d // 2:]                  # plane i = (x_i, x_i+d/2)
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def rope_fwd(x: np.ndarray, B: int, S: int, base: float, interleaved: bool = False) -> np.ndarray:
    """Rotate each plane by +angle[s, i]; x is [T, heads, d]. Plane i is
    (x_i, x_{i+d/2}), or (x_{2i}, x_{2i+1}) when interleaved."""
    return _rope_rotate(x, B, S, base, +1.0, interleaved)


def rope_bwd(dy: np.ndarray, B: int, S: int, base: float, interleaved: bool = False) -> np.ndarray:
    """Gradient of rope_fwd: the rotation is orthogonal, so rotate by -angle."""
    return _rope_rotate(dy, B, S, base, -1.0, interleaved)


# ----------------------------------------------------------------------------
# Causal grouped-query scaled-dot-product attention (capability list:
# "scaled-dot-product attention"; KYNETRA FOUNDRY grouped-query paragraph and
# tiled-attention paragraph: tiling is exact, so this is plain attention with
# the full score matrix materialised).
# Readings: scale 1/sqrt(d); the causal mask keeps keys j <= i (diagonal
# included); query head h reads key/value head floor(h * Hkv / Hq)
# (contiguous groups).
# ----------------------------------------------------------------------------

def _kv_head(h: int, Hq: int, Hkv: int) -> int:
    return (h * Hkv) // Hq


def attention_fwd(q, k, v, B: int, S: int):
    """q [T,Hq,d], k/v [T,Hkv,d] -> (O [T,Hq,d], lse [B,Hq,S])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    O = np.zeros_like(q)
    lse = np.zeros((B, Hq, S))
    mask = np.tril(np.ones((S, S), dtype=bool))
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        for h in range(Hq):
            j = _kv_head(h, Hq, Hkv)
            s = q[rows, h, :] @ k[rows, j, :].T / np.sqrt(d)
            s = np.where(mask, s, -np.inf)
            mx = np.max(s, axis=1, keepdims=True)
            e = np.exp(s - mx)
            den = np.sum(e, axis=1, keepdims=True)
            P = e / den
            O[rows, h, :] = P @ v[rows, j, :]
            lse[b, h, :] = (mx + np.log(den))[:, 0]
    return O, lse


def attention_fwd_rows(q, k, v, B: int, S: int, tokens, heads):
    """Attention output and lse for selected (token, head) pairs only.

    Same definition as attention_fwd, evaluated one query row at a time so a
    full-size run can be sampled. Returns (O_rows [n, d], lse_rows [n]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    outs, lses = [], []
    for t, h in zip(tokens, heads):
        b, s_pos = divmod(int(t), S)
        j = _kv_head(int(h), Hq, Hkv)
        keys = slice(b * S, b * S + s_pos + 1)
        s = k[keys, j, :] @ q[t, h, :] / np.sqrt(d)
        mx = np.max(s)
        e = np.exp(s - mx)
        den = np.sum(e)
        outs.append((e / den) @ v[keys, j, :])
        lses.append(mx + np.log(den))
    return np.array(outs), np.array(lses)


def attention_bwd(q, k, v, dO, B: int, S: int):
    """Gradients of attention_fwd with respect to q, k, v.

    Per head, with P the softmax matrix:
      dV = P^T dO;  dP = dO V^T;  dS = P * (dP - rowsum(P * dP));
      dQ = dS K / sqrt(d);  dK = dS^T Q / sqrt(d);
    dK and dV of a key/value head are summed over its query-head group.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    mask = np.tril(np.ones((S, S), dtype=bool))
    sc = 1.0 / np.sqrt(d)
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        for h in range(Hq):
            j = _kv_head(h, Hq, Hkv)
            s = q[rows, h, :] @ k[rows, j, :].T * sc
            s = np.where(mask, s, -np.inf)
            e = np.exp(s - np.max(s, axis=1, keepdims=True))
            P = e / np.sum(e, axis=1, keepdims=True)
            dv[rows, j, :] += P.T @ dO[rows, h, :]
            dP = dO[rows, h, :] @ v[rows, j, :].T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            dq[rows, h, :] = dS @ k[rows, j, :] * sc
            dk[rows, j, :] += dS.T @ q[rows, h, :] * sc
    return dq, dk, dv


# ----------------------------------------------------------------------------
# SiLU / SwiGLU (capability list: "SiLU / SwiGLU"; KYNETRA FOUNDRY pre-norm
# paragraph: gated SwiGLU feed-forward).  Reading: m = silu(gate) * up.
# ----------------------------------------------------------------------------

def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    x = np.asarray(x, np.float64)
    return x * _sigmoid(x)


def swiglu_fwd(g, u):
    return silu(g) * np.asarray(u, np.float64)


def swiglu_bwd(dm, g, u):
    """dg = dm * u * silu'(g), silu'(g) = s(g) (1 + g (1 - s(g))); du = dm * silu(g)."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    dm = np.asarray(dm, np.float64)
    sg = _sigmoid(g)
    dg = dm * u * sg * (1.0 + g * (1.0 - sg))
    du = dm * g * sg
    return dg, du


# ----------------------------------------------------------------------------
# The decoder layer (KYNETRA FOUNDRY pre-norm paragraph; "From-scratch GPU LLM
# training", "What is built": forward with saved activations, backward to
# 10 tensors = dX, 7 projection gradients and 2 norm-gain gradients, which
# implies no biases and no per-head q/k norms).
# ----------------------------------------------------------------------------

def layer_forward(cfg: LayerConfig, w: dict, X: np.ndarray):
    """Y = x2 + W_down(silu(W_gate h2) * W_up h2), h2 = RMSNorm(x2; gamma2),
    x2 = X + W_o Attn(RoPE(W_q h1), RoPE(W_k h1), W_v h1), h1 = RMSNorm(X; gamma1).

    Returns (Y, saved) with every intermediate in fp64.
    """
    T, Hq, Hkv, d = cfg.T, cfg.Hq, cfg.Hkv, cfg.d
    X = np.asarray(X, np.float64)
    h1, rstd1 = rmsnorm_fwd(X, w["gamma1"], cfg.eps)
    q = linear(h1, w["Wq"]).reshape(T, Hq, d)
    k = linear(h1, w["Wk"]).reshape(T, Hkv, d)
    v = linear(h1, w["Wv"]).reshape(T, Hkv, d)
    extra = {}
    if cfg.qk_norm:
        # each head's d features normalised like the pre-norm RMSNorm, one gain per feature
        qn, rstd_q = rmsnorm_fwd(q, w["gamma_q"], cfg.eps)
        kn, rstd_k = rmsnorm_fwd(k, w["gamma_k"], cfg.eps)
        extra = dict(q_pre=q.reshape(T, Hq * d), k_pre=k.reshape(T, Hkv * d), rstd_q=rstd_q, rstd_k=rstd_k)
        q, k = qn, kn
    qr = rope_fwd(q, cfg.B, cfg.S, cfg.rope_base, cfg.rope_interleaved)
    kr = rope_fwd(k, cfg.B, cfg.S, cfg.rope_base, cfg.rope_interleaved)
    O, lse = attention_fwd(qr, kr, v, cfg.B, cfg.S)
    O2 = O.reshape(T, Hq * d)
    x2 = X + linear(O2, w["Wo"])
    h2, rstd2 = rmsnorm_fwd(x2, w["gamma2"], cfg.eps)
    g = linear(h2, w["Wg"])
    u = linear(h2, w["Wu"])
    m = swiglu_fwd(g, u)
    Y = x2 + linear(m, w["Wd"])
    saved = dict(X=X, h1=h1, rstd1=rstd1, q=qr, k=kr, v=v, o=O2, lse=lse,
                 x2=x2, h2=h2, rstd2=rstd2, g=g, u=u, m=m, **extra)
    return Y, saved


def layer_backward(cfg: LayerConfig, w: dict, saved: dict, dY: np.ndarray):
    """Backward of layer_forward. Returns (dX, grads) with grads keyed like the
    weights: gamma1, Wq, Wk, Wv, Wo, gamma2, Wg, Wu, Wd (and gamma_q, gamma_k
    with qk_norm)."""
    T, Hq, Hkv, d = cfg.T, cfg.Hq, cfg.Hkv, cfg.d
    dY = np.asarray(dY, np.float64)
    s = saved
    # MLP
    dm = dY @ w["Wd"]
    dWd = dY.T @ s["m"]
    dg, du = swiglu_bwd(dm, s["g"], s["u"])
    dh2 = dg @ w["Wg"] + du @ w["Wu"]
    dWg = dg.T @ s["h2"]
    dWu = du.T @ s["h2"]
    dx2_n, dgamma2 = rmsnorm_bwd(dh2, s["x2"], w["gamma2"], s["rstd2"])
    dx2 = dY + dx2_n
    # attention block
    dO = (dx2 @ w["Wo"]).reshape(T, Hq, d)
    dWo = dx2.T @ s["o"]
    dqr, dkr, dv = attention_bwd(s["q"], s["k"], s["v"], dO, cfg.B, cfg.S)
    dq = rope_bwd(dqr, cfg.B, cfg.S, cfg.rope_base, cfg.rope_interleaved)
    dk = rope_bwd(dkr, cfg.B, cfg.S, cfg.rope_base, cfg.rope_interleaved)
    qk_grads = {}
    if cfg.qk_norm:
        dq, qk_grads["gamma_q"] = rmsnorm_bwd(dq, s["q_pre"].reshape(T, Hq, d), w["gamma_q"], s["rstd_q"])
        dk, qk_grads["gamma_k"] = rmsnorm_bwd(dk, s["k_pre"].reshape(T, Hkv, d), w["gamma_k"], s["rstd_k"])
    dq = dq.reshape(T, Hq * d)
    dk = dk.reshape(T, Hkv * d)
    dv = dv.reshape(T, Hkv * d)
    dh1 = dq @ w["Wq"] + dk @ w["Wk"] + dv @ w["Wv"]
    dWq = dq.T @ s["h1"]
    dWk = dk.T @ s["h1"]
    dWv = dv.T @ s["h1"]
    dX_n, dgamma1 = rmsnorm_bwd(dh1, s["X"], w["gamma1"], s["rstd1"])
    dX = dx2 + dX_n
    grads = dict(gamma1=dgamma1, Wq=dWq, Wk=dWk, Wv=dWv, Wo=dWo,
                 gamma2=dgamma2, Wg=dWg, Wu=dWu, Wd=dWd, **qk_grads)
    inter = dict(dm=dm, dg=dg, du=du, dh2=dh2, dx2=dx2, dO=dO.reshape(T, Hq * d),
                 dq=dq, dk=dk, dv=dv, dh1=dh1)
    return dX, grads, inter


# ----------------------------------------------------------------------------
# lm-head softmax cross-entropy with argmax ("From-scratch GPU LLM training",
# capability list: "GPU lm-head - softmax cross-entropy + argmax fused in a
# single launch").
# Readings: loss is the mean over tokens; dlogits = (softmax - onehot) / N;
# argmax is the lowest index attaining the row maximum; no final norm before
# the head; the head weight is untied and stored [V, H].
# ----------------------------------------------------------------------------

def ce_argmax(z: np.ndarray, targets: np.ndarray):
    """Per-row logsumexp, mean loss, argmax and dlogits of logits z [N, V]."""
    z = np.asarray(z, np.float64)
    N, V = z.shape
    tgt = np.asarray(targets, np.int64)
    mx = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - mx)
    den = np.sum(e, axis=1, keepdims=True)
    lse = (mx + np.log(den))[:, 0]
    loss_rows = lse - z[np.arange(N), tgt]
    arg = np.argmax(z, axis=1)          # numpy returns the first maximal index
    dz = e / den
    dz[np.arange(N), tgt] -= 1.0
    dz /= N
    return float(np.mean(loss_rows)), arg.astype(np.int64), dz, lse


def lmhead_ce(X: np.ndarray, W: np.ndarray, targets: np.ndarray):
    """z = X W^T; mean CE loss, argmax, dlogits, dX = dz W, dW = dz^T X."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    z = X @ W.T
    loss, arg, dz, lse = ce_argmax(z, targets)
    dX = dz @ W
    dW = dz.T @ X
    return dict(loss=loss, argmax=arg, z=z, dz=dz, lse=lse, dX=dX, dW=dW)
