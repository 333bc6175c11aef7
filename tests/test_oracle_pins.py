"""Pins for the fp64 oracle: each check ties it to something other than
itself (finite differences, brute-force loops, closed forms, invariants,
special cases). CPU only.

Sources of the properties: "From-scratch GPU LLM training" (every gradient
kernel finite-difference verified; layer backward returns 10 tensors; lm-head
CE with argmax) and "KYNETRA FOUNDRY" (pre-norm decoder wiring, GQA groups,
rotary planes whose score depends only on the offset, tiled attention exact).
"""
import math

import numpy as np
import pytest

import oracle as O
from bwd_qwen3_layer_gb300 import synth

RNG = np.random.default_rng(1234)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _fd_dir(f, x, v, h=1e-5):
    """Central finite difference of scalar f along direction v at x."""
    return (f(x + h * v) - f(x - h * v)) / (2 * h)


def _close(a, b, rtol=1e-6, atol=1e-9):
    return abs(a - b) <= atol + rtol * max(abs(a), abs(b))


# ----------------------------------------------------------------------------
# finite-difference pins of every backward
# ----------------------------------------------------------------------------

def test_rmsnorm_fd():
    x, g, R = _rand(3, 7), 1 + 0.1 * _rand(7), _rand(3, 7)
    eps = 1e-3
    _, rstd = O.rmsnorm_fwd(x, g, eps)
    dx, dg = O.rmsnorm_bwd(R, x, g, rstd)
    for _ in range(3):
        v = _rand(*x.shape)
        fd = _fd_dir(lambda t: np.sum(O.rmsnorm_fwd(t, g, eps)[0] * R), x, v)
        assert _close(fd, np.sum(dx * v))
    for j in range(7):
        e = np.zeros(7)
        e[j] = 1
        fd = _fd_dir(lambda t: np.sum(O.rmsnorm_fwd(x, t, eps)[0] * R), g, e)
        assert _close(fd, dg[j])


def test_rope_fd_and_inverse():
    B, S, nh, d = 2, 5, 3, 8
    x, R = _rand(B * S, nh, d), _rand(B * S, nh, d)
    dx = O.rope_bwd(R, B, S, 100.0)
    for _ in range(3):
        v = _rand(*x.shape)
        fd = _fd_dir(lambda t: np.sum(O.rope_fwd(t, B, S, 100.0) * R), x, v)
        assert _close(fd, np.sum(dx * v))
    y = O.rope_fwd(x, B, S, 100.0)
    np.testing.assert_allclose(O.rope_bwd(y, B, S, 100.0), x, rtol=0, atol=1e-13)


def test_swiglu_fd():
    g, u, R = 3 * _rand(4, 6), _rand(4, 6), _rand(4, 6)
    dg, du = O.swiglu_bwd(R, g, u)
    for _ in range(3):
        v = _rand(*g.shape)
        assert _close(_fd_dir(lambda t: np.sum(O.swiglu_fwd(t, u) * R), g, v), np.sum(dg * v))
        assert _close(_fd_dir(lambda t: np.sum(O.swiglu_fwd(g, t) * R), u, v), np.sum(du * v))


@pytest.mark.parametrize("B,S,Hq,Hkv,d", [(1, 6, 4, 2, 4), (2, 5, 4, 1, 6), (1, 4, 2, 2, 4)])
def test_attention_fd(B, S, Hq, Hkv, d):
    T = B * S
    q, k, v, dO = _rand(T, Hq, d), _rand(T, Hkv, d), _rand(T, Hkv, d), _rand(T, Hq, d)
    dq, dk, dv = O.attention_bwd(q, k, v, dO, B, S)

    def L(qq, kk, vv):
        return np.sum(O.attention_fwd(qq, kk, vv, B, S)[0] * dO)

    for _ in range(2):
        w = _rand(*q.shape)
        assert _close(_fd_dir(lambda t: L(t, k, v), q, w), np.sum(dq * w))
        w = _rand(*k.shape)
        assert _close(_fd_dir(lambda t: L(q, t, v), k, w), np.sum(dk * w))
        w = _rand(*v.shape)
        assert _close(_fd_dir(lambda t: L(q, k, t), v, w), np.sum(dv * w))


def test_ce_fd():
    N, H, V = 5, 6, 11
    X, W = _rand(N, H), 0.5 * _rand(V, H)
    tgt = RNG.integers(0, V, N)
    r = O.lmhead_ce(X, W, tgt)
    for _ in range(3):
        v = _rand(*X.shape)
        fd = _fd_dir(lambda t: O.lmhead_ce(t, W, tgt)["loss"], X, v)
        assert _close(fd, np.sum(r["dX"] * v))
        v = _rand(*W.shape)
        fd = _fd_dir(lambda t: O.lmhead_ce(X, t, tgt)["loss"], W, v)
        assert _close(fd, np.sum(r["dW"] * v))


def _layer_fd_check(cfg, seed, ndir=2, h=1e-5, h_for=None):
    w = synth.layer_weights(seed, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I, qk_norm=cfg.qk_norm)
    inp = synth.layer_inputs(seed, cfg.T, cfg.H)
    X, dY = inp["X"], inp["dY"]
    Y, saved = O.layer_forward(cfg, w, X)
    dX, grads, _ = O.layer_backward(cfg, w, saved, dY)

    def L_x(t):
        return np.sum(O.layer_forward(cfg, w, t)[0] * dY)

    for _ in range(ndir):
        v = _rand(*X.shape)
        assert _close(_fd_dir(L_x, X, v, h=h), np.sum(dX * v), rtol=2e-6)
    assert set(grads) == set(w)
    for name in w:
        def L_w(t, name=name):
            ww = dict(w)
            ww[name] = t
            return np.sum(O.layer_forward(cfg, ww, X)[0] * dY)
        for _ in range(ndir):
            v = _rand(*w[name].shape)
            fd = _fd_dir(L_w, w[name], v, h=(h_for or {}).get(name, h))
            assert _close(fd, np.sum(grads[name] * v), rtol=2e-6), name
    return grads


def test_layer_fd_tiny():
    cfg = O.LayerConfig(B=2, S=3, H=8, Hq=4, Hkv=2, d=4, I=12, eps=1e-6, rope_base=1e4)
    _layer_fd_check(cfg, seed=7, ndir=3)


@pytest.mark.parametrize("qk_norm,interleaved", [(True, False), (False, True), (True, True)])
def test_layer_fd_qk_norm_and_interleaved_rope(qk_norm, interleaved):
    """The per-head q/k RMSNorm (gains gamma_q, gamma_k) and the interleaved
    rotary pairing: every gradient, dX and both new gains, against FD."""
    cfg = O.LayerConfig(B=2, S=3, H=8, Hq=4, Hkv=2, d=4, I=12, eps=1e-6, rope_base=1e4,
                        qk_norm=qk_norm, rope_interleaved=interleaved)
    # the per-head norm of small q / k (projection weights N(0, 0.02)) curves the
    # loss sharply along Wq, Wk: a smaller step keeps the O(h^2) error below 2e-6
    grads = _layer_fd_check(cfg, seed=11, ndir=3, h_for={"Wq": 1e-6, "Wk": 1e-6})
    assert ("gamma_q" in grads) == qk_norm


def test_layer_fd_config_tiny_fp32_dims():
    """The tiny fp32 workload's dims: B1 S32 H64 Hq4 Hkv2 d16 I172."""
    cfg = O.LayerConfig(B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172, eps=1e-6, rope_base=1e6)
    _layer_fd_check(cfg, seed=0, ndir=1)


def test_layer_fd_elementwise_gains():
    """Every entry of both norm-gain gradients against its own FD."""
    cfg = O.LayerConfig(B=1, S=4, H=6, Hq=2, Hkv=1, d=4, I=10)
    w = synth.layer_weights(3, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I)
    inp = synth.layer_inputs(3, cfg.T, cfg.H)
    Y, s = O.layer_forward(cfg, w, inp["X"])
    _, grads, _ = O.layer_backward(cfg, w, s, inp["dY"])
    for name in ("gamma1", "gamma2"):
        for j in range(cfg.H):
            e = np.zeros(cfg.H)
            e[j] = 1

            def L(t):
                ww = dict(w)
                ww[name] = t
                return np.sum(O.layer_forward(cfg, ww, inp["X"])[0] * inp["dY"])
            assert _close(_fd_dir(L, w[name], e), grads[name][j], rtol=2e-6)


def test_stack_fd_and_clip():
    cfg = O.LayerConfig(B=1, S=4, H=8, Hq=2, Hkv=1, d=4, I=10)
    layers = [synth.layer_weights(5, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I, prefix=f"l{i}")
              for i in range(2)]
    V = 13
    X = synth.normal(5, "X", (cfg.T, cfg.H))
    W = synth.normal(5, "lm.W", (V, cfg.H), std=0.3)
    tgt = synth.randint(5, "lm.targets", (cfg.T,), V)
    big = O.stack_fwd_bwd(cfg, layers, W, X, tgt, max_norm=1e9)   # no clipping
    assert big["clip_coef"] == 1.0

    def loss(ls, WW):
        x = X
        for w in ls:
            x, _ = O.layer_forward(cfg, w, x)
        return O.lmhead_ce(x, WW, tgt)["loss"]

    for li in range(2):
        for name in ("Wq", "Wd", "gamma2"):
            v = _rand(*layers[li][name].shape)

            def f(t, li=li, name=name):
                ls = [dict(w) for w in layers]
                ls[li][name] = t
                return loss(ls, W)
            assert _close(_fd_dir(f, layers[li][name], v), np.sum(big["grads"][li][name] * v), rtol=2e-6)
    v = _rand(*W.shape)
    assert _close(_fd_dir(lambda t: loss(layers, t), W, v), np.sum(big["dW_lm"] * v), rtol=2e-6)
    # clipping: the clipped gradients have norm max_norm * n / (n + 1e-6)
    n = big["total_norm"]
    mx = 0.5 * n
    c = O.stack_fwd_bwd(cfg, layers, W, X, tgt, max_norm=mx)
    sq = np.sum(c["dW_lm"] ** 2) + sum(np.sum(g[k] ** 2) for g in c["grads"] for k in g)
    assert math.isclose(math.sqrt(sq), mx * n / (n + 1e-6), rel_tol=1e-12)
    assert math.isclose(c["clip_coef"], mx / (n + 1e-6), rel_tol=1e-15)
    assert c["loss"] == big["loss"]


# ----------------------------------------------------------------------------
# attention: brute force and special cases
# ----------------------------------------------------------------------------

def _attention_loops(q, k, v, B, S):
    """Scalar loops with math.exp: an independent plain implementation."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            j = h // grp
            for i in range(S):
                ti = b * S + i
                scores = []
                for jj in range(i + 1):
                    tj = b * S + jj
                    scores.append(sum(q[ti, h, c] * k[tj, j, c] for c in range(d)) / math.sqrt(d))
                m = max(scores)
                ws = [math.exp(s - m) for s in scores]
                tot = sum(ws)
                for c in range(d):
                    out[ti, h, c] = sum(ws[jj] * v[b * S + jj, j, c] for jj in range(i + 1)) / tot
    return out


def test_attention_bruteforce():
    B, S, Hq, Hkv, d = 2, 5, 4, 2, 3
    q, k, v = _rand(B * S, Hq, d), _rand(B * S, Hkv, d), _rand(B * S, Hkv, d)
    Oa, lse = O.attention_fwd(q, k, v, B, S)
    np.testing.assert_allclose(Oa, _attention_loops(q, k, v, B, S), rtol=1e-12, atol=1e-13)
    # lse by brute force
    for b in range(B):
        for h in range(Hq):
            for i in range(S):
                s = [np.dot(q[b * S + i, h], k[b * S + jj, h // 2]) / math.sqrt(d) for jj in range(i + 1)]
                assert math.isclose(lse[b, h, i], math.log(sum(math.exp(x) for x in s)), rel_tol=1e-12, abs_tol=1e-12)


def test_attention_rows_match_full():
    B, S, Hq, Hkv, d = 2, 9, 4, 2, 8
    q, k, v = _rand(B * S, Hq, d), _rand(B * S, Hkv, d), _rand(B * S, Hkv, d)
    Oa, lse = O.attention_fwd(q, k, v, B, S)
    toks, heads = [0, 5, 9, 17, 12], [0, 3, 1, 2, 3]
    orow, lrow = O.attention_fwd_rows(q, k, v, B, S, toks, heads)
    for n, (t, h) in enumerate(zip(toks, heads)):
        np.testing.assert_allclose(orow[n], Oa[t, h], rtol=1e-12, atol=1e-13)
        assert math.isclose(lrow[n], lse[t // S, h, t % S], rel_tol=1e-12)


def test_attention_special_cases():
    d = 4
    # S = 1: the only key is the token itself, so O = v0 (diagonal included)
    q, k, v = _rand(1, 2, d), _rand(1, 1, d), _rand(1, 1, d)
    Oa, lse = O.attention_fwd(q, k, v, 1, 1)
    np.testing.assert_allclose(Oa[0, 0], v[0, 0], rtol=1e-15)
    np.testing.assert_allclose(Oa[0, 1], v[0, 0], rtol=1e-15)
    # q = 0: uniform weights over the causal prefix -> running mean of v
    S = 6
    q, k, v = np.zeros((S, 1, d)), _rand(S, 1, d), _rand(S, 1, d)
    Oa, lse = O.attention_fwd(q, k, v, 1, S)
    for i in range(S):
        np.testing.assert_allclose(Oa[i, 0], v[: i + 1, 0].mean(axis=0), rtol=1e-13)
        assert math.isclose(lse[0, 0, i], math.log(i + 1), rel_tol=1e-14, abs_tol=1e-15)
    # scale 1/sqrt(d): two tokens, k0 = 0, k1 = a e0, q1 = b e0
    a, b = 1.7, 0.9
    q = np.zeros((2, 1, d)); q[1, 0, 0] = b
    k = np.zeros((2, 1, d)); k[1, 0, 0] = a
    v = _rand(2, 1, d)
    p1 = 1.0 / (1.0 + math.exp(-a * b / math.sqrt(d)))
    Oa, _ = O.attention_fwd(q, k, v, 1, 2)
    np.testing.assert_allclose(Oa[1, 0], (1 - p1) * v[0, 0] + p1 * v[1, 0], rtol=1e-14)


def test_attention_causality():
    B, S, Hq, Hkv, d = 1, 8, 2, 1, 4
    q, k, v = _rand(S, Hq, d), _rand(S, Hkv, d), _rand(S, Hkv, d)
    O1, _ = O.attention_fwd(q, k, v, B, S)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[5:] += 1.0
    k2[5:] -= 2.0
    v2[5:] *= 3.0
    O2, _ = O.attention_fwd(q2, k2, v2, B, S)
    assert np.array_equal(O1[:5], O2[:5])


def test_gqa_contiguous_groups():
    """Hq=4, Hkv=2: heads 0,1 read kv-head 0 and heads 2,3 read kv-head 1."""
    S, d = 3, 4
    q, k = _rand(S, 4, d), _rand(S, 2, d)
    v = np.zeros((S, 2, d))
    v[:, 1, :] = 1.0
    Oa, _ = O.attention_fwd(q, k, v, 1, S)
    assert np.all(Oa[:, :2] == 0.0)
    np.testing.assert_allclose(Oa[:, 2:], 1.0, rtol=1e-15)
    # Hkv = Hq is plain multi-head attention: head h is independent of the rest
    q, k, v = _rand(S, 3, d), _rand(S, 3, d), _rand(S, 3, d)
    Oa, _ = O.attention_fwd(q, k, v, 1, S)
    for h in range(3):
        Oh, _ = O.attention_fwd(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], 1, S)
        np.testing.assert_allclose(Oa[:, h], Oh[:, 0], rtol=1e-15)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def test_rope_position_zero_and_norm():
    B, S, d = 2, 7, 16
    x = _rand(B * S, 3, d)
    y = O.rope_fwd(x, B, S, 1e6)
    for b in range(B):
        np.testing.assert_array_equal(y[b * S], x[b * S])      # position restarts at 0
    # each plane keeps its length
    for i in range(d // 2):
        n0 = x[..., i] ** 2 + x[..., i + d // 2] ** 2
        n1 = y[..., i] ** 2 + y[..., i + d // 2] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-13)


def test_rope_relative_offset():
    """<R_m q, R_n k> depends only on m - n."""
    S, d = 12, 8
    q, k = _rand(d), _rand(d)
    Q = O.rope_fwd(np.tile(q, (S, 1))[:, None, :], 1, S, 1e4)[:, 0]
    K = O.rope_fwd(np.tile(k, (S, 1))[:, None, :], 1, S, 1e4)[:, 0]
    for off in range(0, 5):
        vals = [np.dot(Q[m], K[m - off]) for m in range(off, S)]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-12)
    assert not np.isclose(np.dot(Q[4], K[4]), np.dot(Q[4], K[2]))


def test_rope_plane_angles():
    """Unit vector e_i at position s lands at (cos a, sin a) in plane (i, i+d/2)
    with a = s * base^(-2i/d): planes pair i with i + d/2 and the frequency
    falls geometrically."""
    S, d, base = 9, 8, 1e4
    for i in range(d // 2):
        x = np.zeros((S, 1, d))
        x[:, 0, i] = 1.0
        y = O.rope_fwd(x, 1, S, base)[:, 0]
        for s in range(S):
            a = s * base ** (-2.0 * i / d)
            assert math.isclose(y[s, i], math.cos(a), abs_tol=1e-14)
            assert math.isclose(y[s, i + d // 2], math.sin(a), abs_tol=1e-14)
            others = np.delete(y[s], [i, i + d // 2])
            assert np.all(others == 0.0)


def test_rope_interleaved_is_permuted_half():
    """Pairs (2i, 2i+1) with angle i are the rotate-half pairs (i, i+d/2) after
    moving element 2i to i and 2i+1 to i+d/2."""
    B, S, d = 2, 6, 8
    x = _rand(B * S, 3, d)
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])   # half-layout index -> interleaved index
    inv = np.argsort(perm)
    for fn in (O.rope_fwd, O.rope_bwd):
        y_int = fn(x, B, S, 1e4, interleaved=True)
        y_half = fn(x[..., perm], B, S, 1e4)[..., inv]
        np.testing.assert_allclose(y_int, y_half, rtol=0, atol=1e-15)
    # and it is not the rotate-half map itself
    assert not np.allclose(O.rope_fwd(x, B, S, 1e4, interleaved=True), O.rope_fwd(x, B, S, 1e4))


def test_rope_interleaved_relative_offset():
    S, d = 10, 8
    q, k = _rand(d), _rand(d)
    Q = O.rope_fwd(np.tile(q, (S, 1))[:, None, :], 1, S, 1e4, interleaved=True)[:, 0]
    K = O.rope_fwd(np.tile(k, (S, 1))[:, None, :], 1, S, 1e4, interleaved=True)[:, 0]
    for off in range(0, 4):
        vals = [np.dot(Q[m], K[m - off]) for m in range(off, S)]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-12)


def test_qk_norm_closed_forms():
    """With unit gains each head's normalised q (before the rotation, seen at
    position 0 where the rotation is the identity) has RMS 1/sqrt(1 + eps/mean(q^2));
    with eps = 0 the layer output is invariant to scaling Wq and Wk."""
    cfg = O.LayerConfig(B=1, S=3, H=8, Hq=2, Hkv=1, d=4, I=6, eps=1e-3, qk_norm=True)
    w = synth.layer_weights(2, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I, qk_norm=True)
    w["gamma_q"] = np.ones(cfg.d)
    w["gamma_k"] = np.ones(cfg.d)
    X = synth.layer_inputs(2, cfg.T, cfg.H)["X"]
    _, s = O.layer_forward(cfg, w, X)
    qpre = s["q_pre"].reshape(cfg.T, cfg.Hq, cfg.d)
    rms = np.sqrt(np.mean(s["q"][0] ** 2, axis=-1))
    want = 1.0 / np.sqrt(1.0 + cfg.eps / np.mean(qpre[0] ** 2, axis=-1))
    np.testing.assert_allclose(rms, want, rtol=1e-13)
    cfg0 = O.LayerConfig(B=1, S=3, H=8, Hq=2, Hkv=1, d=4, I=6, eps=0.0, qk_norm=True)
    Y0, _ = O.layer_forward(cfg0, w, X)
    w2 = dict(w, Wq=3.0 * w["Wq"], Wk=0.25 * w["Wk"])
    Y1, _ = O.layer_forward(cfg0, w2, X)
    np.testing.assert_allclose(Y1, Y0, rtol=1e-12, atol=1e-14)
    # without the norm the same scaling changes the output
    cfg1 = O.LayerConfig(B=1, S=3, H=8, Hq=2, Hkv=1, d=4, I=6, eps=0.0)
    assert not np.allclose(O.layer_forward(cfg1, w2, X)[0], O.layer_forward(cfg1, w, X)[0])


# ----------------------------------------------------------------------------
# RMSNorm, SiLU, projections
# ----------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    H, eps = 10, 1e-3
    c = 0.37
    x = np.full((1, H), c)
    g = 1 + 0.1 * _rand(H)
    h, r = O.rmsnorm_fwd(x, g, eps)
    np.testing.assert_allclose(h[0], g * c / math.sqrt(c * c + eps), rtol=1e-15)
    # gain 1: RMS(out) = 1 / sqrt(1 + eps / mean(x^2))
    x = _rand(4, H)
    h, _ = O.rmsnorm_fwd(x, np.ones(H), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(h * h, axis=1)), 1 / np.sqrt(1 + eps / ms), rtol=1e-14)
    # eps = 0: scale invariant
    h0, _ = O.rmsnorm_fwd(x, g, 0.0)
    h1, _ = O.rmsnorm_fwd(7.5 * x, g, 0.0)
    np.testing.assert_allclose(h0, h1, rtol=1e-14)
    # identity <dx, x> = eps * rstd^2 * <dn, n> per row (zero at eps = 0)
    dh = _rand(4, H)
    _, r = O.rmsnorm_fwd(x, g, eps)
    dx, _ = O.rmsnorm_bwd(dh, x, g, r)
    n = x * r[:, None]
    lhs = np.sum(dx * x, axis=1)
    rhs = eps * r ** 2 * np.sum(dh * g * n, axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-9, atol=1e-14)


def test_silu_textbook_values():
    assert O.silu(0.0) == 0.0
    assert math.isclose(O.silu(1.0), 0.7310585786300049, rel_tol=1e-15)
    assert math.isclose(O.silu(-1.0), -0.2689414213699951, rel_tol=1e-15)
    assert math.isclose(O.silu(40.0), 40.0, rel_tol=1e-15)
    assert abs(O.silu(-40.0)) < 1e-15
    # gate goes through silu, up is linear
    assert math.isclose(O.swiglu_fwd(1.0, 3.0), 3 * 0.7310585786300049, rel_tol=1e-15)


def test_linear_orientation():
    """Weights are stored [out, in]: W = e_a e_b^T copies input b to output a."""
    x = _rand(3, 5)
    W = np.zeros((4, 5))
    W[2, 1] = 1.0
    y = O.linear(x, W)
    assert y.shape == (3, 4)
    np.testing.assert_array_equal(y[:, 2], x[:, 1])
    assert np.all(np.delete(y, 2, axis=1) == 0.0)


# ----------------------------------------------------------------------------
# cross entropy
# ----------------------------------------------------------------------------

def test_ce_special_cases():
    N, H, V = 4, 6, 37
    X = _rand(N, H)
    tgt = RNG.integers(0, V, N)
    r = O.lmhead_ce(X, np.zeros((V, H)), tgt)
    assert math.isclose(r["loss"], math.log(V), rel_tol=1e-15)
    assert np.all(r["argmax"] == 0)                      # ties -> lowest index
    np.testing.assert_allclose(r["dz"].sum(axis=1), 0.0, atol=1e-15)
    # dz = (softmax - onehot) / N
    z = _rand(N, V)
    loss, arg, dz, lse = O.ce_argmax(z, tgt)
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    oh = np.zeros_like(z)
    oh[np.arange(N), tgt] = 1
    np.testing.assert_allclose(dz, (p - oh) / N, rtol=1e-12, atol=1e-17)
    assert list(arg) == [int(np.argmax(row)) for row in z]
    # a huge logit on the target: loss ~ 0
    z = np.zeros((2, V))
    z[0, 3] = 200.0
    z[1, 9] = 200.0
    loss, arg, dz, _ = O.ce_argmax(z, np.array([3, 9]))
    assert loss < 1e-80 and list(arg) == [3, 9]
    # tie between two maxima -> lower index
    z = np.zeros((1, V))
    z[0, 7] = z[0, 21] = 5.0
    assert O.ce_argmax(z, np.array([0]))[1][0] == 7


# ----------------------------------------------------------------------------
# whole layer invariants
# ----------------------------------------------------------------------------

def test_layer_zero_output_projections():
    """Wo = Wd = 0: residual identity Y = X, dX = dY, and only dWo, dWd are non-zero."""
    cfg = O.LayerConfig(B=2, S=5, H=16, Hq=4, Hkv=2, d=4, I=24)
    w = synth.layer_weights(11, cfg.H, cfg.Hq, cfg.Hkv, cfg.d, cfg.I)
    w["Wo"] = np.zeros_like(w["Wo"])
    w["Wd"] = np.zeros_like(w["Wd"])
    inp = synth.layer_inputs(11, cfg.T, cfg.H)
    Y, s = O.layer_forward(cfg, w, inp["X"])
    assert np.array_equal(Y, inp["X"])
    dX, g, _ = O.layer_backward(cfg, w, s, inp["dY"])
    assert np.array_equal(dX, inp["dY"])
    for name in ("gamma1", "Wq", "Wk", "Wv", "gamma2", "Wg", "Wu"):
        assert np.all(g[name] == 0.0), name
    assert np.any(g["Wo"] != 0.0) and np.any(g["Wd"] != 0.0)
    assert len(g) + 1 == 10        # dX + 9 parameter gradients


def test_layer_sequences_independent():
    """Batch rows never mix: a two-sequence batch equals two one-sequence runs."""
    cfg2 = O.LayerConfig(B=2, S=4, H=8, Hq=2, Hkv=1, d=4, I=12)
    cfg1 = O.LayerConfig(B=1, S=4, H=8, Hq=2, Hkv=1, d=4, I=12)
    w = synth.layer_weights(2, 8, 2, 1, 4, 12)
    X = _rand(8, 8)
    Y2, _ = O.layer_forward(cfg2, w, X)
    Ya, _ = O.layer_forward(cfg1, w, X[:4])
    Yb, _ = O.layer_forward(cfg1, w, X[4:])
    np.testing.assert_allclose(Y2, np.concatenate([Ya, Yb]), rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------
# the layer's wiring ("KYNETRA FOUNDRY", pre-norm decoder paragraph): RMSNorm
# of the layer input -> attention -> residual onto the layer input (x2); then
# RMSNorm of x2 -> SwiGLU MLP -> residual onto x2. Every expected value below
# is assembled from the separately pinned pieces (rmsnorm_fwd, linear,
# rope_fwd, attention_fwd, swiglu_fwd), never from layer_forward itself.
# ----------------------------------------------------------------------------

_WCFG = O.LayerConfig(B=2, S=5, H=16, Hq=4, Hkv=2, d=4, I=24)


def _wiring_weights(seed):
    w = synth.layer_weights(seed, _WCFG.H, _WCFG.Hq, _WCFG.Hkv, _WCFG.d, _WCFG.I)
    # projections scaled so each branch moves the residual stream by O(1):
    # reading the wrong tensor then changes every output by far more than rounding
    return {k: (v if k.startswith("gamma") else 15.0 * v) for k, v in w.items()}


def _attention_branch(cfg, w, X):
    h1, _ = O.rmsnorm_fwd(X, w["gamma1"], cfg.eps)
    q = O.rope_fwd(O.linear(h1, w["Wq"]).reshape(cfg.T, cfg.Hq, cfg.d), cfg.B, cfg.S, cfg.rope_base)
    k = O.rope_fwd(O.linear(h1, w["Wk"]).reshape(cfg.T, cfg.Hkv, cfg.d), cfg.B, cfg.S, cfg.rope_base)
    v = O.linear(h1, w["Wv"]).reshape(cfg.T, cfg.Hkv, cfg.d)
    o, _ = O.attention_fwd(q, k, v, cfg.B, cfg.S)
    return O.linear(o.reshape(cfg.T, cfg.Hq * cfg.d), w["Wo"])


def _mlp_branch(cfg, w, x):
    h2, _ = O.rmsnorm_fwd(x, w["gamma2"], cfg.eps)
    return O.linear(O.swiglu_fwd(O.linear(h2, w["Wg"]), O.linear(h2, w["Wu"])), w["Wd"])


def _wiring_checks(fwd):
    """The three wiring properties of a layer forward `fwd(cfg, w, X) -> (Y, saved)`;
    returns the names of those that fail."""
    cfg = _WCFG
    w = _wiring_weights(21)
    X = synth.layer_inputs(21, cfg.T, cfg.H)["X"]
    failed = []

    def close(a, b):
        return np.allclose(a, b, rtol=1e-12, atol=1e-12)

    # (i) no MLP contribution (Wd = 0): Y is the layer input plus the attention branch
    Y0, _ = fwd(cfg, dict(w, Wd=np.zeros_like(w["Wd"])), X)
    if not close(Y0, X + _attention_branch(cfg, w, X)):
        failed.append("attention residual")
    # (ii) no attention contribution (Wo = 0): Y is the input plus the MLP of its own norm
    Y1, _ = fwd(cfg, dict(w, Wo=np.zeros_like(w["Wo"])), X)
    if not close(Y1, X + _mlp_branch(cfg, w, X)):
        failed.append("mlp residual")
    # (iii) both branches: the MLP normalises the attention half's output x2 (taken
    # from run (i), which (i) ties to the pieces) and its residual lands on x2
    Y, saved = fwd(cfg, w, X)
    if not (close(Y, Y0 + _mlp_branch(cfg, w, Y0))
            and close(saved["x2"], Y0)
            and close(saved["h2"], O.rmsnorm_fwd(Y0, w["gamma2"], cfg.eps)[0])):
        failed.append("mlp reads x2")
    # and the second norm sees the attention branch at all: a change of Wo moves h2
    _, saved2 = fwd(cfg, dict(w, Wo=1.5 * w["Wo"]), X)
    if np.allclose(saved2["h2"], saved["h2"], rtol=1e-3, atol=1e-3):
        failed.append("h2 independent of Wo")
    return failed


def _miswired_forward(kind):
    """A layer forward assembled from the pinned pieces with one plausible
    wiring mistake, to show that _wiring_checks can tell it from the oracle."""
    def fwd(cfg, w, X):
        h1, _ = O.rmsnorm_fwd(X, w["gamma1"], cfg.eps)
        x2 = (h1 if kind == "attention residual onto h1" else X) + _attention_branch(cfg, w, X)
        norm_in = X if kind == "mlp norm reads X" else x2
        h2, _ = O.rmsnorm_fwd(norm_in, w["gamma2"], cfg.eps)
        mlp = O.linear(O.swiglu_fwd(O.linear(h2, w["Wg"]), O.linear(h2, w["Wu"])), w["Wd"])
        Y = (X if kind == "mlp residual onto X" else x2) + mlp
        return Y, {"x2": x2, "h2": h2}
    return fwd


def test_layer_wiring_from_pinned_pieces():
    """The oracle's layer_forward meets all three wiring properties."""
    assert _wiring_checks(O.layer_forward) == []


@pytest.mark.parametrize("kind", ["mlp norm reads X", "mlp residual onto X", "attention residual onto h1"])
def test_layer_wiring_checks_catch_miswiring(kind):
    """Each plausible miswiring of the second half (or of the first residual)
    fails at least one wiring check, while the correctly wired assembly passes."""
    assert _wiring_checks(_miswired_forward("correct")) == []
    assert _wiring_checks(_miswired_forward(kind)) != []
