"""Pins of the paged-cache oracle (oracle/paged.py) against things other than
itself: the rotary and attention definitions already pinned in
test_oracle_pins.py (identity block tables must reduce to them), invariants of
the indirection (where a block lives in the pool cannot matter), a closed form
(one key), and the training-path forward (feeding a sequence a chunk and then
one token at a time must reproduce its rows). CPU only."""
import numpy as np
import pytest

import oracle as O
from bwd_qwen3_layer_gb300 import synth


def _rand(rng, *shape, std=1.0):
    return std * rng.standard_normal(shape)


def _identity_tables(B, max_blocks, shuffle_rng=None, n_blocks=None):
    """Tables of B sequences over a pool; with a generator the physical blocks
    are a random permutation of the pool (each sequence's blocks disjoint)."""
    n_blocks = n_blocks or B * max_blocks
    perm = np.arange(n_blocks) if shuffle_rng is None else shuffle_rng.permutation(n_blocks)
    return perm[: B * max_blocks].reshape(B, max_blocks).astype(np.int32)


def test_rope_at_reduces_to_rope_fwd():
    rng = np.random.default_rng(0)
    B, S, heads, d = 2, 11, 3, 16
    x = _rand(rng, B * S, heads, d)
    pos = np.tile(np.arange(S), B)
    for inter in (False, True):
        np.testing.assert_allclose(O.rope_at(x, pos, 1e6, inter), O.rope_fwd(x, B, S, 1e6, inter),
                                   rtol=0, atol=1e-13)


def test_positions_and_write_placement():
    rng = np.random.default_rng(1)
    B, bs, maxb, H, d, n_new = 3, 4, 5, 2, 8, 3
    table = _identity_tables(B, maxb, rng)
    ctx = np.array([0, 5, 13])
    kp0 = np.zeros((B * maxb, bs, H, d))
    k_new = _rand(rng, B * n_new, H, d)
    v_new = _rand(rng, B * n_new, H, d)
    kp, vp = O.paged_write(kp0, kp0, table, ctx, k_new, v_new, n_new)
    pos = O.positions(ctx, n_new)
    assert list(pos) == [0, 1, 2, 5, 6, 7, 13, 14, 15]
    for r, p in enumerate(pos):
        b = r // n_new
        blk, slot = table[b][p // bs], p % bs
        assert np.array_equal(kp[blk, slot], k_new[r]) and np.array_equal(vp[blk, slot], v_new[r])
    # nothing else was touched
    assert np.count_nonzero(np.abs(kp).sum(axis=(2, 3))) == len(pos)


@pytest.mark.parametrize("n_new,Hq,Hkv", [(1, 4, 2), (3, 4, 1), (5, 2, 2)])
def test_identity_tables_reduce_to_attention(n_new, Hq, Hkv):
    """With the whole sequence in the cache, the new queries' rows equal the
    last n_new rows of plain causal attention over the sequence."""
    rng = np.random.default_rng(2)
    B, S, d, bs = 2, 13, 16, 4
    maxb = (S + bs - 1) // bs
    q = _rand(rng, B * S, Hq, d)
    k = _rand(rng, B * S, Hkv, d)
    v = _rand(rng, B * S, Hkv, d)
    Oref, lse_ref = O.attention_fwd(q, k, v, B, S)
    table = _identity_tables(B, maxb)
    kp = np.zeros((B * maxb, bs, Hkv, d))
    ctx0 = np.zeros(B, np.int64)
    kp, vp = O.paged_write(kp, kp, table, ctx0, k, v, S)     # the whole sequences
    ctx = np.full(B, S - n_new)
    rows = np.concatenate([np.arange(b * S + S - n_new, (b + 1) * S) for b in range(B)])
    Op, lse_p = O.paged_attention(q[rows], kp, vp, table, ctx, n_new)
    np.testing.assert_allclose(Op, Oref[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_p, lse_ref[:, :, S - n_new:], rtol=0, atol=1e-12)


def test_block_placement_does_not_matter():
    rng = np.random.default_rng(3)
    B, n_new, Hq, Hkv, d, bs, maxb = 3, 2, 4, 2, 8, 4, 6
    ctx = np.array([3, 9, 17])
    q = _rand(rng, B * n_new, Hq, d)
    k_all = _rand(rng, B, maxb * bs, Hkv, d)
    v_all = _rand(rng, B, maxb * bs, Hkv, d)

    def build(table):
        kp = np.zeros((B * maxb + 4, bs, Hkv, d))
        vp = np.zeros_like(kp)
        for b in range(B):
            for p in range(int(ctx[b]) + n_new):
                kp[table[b][p // bs], p % bs] = k_all[b, p]
                vp[table[b][p // bs], p % bs] = v_all[b, p]
        return kp, vp

    t1 = _identity_tables(B, maxb)
    t2 = _identity_tables(B, maxb, np.random.default_rng(7), n_blocks=B * maxb + 4)
    O1, l1 = O.paged_attention(q, *build(t1), t1, ctx, n_new)
    O2, l2 = O.paged_attention(q, *build(t2), t2, ctx, n_new)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_one_key_closed_form():
    """Empty context, one new token: its softmax has a single key, so O = v
    and lse = q.k / sqrt(d)."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, d, bs = 2, 4, 2, 8, 4
    table = _identity_tables(B, 2)
    q = _rand(rng, B, Hq, d)
    k = _rand(rng, B, Hkv, d)
    v = _rand(rng, B, Hkv, d)
    kp, vp = O.paged_write(np.zeros((2 * B, bs, Hkv, d)), np.zeros((2 * B, bs, Hkv, d)), table,
                           np.zeros(B, np.int64), k, v, 1)
    Op, lse = O.paged_attention(q, kp, vp, table, np.zeros(B, np.int64), 1)
    for b in range(B):
        for h in range(Hq):
            j = h * Hkv // Hq
            np.testing.assert_allclose(Op[b, h], v[b, j], rtol=0, atol=1e-15)
            assert abs(lse[b, h, 0] - q[b, h] @ k[b, j] / np.sqrt(d)) < 1e-13


@pytest.mark.parametrize("qk_norm,inter", [(False, False), (True, True)])
def test_incremental_decode_reproduces_the_training_forward(qk_norm, inter):
    """Prefill a chunk, then feed one token at a time through the paged layer:
    every row equals the corresponding row of layer_forward on the whole
    sequence (positions, rotation, cache writes, causal limit all agree)."""
    B, S, H, Hq, Hkv, d, I, bs = 2, 9, 32, 4, 2, 16, 48, 4
    cfg = O.LayerConfig(B=B, S=S, H=H, Hq=Hq, Hkv=Hkv, d=d, I=I, qk_norm=qk_norm, rope_interleaved=inter)
    w = synth.layer_weights(5, H, Hq, Hkv, d, I, qk_norm=qk_norm)
    X = synth.layer_inputs(5, B * S, H)["X"]
    Y_full, _ = O.layer_forward(cfg, w, X)
    maxb = (S + bs - 1) // bs
    table = _identity_tables(B, maxb, np.random.default_rng(9))
    kp = np.zeros((B * maxb, bs, Hkv, d))
    vp = np.zeros_like(kp)
    Xs = X.reshape(B, S, H)
    Yf = Y_full.reshape(B, S, H)
    chunk = 4
    Y, kp, vp, _ = O.layer_forward_paged(cfg, w, Xs[:, :chunk].reshape(-1, H), kp, vp, table,
                                         np.zeros(B, np.int64), chunk)
    np.testing.assert_allclose(Y.reshape(B, chunk, H), Yf[:, :chunk], rtol=0, atol=1e-10)
    for p in range(chunk, S):
        Y, kp, vp, _ = O.layer_forward_paged(cfg, w, Xs[:, p], kp, vp, table, np.full(B, p), 1)
        np.testing.assert_allclose(Y, Yf[:, p], rtol=0, atol=1e-10)
