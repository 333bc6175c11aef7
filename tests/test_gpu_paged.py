"""The forward path with a paged key/value cache through the C ABI against the
oracle (oracle/paged.py): cache writes (exact), decode and chunked attention
over ragged contexts with and without context splits, the paged layer
forward, incremental decode against the training-path forward, and a table
entry outside the pool reported instead of followed."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import layer as L
from bwd_qwen3_layer_gb300 import synth
from _parity import TOL_BF16, assert_rel

pytestmark = pytest.mark.gpu

D = 128


def _bf(a):
    return synth.round_bf16(np.asarray(a, np.float64))


def _dev(a, dtype=torch.bfloat16):
    if dtype == torch.int32:
        return torch.as_tensor(np.asarray(a, np.int32)).cuda()
    return torch.as_tensor(np.asarray(a, np.float64)).to(dtype).cuda()


def _case(seed, B, n_new, Hq, Hkv, bs, ctx, extra_blocks=3):
    """Random bf16 pools with every slot filled, block tables over a shuffled
    pool, and new queries."""
    rng = np.random.default_rng(seed)
    max_blocks = max((c + n_new + bs - 1) // bs for c in ctx)
    n_blocks = B * max_blocks + extra_blocks
    table = rng.permutation(n_blocks)[: B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    kp = _bf(rng.standard_normal((n_blocks, bs, Hkv, D)))
    vp = _bf(rng.standard_normal((n_blocks, bs, Hkv, D)))
    q = _bf(rng.standard_normal((B * n_new, Hq, D)))
    return table, kp, vp, q, max_blocks, n_blocks


@pytest.mark.parametrize("B,n_new,Hq,Hkv,bs,ctx", [
    (3, 1, 8, 1, 16, [0, 17, 300]),          # decode, ragged contexts, one kv head of 8
    (2, 4, 8, 2, 16, [5, 130]),              # chunked prefill rows (4 x 4 = 16 rows per kv head)
    (64, 1, 8, 1, 16, [40] * 64),            # many sequences: no context split
    (1, 1, 64, 8, 32, [2000]),               # one long sequence: context split + combine
    (2, 2, 4, 2, 8, [0, 1]),                 # tiny contexts
    (2, 8, 8, 1, 16, [100, 3]),              # 64 rows per kv head: four row groups
    (6, 1, 16, 2, 16, [0, 1, 63, 64, 65, 1000]),   # ragged around the 64-key tile edge
    (40, 1, 64, 8, 16, [700] * 40),          # runs of several tiles cut items into pieces
    (3, 3, 12, 4, 5, [7, 0, 190]),           # block size 5, three new tokens, 9 rows
])
def test_paged_attention_matches_oracle(kl, B, n_new, Hq, Hkv, bs, ctx):
    table, kp, vp, q, max_blocks, n_blocks = _case(11, B, n_new, Hq, Hkv, bs, ctx)
    pc = kl.PagedCfg(B, n_new, bs, max_blocks, n_blocks)
    Oref, lse_ref = O.paged_attention(q, kp, vp, table, np.array(ctx), n_new)
    qd, kd, vd = _dev(q), _dev(kp), _dev(vp)
    td, cd = _dev(table, torch.int32), _dev(ctx, torch.int32)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, n_new, dtype=torch.float32, device="cuda")
    nb = kl.kl_paged_attention_ws_bytes(pc, Hq, Hkv, D)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    kl.kl_paged_attention(pc, Hq, Hkv, D, kl.KL_BF16, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(),
                          cd.data_ptr(), o.data_ptr(), lse.data_ptr(), ws.data_ptr(), nb)
    torch.cuda.synchronize()
    kl.kl_device_status()
    assert_rel(o.double().cpu().numpy(), Oref, TOL_BF16, "O")
    np.testing.assert_allclose(lse.double().cpu().numpy(), lse_ref, rtol=0, atol=2e-3)


def test_paged_kv_write_is_exact(kl):
    B, n_new, Hkv, bs = 3, 2, 2, 16
    ctx = [0, 15, 33]
    table, kp, vp, _, max_blocks, n_blocks = _case(12, B, n_new, 2, Hkv, bs, ctx)
    rng = np.random.default_rng(13)
    k_new = _bf(rng.standard_normal((B * n_new, Hkv, D)))
    v_new = _bf(rng.standard_normal((B * n_new, Hkv, D)))
    kref, vref = O.paged_write(kp, vp, table, np.array(ctx), k_new, v_new, n_new)
    kd, vd = _dev(kp), _dev(vp)
    kn, vn, td, cd = _dev(k_new), _dev(v_new), _dev(table, torch.int32), _dev(ctx, torch.int32)   # kept alive
    pc = kl.PagedCfg(B, n_new, bs, max_blocks, n_blocks)
    kl.kl_paged_kv_write(pc, Hkv, D, kl.KL_BF16, kn.data_ptr(), vn.data_ptr(), td.data_ptr(), cd.data_ptr(),
                         kd.data_ptr(), vd.data_ptr())
    torch.cuda.synchronize()
    assert np.array_equal(kd.double().cpu().numpy(), kref)
    assert np.array_equal(vd.double().cpu().numpy(), vref)


def _paged_layer(kl, cfg, pc, w_dev, X, kd, vd, td, cd):
    ws = torch.empty(kl.kl_layer_forward_paged_ws_bytes(cfg, pc), dtype=torch.uint8, device="cuda")
    Y = torch.empty_like(X)
    kl.kl_layer_forward_paged(cfg, pc, L.weights_struct(w_dev), X.data_ptr(), Y.data_ptr(), kd.data_ptr(),
                              vd.data_ptr(), td.data_ptr(), cd.data_ptr(), ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    kl.kl_device_status()
    return Y


@pytest.mark.parametrize("n_new,qk_norm,inter", [(1, False, False), (2, True, True)])
def test_paged_layer_forward_matches_oracle(kl, n_new, qk_norm, inter):
    B, H, Hq, Hkv, I, bs = 3, 256, 4, 2, 512, 16
    ctx = [0, 7, 45]
    cfg = L.make_cfg(B, n_new, H, Hq, Hkv, D, I, dtype=kl.KL_BF16, qk_norm=qk_norm, rope_interleaved=inter)
    ocfg = O.LayerConfig(B=B, S=n_new, H=H, Hq=Hq, Hkv=Hkv, d=D, I=I, qk_norm=qk_norm, rope_interleaved=inter)
    w = synth.layer_weights(21, H, Hq, Hkv, D, I, bf16=True, qk_norm=qk_norm)
    X = synth.layer_inputs(21, B * n_new, H, bf16=True)["X"]
    table, kp, vp, _, max_blocks, n_blocks = _case(22, B, n_new, Hq, Hkv, bs, ctx)
    pc = kl.PagedCfg(B, n_new, bs, max_blocks, n_blocks)
    Yref, kref, vref, _ = O.layer_forward_paged(ocfg, w, X, kp, vp, table, np.array(ctx), n_new)
    w_dev = {n: L.to_device(w[L.SYNTH_NAMES[n]], kl.KL_BF16, "cuda") for n in L.weight_fields(cfg)}
    kd, vd = _dev(kp), _dev(vp)
    Xd, td, cd = L.to_device(X, kl.KL_BF16, "cuda"), _dev(table, torch.int32), _dev(ctx, torch.int32)
    Y = _paged_layer(kl, cfg, pc, w_dev, Xd, kd, vd, td, cd)
    assert_rel(Y.double().cpu().numpy(), Yref, TOL_BF16, "Y")
    assert_rel(kd.double().cpu().numpy(), kref, TOL_BF16, "k pool")
    assert_rel(vd.double().cpu().numpy(), vref, TOL_BF16, "v pool")


def test_incremental_decode_matches_training_forward(kl):
    """A prompt chunk, then one token at a time through the paged layer: the
    rows agree with kl_layer_forward over the whole sequences."""
    B, S, H, Hq, Hkv, I, bs, chunk = 2, 24, 256, 4, 2, 512, 16, 16
    w = synth.layer_weights(31, H, Hq, Hkv, D, I, bf16=True)
    X = synth.layer_inputs(31, B * S, H, bf16=True)["X"]
    full = L.run_layer(L.make_cfg(B, S, H, Hq, Hkv, D, I, dtype=kl.KL_BF16), w, X,
                       np.zeros_like(X))["Y"].reshape(B, S, H)
    max_blocks = (S + bs - 1) // bs
    table = np.random.default_rng(32).permutation(B * max_blocks).reshape(B, max_blocks).astype(np.int32)
    kd = torch.zeros(B * max_blocks, bs, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    td = _dev(table, torch.int32)
    w_dev = {n: L.to_device(w[L.SYNTH_NAMES[n]], kl.KL_BF16, "cuda") for n in L.weight_fields(
        L.make_cfg(B, 1, H, Hq, Hkv, D, I))}
    Xs = X.reshape(B, S, H)
    steps = [(0, chunk)] + [(p, 1) for p in range(chunk, S)]
    for start, n in steps:
        cfg = L.make_cfg(B, n, H, Hq, Hkv, D, I, dtype=kl.KL_BF16)
        pc = kl.PagedCfg(B, n, bs, max_blocks, B * max_blocks)
        Xn = L.to_device(Xs[:, start:start + n].reshape(B * n, H), kl.KL_BF16, "cuda")
        cd = _dev([start] * B, torch.int32)
        Y = _paged_layer(kl, cfg, pc, w_dev, Xn, kd, vd, td, cd)
        assert_rel(Y.double().cpu().numpy().reshape(B, n, H), full[:, start:start + n], TOL_BF16,
                   f"rows {start}..{start + n - 1}")


def test_table_entry_outside_the_pool_is_reported(kl):
    B, n_new, Hq, Hkv, bs = 1, 1, 8, 1, 16
    ctx = [20]
    table, kp, vp, q, max_blocks, n_blocks = _case(41, B, n_new, Hq, Hkv, bs, ctx)
    table = table.copy()
    table[0, 1] = n_blocks + 5            # the block holding positions 16..31
    pc = kl.PagedCfg(B, n_new, bs, max_blocks, n_blocks)
    qd, kd, vd = _dev(q), _dev(kp), _dev(vp)
    o = torch.empty_like(qd)
    nb = kl.kl_paged_attention_ws_bytes(pc, Hq, Hkv, D)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    td, cd = _dev(table, torch.int32), _dev(ctx, torch.int32)
    kl.kl_paged_attention(pc, Hq, Hkv, D, kl.KL_BF16, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(),
                          cd.data_ptr(), o.data_ptr(), 0, ws.data_ptr(), nb)
    with pytest.raises(kl.KLError):
        kl.kl_device_status()
    kl.kl_device_status()                 # the word was cleared by the read


def test_layer_step_with_a_table_entry_outside_the_pool_is_reported(kl):
    """The paged layer step's rotation/cache-write launch meets a new token whose
    block-table entry is outside the pool: the write is skipped and the device
    error word says why (the rest of the step still runs)."""
    B, n_new, H, Hq, Hkv, I, bs = 2, 1, 256, 4, 2, 512, 16
    ctx = [5, 20]
    cfg = L.make_cfg(B, n_new, H, Hq, Hkv, D, I, dtype=kl.KL_BF16)
    w = synth.layer_weights(51, H, Hq, Hkv, D, I, bf16=True)
    X = synth.layer_inputs(51, B * n_new, H, bf16=True)["X"]
    table, kp, vp, _, max_blocks, n_blocks = _case(52, B, n_new, Hq, Hkv, bs, ctx)
    table = table.copy()
    table[1, 20 // bs] = n_blocks + 3      # sequence 1's new token (position 20) has no valid block
    pc = kl.PagedCfg(B, n_new, bs, max_blocks, n_blocks)
    w_dev = {n: L.to_device(w[L.SYNTH_NAMES[n]], kl.KL_BF16, "cuda") for n in L.weight_fields(cfg)}
    kd, vd = _dev(kp), _dev(vp)
    Xd, td, cd = L.to_device(X, kl.KL_BF16, "cuda"), _dev(table, torch.int32), _dev(ctx, torch.int32)
    ws = torch.empty(kl.kl_layer_forward_paged_ws_bytes(cfg, pc), dtype=torch.uint8, device="cuda")
    Y = torch.empty_like(Xd)
    kl.kl_layer_forward_paged(cfg, pc, L.weights_struct(w_dev), Xd.data_ptr(), Y.data_ptr(), kd.data_ptr(),
                              vd.data_ptr(), td.data_ptr(), cd.data_ptr(), ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    with pytest.raises(kl.KLError) as e:
        kl.kl_device_status()
    assert e.value.status == kl.KL_ERR_DEVICE
    kl.kl_device_status()                 # the word was cleared by the read
