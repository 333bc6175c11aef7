"""The C ABI: libkl.so loads, exports every entry point include/kl.h declares,
and rejects bad arguments on the host before touching the GPU. CPU only:
no call here launches a kernel."""
import ctypes
import os
import subprocess

import pytest

import bwd_qwen3_layer_gb300 as K


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(K.LIB_PATH):
        import __graft_entry__ as g
        g.build()
    return K.load()


def test_header_declares_the_boundary():
    names = set(K.declared_functions())
    for n in ("kl_layer_forward", "kl_layer_backward", "kl_lmhead_ce_argmax", "kl_stream_create",
              "kl_stream_run", "kl_stream_destroy", "kl_ce_argmax", "kl_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in K.declared_functions() if n not in exported]
    assert not missing, missing
    # and the binding knows the signature of each
    assert set(K.declared_functions()) <= set(K._SIGNATURES)
    for n in K.declared_functions():
        getattr(lib, n)


def test_status_strings(lib):
    assert K.version().startswith("kl ")
    for s in range(7):
        assert lib.kl_status_str(s)
    assert lib.kl_status_str(99) == b"unknown status"


def _cfg(**kw):
    base = dict(B=1, S=2048, H=5120, Hq=64, Hkv=8, d=128, I=25600, eps=1e-6, rope_base=1e6, dtype=K.KL_BF16)
    base.update(kw)
    return K.LayerCfg(**base)


def test_saved_and_workspace_sizes(lib):
    cfg = _cfg()
    T, H, I, Dq, Dkv = 2048, 5120, 25600, 8192, 1024
    # bf16 activations, fp32 rstd1/rstd2 and lse, and the rotary (cos, sin) table [S][64]
    need = (3 * T * H + 2 * T * Dq + 2 * T * Dkv + 3 * T * I) * 2 + 2 * T * 4 + 64 * T * 4 + T * 64 * 8
    got = K.kl_layer_saved_bytes(cfg)
    assert need <= got <= need + 15 * 256
    assert K.kl_layer_bwd_workspace_bytes(cfg) > 3 * T * I * 2
    # fp32 saved set is twice as large (up to alignment)
    cfg32 = _cfg(dtype=K.KL_F32, B=1, S=32, H=64, Hq=4, Hkv=2, d=16, I=172)
    assert K.kl_layer_saved_bytes(cfg32) > 0


def test_bad_configs_rejected_on_host(lib):
    assert K.kl_layer_saved_bytes(_cfg(Hq=6, Hkv=4)) == 0          # Hq % Hkv
    assert K.kl_layer_saved_bytes(_cfg(d=64)) == 0                  # bf16 needs d = 128
    assert K.kl_layer_saved_bytes(_cfg(H=5121)) == 0                # bf16 needs H % 8
    assert K.kl_layer_saved_bytes(_cfg(dtype=7)) == 0
    w = K.LayerWeights()
    s = K.LayerSaved()
    st = lib.kl_layer_forward(ctypes.byref(_cfg()), ctypes.byref(w), None, None, ctypes.byref(s), None, 0, None)
    assert st == K.KL_ERR_INVALID_ARG
    assert "null" in K.last_error()
    st = lib.kl_layer_forward(ctypes.byref(_cfg(d=64)), ctypes.byref(w), None, None, ctypes.byref(s), None, 0, None)
    assert st == K.KL_ERR_UNSUPPORTED


def test_misaligned_pointer_rejected(lib):
    cfg = _cfg()
    w = K.LayerWeights(*([0x1000] * 9))
    w.wq = 0x1008   # 8-byte aligned only
    s = K.LayerSaved()
    st = lib.kl_layer_forward(ctypes.byref(cfg), ctypes.byref(w), 0x2000, 0x3000, ctypes.byref(s), None, 0, None)
    assert st == K.KL_ERR_INVALID_ARG
    assert "aligned" in K.last_error()


def test_backward_workspace_too_small(lib):
    cfg = _cfg()
    w = K.LayerWeights(*([0x1000] * 9))
    s = K.LayerSaved(*([0x1000] * 14))
    g = K.LayerGrads(*([0x1000] * 9), K.KL_BF16)
    st = lib.kl_layer_backward(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(s), 0x2000, 0x3000,
                               ctypes.byref(g), 0x4000, 1024, None)
    assert st == K.KL_ERR_NO_MEMORY


def test_lmhead_and_ce_host_checks(lib):
    c = K.LmheadCfg(4096, 5120, 151936, K.KL_BF16, K.KL_F32)
    nb = K.kl_lmhead_workspace_bytes(c)
    assert nb >= 4096 * 151936 * 4
    assert K.kl_lmhead_workspace_bytes(K.LmheadCfg(4096, 5120, 151937, K.KL_BF16, K.KL_BF16)) == 0
    assert K.kl_lmhead_workspace_bytes(K.LmheadCfg(8, 8, 8, K.KL_F32, K.KL_BF16)) == 0
    assert lib.kl_ce_argmax(0, 10, None, None, None, None, None, K.KL_F32, None, 0, None) == K.KL_ERR_INVALID_ARG
    assert lib.kl_ce_argmax(4, 10, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 5, 0x1000, 1 << 20, None) == K.KL_ERR_INVALID_ARG
    # dlogits overlapping the logits (in place, or bf16 dlogits starting inside z) is rejected
    # before any launch; disjoint buffers pass this check (and would then need a GPU)
    ws = 0x100000
    for dz, dt in ((0x10000, K.KL_F32), (0x10000 + 4 * 40 - 2, K.KL_BF16), (0x10000 - 4 * 40 + 2, K.KL_F32)):
        assert lib.kl_ce_argmax(4, 10, 0x10000, 0x2000, 0x3000, 0x4000, dz, dt, ws, 1 << 20, None) \
            == K.KL_ERR_INVALID_ARG, hex(dz)
        assert "overlaps" in K.last_error()


def test_gemm_host_checks(lib):
    assert lib.kl_gemm(0, 8, 8, K.KL_BF16, 0x1000, 8, 0, 0x1000, 8, 0, 0x1000, 8, K.KL_BF16, None, 0, 0, None) \
        == K.KL_ERR_INVALID_ARG
    # leading dimension smaller than the contiguous extent
    assert lib.kl_gemm(16, 16, 64, K.KL_BF16, 0x1000, 32, 0, 0x1000, 64, 0, 0x1000, 16, K.KL_BF16, None, 0, 0,
                       None) == K.KL_ERR_INVALID_ARG
    # the scratch-taking form: same checks; its scratch size is whole 256-byte blocks
    nb = lib.kl_gemm_scratch_bytes()
    assert nb > 0 and nb % 256 == 0
    assert lib.kl_gemm_ex(0, 8, 8, K.KL_BF16, 0x1000, 8, 0, 0x1000, 8, 0, 0x1000, 8, K.KL_BF16, None, 0, 0,
                          0x1000, nb, None) == K.KL_ERR_INVALID_ARG
    assert lib.kl_gemm_ex(16, 16, 64, K.KL_BF16, 0x1000, 64, 0, 0x1000, 64, 0, 0x1000, 8, K.KL_BF16, None, 0, 0,
                          0x1000, nb, None) == K.KL_ERR_INVALID_ARG      # ldc < N
    assert lib.kl_gemm_ex(16, 16, 64, 7, 0x1000, 64, 0, 0x1000, 64, 0, 0x1000, 16, K.KL_BF16, None, 0, 0,
                          0x1000, nb, None) == K.KL_ERR_INVALID_ARG      # unknown dtype


def test_stream_host_checks(lib):
    layer = _cfg(S=64, H=256, Hq=4, Hkv=2, I=512)
    w = (K.LayerWeights * 1)(K.LayerWeights(*([0x1000] * 9), None, None))
    out = ctypes.c_void_p()
    bad_mode = K.StreamCfg(layer, 1, 1024, 7)
    assert lib.kl_stream_create(ctypes.byref(bad_mode), w, 0x1000, ctypes.byref(out)) == K.KL_ERR_INVALID_ARG
    # a training driver needs the lm-head weight; a forward-only one does not
    train = K.StreamCfg(layer, 1, 1024, K.KL_STREAM_RECOMPUTE)
    assert lib.kl_stream_create(ctypes.byref(train), w, None, ctypes.byref(out)) == K.KL_ERR_INVALID_ARG
    no_layers = K.StreamCfg(layer, 0, 0, K.KL_STREAM_FORWARD)
    assert lib.kl_stream_create(ctypes.byref(no_layers), w, None, ctypes.byref(out)) == K.KL_ERR_INVALID_ARG
    assert lib.kl_stream_forward(None, 0x1000, 0x1000, None) == K.KL_ERR_INVALID_ARG


def test_paged_host_checks(lib):
    pc = K.PagedCfg(4, 1, 16, 8, 64)
    assert K.kl_paged_attention_ws_bytes(pc, 64, 8, 128) >= 0
    assert K.kl_paged_attention_ws_bytes(pc, 64, 8, 64) == 0            # head dim 128 only
    assert K.kl_paged_attention_ws_bytes(K.PagedCfg(4, 9, 16, 8, 64), 64, 8, 128) == 0   # 8 x 9 > 64 rows
    # pool rows past 32-bit indexing are refused
    assert K.kl_paged_attention_ws_bytes(K.PagedCfg(4, 1, 16, 8, 1 << 28), 64, 8, 128) == 0
    assert K.kl_paged_attention_ws_bytes(K.PagedCfg(0, 1, 16, 8, 64), 64, 8, 128) == 0
    # null pointers are refused before any CUDA call
    assert lib.kl_paged_attention(ctypes.byref(pc), 64, 8, 128, K.KL_BF16, None, None, None, None, None, None,
                                  None, None, 0, None) == K.KL_ERR_INVALID_ARG
    assert lib.kl_paged_kv_write(ctypes.byref(pc), 8, 128, K.KL_F32, None, None, None, None, None, None,
                                 None) == K.KL_ERR_UNSUPPORTED
    layer = _cfg(B=4, S=1)
    assert K.kl_layer_forward_paged_ws_bytes(layer, pc) > 0
    assert K.kl_layer_forward_paged_ws_bytes(_cfg(B=4, S=2), pc) == 0    # S must be the step's n_new
