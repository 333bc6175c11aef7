"""Python binding of libkl (include/kl.h): one Qwen3-style decoder layer
forward/backward and the lm-head softmax cross-entropy with argmax on an
NVIDIA GB300 (sm_103a).

Argument marshalling only: every step runs in the CUDA kernels of libkl.so.
The functions keep the C names; tensors are passed as device pointers
(``tensor.data_ptr()``) and streams as ``cudaStream_t`` handles. If the
library has not been built, ``load()`` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkl.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "kl.h")

KL_F32 = 0
KL_BF16 = 1

KL_OK = 0
KL_ERR_INVALID_ARG = 1
KL_ERR_UNSUPPORTED = 2
KL_ERR_CUDA = 3
KL_ERR_TIMEOUT = 4
KL_ERR_NO_MEMORY = 5
KL_ERR_DEVICE = 6

_i32, _i64, _f32, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class LayerCfg(ctypes.Structure):
    _fields_ = [("B", _i32), ("S", _i32), ("H", _i32), ("Hq", _i32), ("Hkv", _i32), ("d", _i32),
                ("I", _i32), ("eps", _f32), ("rope_base", _f32), ("dtype", _i32),
                ("qk_norm", _i32), ("rope_interleaved", _i32)]


WEIGHT_FIELDS = ("gamma1", "wq", "wk", "wv", "wo", "gamma2", "wg", "wu", "wd")
QK_WEIGHT_FIELDS = ("gamma_q", "gamma_k")   # read only with cfg.qk_norm
SAVED_FIELDS = ("x", "h1", "rstd1", "q", "k", "v", "o", "lse", "x2", "h2", "rstd2", "g", "u", "m",
                "q_pre", "k_pre", "rstd_q", "rstd_k", "rope")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in WEIGHT_FIELDS + QK_WEIGHT_FIELDS]


class LayerSaved(ctypes.Structure):
    _fields_ = [(n, _vp) for n in SAVED_FIELDS]


class LayerGrads(ctypes.Structure):
    _fields_ = [(n, _vp) for n in WEIGHT_FIELDS] + [("dtype", _i32)] + [(n, _vp) for n in QK_WEIGHT_FIELDS]


class LmheadCfg(ctypes.Structure):
    _fields_ = [("N", _i32), ("H", _i32), ("V", _i32), ("dtype", _i32), ("dw_dtype", _i32)]


KL_STREAM_SAVE_ALL = 0
KL_STREAM_RECOMPUTE = 1
KL_STREAM_FORWARD = 2


class StreamCfg(ctypes.Structure):
    _fields_ = [("layer", LayerCfg), ("n_layers", _i32), ("V", _i32), ("mode", _i32)]


class PagedCfg(ctypes.Structure):
    _fields_ = [("B", _i32), ("n_new", _i32), ("block_size", _i32), ("max_blocks", _i32), ("n_blocks", _i32)]


class StreamResult(ctypes.Structure):
    _fields_ = [("loss", _f32), ("total_norm", _f32), ("clip_coef", _f32)]


_P = ctypes.POINTER
_SIGNATURES = {
    "kl_version": (ctypes.c_char_p, []),
    "kl_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "kl_last_error": (ctypes.c_char_p, []),
    "kl_device_status": (ctypes.c_int, [_vp, _P(ctypes.c_uint32)]),
    "kl_test_abandon_counters": (ctypes.c_int, []),
    "kl_layer_saved_bytes": (_sz, [_P(LayerCfg)]),
    "kl_layer_saved_carve": (ctypes.c_int, [_P(LayerCfg), _vp, _sz, _P(LayerSaved)]),
    "kl_layer_fwd_workspace_bytes": (_sz, [_P(LayerCfg)]),
    "kl_layer_bwd_workspace_bytes": (_sz, [_P(LayerCfg)]),
    "kl_layer_forward": (ctypes.c_int, [_P(LayerCfg), _P(LayerWeights), _vp, _vp, _P(LayerSaved), _vp, _sz, _vp]),
    "kl_layer_backward": (ctypes.c_int, [_P(LayerCfg), _P(LayerWeights), _P(LayerSaved), _vp, _vp,
                                         _P(LayerGrads), _vp, _sz, _vp]),
    "kl_lmhead_workspace_bytes": (_sz, [_P(LmheadCfg)]),
    "kl_lmhead_ce_argmax": (ctypes.c_int, [_P(LmheadCfg), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kl_ce_workspace_bytes": (_sz, [_i32]),
    "kl_ce_argmax": (ctypes.c_int, [_i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "kl_ce_argmax_noalloc": (ctypes.c_int, [_i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp]),
    "kl_gemm": (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _i32,
                               _vp, _i64, _i32, _vp]),
    "kl_gemm_scratch_bytes": (_sz, []),
    "kl_gemm_ex": (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _i32,
                                  _vp, _i64, _i32, _vp, _sz, _vp]),
    "kl_rmsnorm_fwd": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _f32, _vp, _vp, _vp]),
    "kl_rmsnorm_bwd_ws_bytes": (_sz, [_i32, _i32]),
    "kl_rmsnorm_bwd": (ctypes.c_int, [_i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kl_rope": (ctypes.c_int, [_i32, _i32, _i32, _i32, _f32, _i32, _vp, _i32, _vp]),
    "kl_swiglu_fwd": (ctypes.c_int, [_i64, _i32, _vp, _vp, _vp, _vp]),
    "kl_swiglu_bwd": (ctypes.c_int, [_i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "kl_attention_fwd": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "kl_attention_bwd_ws_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "kl_attention_bwd": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _sz, _vp]),
    "kl_stream_create": (ctypes.c_int, [_P(StreamCfg), _P(LayerWeights), _vp, _P(_vp)]),
    "kl_stream_run": (ctypes.c_int, [_vp, _vp, _vp, _f32, _P(LayerGrads), _vp, _P(StreamResult), _vp]),
    "kl_stream_forward": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
    "kl_stream_device_bytes": (_sz, [_vp]),
    "kl_stream_destroy": (None, [_vp]),
    "kl_paged_kv_write": (ctypes.c_int, [_P(PagedCfg), _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "kl_paged_attention_ws_bytes": (_sz, [_P(PagedCfg), _i32, _i32, _i32]),
    "kl_paged_attention": (ctypes.c_int, [_P(PagedCfg), _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _sz, _vp]),
    "kl_layer_forward_paged_ws_bytes": (_sz, [_P(LayerCfg), _P(PagedCfg)]),
    "kl_layer_forward_paged": (ctypes.c_int, [_P(LayerCfg), _P(PagedCfg), _P(LayerWeights), _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _sz, _vp]),
    "kl_profile_enable": (ctypes.c_int, [_i32]),
    "kl_profile_read": (_i32, [_vp, _i32]),
    "kl_launch_count": (ctypes.c_uint64, []),
}

_lib = None


class KLError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kl status {status}: {msg}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libkl.so (built in-tree). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def declared_functions() -> list:
    """Names of every entry point declared in include/kl.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return re.findall(r"^KL_API\s+[\w\s\*]+?\b(kl_\w+)\s*\(", text, flags=re.M)


def check(status: int) -> None:
    if status != KL_OK:
        raise KLError(status, last_error())


def last_error() -> str:
    return load().kl_last_error().decode()


def version() -> str:
    return load().kl_version().decode()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def ptr(t) -> int:
    """Device pointer of a tensor (or 0 for None)."""
    return 0 if t is None else t.data_ptr()


# --------------------------------------------------------------------------
# entry points (same names as the C functions)
# --------------------------------------------------------------------------

def kl_layer_saved_bytes(cfg: LayerCfg) -> int:
    return load().kl_layer_saved_bytes(ctypes.byref(cfg))


def kl_layer_saved_carve(cfg: LayerCfg, base: int, nbytes: int) -> LayerSaved:
    s = LayerSaved()
    check(load().kl_layer_saved_carve(ctypes.byref(cfg), base, nbytes, ctypes.byref(s)))
    return s


def kl_layer_fwd_workspace_bytes(cfg: LayerCfg) -> int:
    return load().kl_layer_fwd_workspace_bytes(ctypes.byref(cfg))


def kl_layer_bwd_workspace_bytes(cfg: LayerCfg) -> int:
    return load().kl_layer_bwd_workspace_bytes(ctypes.byref(cfg))


def kl_layer_forward(cfg, weights, X: int, Y: int, saved, ws: int, ws_bytes: int, stream=None) -> None:
    check(load().kl_layer_forward(ctypes.byref(cfg), ctypes.byref(weights), X, Y, ctypes.byref(saved),
                                  ws, ws_bytes, _stream(stream)))


def kl_layer_backward(cfg, weights, saved, dY: int, dX: int, grads, ws: int, ws_bytes: int,
                      stream=None) -> None:
    check(load().kl_layer_backward(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(saved), dY, dX,
                                   ctypes.byref(grads), ws, ws_bytes, _stream(stream)))


def kl_lmhead_workspace_bytes(cfg: LmheadCfg) -> int:
    return load().kl_lmhead_workspace_bytes(ctypes.byref(cfg))


def kl_lmhead_ce_argmax(cfg, X, W, targets, loss, argmax, dlogits, dX, dW, ws, ws_bytes, stream=None) -> None:
    check(load().kl_lmhead_ce_argmax(ctypes.byref(cfg), X, W, targets, loss, argmax, dlogits, dX, dW,
                                     ws, ws_bytes, _stream(stream)))


def kl_ce_workspace_bytes(N: int) -> int:
    return load().kl_ce_workspace_bytes(N)


def kl_ce_argmax(N, V, z, targets, loss, argmax, dlogits, dz_dtype, ws, ws_bytes, stream=None) -> None:
    check(load().kl_ce_argmax(N, V, z, targets, loss, argmax, dlogits, dz_dtype, ws, ws_bytes, _stream(stream)))


KL_CE_NOALLOC_MAX_ROWS = 65535


def kl_ce_argmax_noalloc(N, V, z, targets, loss, argmax, dlogits, dz_dtype, stream=None) -> None:
    """kl_ce_argmax without a workspace argument (static scratch inside libkl)."""
    check(load().kl_ce_argmax_noalloc(N, V, z, targets, loss, argmax, dlogits, dz_dtype, _stream(stream)))


def kl_gemm(M, N, K, dtype, A, lda, a_mn, B, ldb, b_mn, C, ldc, c_dtype, R=0, ldr=0, r_dtype=KL_BF16,
            stream=None) -> None:
    check(load().kl_gemm(M, N, K, dtype, A, lda, a_mn, B, ldb, b_mn, C, ldc, c_dtype, R, ldr, r_dtype,
                         _stream(stream)))


def kl_gemm_scratch_bytes() -> int:
    return load().kl_gemm_scratch_bytes()


def kl_gemm_ex(M, N, K, dtype, A, lda, a_mn, B, ldb, b_mn, C, ldc, c_dtype, R=0, ldr=0, r_dtype=KL_BF16,
               ws=0, ws_bytes=0, stream=None) -> None:
    """kl_gemm with a device scratch (last-round K split, few-rows kernel)."""
    check(load().kl_gemm_ex(M, N, K, dtype, A, lda, a_mn, B, ldb, b_mn, C, ldc, c_dtype, R, ldr, r_dtype, ws,
                            ws_bytes, _stream(stream)))


def kl_rmsnorm_fwd(rows, width, dtype, x, gamma, eps, h, rstd, stream=None) -> None:
    check(load().kl_rmsnorm_fwd(rows, width, dtype, x, gamma, eps, h, rstd, _stream(stream)))


def kl_rmsnorm_bwd_ws_bytes(rows, width) -> int:
    return load().kl_rmsnorm_bwd_ws_bytes(rows, width)


def kl_rmsnorm_bwd(rows, width, dtype, dh, dh_dtype, x, gamma, rstd, resid, dx, dgamma, ws, ws_bytes,
                   stream=None) -> None:
    check(load().kl_rmsnorm_bwd(rows, width, dtype, dh, dh_dtype, x, gamma, rstd, resid, dx, dgamma, ws,
                                ws_bytes, _stream(stream)))


def kl_rope(B, S, heads, d, base, dtype, x, direction, stream=None) -> None:
    check(load().kl_rope(B, S, heads, d, base, dtype, x, direction, _stream(stream)))


def kl_swiglu_fwd(n, dtype, g, u, m, stream=None) -> None:
    check(load().kl_swiglu_fwd(n, dtype, g, u, m, _stream(stream)))


def kl_swiglu_bwd(n, dtype, dm, g, u, dg, du, stream=None) -> None:
    check(load().kl_swiglu_bwd(n, dtype, dm, g, u, dg, du, _stream(stream)))


def kl_attention_fwd(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, stream=None) -> None:
    check(load().kl_attention_fwd(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, _stream(stream)))


def kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d) -> int:
    return load().kl_attention_bwd_ws_bytes(B, S, Hq, Hkv, d)


def kl_attention_bwd(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes,
                     stream=None) -> None:
    check(load().kl_attention_bwd(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes,
                                  _stream(stream)))


def kl_paged_kv_write(pc: PagedCfg, Hkv, d, dtype, k_new, v_new, table, ctx, k_pool, v_pool, stream=None) -> None:
    check(load().kl_paged_kv_write(ctypes.byref(pc), Hkv, d, dtype, k_new, v_new, table, ctx, k_pool, v_pool,
                                   _stream(stream)))


def kl_paged_attention_ws_bytes(pc: PagedCfg, Hq, Hkv, d) -> int:
    return load().kl_paged_attention_ws_bytes(ctypes.byref(pc), Hq, Hkv, d)


def kl_paged_attention(pc: PagedCfg, Hq, Hkv, d, dtype, q, k_pool, v_pool, table, ctx, o, lse, ws, ws_bytes,
                       stream=None) -> None:
    check(load().kl_paged_attention(ctypes.byref(pc), Hq, Hkv, d, dtype, q, k_pool, v_pool, table, ctx, o, lse, ws,
                                    ws_bytes, _stream(stream)))


def kl_layer_forward_paged_ws_bytes(cfg: LayerCfg, pc: PagedCfg) -> int:
    return load().kl_layer_forward_paged_ws_bytes(ctypes.byref(cfg), ctypes.byref(pc))


def kl_layer_forward_paged(cfg: LayerCfg, pc: PagedCfg, w: LayerWeights, X, Y, k_pool, v_pool, table, ctx, ws,
                           ws_bytes, stream=None) -> None:
    check(load().kl_layer_forward_paged(ctypes.byref(cfg), ctypes.byref(pc), ctypes.byref(w), X, Y, k_pool, v_pool,
                                        table, ctx, ws, ws_bytes, _stream(stream)))


def kl_device_status(stream=None) -> int:
    bits = ctypes.c_uint32(0)
    check(load().kl_device_status(_stream(stream), ctypes.byref(bits)))
    return bits.value


def kl_test_abandon_counters() -> None:
    check(load().kl_test_abandon_counters())


def kl_stream_create(cfg: StreamCfg, host_layers, host_lm_head: int) -> int:
    arr = (LayerWeights * len(host_layers))(*host_layers)
    out = _vp()
    check(load().kl_stream_create(ctypes.byref(cfg), arr, host_lm_head, ctypes.byref(out)))
    return out.value


def kl_stream_run(handle: int, X: int, targets: int, clip_max_norm: float, grads_list, dW_lm: int,
                  stream=None) -> StreamResult:
    arr = (LayerGrads * len(grads_list))(*grads_list)
    res = StreamResult()
    check(load().kl_stream_run(handle, X, targets, clip_max_norm, arr, dW_lm, ctypes.byref(res),
                               _stream(stream)))
    return res


def kl_stream_forward(handle: int, X: int, Y: int, stream=None) -> None:
    check(load().kl_stream_forward(handle, X, Y, _stream(stream)))


def kl_stream_device_bytes(handle: int) -> int:
    return load().kl_stream_device_bytes(handle)


def kl_stream_destroy(handle: int) -> None:
    load().kl_stream_destroy(handle)


from . import layer  # noqa: E402,F401  (torch-side buffer helpers)
