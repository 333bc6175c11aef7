"""tcgen05 bf16 GEMM and fp32 CUDA-core GEMM against the oracle's matrix
product, for every operand major-ness, with tiles left ragged on M, N and K."""
import numpy as np
import pytest
import torch

import oracle as O
from bwd_qwen3_layer_gb300 import synth
from _parity import assert_rel, dev, host

pytestmark = pytest.mark.gpu

SHAPES = [(200, 296, 136), (256, 512, 1024), (136, 264, 72), (8, 8, 8), (1024, 1280, 320)]


def _operands(M, N, K, seed, bf16=True):
    A = synth.normal(seed, "gemm.A", (M, K))
    B = synth.normal(seed, "gemm.B", (N, K))
    R = synth.normal(seed, "gemm.R", (M, N))
    if bf16:
        A, B, R = synth.round_bf16(A), synth.round_bf16(B), synth.round_bf16(R)
    return A, B, R


def _store(X, mn, dtype):
    """X is the logical [rows, K] operand; MN-major stores its transpose."""
    t = dev(X.T if mn else X, dtype)
    return t, t.shape[1]


@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_bf16_fp32_out(kl, a_mn, b_mn, M, N, K):
    A, B, _ = _operands(M, N, K, 1)
    a, lda = _store(A, a_mn, torch.bfloat16)
    b, ldb = _store(B, b_mn, torch.bfloat16)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    kl.kl_gemm(M, N, K, kl.KL_BF16, a.data_ptr(), lda, a_mn, b.data_ptr(), ldb, b_mn, C.data_ptr(), N,
               kl.KL_F32)
    torch.cuda.synchronize()
    assert_rel(host(C), O.linear(A, B), 1e-5, f"C {M}x{N}x{K} a_mn={a_mn} b_mn={b_mn}")


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
def test_gemm_bf16_out_with_residual(kl, a_mn, b_mn):
    M, N, K = 392, 520, 264
    A, B, R = _operands(M, N, K, 2)
    a, lda = _store(A, a_mn, torch.bfloat16)
    b, ldb = _store(B, b_mn, torch.bfloat16)
    r = dev(R, torch.bfloat16)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    kl.kl_gemm(M, N, K, kl.KL_BF16, a.data_ptr(), lda, a_mn, b.data_ptr(), ldb, b_mn, C.data_ptr(), N,
               kl.KL_BF16, r.data_ptr(), N, kl.KL_BF16)
    torch.cuda.synchronize()
    assert_rel(host(C), O.linear(A, B) + R, 4e-3, "C+R bf16")


@pytest.mark.parametrize("M,N,K,dt", [(392, 520, 264, 1), (2048, 5120, 1024, 1), (64, 1344, 2560, 1),
                                      (200, 296, 136, 0)])
def test_gemm_residual_in_place(kl, M, N, K, dt):
    """R may be C itself (C = A B^T + C): every path reads an element's addend
    before writing it, whole tiles, K-split last-round tiles, the few-rows kernel
    and the fp32 kernel alike. The in-place result equals the out-of-place one
    bit for bit."""
    A, B, R = _operands(M, N, K, 9, bf16=dt == 1)
    tdt = torch.bfloat16 if dt == 1 else torch.float32
    a, b, r = dev(A, tdt), dev(B, tdt), dev(R, tdt)
    nb = kl.kl_gemm_scratch_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=tdt, device="cuda")
    kl.kl_gemm_ex(M, N, K, dt, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, dt,
                  r.data_ptr(), N, dt, ws=ws.data_ptr(), ws_bytes=nb)
    Ci = r.clone()
    kl.kl_gemm_ex(M, N, K, dt, a.data_ptr(), K, 0, b.data_ptr(), K, 0, Ci.data_ptr(), N, dt,
                  Ci.data_ptr(), N, dt, ws=ws.data_ptr(), ws_bytes=nb)
    torch.cuda.synchronize()
    kl.kl_device_status()
    assert_rel(host(C), O.linear(A, B) + R, 4e-3 if dt == 1 else 1e-5, "C+R")
    assert torch.equal(Ci, C)


def test_gemm_bf16_zero_is_exact(kl):
    """A zero operand gives an exact zero product and the residual passes bit-exactly."""
    M, N, K = 256, 256, 128
    _, B, R = _operands(M, N, K, 3)
    a = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    b = dev(B, torch.bfloat16)
    r = dev(R, torch.bfloat16)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    kl.kl_gemm(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, kl.KL_BF16,
               r.data_ptr(), N, kl.KL_BF16)
    torch.cuda.synchronize()
    assert torch.equal(C, r)


@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_gemm_f32(kl, a_mn, b_mn):
    M, N, K = 70, 93, 45
    A, B, R = _operands(M, N, K, 4, bf16=False)
    a, lda = _store(A, a_mn, torch.float32)
    b, ldb = _store(B, b_mn, torch.float32)
    r = dev(R, torch.float32)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    kl.kl_gemm(M, N, K, kl.KL_F32, a.data_ptr(), lda, a_mn, b.data_ptr(), ldb, b_mn, C.data_ptr(), N,
               kl.KL_F32, r.data_ptr(), N, kl.KL_F32)
    torch.cuda.synchronize()
    A32 = A.astype(np.float32).astype(np.float64)
    B32 = B.astype(np.float32).astype(np.float64)
    R32 = R.astype(np.float32).astype(np.float64)
    assert_rel(host(C), O.linear(A32, B32) + R32, 1e-6, "f32")


@pytest.mark.parametrize("a_mn,b_mn,M,N,K", [(0, 0, 264, 520, 20480), (1, 1, 200, 136, 40960), (0, 1, 512, 256, 30720)])
def test_gemm_bf16_long_k(kl, a_mn, b_mn, M, N, K):
    """fp32 output, K >= 16384: every output tile sums its whole K range in one
    fixed order; with a scratch the launch's last (here only) round cuts its
    tiles along K into slices summed in slice order. Either way a repeat gives
    the same bits."""
    A, B, _ = _operands(M, N, K, 5)
    a, lda = _store(A, a_mn, torch.bfloat16)
    b, ldb = _store(B, b_mn, torch.bfloat16)
    ws = torch.empty(kl.kl_gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    # One fp32 accumulation chain of K products per output (the tensor core's
    # accumulator, no K split): its rounding grows like sqrt(K); measured
    # 4.7e-5 at K = 40960. The bound keeps 2x margin there and stays four
    # orders below what a dropped or repeated k-block would give (~1e-1).
    tol = 4e-5 * max(1.0, (K / 8192) ** 0.5)
    for scratch in (False, True):
        outs = []
        for _ in range(2):
            C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
            kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), lda, a_mn, b.data_ptr(), ldb, b_mn, C.data_ptr(), N,
                          kl.KL_F32, 0, 0, kl.KL_BF16, ws.data_ptr() if scratch else 0,
                          ws.numel() if scratch else 0)
            torch.cuda.synchronize()
            assert_rel(host(C), O.linear(A, B), tol, f"C {M}x{N}x{K} scratch {scratch}")
            outs.append(C)
        assert torch.equal(outs[0], outs[1]), f"repeat {M}x{N}x{K} scratch {scratch}"


# few rows (M <= 128, K-major operands) with a scratch: the weights-streaming
# kernel, including tiles whose K range is shared out between CTAs and summed
# from pieces (N ragged on the 128-row tiles, K ragged on the 64-wide blocks)
FEW_ROWS = [(1, 200, 72), (5, 300, 8192), (17, 520, 264), (33, 136, 40), (64, 1344, 2560), (128, 264, 4104)]


@pytest.mark.parametrize("M,N,K", FEW_ROWS)
@pytest.mark.parametrize("out", ["f32", "bf16+R"])
def test_gemm_few_rows_with_scratch(kl, M, N, K, out):
    A, B, R = _operands(M, N, K, 5)
    a, b = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    nb = kl.kl_gemm_scratch_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ref = O.linear(A, B)
    if out == "f32":
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, kl.KL_F32,
                      ws=ws.data_ptr(), ws_bytes=nb)
        tol = 1e-5
    else:
        r = dev(R, torch.bfloat16)
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, kl.KL_BF16,
                      r.data_ptr(), N, kl.KL_BF16, ws=ws.data_ptr(), ws_bytes=nb)
        ref = ref + R
        tol = 4e-3
    torch.cuda.synchronize()
    kl.kl_device_status()
    assert_rel(host(C), ref, tol, f"C {M}x{N}x{K} {out}")
    # the pieces are summed in a fixed order: a second call repeats every bit
    C2 = torch.empty_like(C)
    if out == "f32":
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C2.data_ptr(), N, kl.KL_F32,
                      ws=ws.data_ptr(), ws_bytes=nb)
    else:
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C2.data_ptr(), N, kl.KL_BF16,
                      r.data_ptr(), N, kl.KL_BF16, ws=ws.data_ptr(), ws_bytes=nb)
    torch.cuda.synchronize()
    assert torch.equal(C, C2)


def test_gemm_few_rows_strided_operands(kl):
    """Leading dimensions wider than K and N (views into larger buffers)."""
    M, N, K = 24, 392, 1000
    A, B, R = _operands(M, N, K, 6)
    abuf = torch.zeros((M, K + 24), dtype=torch.bfloat16, device="cuda")
    bbuf = torch.zeros((N, K + 8), dtype=torch.bfloat16, device="cuda")
    abuf[:, :K] = dev(A, torch.bfloat16)
    bbuf[:, :K] = dev(B, torch.bfloat16)
    C = torch.zeros((M, N + 40), dtype=torch.float32, device="cuda")
    nb = kl.kl_gemm_scratch_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    kl.kl_gemm_ex(M, N, K, kl.KL_BF16, abuf.data_ptr(), K + 24, 0, bbuf.data_ptr(), K + 8, 0, C.data_ptr(), N + 40,
                  kl.KL_F32, ws=ws.data_ptr(), ws_bytes=nb)
    torch.cuda.synchronize()
    assert_rel(host(C[:, :N]), O.linear(A, B), 1e-5, "C strided")
    assert torch.count_nonzero(C[:, N:]) == 0          # nothing written past N


def test_gemm_few_rows_counter_slots_rearm(kl):
    """Forty launches in a row cycle the shared-tile arrival counters' slots more
    than twice: each counter must be back at zero when its slot comes round again,
    so every launch gives the same bits (shapes with tiles shared between CTAs)."""
    M, N, K = 64, 1344, 2560
    A, B, _ = _operands(M, N, K, 7)
    a, b = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    nb = kl.kl_gemm_scratch_bytes()
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(40)]
    for C in outs:
        kl.kl_gemm_ex(M, N, K, kl.KL_BF16, a.data_ptr(), K, 0, b.data_ptr(), K, 0, C.data_ptr(), N, kl.KL_F32,
                      ws=ws.data_ptr(), ws_bytes=nb)
    torch.cuda.synchronize()
    kl.kl_device_status()
    assert_rel(host(outs[0]), O.linear(A, B), 1e-5, "first")
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
