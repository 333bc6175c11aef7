// Causal GQA attention forward on the 5th-generation tensor cores ("KYNETRA
// FOUNDRY", tiled-attention paragraph: query tiles stream over key/value tiles
// with a running max and sum, the score matrix never leaves the chip).
//
// One CTA = 128 query rows of one query head (head dim 128), 6 warps:
//   warp 0      TMA: Q once, then K_j / V_j tiles of 128 keys, 2 stages each
//   warp 1      TMEM owner; one thread issues tcgen05.mma:
//                 S_j  = Q K_j^T   -> TMEM S[j%2]  (128 x 128 fp32)
//                 O   += P_j V_j   -> TMEM O       (128 x 128 fp32)
//               S_{j+1} is issued before P_j V_j so the tensor core computes
//               the next scores while the softmax warps work on P_j.
//   warps 2..5  softmax: thread = query row = TMEM lane. Two passes over S_j
//               (row max, then exp2 / row sum / bf16 P written to shared memory
//               in the 128-byte-swizzled K-major layout the MMA reads). The
//               running max is only raised when a row's max grows by more than
//               2^8 (then that warp rescales its O rows in TMEM); otherwise P is
//               taken against the stale max, which the final O / l cancels.
// Every wait is bounded; a timeout records KL_DEVERR_TIMEOUT and unwinds.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int HD = 128;       // head dim
constexpr int BQ = 128;       // query rows per CTA
constexpr int BKV = 128;      // keys per tile
constexpr uint32_t TILE_BYTES = 128 * 128 * 2;   // 32 KB: two 16 KB swizzle blocks of 64 columns
constexpr int THREADS = 192;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float LN2_F = 0.6931471805599453f;

// shared-memory layout (offsets from a 1024-aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;          // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE_BYTES;      // 2 stages
constexpr uint32_t OFF_P = OFF_V + 2 * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_P + TILE_BYTES;
constexpr size_t SMEM_BYTES = 1024 + OFF_BAR + 256;

struct FwdParams {
  CUtensorMap tmQ, tmK, tmV;
  __nv_bfloat16* o;
  float* lse;
  int S, Hq, Hkv;
  float scale_log2;
  uint32_t* err;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// K-major operand of 128 rows x 128 k (two 64-column swizzle blocks): the
// descriptor of k-step kk (16 columns).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
  return smem_desc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (V as B: n = head dim in two 64-wide atoms, k = keys).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 2048, 16384, 1024);
}

__global__ void __launch_bounds__(THREADS, 1) fa_fwd_tc_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + OFF_BAR;
  // barriers
  const uint32_t q_full = bar + 0;
  auto k_full = [&](int s) { return bar + 8 + 8 * s; };
  auto k_empty = [&](int s) { return bar + 24 + 8 * s; };
  auto v_full = [&](int s) { return bar + 40 + 8 * s; };
  auto v_empty = [&](int s) { return bar + 56 + 8 * s; };
  auto s_full = [&](int s) { return bar + 72 + 8 * s; };
  auto s_free = [&](int s) { return bar + 88 + 8 * s; };
  const uint32_t p_full = bar + 104;
  const uint32_t p_free = bar + 112;
  const uint32_t drain = bar + 152;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 164);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (p.S + BQ - 1) / BQ;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x);   // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int j_kv = h * p.Hkv / p.Hq;
  const int q0 = qb * BQ;
  const int row0 = b * p.S;                    // first token row of this sequence
  const int nkb = qb + 1;                      // causal: key tiles 0 .. qb

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 4);
    }
    mbar_init(p_full, 4);
    mbar_init(p_free, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA ----------------
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
    mbar_arrive_expect_tx(q_full, TILE_BYTES);
    tma_load_2d(sb + OFF_Q, &p.tmQ, h * HD, row0 + q0, q_full);
    tma_load_2d(sb + OFF_Q + 16384, &p.tmQ, h * HD + 64, row0 + q0, q_full);
    int issued_k = 0, issued_v = 0;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (*abort_flag || !mbar_wait(k_empty(s), ph ^ 1u, p.err)) { *abort_flag = 1; break; }
      mbar_arrive_expect_tx(k_full(s), TILE_BYTES);
      tma_load_2d(sb + OFF_K + s * TILE_BYTES, &p.tmK, j_kv * HD, row0 + j * BKV, k_full(s));
      tma_load_2d(sb + OFF_K + s * TILE_BYTES + 16384, &p.tmK, j_kv * HD + 64, row0 + j * BKV, k_full(s));
      ++issued_k;
      if (*abort_flag || !mbar_wait(v_empty(s), ph ^ 1u, p.err)) { *abort_flag = 1; break; }
      mbar_arrive_expect_tx(v_full(s), TILE_BYTES);
      tma_load_2d(sb + OFF_V + s * TILE_BYTES, &p.tmV, j_kv * HD, row0 + j * BKV, v_full(s));
      tma_load_2d(sb + OFF_V + s * TILE_BYTES + 16384, &p.tmV, j_kv * HD + 64, row0 + j * BKV, v_full(s));
      ++issued_v;
    }
    // copies still in flight must land before exit
    mbar_wait(q_full, 0, p.err);
    for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j) mbar_wait(k_full(j & 1), (j >> 1) & 1, p.err);
    for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j) mbar_wait(v_full(j & 1), (j >> 1) & 1, p.err);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA ----------------
    const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = mbar_wait(q_full, 0, p.err);
    auto issue_pv = [&](int j) -> bool {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait(p_full, j & 1, p.err)) return false;
      if (!mbar_wait(v_full(s), ph, p.err)) return false;
      tc_fence_after();
      for (int kk = 0; kk < BKV / 16; ++kk)
        umma_bf16(tmem + 256, desc_kmajor(sb + OFF_P, kk), desc_mnmajor(sb + OFF_V + s * TILE_BYTES, kk),
                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit(v_empty(s));
      umma_commit(p_free);
      return true;
    };
    for (int j = 0; ok && j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (*abort_flag || !mbar_wait(k_full(s), ph, p.err) ||
          (j >= 2 && !mbar_wait(s_free(s), ph ^ 1u, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + s * 128;
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16(d, desc_kmajor(sb + OFF_Q, kk), desc_kmajor(sb + OFF_K + s * TILE_BYTES, kk), idesc_s, kk > 0);
      umma_commit(k_empty(s));
      umma_commit(s_full(s));
      if (j >= 1 && !issue_pv(j - 1)) ok = false;
    }
    if (ok && !issue_pv(nkb - 1)) ok = false;
    if (!ok) *abort_flag = 1;
    umma_commit(drain);
    mbar_wait(drain, 0, p.err);
  } else if (warp >= 2) {
    // ---------------- softmax / correction / epilogue ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;           // query row within the tile = TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t oadr = tmem + lane_off + 256;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    uint8_t* prow = smem + OFF_P + r * 128;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (*abort_flag || !mbar_wait(s_full(s), ph, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sadr = tmem + lane_off + s * 128;
      const bool diag = (j == nkb - 1);
      // pass 1: row max of the scaled, masked scores
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(sadr + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = j * BKV + c * 32 + e;
          float x = __uint_as_float(v[e]) * p.scale_log2;
          if (diag && key > qrow) x = -INFINITY;
          mx = fmaxf(mx, x);
        }
      }
      // raise the running max only when it grows by more than 2^8
      const bool raise = mx > m + 8.0f;
      const float m_new = raise ? mx : m;
      const float alpha = raise ? exp2f(m - m_new) : 1.0f;
      // O and the P buffer are stable once the previous P V product is done
      if (j >= 1 && !mbar_wait(p_free, (j - 1) & 1, p.err)) { ok = false; break; }
      if (j >= 1 && __any_sync(0xffffffffu, raise)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(oadr + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st_32x32b_x32(oadr + c * 32, v);
        }
        tmem_st_wait();
      }
      // pass 2: probabilities, row sum, bf16 P into the swizzled K-major tile
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(sadr + c * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int key = j * BKV + c * 32 + e;
          const float x0 = __uint_as_float(v[e]) * p.scale_log2;
          const float x1 = __uint_as_float(v[e + 1]) * p.scale_log2;
          const float p0 = (diag && key > qrow) ? 0.f : exp2f(x0 - m_new);
          const float p1 = (diag && key + 1 > qrow) ? 0.f : exp2f(x1 - m_new);
          rs += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        uint8_t* blk = prow + (c >> 1) * 16384;   // 64-key swizzle block
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (c & 1) * 4 + q;
          *reinterpret_cast<uint4*>(blk + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      l = l * alpha + rs;
      m = m_new;
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(s_free(s));
        mbar_arrive(p_full);
      }
    }
    // O / l and lse once the last P V product is done
    if (ok && mbar_wait(p_free, (nkb - 1) & 1, p.err)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(row0 + qrow) * p.Hq + h) * HD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(oadr + c * 32, v);
        tmem_ld_wait();
        if (qrow < p.S) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = w;
          }
        }
      }
      if (qrow < p.S) p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.S + qrow] = (m + log2f(l)) * LN2_F;
    } else {
      ok = false;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [rows, cols] bf16 row-major, box 64 columns x 128 rows, 128-byte swizzle.
kl_status map_rows(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  auto fn = encode();
  if (!fn) return set_error(KL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(KL_ERR_INVALID_ARG, "attention tensor map encode failed (%d)", (int)r);
  return KL_OK;
}

}  // namespace

kl_status attention_fwd_tc(int B, int S, int Hq, int Hkv, const void* q, const void* k, const void* v, void* o,
                           float* lse, cudaStream_t st) {
  FwdParams p;
  memset(&p, 0, sizeof(p));
  const uint64_t T = static_cast<uint64_t>(B) * S;
  KL_TRY(map_rows(&p.tmQ, q, static_cast<uint64_t>(Hq) * HD, T));
  KL_TRY(map_rows(&p.tmK, k, static_cast<uint64_t>(Hkv) * HD, T));
  KL_TRY(map_rows(&p.tmV, v, static_cast<uint64_t>(Hkv) * HD, T));
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.S = S;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2 = LOG2E_F / sqrtf(static_cast<float>(HD));
  p.err = device_error_word();
  static uint64_t attr_done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(fa_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_BYTES)));
    attr_done |= uint64_t(1) << dev;
  }
  dim3 grid((S + BQ - 1) / BQ, Hq, B);
  fa_fwd_tc_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(p);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
