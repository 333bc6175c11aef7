// Causal GQA attention forward on the 5th-generation tensor cores ("KYNETRA
// FOUNDRY", tiled-attention paragraph: query tiles stream over key/value tiles
// with a running max and sum, the score matrix never leaves the chip).
//
// One CTA = 128 query rows of one query head (head dim 128). For short
// sequences a persistent form (fa_fwd_tc_persist_kernel) has one CTA per SM
// work through such items, longest first in a snake order: the K/V ring, the
// score buffers and the P hand-off keep their phases across items, Q is
// reloaded as soon as an item's last score product has used it, and O
// alternates between two TMEM buffers, so an item's epilogue overlaps the next
// item's loads and first score product. 6 warps:
//   warp 0      TMA: Q (per item), then K_j / V_j tiles of 128 keys, 2 stages each
//   warp 1      TMEM owner; one thread issues tcgen05.mma:
//                 S_j  = Q K_j^T   -> TMEM S[j%2]  (128 x 128 fp32)
//                 O   += P_j V_j   -> TMEM O[item%2] (128 x 128 fp32)
//               S_{j+1} is issued before P_j V_j so the tensor core computes
//               the next scores while the softmax warps work on P_j. P_j is
//               the TMEM A operand of its product (the one-CTA-per-item form
//               also holds Q in TMEM), so the products read only K and V from
//               shared memory.
//   warps 2..5  softmax: thread = query row = TMEM lane. Two passes over S_j
//               (row max, then exp2 / row sum / bf16 P written with tcgen05.st
//               into the first 64 columns of S_j's own buffer). The running
//               max is only raised when a row's max grows by more than 2^8
//               (then that warp rescales its O rows in TMEM); otherwise P is
//               taken against the stale max, which the final O / l cancels.
// Every wait is bounded; a timeout records KL_DEVERR_TIMEOUT and unwinds.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int HD = 128;       // head dim
constexpr int BQ = 128;       // query rows per CTA
constexpr int BKV = 128;      // keys per tile
constexpr uint32_t TILE_BYTES = 128 * 128 * 2;   // 32 KB: two 16 KB swizzle blocks of 64 columns
constexpr int THREADS = 192;
// Backward kernels: TMA warp, MMA warp and 8 elementwise warps, two per TMEM
// lane quarter, each taking 32 of a step's 64 columns (one warp per scheduler
// left the exp / multiply / store chain of a step unhidden).
constexpr int BWD_THREADS = 320;
constexpr int BWD_EW = 8;                     // elementwise warps
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float LN2_F = 0.6931471805599453f;

// shared-memory layout (offsets from a 1024-aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;          // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE_BYTES;      // 2 stages
constexpr uint32_t OFF_BAR = OFF_V + 2 * TILE_BYTES;
// tensor memory of the one-CTA-per-item form: S[0], S[1] (P in the first 64
// columns of each), O, and Q as bf16 pairs (the A operand of S = Q K^T)
constexpr uint32_t TM_QF = 384;
constexpr size_t SMEM_BYTES = 1024 + OFF_BAR + 256;

struct FwdParams {
  CUtensorMap tmQ, tmK, tmV;
  __nv_bfloat16* o;
  float* lse;
  int S, Hq, Hkv, B;
  int items;                  // B * Hq * query tiles
  float scale_log2;
  uint32_t* err;
};

// 2^x with the hardware approximation (about 2 ulp; 0 for -inf).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// The query tiles of every (sequence, head), longest first: position t holds
// query tile nqb-1 - t / (B Hq) of head t % Hq of sequence (t / Hq) % B.
struct FwdItem {
  int b, h, qb;
};
__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int t) {
  const int nqb = (p.S + BQ - 1) / BQ;
  const int per = p.Hq * p.B;
  const int y = t / per, rem = t - y * per;
  const int b = rem / p.Hq;
  return {b, rem - b * p.Hq, nqb - 1 - y};
}
// The k-th item of CTA c of G: a snake over the longest-first list (rounds of
// G items, every other round reversed), so the CTAs' key-tile counts even out.
__device__ __forceinline__ int fwd_item_index(int c, int k, int G) { return k * G + ((k & 1) ? G - 1 - c : c); }

__global__ void __launch_bounds__(THREADS, 1) fa_fwd_tc_kernel(const __grid_constant__ FwdParams p) {
  pdl_enter();
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
  const uint32_t q_tm = bar + 120;     // Q copied into tensor memory
  const uint32_t drain = bar + 152;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 164);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (p.S + BQ - 1) / BQ;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.y);   // longest rows first (all heads)
  const int h = blockIdx.x, b = blockIdx.z;
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
    mbar_init(q_tm, 4);
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

  if (warp == 0) {
    // ---------------- TMA (whole warp; the elected lane issues) ----------------
    const bool el = elect_one();
    if (el) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      mbar_arrive_expect_tx(q_full, TILE_BYTES);
      tma_load_2d(sb + OFF_Q, &p.tmQ, h * HD, row0 + q0, q_full);
      tma_load_2d(sb + OFF_Q + 16384, &p.tmQ, h * HD + 64, row0 + q0, q_full);
    }
    __syncwarp();
    int issued_k = 0, issued_v = 0;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(k_empty(s), ph ^ 1u, p.err, abort_flag)) { *abort_flag = 1; break; }
      if (el) {
        mbar_arrive_expect_tx(k_full(s), TILE_BYTES);
        tma_load_2d(sb + OFF_K + s * TILE_BYTES, &p.tmK, j_kv * HD, row0 + j * BKV, k_full(s));
        tma_load_2d(sb + OFF_K + s * TILE_BYTES + 16384, &p.tmK, j_kv * HD + 64, row0 + j * BKV, k_full(s));
      }
      __syncwarp();
      ++issued_k;
      if (!mbar_wait_warp(v_empty(s), ph ^ 1u, p.err, abort_flag)) { *abort_flag = 1; break; }
      if (el) {
        mbar_arrive_expect_tx(v_full(s), TILE_BYTES);
        tma_load_2d(sb + OFF_V + s * TILE_BYTES, &p.tmV, j_kv * HD, row0 + j * BKV, v_full(s));
        tma_load_2d(sb + OFF_V + s * TILE_BYTES + 16384, &p.tmV, j_kv * HD + 64, row0 + j * BKV, v_full(s));
      }
      __syncwarp();
      ++issued_v;
    }
    // copies still in flight must land before exit
    mbar_wait(q_full, 0, p.err);
    for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j) mbar_wait(k_full(j & 1), (j >> 1) & 1, p.err);
    for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j) mbar_wait(v_full(j & 1), (j >> 1) & 1, p.err);
  } else if (warp == 1) {
    // ---------------- MMA (whole warp; the elected lane issues) ----------------
    const bool el = elect_one();
    const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = mbar_wait_warp(q_tm, 0, p.err, abort_flag);
    auto issue_pv = [&](int j) -> bool {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(p_full, j & 1, p.err, abort_flag)) return false;
      if (!mbar_wait_warp(v_full(s), ph, p.err, abort_flag)) return false;
      tc_fence_after();
      if (el) {
        for (int kk = 0; kk < BKV / 16; ++kk)   // P from TMEM (the first 64 columns of S[s])
          umma_bf16_ta(tmem + 256, tmem + s * 128 + kk * 8, desc_mnmajor(sb + OFF_V + s * TILE_BYTES, kk),
                       idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(v_empty(s));
        umma_commit(p_free);
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; ok && j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(k_full(s), ph, p.err, abort_flag) ||
          (j >= 2 && !mbar_wait_warp(s_free(s), ph ^ 1u, p.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + s * 128;
      if (el) {
        for (int kk = 0; kk < HD / 16; ++kk)   // Q from TMEM
          umma_bf16_ta(d, tmem + TM_QF + kk * 8, desc_kmajor(sb + OFF_K + s * TILE_BYTES, kk), idesc_s, kk > 0);
        umma_commit(k_empty(s));
        umma_commit(s_full(s));
      }
      __syncwarp();
      if (j >= 1 && !issue_pv(j - 1)) ok = false;
    }
    if (ok && !issue_pv(nkb - 1)) ok = false;
    if (!ok) *abort_flag = 1;
    if (el) umma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err);
  } else if (warp >= 2) {
    // ---------------- softmax / correction / epilogue ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;           // query row within the tile = TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t oadr = tmem + lane_off + 256;
    float m = -INFINITY, l = 0.f;
    bool ok = mbar_wait_warp(q_full, 0, p.err, abort_flag);
    if (ok) {
      // this row's Q (two 128-byte-swizzled 64-column blocks) into TMEM columns
      // TM_QF .. + 63 as bf16 pairs: the A operand of every S = Q K^T
      uint32_t qa[32], qb[32];
      const uint8_t* qs = smem + OFF_Q + r * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int off = (e ^ (r & 7)) << 4;
        const uint4 x = *reinterpret_cast<const uint4*>(qs + off), y = *reinterpret_cast<const uint4*>(qs + 16384 + off);
        qa[4 * e] = x.x; qa[4 * e + 1] = x.y; qa[4 * e + 2] = x.z; qa[4 * e + 3] = x.w;
        qb[4 * e] = y.x; qb[4 * e + 1] = y.y; qb[4 * e + 2] = y.z; qb[4 * e + 3] = y.w;
      }
      tmem_st_32x32b_x32(tmem + lane_off + TM_QF, qa);
      tmem_st_32x32b_x32(tmem + lane_off + TM_QF + 32, qb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_tm);
    }
    for (int j = 0; ok && j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(s_full(s), ph, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sadr = tmem + lane_off + s * 128;
      // the whole score row in registers: one TMEM round trip
      uint32_t sv[BKV];
      tmem_ld_32x32b_x32(sadr + 0, *reinterpret_cast<uint32_t(*)[32]>(sv + 0));
      tmem_ld_32x32b_x32(sadr + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_ld_32x32b_x32(sadr + 64, *reinterpret_cast<uint32_t(*)[32]>(sv + 64));
      tmem_ld_32x32b_x32(sadr + 96, *reinterpret_cast<uint32_t(*)[32]>(sv + 96));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(s));   // S[s] may be overwritten from here on
      if (j == nkb - 1) {                      // diagonal tile: keys after the row are masked
        const int lim = qrow - j * BKV;        // keys 0 .. lim are kept
#pragma unroll
        for (int e = 0; e < BKV; ++e)
          if (e > lim) sv[e] = __float_as_uint(-INFINITY);
      }
      float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
      for (int e = 0; e < BKV; e += 4) {
        m0 = fmaxf(m0, __uint_as_float(sv[e]));
        m1 = fmaxf(m1, __uint_as_float(sv[e + 1]));
        m2 = fmaxf(m2, __uint_as_float(sv[e + 2]));
        m3 = fmaxf(m3, __uint_as_float(sv[e + 3]));
      }
      const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * p.scale_log2;
      // raise the running max only when it grows by more than 2^8
      const bool raise = mx > m + 8.0f;
      const float m_new = raise ? mx : m;
      const float alpha = raise ? ex2_approx(m - m_new) : 1.0f;
      // O is stable for a rescale once the previous P V product is done (P
      // goes into this step's S buffer, which S's completion shows free)
      if (j >= 1 && __any_sync(0xffffffffu, raise)) {
        if (!mbar_wait_warp(p_free, (j - 1) & 1, p.err, abort_flag)) { ok = false; break; }
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
      // probabilities (one FFMA + one ex2 each), row sum, bf16 P packed two
      // keys per column into the first 64 columns of S[s] (the A operand of
      // the P V product; S has been read into registers)
      const float neg = -m_new;
      const float sc = p.scale_log2;
      float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int e = 0; e < BKV; e += 4) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), sc, neg));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), sc, neg));
        const float p2 = ex2_approx(fmaf(__uint_as_float(sv[e + 2]), sc, neg));
        const float p3 = ex2_approx(fmaf(__uint_as_float(sv[e + 3]), sc, neg));
        r0 += p0;
        r1 += p1;
        r2 += p2;
        r3 += p3;
        pk[e >> 1] = pack_bf16x2(p0, p1);
        pk[(e >> 1) + 1] = pack_bf16x2(p2, p3);
      }
      tmem_st_32x32b_x32(sadr, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st_32x32b_x32(sadr + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      l = l * alpha + ((r0 + r1) + (r2 + r3));
      m = m_new;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // O / l and lse once the last P V product is done. p_free completes once per
    // P V product, and the last scores' completion shows only the product two
    // steps back done (the one before is issued after those scores): a parity
    // wait for the last one alone would pass while the barrier is still a phase
    // behind it, so the product before it is waited for first.
    if (ok && (nkb < 2 || mbar_wait_warp(p_free, (nkb - 2) & 1, p.err, abort_flag)) &&
        mbar_wait_warp(p_free, (nkb - 1) & 1, p.err, abort_flag)) {
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

// Persistent form for short sequences (see the file comment): CTA c works
// through items c, then the snake's later ones.
__global__ void __launch_bounds__(THREADS, 1) fa_fwd_tc_persist_kernel(const __grid_constant__ FwdParams p) {
  pdl_enter();
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
  const uint32_t q_empty = bar + 120;
  auto o_empty = [&](int s) { return bar + 128 + 8 * s; };
  const uint32_t drain = bar + 152;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 160);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 164);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  auto item_of = [&](int k) { return fwd_item_index(cta, k, G); };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 4);
      mbar_init(o_empty(s), 4);
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
  const uint32_t tmem = *tmem_holder;   // S[0] at column 0, S[1] at 128, O[0] at 256, O[1] at 384

  if (warp == 0) {
    // ---------------- TMA (whole warp; the elected lane issues) ----------------
    const bool el = elect_one();
    if (el) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
    }
    int issued_q = 0, issued_k = 0, issued_v = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int t = item_of(k);
      if (t >= p.items) break;
      const FwdItem f = fwd_item(p, t);
      const int row0 = f.b * p.S, j_kv = f.h * p.Hkv / p.Hq, nkb = f.qb + 1;
      // Q: the buffer is free once the previous item's last S product is done
      if (!mbar_wait_warp(q_empty, (k & 1) ^ 1u, p.err, abort_flag)) { ok = false; break; }
      if (el) {
        mbar_arrive_expect_tx(q_full, TILE_BYTES);
        tma_load_2d(sb + OFF_Q, &p.tmQ, f.h * HD, row0 + f.qb * BQ, q_full);
        tma_load_2d(sb + OFF_Q + 16384, &p.tmQ, f.h * HD + 64, row0 + f.qb * BQ, q_full);
      }
      __syncwarp();
      ++issued_q;
      for (int j = 0; j < nkb; ++j) {
        const int s = issued_k & 1;
        const uint32_t ph = (issued_k >> 1) & 1;
        if (!mbar_wait_warp(k_empty(s), ph ^ 1u, p.err, abort_flag)) { ok = false; break; }
        if (el) {
          mbar_arrive_expect_tx(k_full(s), TILE_BYTES);
          tma_load_2d(sb + OFF_K + s * TILE_BYTES, &p.tmK, j_kv * HD, row0 + j * BKV, k_full(s));
          tma_load_2d(sb + OFF_K + s * TILE_BYTES + 16384, &p.tmK, j_kv * HD + 64, row0 + j * BKV, k_full(s));
        }
        __syncwarp();
        ++issued_k;
        if (!mbar_wait_warp(v_empty(s), ph ^ 1u, p.err, abort_flag)) { ok = false; break; }
        if (el) {
          mbar_arrive_expect_tx(v_full(s), TILE_BYTES);
          tma_load_2d(sb + OFF_V + s * TILE_BYTES, &p.tmV, j_kv * HD, row0 + j * BKV, v_full(s));
          tma_load_2d(sb + OFF_V + s * TILE_BYTES + 16384, &p.tmV, j_kv * HD + 64, row0 + j * BKV, v_full(s));
        }
        __syncwarp();
        ++issued_v;
      }
    }
    if (!ok) *abort_flag = 1;
    // copies still in flight must land before exit
    if (issued_q > 0) mbar_wait(q_full, (issued_q - 1) & 1, p.err);
    for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j) mbar_wait(k_full(j & 1), (j >> 1) & 1, p.err);
    for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j) mbar_wait(v_full(j & 1), (j >> 1) & 1, p.err);
  } else if (warp == 1) {
    // ---------------- MMA (whole warp; the elected lane issues) ----------------
    // Step g (over all items) issues S_g, then the P V product of step g - 1,
    // which may be the previous item's last: the tensor core computes the next
    // scores while the softmax warps work on the current ones.
    const bool el = elect_one();
    const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);
    auto issue_pv = [&](int gp, int ob, bool first) -> bool {
      const int s = gp & 1;
      const uint32_t ph = (gp >> 1) & 1;
      if (!mbar_wait_warp(p_full, gp & 1, p.err, abort_flag)) return false;
      if (!mbar_wait_warp(v_full(s), ph, p.err, abort_flag)) return false;
      tc_fence_after();
      if (el) {
        for (int kk = 0; kk < BKV / 16; ++kk)   // P from TMEM (the first 64 columns of S[s])
          umma_bf16_ta(tmem + 256 + ob * 128, tmem + s * 128 + kk * 8, desc_mnmajor(sb + OFF_V + s * TILE_BYTES, kk),
                       idesc_pv, (!first || kk > 0) ? 1u : 0u);
        umma_commit(v_empty(s));
        umma_commit(p_free);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    int g = 0, pend_g = -1, pend_ob = 0;
    bool pend_first = false;
    for (int k = 0; ok; ++k) {
      const int t = item_of(k);
      if (t >= p.items) break;
      const int nkb = fwd_item(p, t).qb + 1, ob = k & 1;
      if (!mbar_wait_warp(q_full, k & 1, p.err, abort_flag)) { ok = false; break; }
      for (int j = 0; j < nkb; ++j, ++g) {
        const int s = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        if (!mbar_wait_warp(k_full(s), ph, p.err, abort_flag) ||
            (g >= 2 && !mbar_wait_warp(s_free(s), ph ^ 1u, p.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (el) {
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(tmem + s * 128, desc_kmajor(sb + OFF_Q, kk), desc_kmajor(sb + OFF_K + s * TILE_BYTES, kk), idesc_s,
                      kk > 0);
          umma_commit(k_empty(s));
          umma_commit(s_full(s));
          if (j == nkb - 1) umma_commit(q_empty);   // the item's last use of Q
        }
        __syncwarp();
        if (pend_g >= 0 && !issue_pv(pend_g, pend_ob, pend_first)) { ok = false; break; }
        // O[ob] takes this item's first P V: the epilogue of item k - 2 must have read it
        if (j == 0 && !mbar_wait_warp(o_empty(ob), ((k >> 1) & 1) ^ 1u, p.err, abort_flag)) { ok = false; break; }
        pend_g = g;
        pend_ob = ob;
        pend_first = j == 0;
      }
    }
    if (ok && pend_g >= 0 && !issue_pv(pend_g, pend_ob, pend_first)) ok = false;
    if (!ok) *abort_flag = 1;
    if (el) umma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err);
  } else if (warp >= 2) {
    // ---------------- softmax / correction / epilogue ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;           // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int t = item_of(k);
      if (t >= p.items) break;
      const FwdItem f = fwd_item(p, t);
      const int nkb = f.qb + 1, ob = k & 1;
      const int qrow = f.qb * BQ + r;
      const uint32_t oadr = tmem + lane_off + 256 + ob * 128;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkb; ++j, ++g) {
        const int s = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        if (!mbar_wait_warp(s_full(s), ph, p.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sadr = tmem + lane_off + s * 128;
        // the whole score row in registers: one TMEM round trip
        uint32_t sv[BKV];
        tmem_ld_32x32b_x32(sadr, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld_32x32b_x32(sadr + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_ld_32x32b_x32(sadr + 64, *reinterpret_cast<uint32_t(*)[32]>(sv + 64));
        tmem_ld_32x32b_x32(sadr + 96, *reinterpret_cast<uint32_t(*)[32]>(sv + 96));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free(s));   // S[s] may be overwritten from here on
        if (j == nkb - 1) {                      // diagonal tile: keys after the row are masked
          const int lim = qrow - j * BKV;        // keys 0 .. lim are kept
#pragma unroll
          for (int e = 0; e < BKV; ++e)
            if (e > lim) sv[e] = __float_as_uint(-INFINITY);
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < BKV; e += 4) {
          m0 = fmaxf(m0, __uint_as_float(sv[e]));
          m1 = fmaxf(m1, __uint_as_float(sv[e + 1]));
          m2 = fmaxf(m2, __uint_as_float(sv[e + 2]));
          m3 = fmaxf(m3, __uint_as_float(sv[e + 3]));
        }
        const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * p.scale_log2;
        // raise the running max only when it grows by more than 2^8
        const bool raise = mx > m + 8.0f;
        const float m_new = raise ? mx : m;
        const float alpha = raise ? ex2_approx(m - m_new) : 1.0f;
        // O is stable for a rescale once the previous P V product is done (P
        // goes into this step's S buffer, which S's completion shows free)
        if (j >= 1 && __any_sync(0xffffffffu, raise)) {
          if (!mbar_wait_warp(p_free, (g - 1) & 1, p.err, abort_flag)) { ok = false; break; }
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
        // probabilities (one FFMA + one ex2 each), row sum, bf16 P packed two
        // keys per column into the first 64 columns of S[s] (the A operand of
        // the P V product; S has been read into registers)
        const float neg = -m_new;
        const float sc = p.scale_log2;
        float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int e = 0; e < BKV; e += 4) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), sc, neg));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), sc, neg));
          const float p2 = ex2_approx(fmaf(__uint_as_float(sv[e + 2]), sc, neg));
          const float p3 = ex2_approx(fmaf(__uint_as_float(sv[e + 3]), sc, neg));
          r0 += p0;
          r1 += p1;
          r2 += p2;
          r3 += p3;
          pk[e >> 1] = pack_bf16x2(p0, p1);
          pk[(e >> 1) + 1] = pack_bf16x2(p2, p3);
        }
        tmem_st_32x32b_x32(sadr, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st_32x32b_x32(sadr + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        l = l * alpha + ((r0 + r1) + (r2 + r3));
        m = m_new;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      // O / l and lse once the item's last P V product (step g - 1) is done. p_free
      // completes once per P V product; step g - 1's scores completing shows only
      // step g - 3's product done (step g - 2's is issued after those scores), and a
      // parity wait for step g - 1's alone would pass while the barrier is still at
      // step g - 2's phase: wait for that one first.
      if (g >= 2 && !mbar_wait_warp(p_free, (g - 2) & 1, p.err, abort_flag)) { ok = false; break; }
      if (!mbar_wait_warp(p_free, (g - 1) & 1, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(f.b * p.S + qrow) * p.Hq + f.h) * HD;
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(ob));   // O[ob] may take item k + 2's products
      if (qrow < p.S) p.lse[(static_cast<int64_t>(f.b) * p.Hq + f.h) * p.S + qrow] = (m + log2f(l)) * LN2_F;
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


// ===========================================================================
// Backward on the tensor cores. Two kernels, both recomputing P from lse:
//   dK/dV: CTA = 128 keys of one kv head, walking 64-query tiles of every
//          query head of its GQA group from the diagonal on (at short
//          sequences the group is split over a 2- or 4-CTA cluster).
//          S^T = K Q^T and dP^T = V dO^T in TMEM (K and V are TMEM A
//          operands); thread = key row builds P^T and dS^T = P^T (dP^T - D)
//          as bf16 in swizzled shared memory; dV += P^T dO and dK += dS^T Q
//          accumulate in TMEM across the group and are written once as bf16.
//   dQ:    CTA = 128 queries of one head; 64-key tiles up to the diagonal.
//          S = Q K^T and dP = dO V^T (Q and dO are TMEM A operands); thread =
//          query row builds dS into TMEM; dQ += dS K accumulates in TMEM and
//          is written once (no atomics).
// ===========================================================================
constexpr uint32_t T64 = 64 * 128 * 2;   // 16 KB: a 64-row x 128-column bf16 tile (two 8 KB blocks)

// K-major operand: R rows x 128 columns stored as two 64-column swizzle blocks
// of R x 128 bytes; descriptor of k-step kk.
__device__ __forceinline__ uint64_t desc_k128(uint32_t base, uint32_t block_bytes, int kk) {
  return smem_desc_sw128(base + (kk >> 2) * block_bytes + (kk & 3) * 32, 16, 1024);
}
// K-major operand: R rows x 64 columns (one swizzle block).
__device__ __forceinline__ uint64_t desc_k64(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 32, 16, 1024);
}
// MN-major view of a [K rows x 128 columns] tile (two 64-column blocks of
// K x 128 bytes): N = the 128 columns, k-step kk = 16 rows.
__device__ __forceinline__ uint64_t desc_mn128(uint32_t base, uint32_t block_bytes, int kk) {
  return smem_desc_sw128(base + kk * 2048, block_bytes, 1024);
}

struct BwdParams {
  CUtensorMap tmQ, tmK, tmV, tmdO;   // box rows: see the kernels
  const float* lse;                  // [B, Hq, S]
  const float* Dd;                   // [B, Hq, S]
  float* dq_acc;                     // [T, Hq*128] fp32 (when dq_out is null)
  __nv_bfloat16* dq_out;             // [T, Hq*128] bf16 final dQ, or null
  __nv_bfloat16* dk_out;             // [T, Hkv*128] bf16 final dK
  __nv_bfloat16* dv_out;             // [T, Hkv*128] bf16 final dV
  const float2* rope_cs;             // [S][64] cos/sin: dQ (with dq_out) and dK turned back by -angle, or null
  const __nv_bfloat16* kg;           // [T, Hkv*128] K and V (dK/dV kernel: rows read into TMEM)
  const __nv_bfloat16* vg;
  int S, Hq, Hkv;
  int nsplit;                        // CTAs (one cluster) sharing a kv head's key tile; heads split between them
  float scale_log2, scale;
  uint32_t* err;
};

// ---------------------------------------------------------------------------
// dK / dV, one CTA per (kv head, 128-key tile) walking its query-head group
// ---------------------------------------------------------------------------
// The kv head's K and V tiles are loaded once; the CTA then steps through
// 64-query tiles of every query head of its share of the group (each head from
// the diagonal to the end of the sequence) with dV and dK accumulating in TMEM
// across all of them. When the group is split over a cluster of nsplit CTAs
// (short sequences: the causal work per key tile is uneven and few tiles
// exist), the CTAs' partial sums meet in distributed shared memory: CTA o owns
// head-dim columns [W o, W o + W) and [64 + W o, ...) (W = 64 / nsplit, so a
// rotary plane's two columns stay together) and adds the nsplit partials of
// those columns in rank order. dK (times the softmax scale, turned back by the
// key position's rotary angle when a table is given) and dV are written once,
// as bf16: no atomics, and the same bits on every run.
//
// K and V are the A operands of S^T = K Q^T and dP^T = V dO^T and stay the same
// for the whole CTA, so they live in tensor memory (loaded once by the
// elementwise warps): each step's products then read only Q, dO, P^T and dS^T
// from shared memory, which bounds these N = 64 products when both operands
// come from shared memory. Tensor memory: S^T | dP^T (one buffer, 64 columns
// each), K | V (bf16, 64 columns each), dV, dK (128 fp32 columns each).
// Shared memory: a 4-stage Q / dO ring with the stage's lse / D rows, and
// double-buffered P^T / dS^T. The dynamic shared memory is taken as 1024-byte
// aligned (checked at entry).
constexpr int KV_QS = 4;                                      // stages of the Q / dO / lse / D ring
constexpr uint32_t KV_OFF_Q = 0;                              // KV_QS stages of T64
constexpr uint32_t KV_OFF_DO = KV_OFF_Q + KV_QS * T64;       // KV_QS stages of T64
constexpr uint32_t PT_BYTES = 128 * 64 * 2;                   // 16 KB: 128 key rows x 64 queries
constexpr uint32_t KV_OFF_P = KV_OFF_DO + KV_QS * T64;       // 2 buffers of P^T
constexpr uint32_t KV_OFF_DS = KV_OFF_P + 2 * PT_BYTES;      // 2 buffers of dS^T
constexpr uint32_t KV_OFF_STAT = KV_OFF_DS + 2 * PT_BYTES;  // KV_QS stages: lse[64], D[64] (fp32)
constexpr uint32_t KV_OFF_BAR = KV_OFF_STAT + KV_QS * 512;
constexpr size_t KV_SMEM = KV_OFF_BAR + 256;
constexpr uint32_t TM_ST = 0, TM_DPT = 64, TM_K = 128, TM_V = 192, TM_DV = 256, TM_DK = 384;
// The partial-sum exchange reuses the Q / dO ring: nsplit slots of 128 rows x
// 4W fp32 (dV low, dV high, dK low, dK high columns) = 128 KB.
constexpr uint32_t KV_OFF_XCH = 0;
constexpr uint32_t KV_XCH_BYTES = 128 * 256 * 4;
static_assert(KV_XCH_BYTES <= KV_OFF_P, "exchange slots overlap the P^T buffers");
static_assert(KV_SMEM <= 232448, "dK/dV shared memory above the per-CTA limit");

// Writes one key row's finished dV or dK columns [c0, c0 + W) and [64 + c0, ...)
// as bf16 (dK: times the scale, turned back by the key position's rotary angle).
template <int W>
__device__ __forceinline__ void dkdv_store_row(__nv_bfloat16* row, int c0, const float (&lo)[W],
                                               const float (&hi)[W], bool is_k, float scale,
                                               const float2* cs) {
  float a[W], bb[W];
#pragma unroll
  for (int e = 0; e < W; ++e) {
    if (is_k) {
      const float x = lo[e] * scale, y = hi[e] * scale;
      if (cs) {
        const float2 t = cs[c0 + e];
        a[e] = x * t.x + y * t.y;
        bb[e] = y * t.x - x * t.y;
      } else {
        a[e] = x;
        bb[e] = y;
      }
    } else {
      a[e] = lo[e];
      bb[e] = hi[e];
    }
  }
#pragma unroll
  for (int e = 0; e < W; e += 8) {
    uint4 wa, wb;
    wa.x = pack_bf16x2(a[e], a[e + 1]); wa.y = pack_bf16x2(a[e + 2], a[e + 3]);
    wa.z = pack_bf16x2(a[e + 4], a[e + 5]); wa.w = pack_bf16x2(a[e + 6], a[e + 7]);
    wb.x = pack_bf16x2(bb[e], bb[e + 1]); wb.y = pack_bf16x2(bb[e + 2], bb[e + 3]);
    wb.z = pack_bf16x2(bb[e + 4], bb[e + 5]); wb.w = pack_bf16x2(bb[e + 6], bb[e + 7]);
    *reinterpret_cast<uint4*>(row + c0 + e) = wa;
    *reinterpret_cast<uint4*>(row + 64 + c0 + e) = wb;
  }
}

// TMEM columns [col, col + W) of this warp's 32 lanes (W = 16, 32 or 64).
template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[W]) {
  if constexpr (W == 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
  } else {
#pragma unroll
    for (int c = 0; c < W; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) v[c + e] = __uint_as_float(r[e]);
    }
  }
}

// The end of the dK/dV kernel for one elementwise thread: key row r (TMEM lane),
// matrix is_k (dK at TMEM column 384, else dV at 256). With a cluster, the
// thread first sends its row's columns of every owner to that owner's slot
// `rank` (between the two cluster barriers the caller places around it), then
// adds its own columns' slots in rank order.
template <int W>
__device__ __forceinline__ void dkdv_send(uint32_t tmem_row, uint32_t sb, int r, bool is_k, int nsplit,
                                          uint32_t rank) {
  const uint32_t slot_bytes = 128u * 16u * W;
  for (int o = 0; o < nsplit; ++o) {
    float lo[W], hi[W];
    tmem_ld_cols<W>(tmem_row + W * o, lo);
    tmem_ld_cols<W>(tmem_row + 64 + W * o, hi);
    // row r of slot `rank`: 4W floats (dV lo, dV hi, dK lo, dK hi), 16-byte granules XOR-swizzled by row
    const uint32_t rowb = sb + KV_OFF_XCH + rank * slot_bytes + static_cast<uint32_t>(r) * 16u * W;
    const uint32_t dst = mapa_shared(rowb, static_cast<uint32_t>(o));
#pragma unroll
    for (int g = 0; g < W / 4; ++g) {
      const int ga = (is_k ? W / 2 : 0) + g, gb = (is_k ? W / 2 : 0) + W / 4 + g;
      st_cluster_v4(dst + ((ga ^ (r & 7)) << 4), lo[4 * g], lo[4 * g + 1], lo[4 * g + 2], lo[4 * g + 3]);
      st_cluster_v4(dst + ((gb ^ (r & 7)) << 4), hi[4 * g], hi[4 * g + 1], hi[4 * g + 2], hi[4 * g + 3]);
    }
  }
}

template <int W>
__device__ __forceinline__ void dkdv_reduce_store(const uint8_t* smem, int r, bool is_k, int nsplit, uint32_t rank,
                                                  __nv_bfloat16* row, float scale, const float2* cs) {
  const uint32_t slot_bytes = 128u * 16u * W;
  float lo[W], hi[W];
#pragma unroll
  for (int e = 0; e < W; ++e) lo[e] = hi[e] = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const uint8_t* rowp = smem + KV_OFF_XCH + s * slot_bytes + static_cast<uint32_t>(r) * 16u * W;
#pragma unroll
    for (int g = 0; g < W / 4; ++g) {
      const int ga = (is_k ? W / 2 : 0) + g, gb = (is_k ? W / 2 : 0) + W / 4 + g;
      const float4 a = *reinterpret_cast<const float4*>(rowp + ((ga ^ (r & 7)) << 4));
      const float4 b = *reinterpret_cast<const float4*>(rowp + ((gb ^ (r & 7)) << 4));
      lo[4 * g] += a.x; lo[4 * g + 1] += a.y; lo[4 * g + 2] += a.z; lo[4 * g + 3] += a.w;
      hi[4 * g] += b.x; hi[4 * g + 1] += b.y; hi[4 * g + 2] += b.z; hi[4 * g + 3] += b.w;
    }
  }
  if (row) dkdv_store_row<W>(row, W * static_cast<int>(rank), lo, hi, is_k, scale, cs);
}

// Bounded wait by one thread that also gives up when the CTA's abort flag is
// set (another role stopped): false then, or on timeout (recorded).
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, uint32_t* err,
                                                   volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > KL_WAIT_LIMIT_NS) {
        record_error(err, KL_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__global__ void __launch_bounds__(BWD_THREADS, 1) fa_bwd_dkdv_tc_kernel(const __grid_constant__ BwdParams p) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t kv_smem_raw[];
  const int nsplit = p.nsplit;
  if (smem_u32(kv_smem_raw) & 1023u) {   // the layout has no alignment slack (CTA-uniform exit)
    if (threadIdx.x == 0) record_error(p.err, KL_DEVERR_SMEM);
    if (nsplit > 1) {                    // the cluster's barriers still see every thread
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }
  uint8_t* smem = kv_smem_raw;
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + KV_OFF_BAR;
  auto q_full = [&](int s) { return bar + 8 * s; };                   // KV_QS of each ring barrier
  auto q_free = [&](int s) { return bar + 8 * KV_QS + 8 * s; };
  const uint32_t st_full = bar + 16 * KV_QS;                          // S^T / dP^T in TMEM
  const uint32_t st_free = bar + 16 * KV_QS + 8;
  auto p_full = [&](int s) { return bar + 16 * KV_QS + 16 + 8 * s; }; // 2 P^T / dS^T buffers
  auto p_free = [&](int s) { return bar + 16 * KV_QS + 32 + 8 * s; };
  const uint32_t kv_ready = bar + 16 * KV_QS + 48;                    // K, V written into TMEM
  const uint32_t done = bar + 16 * KV_QS + 56;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + KV_OFF_BAR + 16 * KV_QS + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + KV_OFF_BAR + 16 * KV_QS + 68);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.y;                 // key tiles near the start see the most queries
  const int jh = static_cast<int>(blockIdx.x) / nsplit, b = blockIdx.z;
  const uint32_t rank = nsplit > 1 ? cluster_ctarank() : 0u;
  const int G = p.Hq / p.Hkv;                // query heads of the kv head
  const int gh = G / nsplit;                 // of them, this CTA's
  const int h_first = jh * G + static_cast<int>(rank) * gh;
  const int k0 = kb * BKV;
  const int row0 = b * p.S;
  const int nit = (p.S - k0 + 63) / 64;      // 64-query tiles from the diagonal to the end, per head
  const int nsteps = gh * nit;               // step g: head h_first + g / nit, query tile g % nit
  // lse / D rows staged in shared memory by bulk copies when they are 16-byte aligned
  const bool stat_smem = (p.S & 3) == 0 && (reinterpret_cast<uintptr_t>(p.lse) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.Dd) & 15u) == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KV_QS; ++s) {
      mbar_init(q_full(s), 1);
      mbar_init(q_free(s), 1);
    }
    mbar_init(st_full, 1);
    mbar_init(st_free, BWD_EW);
    for (int s = 0; s < 2; ++s) {
      mbar_init(p_full(s), BWD_EW);
      mbar_init(p_free(s), 1);
    }
    mbar_init(kv_ready, BWD_EW);
    mbar_init(done, 1);
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
  bool fin = false;                          // elementwise warps: every MMA of the CTA completed

  if (warp == 0) {
    // ---------------- TMA: Q / dO tiles and lse / D rows (the elected lane issues) ----------------
    const bool el = elect_one();
    int issued = 0;
    for (int g = 0; g < nsteps; ++g) {
      const int s = g % KV_QS;
      const uint32_t ph = (g / KV_QS) & 1;
      if (!mbar_wait_warp(q_free(s), ph ^ 1u, p.err, abort_flag)) { *abort_flag = 1; break; }
      const int h = h_first + g / nit;
      const int q0 = k0 + (g % nit) * 64;
      const int qr = row0 + q0;
      if (el) {
        // lse and D of the tile's queries (those inside the sequence) ride with Q and dO
        const int nq = p.S - q0 < 64 ? p.S - q0 : 64;
        const uint32_t stat_bytes = stat_smem ? static_cast<uint32_t>(nq) * 4u : 0u;
        mbar_arrive_expect_tx(q_full(s), 2 * T64 + 2 * stat_bytes);
        if (stat_smem) {
          const int64_t so = (static_cast<int64_t>(b) * p.Hq + h) * p.S + q0;
          bulk_copy_g2s(sb + KV_OFF_STAT + s * 512, p.lse + so, stat_bytes, q_full(s));
          bulk_copy_g2s(sb + KV_OFF_STAT + s * 512 + 256, p.Dd + so, stat_bytes, q_full(s));
        }
        tma_load_2d(sb + KV_OFF_Q + s * T64, &p.tmQ, h * HD, qr, q_full(s));
        tma_load_2d(sb + KV_OFF_Q + s * T64 + 8192, &p.tmQ, h * HD + 64, qr, q_full(s));
        tma_load_2d(sb + KV_OFF_DO + s * T64, &p.tmdO, h * HD, qr, q_full(s));
        tma_load_2d(sb + KV_OFF_DO + s * T64 + 8192, &p.tmdO, h * HD + 64, qr, q_full(s));
      }
      __syncwarp();
      ++issued;
    }
    for (int g = (issued > KV_QS ? issued - KV_QS : 0); g < issued; ++g)
      mbar_wait(q_full(g % KV_QS), (g / KV_QS) & 1, p.err);
  } else if (warp == 1) {
    // ---------------- MMA (the elected lane issues) ----------------
    // S^T / dP^T of step j go out once the elementwise warps have read step
    // j - 1's (one TMEM buffer) and step j's Q / dO have landed; the gradient
    // products of step j - 1 once its P^T / dS^T are written. The elementwise
    // warps read a step's scores before they write its P^T / dS^T and finish a
    // step before they read the next one's, so the issuer waits for the events
    // in that order (S^T of step j, then the gradients of step j - 1) with
    // blocking, bounded waits instead of polling both conditions (~1 % faster
    // at 32768 tokens). The next scores stay one step ahead.
    const bool el = elect_one();
    const uint32_t id_st = idesc_bf16_f32(128, 64, 0, 0);
    const uint32_t id_gr = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = mbar_wait_warp(kv_ready, 0, p.err, abort_flag);
    if (ok) tc_fence_after();
    if (el && ok) {
      for (int j = 0; j <= nsteps; ++j) {
        if (j < nsteps) {
          const int qs = j % KV_QS;
          if (!mbar_wait_or_abort(q_full(qs), (j / KV_QS) & 1, p.err, abort_flag) ||
              (j > 0 && !mbar_wait_or_abort(st_free, (j - 1) & 1, p.err, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sq = sb + KV_OFF_Q + qs * T64, sdo = sb + KV_OFF_DO + qs * T64;
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16_ta(tmem + TM_ST, tmem + TM_K + kk * 8, desc_k128(sq, 8192, kk), id_st, kk > 0);
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16_ta(tmem + TM_DPT, tmem + TM_V + kk * 8, desc_k128(sdo, 8192, kk), id_st, kk > 0);
          umma_commit(st_full);
        }
        if (j > 0) {
          const int g = j - 1;
          if (!mbar_wait_or_abort(p_full(g & 1), (g >> 1) & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int qs = g % KV_QS, pb = g & 1;
          const uint32_t sq = sb + KV_OFF_Q + qs * T64, sdo = sb + KV_OFF_DO + qs * T64;
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + TM_DV, desc_k64(sb + KV_OFF_P + pb * PT_BYTES, kk), desc_mn128(sdo, 8192, kk), id_gr,
                      (g > 0 || kk > 0) ? 1u : 0u);
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + TM_DK, desc_k64(sb + KV_OFF_DS + pb * PT_BYTES, kk), desc_mn128(sq, 8192, kk), id_gr,
                      (g > 0 || kk > 0) ? 1u : 0u);
          umma_commit(q_free(qs));
          umma_commit(p_free(pb));
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, __ffs(__ballot_sync(0xffffffffu, el)) - 1) != 0;
    if (!ok) *abort_flag = 1;
    if (el) umma_commit(done);
    __syncwarp();
    mbar_wait(done, 0, p.err);
  } else if (warp >= 2) {
    // ---------------- K, V into TMEM; then P^T, dS^T (thread = key row) ----------------
    // warp 2 + 4 * half + i: lane quarter (warp & 3), queries 32 * half .. + 31 of a step
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int col0 = half * 32;
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    {
      // this row's head-dim columns 64 * half .. + 63 of K and V (zero past the sequence),
      // packed bf16 pairs into TMEM columns TM_K / TM_V + 32 * half .. + 31
      uint32_t kr[32], vr[32];
      if (key < p.S) {
        const int64_t o = (static_cast<int64_t>(row0 + key) * p.Hkv + jh) * HD + half * 64;
        const uint4* kp = reinterpret_cast<const uint4*>(p.kg + o);
        const uint4* vp = reinterpret_cast<const uint4*>(p.vg + o);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 a = kp[e], c = vp[e];
          kr[4 * e] = a.x; kr[4 * e + 1] = a.y; kr[4 * e + 2] = a.z; kr[4 * e + 3] = a.w;
          vr[4 * e] = c.x; vr[4 * e + 1] = c.y; vr[4 * e + 2] = c.z; vr[4 * e + 3] = c.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;
      }
      tmem_st_32x32b_x32(tmem + lane_off + TM_K + half * 32, kr);
      tmem_st_32x32b_x32(tmem + lane_off + TM_V + half * 32, vr);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_ready);
    }
    const bool vec_stat = (p.S & 3) == 0;     // rows of lse / D are 16-byte aligned
    bool ok = true;
    for (int g = 0; g < nsteps; ++g) {
      const int h = h_first + g / nit;
      const int q0 = k0 + (g % nit) * 64;
      const float* lrow = p.lse + (static_cast<int64_t>(b) * p.Hq + h) * p.S;
      const float* drow = p.Dd + (static_cast<int64_t>(b) * p.Hq + h) * p.S;
      if (!mbar_wait_warp(st_full, g & 1, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[32], dv[32];
      tmem_ld_32x32b_x32(tmem + lane_off + TM_ST + col0, sv);
      tmem_ld_32x32b_x32(tmem + lane_off + TM_DPT + col0, dv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(st_free);
      const int lim = key - q0;              // queries q0 + c with c >= lim see this key
      const int pb = g & 1;
      uint8_t* prow = smem + KV_OFF_P + pb * PT_BYTES + r * 128;
      uint8_t* drw = smem + KV_OFF_DS + pb * PT_BYTES + r * 128;
      uint4 pst[4], dst[4];                  // this warp's 4 chunks of the row
      // the stage's lse / D copies completed with its Q / dO (q_full), before S^T
      if (stat_smem && !mbar_wait_warp(q_full(g % KV_QS), (g / KV_QS) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      const float* sl = reinterpret_cast<const float*>(smem + KV_OFF_STAT + (g % KV_QS) * 512);
      // the causal mask only reaches the steps at the diagonal: the others take the unmasked body
      auto step = [&](auto masked) {
      constexpr bool MASK = decltype(masked)::value;
#pragma unroll
      for (int c8l = 0; c8l < 4; ++c8l) {
        const int c8 = half * 4 + c8l;
        // lse (log2 units, +inf past the sequence end) and D of these 8 queries
        float l8[8], d8[8];
        const int qa = q0 + c8 * 8;
        if (stat_smem && qa + 8 <= p.S) {
          const float4 la = *reinterpret_cast<const float4*>(sl + c8 * 8);
          const float4 lb = *reinterpret_cast<const float4*>(sl + c8 * 8 + 4);
          const float4 da = *reinterpret_cast<const float4*>(sl + 64 + c8 * 8);
          const float4 db = *reinterpret_cast<const float4*>(sl + 64 + c8 * 8 + 4);
          l8[0] = la.x; l8[1] = la.y; l8[2] = la.z; l8[3] = la.w;
          l8[4] = lb.x; l8[5] = lb.y; l8[6] = lb.z; l8[7] = lb.w;
          d8[0] = da.x; d8[1] = da.y; d8[2] = da.z; d8[3] = da.w;
          d8[4] = db.x; d8[5] = db.y; d8[6] = db.z; d8[7] = db.w;
#pragma unroll
          for (int e = 0; e < 8; ++e) l8[e] *= LOG2E_F;
        } else if (vec_stat && qa + 8 <= p.S) {
          const float4 la = *reinterpret_cast<const float4*>(lrow + qa);
          const float4 lb = *reinterpret_cast<const float4*>(lrow + qa + 4);
          const float4 da = *reinterpret_cast<const float4*>(drow + qa);
          const float4 db = *reinterpret_cast<const float4*>(drow + qa + 4);
          l8[0] = la.x; l8[1] = la.y; l8[2] = la.z; l8[3] = la.w;
          l8[4] = lb.x; l8[5] = lb.y; l8[6] = lb.z; l8[7] = lb.w;
          d8[0] = da.x; d8[1] = da.y; d8[2] = da.z; d8[3] = da.w;
          d8[4] = db.x; d8[5] = db.y; d8[6] = db.z; d8[7] = db.w;
#pragma unroll
          for (int e = 0; e < 8; ++e) l8[e] *= LOG2E_F;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool in = qa + e < p.S;
            l8[e] = in ? lrow[qa + e] * LOG2E_F : INFINITY;
            d8[e] = in ? drow[qa + e] : 0.f;
          }
        }
        uint32_t pk[4], dk4[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int c = c8 * 8 + e, cl = c8l * 8 + e;   // step column, column within this warp's half
          float p0 = ex2_approx(fmaf(__uint_as_float(sv[cl]), p.scale_log2, -l8[e]));
          float p1 = ex2_approx(fmaf(__uint_as_float(sv[cl + 1]), p.scale_log2, -l8[e + 1]));
          if (MASK && c < lim) p0 = 0.f;
          if (MASK && c + 1 < lim) p1 = 0.f;
          const float d0 = p0 * (__uint_as_float(dv[cl]) - d8[e]);
          const float d1 = p1 * (__uint_as_float(dv[cl + 1]) - d8[e + 1]);
          pk[e >> 1] = pack_bf16x2(p0, p1);
          dk4[e >> 1] = pack_bf16x2(d0, d1);
        }
        pst[c8l] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[c8l] = make_uint4(dk4[0], dk4[1], dk4[2], dk4[3]);
      }
      };
      if (__any_sync(0xffffffffu, lim > col0)) step(std::true_type{});
      else step(std::false_type{});
      // buffer pb is free once step g - 2's gradient products completed
      if (g >= 2 && !mbar_wait_warp(p_free(pb), ((g >> 1) - 1) & 1, p.err, abort_flag)) { ok = false; break; }
#pragma unroll
      for (int c8l = 0; c8l < 4; ++c8l) {
        const int off = (((half * 4 + c8l) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(prow + off) = pst[c8l];
        *reinterpret_cast<uint4*>(drw + off) = dst[c8l];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(pb));
    }
    fin = ok && mbar_wait_warp(done, 0, p.err, abort_flag);
    if (!fin) *abort_flag = 1;
    if (fin) tc_fence_after();
  }

  // ---------------- dK, dV: written once, as bf16 ----------------
  // Elementwise warp 2 + 4 * half + i: key row r = its TMEM lane; half 0 finishes
  // dV, half 1 dK. The TMEM loads are warp-collective: every lane takes part,
  // only rows inside the sequence store.
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const int key = k0 + r;
  const bool is_k = warp >= 6;
  const uint32_t tmem_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + (is_k ? TM_DK : TM_DV);
  __nv_bfloat16* orow = nullptr;
  const float2* cs = nullptr;
  if (warp >= 2 && key < p.S) {
    orow = (is_k ? p.dk_out : p.dv_out) + (static_cast<int64_t>(row0 + key) * p.Hkv + jh) * HD;
    if (is_k && p.rope_cs) cs = p.rope_cs + static_cast<int64_t>(key) * 64;
  }
  if (nsplit == 1) {
    if (fin) {
      float lo[32], hi[32];
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        tmem_ld_cols<32>(tmem_row + c, lo);
        tmem_ld_cols<32>(tmem_row + 64 + c, hi);
        if (orow) dkdv_store_row<32>(orow, c, lo, hi, is_k, p.scale, cs);
      }
    }
  } else {
    // every CTA of the cluster has finished its MMAs and copies: the Q / dO
    // ring is free to take the partial sums
    cluster_sync_all();
    if (warp >= 2 && fin) {
      if (nsplit == 2) dkdv_send<32>(tmem_row, sb, r, is_k, 2, rank);
      else dkdv_send<16>(tmem_row, sb, r, is_k, 4, rank);
    }
    cluster_sync_all();
    if (warp >= 2 && fin) {
      if (nsplit == 2) dkdv_reduce_store<32>(smem, r, is_k, 2, rank, orow, p.scale, cs);
      else dkdv_reduce_store<16>(smem, r, is_k, 4, rank, orow, p.scale, cs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------
// Q and dO, the A operands of S = Q K^T and dP = dO V^T, are the same for the
// whole CTA and live in tensor memory: the TMA warp stages them in the K / V
// ring's last two stages, the elementwise warps copy each row into tensor
// memory, and those stages then join the ring. dS, the A operand of
// dQ += dS K, also lives in tensor memory: the warp holding keys 32 h .. 32 h +
// 31 of a step writes their bf16 pairs into the first 16 of its own 32 columns
// of the step's S buffer once it has read them (so S of step j + 2 is issued
// only after the dQ product of step j, which reads them). Shared memory holds
// only the K / V ring. Tensor memory: S (2 x 64 columns, dS inside), dP
// (2 x 64), dQ (128), Q and dO (bf16, 64 each).
constexpr int DQ_KS = 6;                                     // stages of the K / V ring
constexpr uint32_t DQ_TM_DQ = 256, DQ_TM_Q = 384, DQ_TM_DO = 448;
constexpr uint32_t DQ_OFF_K = 0;                             // DQ_KS stages of T64
constexpr uint32_t DQ_OFF_V = DQ_OFF_K + DQ_KS * T64;       // DQ_KS stages of T64
constexpr uint32_t DQ_OFF_BAR = DQ_OFF_V + DQ_KS * T64;
constexpr size_t DQ_SMEM = 1024 + DQ_OFF_BAR + 256;
static_assert(DQ_SMEM <= 232448, "dQ shared memory above the per-CTA limit");
static_assert(DQ_KS >= 4, "Q and dO are staged in the ring's last two stages");
// staging of Q / dO (128 rows x 128 columns each, two 64-column swizzle blocks of
// 16 KB): ring stages DQ_KS - 2 and DQ_KS - 1 (a stage is 2 x T64 = 32 KB)
constexpr uint32_t DQ_STAGE_Q = DQ_OFF_K + (DQ_KS - 2) * T64;     // K slots of the last two stages
constexpr uint32_t DQ_STAGE_DO = DQ_OFF_V + (DQ_KS - 2) * T64;    // V slots of the last two stages

__global__ void __launch_bounds__(BWD_THREADS, 1) fa_bwd_dq_tc_kernel(const __grid_constant__ BwdParams p) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + DQ_OFF_BAR;
  const uint32_t q_ready = bar;                                      // Q, dO written into TMEM
  auto kv_full = [&](int s) { return bar + 8 + 8 * s; };             // DQ_KS of each ring barrier
  auto kv_free = [&](int s) { return bar + 8 + 8 * DQ_KS + 8 * s; };
  const uint32_t b2 = bar + 8 + 16 * DQ_KS;
  auto sd_full = [&](int s) { return b2 + 8 * s; };                   // 2 of each TMEM / dS barrier
  auto ds_full = [&](int s) { return b2 + 32 + 8 * s; };
  const uint32_t done = b2 + 64;
  const uint32_t q_staged = b2 + 72;                                 // Q, dO copied into the staging
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + DQ_OFF_BAR + 8 + 16 * DQ_KS + 80);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + DQ_OFF_BAR + 8 + 16 * DQ_KS + 84);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (p.S + BQ - 1) / BQ;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.y);   // longest rows first (all heads)
  const int h = blockIdx.x, b = blockIdx.z;
  const int jh = h * p.Hkv / p.Hq;
  const int q0 = qb * BQ;
  const int row0 = b * p.S;
  const int nkb = (min(q0 + BQ, p.S) + 63) / 64;            // 64-key tiles up to the diagonal

  if (threadIdx.x == 0) {
    mbar_init(q_ready, BWD_EW);
    mbar_init(q_staged, 1);
    for (int s = 0; s < DQ_KS; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_free(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sd_full(s), 1);
      mbar_init(ds_full(s), BWD_EW);
    }
    mbar_init(done, 1);
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

  if (warp == 0) {
    // ---------------- TMA (whole warp; the elected lane issues) ----------------
    const bool el = elect_one();
    if (el) {
      mbar_arrive_expect_tx(q_staged, 2 * TILE_BYTES);
      tma_load_2d(sb + DQ_STAGE_Q, &p.tmQ, h * HD, row0 + q0, q_staged);
      tma_load_2d(sb + DQ_STAGE_Q + 16384, &p.tmQ, h * HD + 64, row0 + q0, q_staged);
      tma_load_2d(sb + DQ_STAGE_DO, &p.tmdO, h * HD, row0 + q0, q_staged);
      tma_load_2d(sb + DQ_STAGE_DO + 16384, &p.tmdO, h * HD + 64, row0 + q0, q_staged);
    }
    __syncwarp();
    int issued = 0;
    for (int j = 0; j < nkb; ++j) {
      const int s = j % DQ_KS;
      const uint32_t ph = (j / DQ_KS) & 1;
      // the last two stages hold the Q / dO staging until it is in tensor memory
      if (j == DQ_KS - 2 && !mbar_wait_warp(q_ready, 0, p.err, abort_flag)) { *abort_flag = 1; break; }
      if (!mbar_wait_warp(kv_free(s), ph ^ 1u, p.err, abort_flag)) { *abort_flag = 1; break; }
      const int kr = row0 + j * 64;
      if (el) {
        mbar_arrive_expect_tx(kv_full(s), 2 * T64);
        tma_load_2d(sb + DQ_OFF_K + s * T64, &p.tmK, jh * HD, kr, kv_full(s));
        tma_load_2d(sb + DQ_OFF_K + s * T64 + 8192, &p.tmK, jh * HD + 64, kr, kv_full(s));
        tma_load_2d(sb + DQ_OFF_V + s * T64, &p.tmV, jh * HD, kr, kv_full(s));
        tma_load_2d(sb + DQ_OFF_V + s * T64 + 8192, &p.tmV, jh * HD + 64, kr, kv_full(s));
      }
      __syncwarp();
      ++issued;
    }
    mbar_wait(q_staged, 0, p.err);
    for (int j = (issued > DQ_KS ? issued - DQ_KS : 0); j < issued; ++j)
      mbar_wait(kv_full(j % DQ_KS), (j / DQ_KS) & 1, p.err);
  } else if (warp == 1) {
    // ---------------- MMA (the elected lane issues) ----------------
    // S / dP of step j go out as soon as their TMEM buffer (j & 1) is free and
    // the step's K / V have landed; dQ += dS K of step j as soon as its dS is
    // written (see the dK / dV kernel for why the two streams are not ordered).
    const bool el = elect_one();
    const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
    const uint32_t id_q = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = mbar_wait_warp(q_ready, 0, p.err, abort_flag);
    if (ok) tc_fence_after();
    if (el && ok) {
      int ns = 0, ng = 0;          // next step whose S / dP, whose dQ product, goes out
      uint32_t idle = 0;
      uint64_t since = 0;
      while (ng < nkb) {
        bool prog = false;
        if (ng < ns && mbar_test_wait(ds_full(ng & 1), (ng >> 1) & 1)) {
          tc_fence_after();
          const int sg = ng & 1, ks = ng % DQ_KS;
          // dS from TMEM: keys 16 kk .. 16 kk + 15 in S[sg] columns 32 (kk / 2) + 8 (kk % 2) ..
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ta(tmem + DQ_TM_DQ, tmem + sg * 64 + (kk >> 1) * 32 + (kk & 1) * 8,
                         desc_mn128(sb + DQ_OFF_K + ks * T64, 8192, kk), id_q, (ng > 0 || kk > 0) ? 1u : 0u);
          umma_commit(kv_free(ks));
          ++ng;
          prog = true;
        }
        // S / dP of step ns overwrite the buffers of step ns - 2: after its dQ
        // product (issued in order; its dS was written after S and dP were read)
        if (ns < nkb && ng >= ns - 1 && mbar_test_wait(kv_full(ns % DQ_KS), (ns / DQ_KS) & 1)) {
          tc_fence_after();
          const int ss = ns & 1, ks = ns % DQ_KS;
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16_ta(tmem + ss * 64, tmem + DQ_TM_Q + kk * 8, desc_k128(sb + DQ_OFF_K + ks * T64, 8192, kk),
                         id_s, kk > 0);
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16_ta(tmem + 128 + ss * 64, tmem + DQ_TM_DO + kk * 8,
                         desc_k128(sb + DQ_OFF_V + ks * T64, 8192, kk), id_s, kk > 0);
          umma_commit(sd_full(ss));
          ++ns;
          prog = true;
        }
        if (prog) {
          idle = 0;
          since = 0;
          continue;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        if ((++idle & 1023u) == 0) {
          const uint64_t now = global_timer_ns();
          if (since == 0) {
            since = now;
          } else if (now - since > KL_WAIT_LIMIT_NS) {
            record_error(p.err, KL_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, __ffs(__ballot_sync(0xffffffffu, el)) - 1) != 0;
    if (!ok) *abort_flag = 1;
    if (el) umma_commit(done);
    __syncwarp();
    mbar_wait(done, 0, p.err);
  } else if (warp >= 2) {
    // warp 2 + 4 * half + i: lane quarter (warp & 3), keys 32 * half .. + 31 of a step,
    // and at the end rotary planes 32 * half .. + 31 (with their partners at +64)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int col0 = half * 32;
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    {
      // this query row's head-dim columns 64 * half .. + 63 of Q and dO (the staged
      // 128-byte-swizzled block `half`, zero past the sequence), packed bf16 pairs into
      // TMEM columns DQ_TM_Q / DQ_TM_DO + 32 * half .. + 31
      uint32_t qv[32], ov[32];
      const bool staged = mbar_wait_warp(q_staged, 0, p.err, abort_flag);
      const uint8_t* qs = smem + DQ_STAGE_Q + half * 16384 + r * 128;
      const uint8_t* os = smem + DQ_STAGE_DO + half * 16384 + r * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int off = (e ^ (r & 7)) << 4;
        const uint4 a = *reinterpret_cast<const uint4*>(qs + off), c = *reinterpret_cast<const uint4*>(os + off);
        qv[4 * e] = a.x; qv[4 * e + 1] = a.y; qv[4 * e + 2] = a.z; qv[4 * e + 3] = a.w;
        ov[4 * e] = c.x; ov[4 * e + 1] = c.y; ov[4 * e + 2] = c.z; ov[4 * e + 3] = c.w;
      }
      tmem_st_32x32b_x32(tmem + lane_off + DQ_TM_Q + half * 32, qv);
      tmem_st_32x32b_x32(tmem + lane_off + DQ_TM_DO + half * 32, ov);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
      if (!staged) *abort_flag = 1;
    }
    const int64_t li = (static_cast<int64_t>(b) * p.Hq + h) * p.S + qrow;
    const float l2 = qrow < p.S ? p.lse[li] * LOG2E_F : INFINITY;
    const float Dq = qrow < p.S ? p.Dd[li] : 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(sd_full(s), ph, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[32], dv[32];
      tmem_ld_32x32b_x32(tmem + lane_off + s * 64 + col0, sv);
      tmem_ld_32x32b_x32(tmem + lane_off + 128 + s * 64 + col0, dv);
      tmem_ld_wait();
      const int lim = qrow - j * 64;          // keys j*64 + c with c <= lim are kept
      uint32_t pk[16];                        // dS of this warp's 32 keys, bf16 pairs
      auto step = [&](auto masked) {
      constexpr bool MASK = decltype(masked)::value;
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int c = col0 + e;               // step column
        float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), p.scale_log2, -l2));
        float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), p.scale_log2, -l2));
        if (MASK && c > lim) p0 = 0.f;
        if (MASK && c + 1 > lim) p1 = 0.f;
        pk[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dv[e]) - Dq), p1 * (__uint_as_float(dv[e + 1]) - Dq));
      }
      };
      // keys j*64 + c with c > lim are masked: only the steps at the diagonal have any
      if (__any_sync(0xffffffffu, lim < col0 + 31)) step(std::true_type{});
      else step(std::false_type{});
      tmem_st_32x32b_x16(tmem + lane_off + s * 64 + col0, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full(s));
    }
    // the query's rotary cos/sin of this warp's planes are fetched before the wait for the last MMA
    const float2* cs = p.rope_cs ? p.rope_cs + static_cast<int64_t>(qrow < p.S ? qrow : 0) * 64 : nullptr;
    float4 csc[16];
    if (cs) {
#pragma unroll
      for (int e = 0; e < 16; ++e) csc[e] = reinterpret_cast<const float4*>(cs)[16 * half + e];
    }
    const bool fin = ok && mbar_wait_warp(done, 0, p.err, abort_flag);
    if (fin && p.dq_out) {
      // bf16 dQ, turned back by the rotary angle of the query's position when a table is given
      tc_fence_after();
      __nv_bfloat16* orow = p.dq_out + (static_cast<int64_t>(row0 + qrow) * p.Hq + h) * HD;
      {
        const int c = half;
        uint32_t va[32], vb[32];   // planes 32c .. 32c+31 and their partners at +64
        tmem_ld_32x32b_x32(tmem + lane_off + DQ_TM_DQ + c * 32, va);
        tmem_ld_32x32b_x32(tmem + lane_off + DQ_TM_DQ + 64 + c * 32, vb);
        tmem_ld_wait();
        if (qrow < p.S) {
          float xa[32], xb[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(va[e]) * p.scale, y = __uint_as_float(vb[e]) * p.scale;
            if (cs) {
              const float4 q4 = csc[e >> 1];
              const float tc = (e & 1) ? q4.z : q4.x, ts = (e & 1) ? q4.w : q4.y;
              xa[e] = x * tc + y * ts;
              xb[e] = y * tc - x * ts;
            } else {
              xa[e] = x;
              xb[e] = y;
            }
          }
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 wa, wb;
            wa.x = pack_bf16x2(xa[e], xa[e + 1]); wa.y = pack_bf16x2(xa[e + 2], xa[e + 3]);
            wa.z = pack_bf16x2(xa[e + 4], xa[e + 5]); wa.w = pack_bf16x2(xa[e + 6], xa[e + 7]);
            wb.x = pack_bf16x2(xb[e], xb[e + 1]); wb.y = pack_bf16x2(xb[e + 2], xb[e + 3]);
            wb.z = pack_bf16x2(xb[e + 4], xb[e + 5]); wb.w = pack_bf16x2(xb[e + 6], xb[e + 7]);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = wa;
            *reinterpret_cast<uint4*>(orow + 64 + c * 32 + e) = wb;
          }
        }
      }
    } else if (fin) {
      // fp32 accumulator
      tc_fence_after();
      float* orow = p.dq_acc + (static_cast<int64_t>(row0 + qrow) * p.Hq + h) * HD;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = half * 2 + cc;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_off + DQ_TM_DQ + c * 32, v);
        tmem_ld_wait();
        if (qrow < p.S) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + c * 32 + e) =
                make_float4(__uint_as_float(v[e]) * p.scale, __uint_as_float(v[e + 1]) * p.scale,
                            __uint_as_float(v[e + 2]) * p.scale, __uint_as_float(v[e + 3]) * p.scale);
        }
      }
    } else {
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// [rows, cols] bf16 row-major, box 64 columns x box_rows rows, 128-byte swizzle.
kl_status map_rows(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows = 128) {
  auto fn = tensor_map_encoder();
  if (!fn) return set_error(KL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
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
    KL_CUDA(cudaFuncSetAttribute(fa_fwd_tc_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_BYTES)));
    attr_done |= uint64_t(1) << dev;
  }
  p.B = B;
  p.items = B * Hq * ((S + BQ - 1) / BQ);
  // Short sequences: the persistent kernel, one CTA per SM through all items,
  // so an item's start and end overlap its neighbours' (at 2048 tokens an item
  // is ~8 key tiles; 0.098 -> 0.089 ms). Long ones: one CTA per item, the
  // hardware handing out the next as each finishes (there the persistent
  // kernel's steps measured ~4 % slower than this one's).
  const int nqb = (S + BQ - 1) / BQ;
  if (nqb <= 32 && p.items > num_sms())
    launch_pdl(fa_fwd_tc_persist_kernel, num_sms(), THREADS, SMEM_BYTES, st, p);
  else
    launch_pdl(fa_fwd_tc_kernel, dim3(Hq, nqb, B), THREADS, SMEM_BYTES, st, p);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl

namespace kl {

int attention_dkdv_split(int B, int S, int Hq, int Hkv, int sms) {
  // Causal work per (head, key tile kb): ceil((S - 128 kb) / 64) query steps.
  // Split a kv head's query-head group over 2 or 4 CTAs of a cluster until the
  // longest key tile's share is at most 1.2x the mean work per SM (measured at
  // 2048 tokens, 64 / 8 heads: 0.309 ms unsplit, 0.179 ms in pairs, 0.233 ms
  // in fours); long sequences stay unsplit.
  const int G = Hq / Hkv;
  const int nkb = (S + BKV - 1) / BKV;
  double total = 0.0;
  for (int kb = 0; kb < nkb; ++kb) total += (S - kb * BKV + 63) / 64;
  total *= static_cast<double>(B) * Hq;
  const double per_sm = total / (sms > 0 ? sms : 1);
  const int nit0 = (S + 63) / 64;
  int best = 1;
  for (int n = 1; n <= 4; n *= 2) {
    if (G % n) continue;
    best = n;
    if (static_cast<double>(G / n) * nit0 <= 1.2 * per_sm) break;
  }
  return best;
}

// A second stream per device, with a fork and a join event (created on first
// use, kept until exit): the dK / dV and dQ kernels read the same inputs and
// write different outputs, so at long sequences dK / dV runs on it beside dQ
// on the caller's stream, and the SMs that one kernel's uneven causal tail
// leaves idle take the other's CTAs (32768 tokens: 56.3 -> 54.9 ms per
// attention fwd+bwd; at 2048 tokens, 256 dK / dV CTAs, no gain, so one after
// the other there). The caller's stream waits for both before it goes on.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
kl_status side_stream(SideStream** out) {
  static std::mutex mu;
  static SideStream side[64];
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(KL_ERR_UNSUPPORTED, "attention_bwd: device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  SideStream& d = side[dev];
  if (!d.s) {
    KL_CUDA(cudaStreamCreateWithFlags(&d.s, cudaStreamNonBlocking));
    KL_CUDA(cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming));
    KL_CUDA(cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming));
  }
  *out = &d;
  return KL_OK;
}

kl_status attention_bwd_tc(int B, int S, int Hq, int Hkv, const void* q, const void* k, const void* v,
                           const void* dout, const float* lse, const float* Dd, float* dq_acc, void* dq_out,
                           void* dk_out, void* dv_out, const float2* rope_cs, cudaStream_t st) {
  if (!dk_out || !dv_out || (!dq_out && !dq_acc))
    return set_error(KL_ERR_INVALID_ARG, "attention_bwd: null output");
  if (((reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) & 15u) != 0)
    return set_error(KL_ERR_INVALID_ARG, "attention_bwd: dk / dv not 16-byte aligned");
  const uint64_t T = static_cast<uint64_t>(B) * S;
  static uint64_t attr_done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(fa_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(KV_SMEM)));
    KL_CUDA(cudaFuncSetAttribute(fa_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(DQ_SMEM)));
    attr_done |= uint64_t(1) << dev;
  }
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.Dd = Dd;
  p.dq_acc = dq_acc;
  p.dq_out = static_cast<__nv_bfloat16*>(dq_out);
  p.dk_out = static_cast<__nv_bfloat16*>(dk_out);
  p.dv_out = static_cast<__nv_bfloat16*>(dv_out);
  p.rope_cs = rope_cs;
  p.kg = static_cast<const __nv_bfloat16*>(k);
  p.vg = static_cast<const __nv_bfloat16*>(v);
  p.S = S;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.nsplit = attention_dkdv_split(B, S, Hq, Hkv, num_sms());
  // tuning override: KL_ATTN_DKDV_SPLIT = 1, 2 or 4 (a divisor of the query-head group)
  if (const char* e = getenv("KL_ATTN_DKDV_SPLIT")) {
    const int v = atoi(e);
    if ((v == 1 || v == 2 || v == 4) && (Hq / Hkv) % v == 0) p.nsplit = v;
  }
  p.scale_log2 = LOG2E_F / sqrtf(static_cast<float>(HD));
  p.scale = 1.0f / sqrtf(static_cast<float>(HD));
  p.err = device_error_word();
  const double pairs = 0.5 * static_cast<double>(S) * (S + 1);
  // dQ: Q and dO tiles of 128 rows (staged, then moved into TMEM), K and V tiles of 64 rows
  BwdParams pq = p;
  KL_TRY(map_rows(&pq.tmQ, q, static_cast<uint64_t>(Hq) * HD, T, 128));
  KL_TRY(map_rows(&pq.tmdO, dout, static_cast<uint64_t>(Hq) * HD, T, 128));
  KL_TRY(map_rows(&pq.tmK, k, static_cast<uint64_t>(Hkv) * HD, T, 64));
  KL_TRY(map_rows(&pq.tmV, v, static_cast<uint64_t>(Hkv) * HD, T, 64));
  // dK / dV: Q and dO tiles of 64 rows (K and V rows are read into TMEM by the kernel)
  KL_TRY(map_rows(&p.tmQ, q, static_cast<uint64_t>(Hq) * HD, T, 64));
  KL_TRY(map_rows(&p.tmdO, dout, static_cast<uint64_t>(Hq) * HD, T, 64));
  const dim3 kv_grid(Hkv * p.nsplit, (S + BKV - 1) / BKV, B);
  const bool overlap =
      static_cast<uint64_t>(kv_grid.x) * kv_grid.y * kv_grid.z >= 4ull * num_sms() && !profiling_on();
  SideStream* side = nullptr;
  cudaStream_t kv_st = st;
  if (overlap) {
    KL_TRY(side_stream(&side));
    // from here on both kernels are launched and the caller's stream joins the side stream
    KL_CUDA(cudaEventRecord(side->fork, st));
    KL_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    kv_st = side->s;
  }
  cudaError_t e_kv, e_q;
  {
    ProfScope ps("attn_bwd_dkdv_tc", kv_st, 8.0 * B * Hq * HD * pairs, 0.0);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_enter
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.nsplit);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = kv_grid;
    cfg.blockDim = dim3(BWD_THREADS);
    cfg.dynamicSmemBytes = KV_SMEM;                                    // alignment checked in-kernel
    cfg.stream = kv_st;
    cfg.attrs = attr;
    cfg.numAttrs = p.nsplit > 1 ? 2 : 1;
    e_kv = cudaLaunchKernelEx(&cfg, fa_bwd_dkdv_tc_kernel, p);
  }
  {
    // only the dQ product is algorithmic work here; S and dP are recomputed
    ProfScope ps("attn_bwd_dq_tc", st, 2.0 * B * Hq * HD * pairs, 0.0);
    dim3 grid(Hq, (S + BQ - 1) / BQ, B);
    e_q = launch_pdl(fa_bwd_dq_tc_kernel, grid, BWD_THREADS, DQ_SMEM, st, pq);
  }
  const cudaError_t e_r = overlap ? cudaEventRecord(side->join, side->s) : cudaSuccess;
  const cudaError_t e_w = overlap ? cudaStreamWaitEvent(st, side->join, 0) : cudaSuccess;
  KL_CUDA(e_kv);
  KL_CUDA(e_q);
  KL_CUDA(e_r);
  KL_CUDA(e_w);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
