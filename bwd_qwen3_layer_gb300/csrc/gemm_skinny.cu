// GEMM for few rows (M <= 128): C[M, N] = A[M, K] B[N, K]^T (+ R), or the
// SwiGLU pair (g = A Bg^T, u = A Bu^T, m = silu(g) u), with both operands
// K-major. The projections of a decode step ("From-scratch GPU LLM training",
// "What is built": the forward path with a paged key-value cache) have M = the
// step's tokens, tens, against weights of 5120 x 25600: the weights are read
// once and nothing else matters, so the work is laid out around them.
//
//   * Operands swapped: the MMA's M is 128 weight rows (a tile), its N the
//     activation rows rounded up to 32. tcgen05.mma cta_group::1, kind::f16,
//     M = 128, N = Mpad, K = 16; fp32 accumulators in TMEM (double-buffered
//     so a tile's epilogue overlaps the next tile's loads).
//   * Work units are (weight tile, 64-wide k-block); the W units, tile-major,
//     are dealt in equal runs of P to one CTA per SM (stream-K), so every SM
//     streams the same bytes whatever N and K are.
//   * Weights that no earlier kernel writes (GemmSpec::b_const) start
//     streaming before the wait for the preceding kernel: the first ring
//     stages' weight tiles are copied, then the wait, then their activations.
//   * A tile held whole by one CTA is written by it. A tile shared by two or
//     more CTAs leaves one fp32 piece per CTA; per 32-row quarter of the
//     tile, the warp that brings its arrival counter to the number of pieces
//     sums them in CTA order (deterministic), finishes and stores the rows,
//     and re-arms the counter.
//
// Roles: warp 0 issues the TMA copies (weights and activations into a
// multi-stage ring), warp 1 the MMAs, warps 2..5 the epilogue (TMEM lane
// quarter = warp % 4). Every wait is bounded (KL_DEVERR_TIMEOUT) and a role
// that gives up raises the shared abort flag; the teardown waits for copies
// and MMAs in flight before TMEM is freed.
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int SK_THREADS = 192;
constexpr int SK_BK = 64;                 // k per unit: one 128-byte swizzle row of bf16
constexpr int SK_BN = 128;                // weight rows per tile
constexpr int SK_MAXP = 4;                // problems per launch
constexpr int SK_MAX_STAGES = 8;
constexpr int SK_SMEM_BUDGET = 200 * 1024;
constexpr int SK_W_BYTES = SK_BN * SK_BK * 2;   // one weight tile of a unit: 16 KB
constexpr int SK_CNT_SLOTS = 16;
constexpr int SK_CNT_TILES = 1024;              // tiles per launch at most

struct SkProb {
  int M, N, K, kb, nt;        // rows, columns, depth, k-blocks, weight tiles
  int unit_begin, tile_begin;
  void* C;
  void* C2;
  void* C3;
  int64_t ldc;
  int c_f32;
  const void* R;
  int64_t ldr;
  int r_f32;
};

struct SkParams {
  CUtensorMap tmA[SK_MAXP];   // activations [M][K], box {64, Mpad}
  CUtensorMap tmB[SK_MAXP];   // weights [N][K], box {64, 128}
  CUtensorMap tmB2[SK_MAXP];  // up weights (SwiGLU)
  SkProb prob[SK_MAXP];
  int nprob, W, P, stages, mpad, glu, stage_bytes;
  int b_early;                // the weights may be copied before the dependency wait
  float* pieces;              // [2 * grid][1 + glu][mpad / 4][128][4] fp32 (16-byte granules, row fastest)
  unsigned int* cnt;          // [tiles][4] arrival counters (zero between launches)
  uint32_t* err;
};

struct SkUnit {
  int p, tile, kbi;
};

__device__ __forceinline__ SkUnit sk_decode(const SkParams& P, int u) {
  int p = 0;
  while (p + 1 < P.nprob && u >= P.prob[p + 1].unit_begin) ++p;
  const int local = u - P.prob[p].unit_begin;
  const int t = local / P.prob[p].kb;
  return {p, t, local - t * P.prob[p].kb};
}

__device__ __forceinline__ float sk_sigmoid(float g) { return 1.0f / (1.0f + expf(-g)); }

// One row n of the output (this thread's weight row) for tokens m0 .. m0+31:
// the finished values, stored (with the residual) or, for SwiGLU, g, u and m.
// The residual's 32 loads are all issued before the first store (the compiler
// must assume C may alias R, so a load after a store would wait for it).
__device__ __forceinline__ void sk_store_final(const SkProb& pr, int glu, int n, int m0, const float (&g)[32],
                                               const float (&u)[32]) {
  if (n >= pr.N) return;
  if (glu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (m0 + j >= pr.M) continue;
      const int64_t o = static_cast<int64_t>(m0 + j) * pr.ldc + n;
      const float mm = g[j] * sk_sigmoid(g[j]) * u[j];
      static_cast<__nv_bfloat16*>(pr.C)[o] = __float2bfloat16_rn(g[j]);
      static_cast<__nv_bfloat16*>(pr.C2)[o] = __float2bfloat16_rn(u[j]);
      static_cast<__nv_bfloat16*>(pr.C3)[o] = __float2bfloat16_rn(mm);
    }
    return;
  }
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = g[j];
  if (pr.R) {
    // unconditional loads (rows past M clamped to a valid row, their sums never
    // stored), one dtype per loop: straight-line code keeps all 32 in flight
    float rv[32];
    if (pr.r_f32) {
      const float* R = static_cast<const float*>(pr.R) + n;
#pragma unroll
      for (int j = 0; j < 32; ++j) rv[j] = R[static_cast<int64_t>(min(m0 + j, pr.M - 1)) * pr.ldr];
    } else {
      const __nv_bfloat16* R = static_cast<const __nv_bfloat16*>(pr.R) + n;
#pragma unroll
      for (int j = 0; j < 32; ++j) rv[j] = __bfloat162float(R[static_cast<int64_t>(min(m0 + j, pr.M - 1)) * pr.ldr]);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += rv[j];
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (m0 + j >= pr.M) continue;
    const int64_t o = static_cast<int64_t>(m0 + j) * pr.ldc + n;
    if (pr.c_f32) static_cast<float*>(pr.C)[o] = v[j];
    else static_cast<__nv_bfloat16*>(pr.C)[o] = __float2bfloat16_rn(v[j]);
  }
}

__global__ void __launch_bounds__(SK_THREADS, 1) gemm_skinny_kernel(const __grid_constant__ SkParams p) {
  // No global access before the dependency wait except the weights' first
  // copies (warp 0 below): no earlier kernel writes them.
  extern __shared__ uint8_t sk_smem[];
  __shared__ __align__(8) uint64_t bars[2 * SK_MAX_STAGES + 5];
  __shared__ uint32_t tmem_holder;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = blockIdx.x * p.P;
  const int u1 = min(p.W, u0 + p.P);
  const int S = p.stages;
  const int nacc = 1 + p.glu;
  const uint32_t cols_needed = 2u * nacc * p.mpad;
  uint32_t tmem_cols = 32;
  while (tmem_cols < cols_needed) tmem_cols <<= 1;
  const uint32_t sbase = (smem_u32(sk_smem) + 1023u) & ~1023u;   // 128-byte swizzle atoms: 1 KB aligned
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[SK_MAX_STAGES + s]); };
  auto afull_bar = [&](int b) { return smem_u32(&bars[2 * SK_MAX_STAGES + b]); };
  auto aempty_bar = [&](int b) { return smem_u32(&bars[2 * SK_MAX_STAGES + 2 + b]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * SK_MAX_STAGES + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull_bar(b), 1);
      mbar_init(aempty_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;

  if (warp == 0) {
    // ---------------- TMA: the unit's weight tile(s) and activation rows ----------------
    const bool el = elect_one();
    if (el)
      for (int i = 0; i < p.nprob; ++i) {
        tma_prefetch_desc(&p.tmA[i]);
        tma_prefetch_desc(&p.tmB[i]);
        if (p.glu) tma_prefetch_desc(&p.tmB2[i]);
      }
    const uint32_t tx = static_cast<uint32_t>(nacc * SK_W_BYTES + p.mpad * SK_BK * 2);
    // the first stages' weights go out before the wait for the preceding kernel
    // (their stages are free: the ring is fresh); their activation rows after it
    const int pre = p.b_early ? min(S, u1 - u0) : 0;
    if (el)
      for (int i = 0; i < pre; ++i) {
        const SkUnit un = sk_decode(p, u0 + i);
        const uint32_t s = sbase + i * p.stage_bytes;
        mbar_arrive_expect_tx(full_bar(i), tx);
        tma_load_2d(s, &p.tmB[un.p], un.kbi * SK_BK, un.tile * SK_BN, full_bar(i));
        if (p.glu) tma_load_2d(s + SK_W_BYTES, &p.tmB2[un.p], un.kbi * SK_BK, un.tile * SK_BN, full_bar(i));
      }
    __syncwarp();
    pdl_wait();
    pdl_launch_dependents();
    if (el)
      for (int i = 0; i < pre; ++i) {
        const SkUnit un = sk_decode(p, u0 + i);
        tma_load_2d(sbase + i * p.stage_bytes + nacc * SK_W_BYTES, &p.tmA[un.p], un.kbi * SK_BK, 0, full_bar(i));
      }
    __syncwarp();
    int stage = pre % S;
    uint32_t phase = pre == S ? 1u : 0u;
    int issued = pre;
    for (int u = u0 + pre; u < u1; ++u) {
      if (!mbar_wait_warp(empty_bar(stage), phase ^ 1u, p.err, &abort_flag)) {
        abort_flag = 1;
        break;
      }
      if (el) {
        const SkUnit un = sk_decode(p, u);
        const uint32_t s = sbase + stage * p.stage_bytes;
        const int k0 = un.kbi * SK_BK, n0 = un.tile * SK_BN;
        mbar_arrive_expect_tx(full_bar(stage), tx);
        tma_load_2d(s, &p.tmB[un.p], k0, n0, full_bar(stage));
        if (p.glu) tma_load_2d(s + SK_W_BYTES, &p.tmB2[un.p], k0, n0, full_bar(stage));
        tma_load_2d(s + nacc * SK_W_BYTES, &p.tmA[un.p], k0, 0, full_bar(stage));
      }
      __syncwarp();
      ++issued;
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // the copies still landing: wait for them before the CTA may leave
    const int outstanding = issued < S ? issued : S;
    for (int i = 0; i < outstanding; ++i) {
      if (stage == 0) {
        stage = S - 1;
        phase ^= 1u;
      } else {
        --stage;
      }
      mbar_wait(full_bar(stage), phase, p.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    const bool el = elect_one();
    const uint32_t idesc = idesc_bf16_f32(SK_BN, p.mpad, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    int seg = -1;
    uint32_t d = 0, accumulate = 0;
    for (int u = u0; u < u1; ++u) {
      const SkUnit un = sk_decode(p, u);
      const int kb = p.prob[un.p].kb;
      if (u == u0 || un.kbi == 0) {   // a segment (this CTA's part of one tile) starts
        ++seg;
        const int b = seg & 1;
        if (!mbar_wait_warp(aempty_bar(b), ((static_cast<uint32_t>(seg) >> 1) & 1u) ^ 1u, p.err, &abort_flag)) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        d = tmem_base + static_cast<uint32_t>(b * nacc * p.mpad);
        accumulate = 0;
      }
      if (!mbar_wait_warp(full_bar(stage), phase, p.err, &abort_flag)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (el) {
        const uint32_t s = sbase + stage * p.stage_bytes;
        const uint32_t sx = s + nacc * SK_W_BYTES;
#pragma unroll
        for (int k = 0; k < SK_BK / 16; ++k)
          umma_bf16(d, smem_desc_sw128(s + 32 * k, 16, 1024), smem_desc_sw128(sx + 32 * k, 16, 1024), idesc,
                    accumulate | static_cast<uint32_t>(k));
        if (p.glu) {
#pragma unroll
          for (int k = 0; k < SK_BK / 16; ++k)
            umma_bf16(d + static_cast<uint32_t>(p.mpad), smem_desc_sw128(s + SK_W_BYTES + 32 * k, 16, 1024),
                      smem_desc_sw128(sx + 32 * k, 16, 1024), idesc, accumulate | static_cast<uint32_t>(k));
        }
        umma_commit(empty_bar(stage));
        if (u + 1 == u1 || un.kbi == kb - 1) umma_commit(afull_bar(seg & 1));
      }
      __syncwarp();
      accumulate = 1;
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (el) umma_commit(drain_bar);   // every MMA issued above has completed once this arrives
    __syncwarp();
    mbar_wait(drain_bar, 0, p.err);
  } else {
    // ---------------- epilogue: warp w owns TMEM lanes (rows) 32 (w % 4) .. +31 ----------------
    pdl_wait();
    const int q = warp & 3;
    const int r = 32 * q + lane;                 // row of the weight tile
    const size_t piece_floats = static_cast<size_t>(nacc) * p.mpad * SK_BN;
    int seg = 0;
    for (int s0 = u0; s0 < u1; ++seg) {
      const SkUnit un = sk_decode(p, s0);
      // a copy in registers: through a reference into the parameters, every
      // global store below would force the fields to be loaded again
      const SkProb pr = p.prob[un.p];
      const int s1 = min(u1, s0 + (pr.kb - un.kbi));
      const int b = seg & 1;
      if (!mbar_wait_warp(afull_bar(b), (static_cast<uint32_t>(seg) >> 1) & 1u, p.err, &abort_flag)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int tfu = pr.unit_begin + un.tile * pr.kb;   // the tile's first unit
      const int first = tfu / p.P, last = (tfu + pr.kb - 1) / p.P;
      const bool whole = first == last;
      const int n = un.tile * SK_BN + r;
      float* piece = p.pieces + (2 * static_cast<size_t>(blockIdx.x) + (s0 == u0 ? 0 : 1)) * piece_floats;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * nacc * p.mpad);
      for (int c = 0; c < p.mpad / 32; ++c) {
        uint32_t vg[32], vu[32];
        tmem_ld_32x32b_x32(tb + 32 * c, vg);
        if (p.glu) tmem_ld_32x32b_x32(tb + p.mpad + 32 * c, vu);
        tmem_ld_wait();
        float g[32], uu[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] = __uint_as_float(vg[j]);
          uu[j] = p.glu ? __uint_as_float(vu[j]) : 0.f;
        }
        if (whole) {
          sk_store_final(pr, p.glu, n, 32 * c, g, uu);
        } else {
          // granule (m / 4, r) holds tokens m .. m+3 of row r: a warp writes 512 contiguous bytes
          float4* pg = reinterpret_cast<float4*>(piece) + static_cast<size_t>(8 * c) * SK_BN + r;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            pg[q4 * SK_BN] = make_float4(g[4 * q4], g[4 * q4 + 1], g[4 * q4 + 2], g[4 * q4 + 3]);
          if (p.glu) {
            float4* pu = pg + static_cast<size_t>(p.mpad / 4) * SK_BN;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              pu[q4 * SK_BN] = make_float4(uu[4 * q4], uu[4 * q4 + 1], uu[4 * q4 + 2], uu[4 * q4 + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty_bar(b));
      if (!whole) {
        // this quarter's piece is out: count it; the last of the tile's CTAs finishes the rows
        __threadfence();
        __syncwarp();
        unsigned int* cnt = p.cnt + (static_cast<size_t>(pr.tile_begin) + un.tile) * 4 + q;
        const unsigned np = static_cast<unsigned>(last - first + 1);
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(cnt, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == np - 1) {
          __threadfence();
          for (int mc = 0; mc < pr.M; mc += 32) {
            float g[32], uu[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = uu[j] = 0.f;
            for (int c = first; c <= last; ++c) {
              // CTA c's piece of this tile: its first segment unless the tile began before c's run.
              // Tokens mc .. mc+31 lie inside the piece (mpad is a multiple of 32; every CTA
              // writes all mpad tokens, those past M as zeros, never stored).
              const int slot = 2 * c + ((c == first && c * p.P != tfu) ? 1 : 0);
              const float4* pc = reinterpret_cast<const float4*>(p.pieces + static_cast<size_t>(slot) * piece_floats) +
                                 static_cast<size_t>(mc / 4) * SK_BN + r;
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const float4 v = __ldcg(pc + q4 * SK_BN);
                g[4 * q4] += v.x;
                g[4 * q4 + 1] += v.y;
                g[4 * q4 + 2] += v.z;
                g[4 * q4 + 3] += v.w;
              }
              if (p.glu) {
                const float4* pu = pc + static_cast<size_t>(p.mpad / 4) * SK_BN;
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  const float4 v = __ldcg(pu + q4 * SK_BN);
                  uu[4 * q4] += v.x;
                  uu[4 * q4 + 1] += v.y;
                  uu[4 * q4 + 2] += v.z;
                  uu[4 * q4 + 3] += v.w;
                }
              }
            }
            sk_store_final(pr, p.glu, n, mc, g, uu);
          }
          __syncwarp();
          if (lane == 0) atomicExch(cnt, 0u);   // re-armed for the next launch that uses this slot
        }
      }
      s0 = s1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// Arrival counters, one slot per launch, reused round-robin; each counter is
// re-armed by the warp that finishes its rows, so a slot is all zeros again
// once its launch has ended. A launch that gave up on a wait can leave counts
// behind; it has also set the sticky timeout bit of the device error word, and
// skinny_cnt_reset() (called when kl_device_status reads that bit) clears every
// slot before the next launch.
__device__ unsigned int g_skinny_cnt[SK_CNT_SLOTS][SK_CNT_TILES * 4];

unsigned int* skinny_cnt_slot() {
  static unsigned int* base[64] = {};
  static std::atomic<unsigned> seq{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!base[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_skinny_cnt) != cudaSuccess) return nullptr;
    base[dev] = static_cast<unsigned int*>(ptr);
  }
  return base[dev] + static_cast<size_t>(seq.fetch_add(1) % SK_CNT_SLOTS) * SK_CNT_TILES * 4;
}

// K-major bf16 operand [rows][K] (row stride ld elements), box {64, box_rows},
// 128-byte swizzle, zero fill outside.
bool sk_map(CUtensorMap* m, const void* ptr, int K, int rows, int64_t ld, int box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {SK_BK, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct SkPlan {
  int mpad, glu, W, P, grid, stages, stage_bytes, tiles;
  size_t piece_bytes;
};

// The launch shape, or false when the problems do not suit this kernel.
bool skinny_plan(const GemmSpec* s, int n, SkPlan* pl) {
  if (n < 1 || n > SK_MAXP) return false;
  const int glu = s[0].epi == GEMM_EPI_SWIGLU;
  int mmax = 0, W = 0, tiles = 0;
  for (int i = 0; i < n; ++i) {
    const GemmSpec& g = s[i];
    if (g.M < 1 || g.M > 128 || g.N < 1 || g.nseg != 1 || g.K[0] < 1 || g.a_mn || g.b_mn) return false;
    if ((g.epi == GEMM_EPI_SWIGLU) != (glu != 0)) return false;
    if (g.epi != GEMM_EPI_STORE && g.epi != GEMM_EPI_SWIGLU) return false;
    if (!g.A[0] || !g.B[0] || !g.C || !al16(g.A[0]) || !al16(g.B[0]) || g.lda[0] % 8 || g.ldb[0] % 8) return false;
    if (g.lda[0] < g.K[0] || g.ldb[0] < g.K[0] || g.ldc < g.N) return false;
    if (glu && (!g.B2 || !al16(g.B2) || !g.C2 || !g.C3 || g.R || g.c_dtype != KL_BF16)) return false;
    if (g.c_dtype != KL_BF16 && g.c_dtype != KL_F32) return false;
    if (g.R && g.ldr < g.N) return false;
    mmax = g.M > mmax ? g.M : mmax;
    const long long units = static_cast<long long>((g.N + SK_BN - 1) / SK_BN) * ((g.K[0] + SK_BK - 1) / SK_BK);
    if (W + units > (1ll << 30)) return false;
    W += static_cast<int>(units);
    tiles += (g.N + SK_BN - 1) / SK_BN;
  }
  if (tiles > SK_CNT_TILES) return false;
  pl->glu = glu;
  pl->mpad = (mmax + 31) / 32 * 32;
  pl->W = W;
  pl->tiles = tiles;
  const int sms = num_sms();
  const int grid0 = W < sms ? W : sms;
  pl->P = (W + grid0 - 1) / grid0;
  pl->grid = (W + pl->P - 1) / pl->P;
  pl->stage_bytes = (1 + glu) * SK_W_BYTES + pl->mpad * SK_BK * 2;
  int st = SK_SMEM_BUDGET / pl->stage_bytes;
  pl->stages = st > SK_MAX_STAGES ? SK_MAX_STAGES : st;
  pl->piece_bytes = static_cast<size_t>(1 + glu) * pl->mpad * SK_BN * 4;
  return pl->stages >= 2;
}

}  // namespace

kl_status skinny_cnt_reset() {
  void* ptr = nullptr;
  KL_CUDA(cudaGetSymbolAddress(&ptr, g_skinny_cnt));
  KL_CUDA(cudaMemset(ptr, 0, sizeof(g_skinny_cnt)));
  return KL_OK;
}

kl_status skinny_cnt_abandon() {
  // one piece counted on every tile of every slot, the tile never finished
  std::vector<unsigned int> ones(sizeof(g_skinny_cnt) / sizeof(unsigned int), 1u);
  KL_CUDA(cudaMemcpyToSymbol(g_skinny_cnt, ones.data(), sizeof(g_skinny_cnt)));
  return KL_OK;
}

bool gemm_skinny_fits(const GemmSpec* specs, int nspec) {
  SkPlan pl;
  if (!skinny_plan(specs, nspec, &pl)) return false;
  const size_t need = 2 * static_cast<size_t>(pl.grid) * pl.piece_bytes;
  return specs[0].tail_ws && al16(specs[0].tail_ws) && specs[0].tail_ws_bytes >= need;
}

kl_status gemm_skinny(const GemmSpec* specs, int nspec, cudaStream_t st, const char* label) {
  SkPlan pl;
  if (!skinny_plan(specs, nspec, &pl)) return set_error(KL_ERR_UNSUPPORTED, "gemm (few rows): unsuitable problems");
  const size_t need = 2 * static_cast<size_t>(pl.grid) * pl.piece_bytes;
  if (!specs[0].tail_ws || specs[0].tail_ws_bytes < need)
    return set_error(KL_ERR_NO_MEMORY, "gemm (few rows): scratch of %zu bytes needed", need);
  SkParams p;
  memset(&p, 0, sizeof(p));
  double flops = 0.0, bytes = 0.0;
  int ub = 0, tb = 0;
  for (int i = 0; i < nspec; ++i) {
    const GemmSpec& g = specs[i];
    SkProb& pr = p.prob[i];
    pr.M = g.M;
    pr.N = g.N;
    pr.K = g.K[0];
    pr.kb = (g.K[0] + SK_BK - 1) / SK_BK;
    pr.nt = (g.N + SK_BN - 1) / SK_BN;
    pr.unit_begin = ub;
    pr.tile_begin = tb;
    ub += pr.kb * pr.nt;
    tb += pr.nt;
    pr.C = g.C;
    pr.C2 = g.C2;
    pr.C3 = g.C3;
    pr.ldc = g.ldc;
    pr.c_f32 = g.c_dtype == KL_F32;
    pr.R = g.R;
    pr.ldr = g.ldr;
    pr.r_f32 = g.r_dtype == KL_F32;
    if (!sk_map(&p.tmA[i], g.A[0], g.K[0], g.M, g.lda[0], pl.mpad) ||
        !sk_map(&p.tmB[i], g.B[0], g.K[0], g.N, g.ldb[0], SK_BN) ||
        (pl.glu && !sk_map(&p.tmB2[i], g.B2, g.K[0], g.N, g.ldb[0], SK_BN)))
      return set_error(KL_ERR_INVALID_ARG, "gemm (few rows): tensor map encode failed (problem %d)", i);
    const double nmul = pl.glu ? 2.0 : 1.0;
    flops += 2.0 * g.M * g.N * nmul * g.K[0];
    bytes += 2.0 * (g.M + nmul * g.N) * g.K[0] +
             static_cast<double>(g.M) * g.N * dtype_size(g.c_dtype) * (pl.glu ? 3.0 : 1.0) +
             (g.R ? static_cast<double>(g.M) * g.N * dtype_size(g.r_dtype) : 0.0);
  }
  p.nprob = nspec;
  p.W = pl.W;
  p.P = pl.P;
  p.stages = pl.stages;
  p.mpad = pl.mpad;
  p.glu = pl.glu;
  p.stage_bytes = pl.stage_bytes;
  p.b_early = 1;
  for (int i = 0; i < nspec; ++i) p.b_early &= specs[i].b_const ? 1 : 0;
  p.pieces = specs[0].tail_ws;
  p.cnt = skinny_cnt_slot();
  p.err = device_error_word();
  if (!p.cnt) return set_error(KL_ERR_CUDA, "gemm (few rows): arrival counters unavailable");
  const size_t smem = static_cast<size_t>(pl.stages) * pl.stage_bytes + 1024;
  static uint64_t attr_done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(gemm_skinny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SK_SMEM_BUDGET + 1024));
    attr_done |= uint64_t(1) << dev;
  }
  {
    ProfScope ps(label, st, flops, bytes);
    KL_CUDA(launch_pdl(gemm_skinny_kernel, pl.grid, SK_THREADS, smem, st, p));
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
