// Matrix products of the layer ("From-scratch GPU LLM training", capability
// list: the matrix-multiply gradient kernel): every projection forward
// (y = x W^T), its input gradient (dx = dy W) and its weight gradient
// (dW = dy^T x), and the lm-head products.
//
// bf16 path: one persistent, warp-specialised tcgen05 kernel on CTA pairs
// (cta_group::2, 256 x 256 output tiles; the pair form is described above the
// kernel). Per k-block of 64 each CTA stages a 128 x 64 half of A and of B with
// 128-byte swizzle in a 6-stage mbarrier ring; tcgen05.mma M=256 N=256 K=16
// accumulates in TMEM (two 256-column fp32 accumulators per CTA, so one tile's
// epilogue overlaps the next tile's main loop); four epilogue warps read their
// TMEM lane quarter (tcgen05.ld 32x32b.x32), add the optional residual,
// convert and store. Work units (whole output tiles, each summed over its
// whole K range in one order; when the last round would leave pairs idle, its
// tiles split along K into per-range fp32 slices that gemm_tail_finalize_kernel
// sums in range order) are handed out by a global atomic counter, heaviest
// problems first.
// Operands may be K-major or MN-major (the transpose bits of the instruction
// descriptor), so dX and dW need no transposed copies. Up to four problems
// share one launch (for example the q/k/v projections, or a dX and a dW
// product), and one problem may accumulate up to three (A, B) segments (the
// input gradient of the fused q/k/v projection).
//
// fp32 path: a plain shared-memory tiled FFMA kernel (no TF32).
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int BN = 256;                    // output tile columns
constexpr int BK = 64;                     // k-block: one 128-byte swizzle atom of bf16
constexpr uint32_t TMEM_COLS = 2 * BN;     // two fp32 accumulators
constexpr int SCHED_Q = 8;                 // depth of the unit-id ring

struct GemmProb {
  int M, N;
  int nseg;
  int kb[GEMM_MAX_SEG];   // k-blocks of each (A, B) segment
  int kb_total;
  int a_mn, b_mn;
  int a3d, b3d;           // MN-major operand staged by one 3-D copy (both 64-wide atoms)
  int m_tiles, n_tiles;
  int n_fast;             // tile order: n fastest (1) or m fastest (0)
  int unit_begin;         // first global work-unit index of this problem
  int tmap_base;
  void* C;
  int64_t ldc;
  int c_f32;
  int vec_ok;
  const void* R;
  int64_t ldr;
  int r_f32;
  int epi;                // GEMM_EPI_*
  int n_step;             // output columns per tile: 256, or 128 for GEMM_EPI_SWIGLU
  int nmaps;              // tensor-map slots used (segments, or 2 B maps for GEMM_EPI_SWIGLU)
  void* C2;
  void* C3;
  const void* X1;
  const void* X2;
  float* dot_out;
  int dot_S;
  const float2* rope_cs;  // GEMM_EPI_ROPE: [rope_S][64] cos/sin
  int rope_S;
  int tma_c;              // outputs leave through shared memory and TMA stores (maps tmC[problem][0..2])
  int whole_tiles;        // tiles computed whole; the rest (tail) are split along K
  int tail_tiles, tail_splits;
  float* tail_acc;        // [tail_splits][tail_tiles][256][256] fp32, one slice per K range
};

struct GemmParams {
  CUtensorMap tmA[GEMM_MAX_PROB * GEMM_MAX_SEG];
  CUtensorMap tmB[GEMM_MAX_PROB * GEMM_MAX_SEG];
  CUtensorMap tmC[GEMM_MAX_PROB][3];   // output maps (C, C2, C3) of the problems with tma_c (box 32 x 32)
  GemmProb prob[GEMM_MAX_PROB];
  int nprob;
  int total_units;
  unsigned int* sched;    // [0] next unit to hand out, [1] CTAs finished
  uint32_t* err;
};

// A work unit: one K-range of one output tile of one problem.
struct Unit {
  int p;
  int m0, n0;
  int kb_lo, kb_hi;
  int tail;               // scratch slice of a split last-round tile (split * tail_tiles + tile), or -1
};


__device__ __forceinline__ void store_chunk(const GemmProb& pr, int row, int col0,
                                            const uint32_t (&v)[32]) {
  float f[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
  const int ncols = min(32, pr.N - col0);
  const bool vec = pr.vec_ok && ncols == 32;
  if (pr.R) {
    if (pr.r_f32) {
      const float* r = static_cast<const float*>(pr.R) + row * pr.ldr + col0;
      if (vec) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 a = *reinterpret_cast<const float4*>(r + j);
          f[j] += a.x; f[j + 1] += a.y; f[j + 2] += a.z; f[j + 3] += a.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncols) f[j] += r[j];
      }
    } else {
      const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(pr.R) + row * pr.ldr + col0;
      if (vec) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 a = *reinterpret_cast<const uint4*>(r + j);
          float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y), x2 = unpack_bf16x2(a.z),
                 x3 = unpack_bf16x2(a.w);
          f[j] += x0.x; f[j + 1] += x0.y; f[j + 2] += x1.x; f[j + 3] += x1.y;
          f[j + 4] += x2.x; f[j + 5] += x2.y; f[j + 6] += x3.x; f[j + 7] += x3.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncols) f[j] += __bfloat162float(r[j]);
      }
    }
  }
  if (pr.c_f32) {
    float* c = static_cast<float*>(pr.C) + row * pr.ldc + col0;
    if (vec) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(c + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncols) c[j] = f[j];
    }
  } else {
    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(pr.C) + row * pr.ldc + col0;
    if (vec) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 o;
        o.x = pack_bf16x2(f[j], f[j + 1]);
        o.y = pack_bf16x2(f[j + 2], f[j + 3]);
        o.z = pack_bf16x2(f[j + 4], f[j + 5]);
        o.w = pack_bf16x2(f[j + 6], f[j + 7]);
        *reinterpret_cast<uint4*>(c + j) = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncols) c[j] = __float2bfloat16_rn(f[j]);
    }
  }
}

// f += the addend R's 32 columns col0.. of `row` (bf16 or fp32).
__device__ __forceinline__ void add_residual(const GemmProb& pr, int row, int col0, float (&f)[32]) {
  const int ncols = min(32, pr.N - col0);
  const bool vec = pr.vec_ok && ncols == 32;
  if (pr.r_f32) {
    const float* r = static_cast<const float*>(pr.R) + row * pr.ldr + col0;
    if (vec) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 a = *reinterpret_cast<const float4*>(r + j);
        f[j] += a.x; f[j + 1] += a.y; f[j + 2] += a.z; f[j + 3] += a.w;
      }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncols) f[j] += r[j];
    }
  } else {
    const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(pr.R) + row * pr.ldr + col0;
    if (vec) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(r + j);
        const float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y), x2 = unpack_bf16x2(a.z),
                     x3 = unpack_bf16x2(a.w);
        f[j] += x0.x; f[j + 1] += x0.y; f[j + 2] += x1.x; f[j + 3] += x1.y;
        f[j + 4] += x2.x; f[j + 5] += x2.y; f[j + 6] += x3.x; f[j + 7] += x3.y;
      }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncols) f[j] += __bfloat162float(r[j]);
    }
  }
}

// sigmoid(g) = 1 / (1 + e^-g) = 1 / (1 + 2^(-g log2 e)) from the two hardware
// approximations (ex2.approx, rcp.approx: a few ulp, far below the bf16 the
// SwiGLU epilogues store; g -> -inf gives 2^+inf = inf and 1/inf = 0). The
// IEEE expf and division took ~45 instructions per element and slowed the
// down projection's backward (SwiGLU backward epilogue) by ~7 %.
__device__ __forceinline__ float sigmoid_f(float g) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, bool vec, int ncols, float (&f)[32]) {
  if (vec) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(p + j);
      const float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y), x2 = unpack_bf16x2(a.z),
                   x3 = unpack_bf16x2(a.w);
      f[j] = x0.x; f[j + 1] = x0.y; f[j + 2] = x1.x; f[j + 3] = x1.y;
      f[j + 4] = x2.x; f[j + 5] = x2.y; f[j + 6] = x3.x; f[j + 7] = x3.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = j < ncols ? __bfloat162float(p[j]) : 0.f;
  }
}
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, bool vec, int ncols, const float (&f)[32]) {
  if (vec) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      uint4 o;
      o.x = pack_bf16x2(f[j], f[j + 1]);
      o.y = pack_bf16x2(f[j + 2], f[j + 3]);
      o.z = pack_bf16x2(f[j + 4], f[j + 5]);
      o.w = pack_bf16x2(f[j + 6], f[j + 7]);
      *reinterpret_cast<uint4*>(p + j) = o;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < ncols) p[j] = __float2bfloat16_rn(f[j]);
  }
}

// GEMM_EPI_SWIGLU: 32 columns of g and of u (fp32 accumulators) -> g, u, m.
__device__ __forceinline__ void store_swiglu(const GemmProb& pr, int row, int col0, const uint32_t (&vg)[32],
                                             const uint32_t (&vu)[32]) {
  const int ncols = min(32, pr.N - col0);
  const bool vec = pr.vec_ok && ncols == 32;
  const int64_t o = static_cast<int64_t>(row) * pr.ldc + col0;
  float g[32], u[32], m[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    g[j] = __uint_as_float(vg[j]);
    u[j] = __uint_as_float(vu[j]);
    m[j] = g[j] * sigmoid_f(g[j]) * u[j];
  }
  store_bf16x32(static_cast<__nv_bfloat16*>(pr.C) + o, vec, ncols, g);
  store_bf16x32(static_cast<__nv_bfloat16*>(pr.C2) + o, vec, ncols, u);
  store_bf16x32(static_cast<__nv_bfloat16*>(pr.C3) + o, vec, ncols, m);
}

// GEMM_EPI_SWIGLU_BWD: the saved g, u of one 32-column chunk, as raw bf16
// (loaded a chunk ahead so the epilogue does not wait on HBM for each chunk).
struct GluRaw {
  uint4 g[4], u[4];
};
__device__ __forceinline__ void glu_load(const GemmProb& pr, int row, int col0, GluRaw& r) {
  const int ncols = min(32, pr.N - col0);
  if (row >= pr.M || ncols <= 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) r.g[j] = r.u[j] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int64_t o = static_cast<int64_t>(row) * pr.ldc + col0;
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(pr.X1) + o;
  const __nv_bfloat16* u = static_cast<const __nv_bfloat16*>(pr.X2) + o;
  if (pr.vec_ok && ncols == 32) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r.g[j] = *reinterpret_cast<const uint4*>(g + 8 * j);
      r.u[j] = *reinterpret_cast<const uint4*>(u + 8 * j);
    }
  } else {
    __nv_bfloat16 tg[32], tu[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      tg[j] = j < ncols ? g[j] : __float2bfloat16_rn(0.f);
      tu[j] = j < ncols ? u[j] : __float2bfloat16_rn(0.f);
    }
    memcpy(r.g, tg, sizeof(tg));
    memcpy(r.u, tu, sizeof(tu));
  }
}
// 32 columns of dm (fp32) with the saved g, u -> dg = dm u s (1 + g (1 - s)), du = dm g s (into g, u).
__device__ __forceinline__ void swiglu_bwd_math(const uint32_t (&v)[32], const GluRaw& r, float (&g)[32],
                                                float (&u)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t gw[4] = {r.g[j].x, r.g[j].y, r.g[j].z, r.g[j].w};
    const uint32_t uw[4] = {r.u[j].x, r.u[j].y, r.u[j].z, r.u[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 gf = unpack_bf16x2(gw[e]), uf = unpack_bf16x2(uw[e]);
      g[8 * j + 2 * e] = gf.x;
      g[8 * j + 2 * e + 1] = gf.y;
      u[8 * j + 2 * e] = uf.x;
      u[8 * j + 2 * e + 1] = uf.y;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float dm = __uint_as_float(v[j]);
    const float sg = sigmoid_f(g[j]);
    const float dg = dm * u[j] * sg * (1.0f + g[j] * (1.0f - sg));
    u[j] = dm * g[j] * sg;   // du
    g[j] = dg;
  }
}
__device__ __forceinline__ void store_swiglu_bwd(const GemmProb& pr, int row, int col0, const uint32_t (&v)[32],
                                                 const GluRaw& r) {
  const int ncols = min(32, pr.N - col0);
  const bool vec = pr.vec_ok && ncols == 32;
  const int64_t o = static_cast<int64_t>(row) * pr.ldc + col0;
  float g[32], u[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t gw[4] = {r.g[j].x, r.g[j].y, r.g[j].z, r.g[j].w};
    const uint32_t uw[4] = {r.u[j].x, r.u[j].y, r.u[j].z, r.u[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 gf = unpack_bf16x2(gw[e]), uf = unpack_bf16x2(uw[e]);
      g[8 * j + 2 * e] = gf.x;
      g[8 * j + 2 * e + 1] = gf.y;
      u[8 * j + 2 * e] = uf.x;
      u[8 * j + 2 * e + 1] = uf.y;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float dm = __uint_as_float(v[j]);
    const float sg = sigmoid_f(g[j]);
    const float dg = dm * u[j] * sg * (1.0f + g[j] * (1.0f - sg));
    u[j] = dm * g[j] * sg;   // du
    g[j] = dg;
  }
  store_bf16x32(static_cast<__nv_bfloat16*>(pr.C) + o, vec, ncols, g);
  store_bf16x32(static_cast<__nv_bfloat16*>(pr.C2) + o, vec, ncols, u);
}

// GEMM_EPI_ROPE: planes 0..31 of a 32-column chunk (va) and their partners 64
// columns on (vb), turned by the angles cs[0..31] of the row's position.
__device__ __forceinline__ void store_rope(const GemmProb& pr, int row, int colA, const uint32_t (&va)[32],
                                           const uint32_t (&vb)[32], const float2* cs) {
  float xa[32], xb[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float2 t = cs[j];
    const float x = __uint_as_float(va[j]), y = __uint_as_float(vb[j]);
    xa[j] = x * t.x - y * t.y;
    xb[j] = x * t.y + y * t.x;
  }
  __nv_bfloat16* c = static_cast<__nv_bfloat16*>(pr.C) + static_cast<int64_t>(row) * pr.ldc + colA;
  store_bf16x32(c, pr.vec_ok, 32, xa);
  store_bf16x32(c + 64, pr.vec_ok, 32, xb);
}

// GEMM_EPI_ROWDOT: sum over 32 columns of bf16(product) * X1.
__device__ __forceinline__ float chunk_rowdot(const GemmProb& pr, int row, int col0, const uint32_t (&v)[32]) {
  const int ncols = min(32, pr.N - col0);
  const bool vec = pr.vec_ok && ncols == 32;
  float x[32];
  load_bf16x32(static_cast<const __nv_bfloat16*>(pr.X1) + static_cast<int64_t>(row) * pr.ldc + col0, vec, ncols, x);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    a0 = fmaf(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[j]))), x[j], a0);
    a1 = fmaf(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[j + 1]))), x[j + 1], a1);
    a2 = fmaf(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[j + 2]))), x[j + 2], a2);
    a3 = fmaf(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[j + 3]))), x[j + 3], a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// ---------------------------------------------------------------------------
// Pair form (cta_group::2): a cluster of two CTAs computes 256 x 256 tiles.
//   Per k-block each CTA stages its 128-row half of A (16 KB) and its 128-row
//   half of B (16 KB); 6 stages. The leader (rank 0) issues tcgen05.mma
//   M=256 N=256, which reads both CTAs' halves and leaves rows 0..127 of the
//   tile in the leader's TMEM and rows 128..255 in the follower's.
//   leader    warp 0: scheduler (unit ids to both CTAs through DSMEM) + A copies
//   follower  warp 0: A copies, completing on the leader's barrier
//   both      warp 6: B copies (two producer threads: one thread issuing every
//                     tensor copy of a stage serialises them)
//   leader    warp 1: TMEM (both CTAs allocate together) + MMA issue
//   both      warps 2..5: epilogue of their own 128 rows
// The issuing roles run as whole warps; one elected lane issues.
// ---------------------------------------------------------------------------
// k-blocks (of BK) per pipeline stage, and stages in the ring
#ifndef KL_GEMM_KPS
#define KL_GEMM_KPS 1
#endif
#ifndef KL_GEMM_PAIR_STAGES
#define KL_GEMM_PAIR_STAGES (6 / KL_GEMM_KPS)
#endif
constexpr int KPS = KL_GEMM_KPS;
constexpr int STAGES2 = KL_GEMM_PAIR_STAGES;
// A and B tiles are issued by two producer threads in different warps (warp 0
// and warp 6): one thread issuing every tensor copy of a stage serialises them.
#ifndef KL_GEMM_SPLIT_PRODUCER
#define KL_GEMM_SPLIT_PRODUCER 1
#endif
constexpr bool SPLIT_PRODUCER = KL_GEMM_SPLIT_PRODUCER != 0;
constexpr int PAIR_THREADS = SPLIT_PRODUCER ? 224 : 192;
constexpr uint32_t HALF_BYTES = 128 * BK * 2;            // 16 KB
constexpr uint32_t KB2_BYTES = 2 * HALF_BYTES;           // one k-block: A half + B half
constexpr uint32_t STAGE2_BYTES = KPS * KB2_BYTES;
// Output staging of the plain-store epilogue: per epilogue warp two buffers of
// 32 rows x 32 columns (4 KB for fp32), filled in the TMA store's swizzled
// layout (64-byte swizzle for bf16 rows of 64 bytes, 128-byte for fp32 rows).
constexpr uint32_t STG_BUF = 32 * 32 * 4;
constexpr uint32_t STG_BYTES = 4 * 2 * STG_BUF;
constexpr uint32_t BAR_BYTES = 1024;   // barriers and scheduler slots; keeps the staging 1024-aligned
constexpr size_t SMEM2_BYTES = 1024 + STAGES2 * STAGE2_BYTES + BAR_BYTES + STG_BYTES;
static_assert(SMEM2_BYTES <= 232448, "pair-kernel shared memory above the per-CTA limit");

// Stages this warp's 32 x 32 output chunk f (row = lane) in its next staging
// slot (two per warp at wbase) and TMA-stores it through `map` at {col0,
// wrow0}, as fp32 or bf16. A slot is rewritten only after the store two
// chunks back has finished reading it.
__device__ __forceinline__ void stage_store(uint32_t wbase, uint32_t& n, int lane, const CUtensorMap* map, bool f32,
                                            int col0, int wrow0, const float (&f)[32]) {
  const uint32_t buf = wbase + (n & 1u) * STG_BUF;
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
  if (f32) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), __float_as_uint(f[4 * j]), __float_as_uint(f[4 * j + 1]),
                   __float_as_uint(f[4 * j + 2]), __float_as_uint(f[4 * j + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_v4(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pack_bf16x2(f[8 * j], f[8 * j + 1]),
                   pack_bf16x2(f[8 * j + 2], f[8 * j + 3]), pack_bf16x2(f[8 * j + 4], f[8 * j + 5]),
                   pack_bf16x2(f[8 * j + 6], f[8 * j + 7]));
  }
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, col0, wrow0, buf);
    bulk_commit_group();
  }
  ++n;
}

__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals may come from other CTAs).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait_cl(bar, parity)) {
    if ((++n & 255u) == 0 && global_timer_ns() - t0 > KL_WAIT_LIMIT_NS) {
      record_error(err, KL_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_cl_warp(uint32_t bar, uint32_t parity, uint32_t* err,
                                                  volatile int* abort_flag) {
  const bool ok = !*abort_flag && mbar_wait_cl(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}
// Ring-stage wait (full / empty barriers, one use per k-block): first one
// CTA-scope try_wait by every lane, which is the common case and keeps the
// stage hand-off short; only if that fails the bounded, abort-aware loop.
// (+4 % on K = 5120 products, +12 % on K = 2048 ones, measured alone.)
__device__ __forceinline__ bool stage_wait_warp(uint32_t bar, uint32_t parity, uint32_t* err,
                                                volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return mbar_wait_cl_warp(bar, parity, err, abort_flag);
}
// Tile load into this CTA's shared memory, completing on the pair leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                 uint32_t leader_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(leader_bar)
      : "memory");
}
// Both 64-wide atoms of an MN-major half in one copy: 3-D map [MN/64][K][64],
// box {64, 64, 2}, lands exactly as two 2-D {64, 64} copies 8 KB apart.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                                 uint32_t leader_bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(leader_bar)
      : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` when this thread's MMAs complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Unit decode for 256 x 256 tiles.
__device__ __forceinline__ Unit decode_unit_cl(const GemmParams& P, int u) {
  int p = 0;
  while (p + 1 < P.nprob && u >= P.prob[p + 1].unit_begin) ++p;
  const GemmProb& pr = P.prob[p];
  const int local = u - pr.unit_begin;
  // last-round K splits are the slowest index: the units in flight share one
  // K range, so the operand slices they stream stay resident in L2
  int si, tile, nsplit;
  Unit r;
  r.p = p;
  r.tail = -1;
  if (pr.tail_splits > 1 && local >= pr.whole_tiles) {
    // last-round tiles, split along K (split-major as well)
    const int t = local - pr.whole_tiles;
    si = t / pr.tail_tiles;
    r.tail = t;
    tile = pr.whole_tiles + (t - si * pr.tail_tiles);
    nsplit = pr.tail_splits;
  } else {
    si = 0;
    tile = local;
    nsplit = 1;
  }
  if (pr.n_fast) {
    r.n0 = (tile % pr.n_tiles) * pr.n_step;
    r.m0 = (tile / pr.n_tiles) * 256;
  } else {
    r.m0 = (tile % pr.m_tiles) * 256;
    r.n0 = (tile / pr.m_tiles) * pr.n_step;
  }
  r.kb_lo = static_cast<int>(static_cast<int64_t>(si) * pr.kb_total / nsplit);
  r.kb_hi = static_cast<int>(static_cast<int64_t>(si + 1) * pr.kb_total / nsplit);
  return r;
}

__global__ void __launch_bounds__(PAIR_THREADS, 1) gemm_bf16_tcp_kernel(const __grid_constant__ GemmParams p) {
  pdl_enter();
  constexpr int CL = 2;                                        // CTAs per cluster
  // consumers of each unit id: epilogue warps, producers (all but the
  // scheduler's own, plus the B producers), the MMA issuer
  constexpr int QEMPTY_COUNT = 4 * CL + (CL - 1) + (SPLIT_PRODUCER ? CL : 0) + 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES2 * STAGE2_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES2 + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES2 + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES2 + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES2 + 4);
  auto qfull_bar = [&](int q) { return bar0 + 8u * (2 * STAGES2 + 5 + q); };
  auto qempty_bar = [&](int q) { return bar0 + 8u * (2 * STAGES2 + 5 + SCHED_Q + q); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES2 + 5 + 2 * SCHED_Q);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* qids = reinterpret_cast<volatile int*>(tmem_holder + 2);
  const uint32_t stg_base = sbase + STAGES2 * STAGE2_BYTES + BAR_BYTES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank;                                  // 0: leader, 1: follower
  const bool pair_leader = peer == 0;
  const uint16_t pair_mask = 3u;                               // both CTAs of the pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);    // the MMA commit (multicast to both CTAs)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);   // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(drain_bar, 1);
    for (int q = 0; q < SCHED_Q; ++q) {
      mbar_init(qfull_bar(q), 1);
      mbar_init(qempty_bar(q), QEMPTY_COUNT);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // every CTA's barriers exist before any CTA signals another
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t sched_qempty0 = mapa_rank(qempty_bar(0), 0);
  const uint32_t lead_tempty0 = mapa_rank(tempty_bar(0), 0);
  const uint32_t lead_full0 = mapa_rank(full_bar(0), 0);

  const bool b_producer = SPLIT_PRODUCER && warp == 6;
  if (warp == 0 || b_producer) {
    const bool el = elect_one();
    // ---------------- scheduler (rank 0) + TMA (every CTA) ----------------
    // warp 0: scheduler on rank 0, A tiles (and B tiles unless split);
    // warp 6: B tiles when split.
    if (el)
      for (int i = 0; i < p.nprob; ++i)
        for (int s = 0; s < p.prob[i].nmaps; ++s) {
          tma_prefetch_desc(&p.tmA[p.prob[i].tmap_base + s]);
          tma_prefetch_desc(&p.tmB[p.prob[i].tmap_base + s]);
        }
    int stage = 0;
    uint32_t phase = 0;
    int q = 0;
    uint32_t qphase = 0;
    long issued = 0;
    bool ok = true;
    while (ok) {
      int u = 0;
      if (rank == 0 && !b_producer) {
        if (el) {
          u = static_cast<int>(atomicAdd(&p.sched[0], 1u));
          if (u >= p.total_units) u = -1;
        }
        u = __shfl_sync(0xffffffffu, u, 0);
        if (!mbar_wait_cl_warp(qempty_bar(q), qphase ^ 1u, p.err, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        if (el) {
          qids[q] = u;
          mbar_arrive(qfull_bar(q));
#pragma unroll
          for (int r = 1; r < CL; ++r) {
            const uint32_t rq = mapa_rank(smem_u32(const_cast<int*>(qids)), r) + 4u * q;
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(rq), "r"(u) : "memory");
            mbar_arrive_cluster(mapa_rank(qfull_bar(q), r));
          }
        }
        __syncwarp();
      } else {
        if (!mbar_wait_cl_warp(qfull_bar(q), qphase, p.err, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        u = qids[q];
        __syncwarp();
        if (el) mbar_arrive_cluster(sched_qempty0 + 8u * q);
      }
      if (++q == SCHED_Q) {
        q = 0;
        qphase ^= 1u;
      }
      if (u < 0) break;
      const Unit un = decode_unit_cl(p, u);
      const GemmProb& pr = p.prob[un.p];
      const int mh = un.m0 + 128 * static_cast<int>(peer);   // this CTA's rows of A
      // this CTA's rows of B: its half of the tile's 256 columns, or (SwiGLU) the
      // tile's 128 columns of the gate (leader) or up (follower) weights
      const bool glu = pr.epi == GEMM_EPI_SWIGLU;
      const int nh = glu ? un.n0 : un.n0 + 128 * static_cast<int>(peer);
      int s = 0, off = 0;
      while (un.kb_lo >= off + pr.kb[s]) off += pr.kb[s++];
      int kl = un.kb_lo - off;
      for (int kbg = un.kb_lo; kbg < un.kb_hi; kbg += KPS) {
        const int nk = un.kb_hi - kbg < KPS ? un.kb_hi - kbg : KPS;
        if (!stage_wait_warp(empty_bar(stage), phase ^ 1u, p.err, abort_flag)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        const uint32_t fb = lead_full0 + 8u * stage;
        if (pair_leader && !b_producer && el)
          mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(nk) * 2 * KB2_BYTES);
        for (int j = 0; j < nk; ++j, ++kl) {
          if (kl == pr.kb[s]) {
            ++s;
            kl = 0;
          }
          const CUtensorMap* ta = &p.tmA[pr.tmap_base + s];
          const CUtensorMap* tb = &p.tmB[pr.tmap_base + (glu ? static_cast<int>(peer) : s)];
          const uint32_t sa = sbase + stage * STAGE2_BYTES + j * KB2_BYTES;
          const uint32_t sb = sa + HALF_BYTES;
          const int k0 = kl * BK;
          if (!el) {
            // only the elected lane issues
          } else if (!b_producer) {
            if (!pr.a_mn) {
              tma_load_2d_pair(sa, ta, k0, mh, fb);
            } else if (pr.a3d) {
              tma_load_3d_pair(sa, ta, 0, k0, mh >> 6, fb);
            } else {
              tma_load_2d_pair(sa, ta, mh, k0, fb);
              tma_load_2d_pair(sa + 8192, ta, mh + 64, k0, fb);
            }
          }
          if (!el || (SPLIT_PRODUCER && !b_producer)) {
            // B is issued by warp 6 (by its elected lane)
          } else if (!pr.b_mn) {
            tma_load_2d_pair(sb, tb, k0, nh, fb);
          } else if (pr.b3d) {
            tma_load_3d_pair(sb, tb, 0, k0, nh >> 6, fb);
          } else {
            tma_load_2d_pair(sb, tb, nh, k0, fb);
            tma_load_2d_pair(sb + 8192, tb, nh + 64, k0, fb);
          }
        }
        ++issued;
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (pair_leader && !b_producer) {
      // the leader's full barriers see every copy into its pair: wait for the last ones
      const long outstanding = issued < STAGES2 ? issued : STAGES2;
      for (long i = 0; i < outstanding; ++i) {
        if (stage == 0) {
          stage = STAGES2 - 1;
          phase ^= 1u;
        } else {
          --stage;
        }
        mbar_wait_cl(full_bar(stage), phase, p.err);
      }
    }
  } else if (warp == 1 && pair_leader) {
    // ---------------- MMA issuer (pair leaders; one elected lane issues) ----------------
    const bool el = elect_one();
    int stage = 0;
    uint32_t phase = 0;
    int q = 0;
    uint32_t qphase = 0;
    int it = 0;
    bool ok = true;
    while (ok) {
      if (!mbar_wait_cl_warp(qfull_bar(q), qphase, p.err, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      const int u = qids[q];
      __syncwarp();
      if (el) mbar_arrive_cluster(sched_qempty0 + 8u * q);
      if (++q == SCHED_Q) {
        q = 0;
        qphase ^= 1u;
      }
      if (u < 0) break;
      const Unit un = decode_unit_cl(p, u);
      const GemmProb& pr = p.prob[un.p];
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait_cl_warp(tempty_bar(acc), (use & 1u) ^ 1u, p.err, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
      const uint32_t idesc = idesc_bf16_f32(256, 256, pr.a_mn, pr.b_mn);
      uint32_t accumulate = 0;
      for (int kbg = un.kb_lo; kbg < un.kb_hi; kbg += KPS) {
        const int nk = un.kb_hi - kbg < KPS ? un.kb_hi - kbg : KPS;
        if (!stage_wait_warp(full_bar(stage), phase, p.err, abort_flag)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        if (el) {
        for (int j = 0; j < nk; ++j) {
          const uint32_t sa = sbase + stage * STAGE2_BYTES + j * KB2_BYTES;
          const uint32_t sb = sa + HALF_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = pr.a_mn ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                        : smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bd = pr.b_mn ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                                        : smem_desc_sw128(sb + k * 32, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
            accumulate = 1;
          }
        }
        umma_commit_pair(empty_bar(stage), pair_mask);
        }
        __syncwarp();
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && el) umma_commit_pair(tfull_bar(acc), pair_mask);
      __syncwarp();
      ++it;
    }
    if (el) umma_commit_pair_local(drain_bar);
    __syncwarp();
    mbar_wait(drain_bar, 0, p.err);
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue (every CTA, its own 128 rows) ----------------
    const int quarter = warp & 3;
    int q = 0;
    uint32_t qphase = 0;
    int it = 0;
    uint32_t stg_n = 0;   // chunks this warp has staged (slot = stg_n & 1)
    const uint32_t wstg = stg_base + static_cast<uint32_t>(quarter) * 2 * STG_BUF;
    while (true) {
      if (!mbar_wait_cl_warp(qfull_bar(q), qphase, p.err, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      const int u = qids[q];
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(sched_qempty0 + 8u * q);
      if (++q == SCHED_Q) {
        q = 0;
        qphase ^= 1u;
      }
      if (u < 0) break;
      const Unit un = decode_unit_cl(p, u);
      const GemmProb& pr = p.prob[un.p];
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      const int row = un.m0 + 128 * static_cast<int>(peer) + quarter * 32 + lane;
      GluRaw glu_next;
      if (pr.epi == GEMM_EPI_SWIGLU_BWD) glu_load(pr, row, un.n0, glu_next);   // overlaps the wait below
      if (!mbar_wait_cl_warp(tfull_bar(acc), use & 1u, p.err, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * 256);
      // outputs through staged TMA stores (rows and columns past the output are clipped);
      // a follower half wholly below the output stores nothing
      const bool staged = pr.tma_c && un.tail < 0;
      const int wrow0 = un.m0 + 128 * static_cast<int>(peer) + quarter * 32;   // this warp's first row
      const bool live = wrow0 < pr.M;
      const CUtensorMap* tmc = p.tmC[un.p];
      if (pr.epi == GEMM_EPI_SWIGLU) {
        // columns 0..127 of the accumulator are g, 128..255 are u, of the same 128 outputs
        for (int c = 0; c < 4; ++c) {
          const int col0 = un.n0 + c * 32;
          if (col0 >= pr.N) break;
          uint32_t vg[32], vu[32];
          tmem_ld_32x32b_x32(tacc + c * 32, vg);
          tmem_ld_32x32b_x32(tacc + 128 + c * 32, vu);
          tmem_ld_wait();
          if (staged) {
            if (live) {
              float g[32], u[32], m[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                g[j] = __uint_as_float(vg[j]);
                u[j] = __uint_as_float(vu[j]);
                m[j] = g[j] * sigmoid_f(g[j]) * u[j];
              }
              stage_store(wstg, stg_n, lane, &tmc[0], false, col0, wrow0, g);
              stage_store(wstg, stg_n, lane, &tmc[1], false, col0, wrow0, u);
              stage_store(wstg, stg_n, lane, &tmc[2], false, col0, wrow0, m);
            }
          } else if (row < pr.M) {
            store_swiglu(pr, row, col0, vg, vu);
          }
        }
      } else if (pr.epi == GEMM_EPI_ROPE) {
        // two heads of 128 columns; plane i pairs column i with i + 64 of its head
        const float2* cs = pr.rope_cs + static_cast<int64_t>((row < pr.M ? row : 0) % pr.rope_S) * 64;
        for (int hl = 0; hl < 2; ++hl) {
          for (int c = 0; c < 2; ++c) {
            const int colA = un.n0 + 128 * hl + 32 * c;
            if (colA >= pr.N) break;
            uint32_t va[32], vb[32];
            tmem_ld_32x32b_x32(tacc + 128 * hl + 32 * c, va);
            tmem_ld_32x32b_x32(tacc + 128 * hl + 64 + 32 * c, vb);
            tmem_ld_wait();
            if (staged) {
              if (live) {
                float xa[32], xb[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float2 t = cs[32 * c + j];
                  const float x = __uint_as_float(va[j]), y = __uint_as_float(vb[j]);
                  xa[j] = x * t.x - y * t.y;
                  xb[j] = x * t.y + y * t.x;
                }
                stage_store(wstg, stg_n, lane, &tmc[0], false, colA, wrow0, xa);
                stage_store(wstg, stg_n, lane, &tmc[0], false, colA + 64, wrow0, xb);
              }
            } else if (row < pr.M) {
              store_rope(pr, row, colA, va, vb, cs + 32 * c);
            }
          }
        }
      } else {
        float dot = 0.f;
        for (int c = 0; c < 256 / 32; ++c) {
          const int col0 = un.n0 + c * 32;
          if (col0 >= pr.N) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_ld_wait();
          if (pr.epi == GEMM_EPI_SWIGLU_BWD) {
            const GluRaw cur = glu_next;
            if (c + 1 < 256 / 32) glu_load(pr, row, col0 + 32, glu_next);   // next chunk in flight
            if (staged) {
              if (live) {
                float dg[32], du[32];
                swiglu_bwd_math(v, cur, dg, du);
                stage_store(wstg, stg_n, lane, &tmc[0], false, col0, wrow0, dg);
                stage_store(wstg, stg_n, lane, &tmc[1], false, col0, wrow0, du);
              }
            } else if (row < pr.M) {
              store_swiglu_bwd(pr, row, col0, v, cur);
            }
          } else if (un.tail >= 0) {
            if (row < pr.M) {
              // a K range of a last-round tile: its own fp32 scratch slice (summed in a fixed order later)
              float4* a = reinterpret_cast<float4*>(pr.tail_acc + (static_cast<int64_t>(un.tail) * 256 + (row - un.m0)) *
                                                                      256 + (col0 - un.n0));
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                a[j / 4] = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                       __uint_as_float(v[j + 3]));
            }
          } else if (staged) {
            if (live) {
              float f[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
              if (pr.R && row < pr.M) add_residual(pr, row, col0, f);
              stage_store(wstg, stg_n, lane, &tmc[0], pr.c_f32 != 0, col0, wrow0, f);
            }
          } else if (row < pr.M) {
            store_chunk(pr, row, col0, v);
          }
          if (pr.epi == GEMM_EPI_ROWDOT && un.tail < 0) {
            if (row < pr.M) dot += chunk_rowdot(pr, row, col0, v);
            if ((c & 3) == 3) {   // the 128 columns of one head are done
              if (row < pr.M) {
                const int heads = pr.N >> 7, h = (col0 - 96) >> 7;
                const int b = row / pr.dot_S, t = row - b * pr.dot_S;
                pr.dot_out[(static_cast<int64_t>(b) * heads + h) * pr.dot_S + t] = dot;
              }
              dot = 0.f;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_tempty0 + 8u * acc);
      ++it;
    }
    if (lane == 0) bulk_wait_all();   // every TMA store of this warp has written its tile
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // no CTA leaves while another may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
  }
  if (threadIdx.x == 0 && rank == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&p.sched[1], 1u);
    if (prev == gridDim.x / CL - 1) {
      atomicExch(&p.sched[0], 0u);
      atomicExch(&p.sched[1], 0u);
      __threadfence();
    }
  }
}

// Finishes the split last-round tiles of one problem: C = (sum of the K-range
// slices, in split order) + R, converted. Deterministic: no atomics anywhere.
struct TailFin {
  int M, N, m_tiles, n_tiles, n_fast, whole, tiles, splits;
  const float* acc;
  void* C;
  int64_t ldc;
  int c_f32;
  const void* R;
  int64_t ldr;
  int r_f32;
};
__global__ void __launch_bounds__(256) gemm_tail_finalize_kernel(const TailFin f) {
  pdl_enter();
  const int t = blockIdx.x;                      // tail tile
  const int tile = f.whole + t;
  int m0, n0;
  if (f.n_fast) {
    n0 = (tile % f.n_tiles) * 256;
    m0 = (tile / f.n_tiles) * 256;
  } else {
    m0 = (tile % f.m_tiles) * 256;
    n0 = (tile / f.m_tiles) * 256;
  }
  const int r = blockIdx.y * 4 + (threadIdx.x >> 6);  // 4 rows per block, 64 threads x 4 columns per row
  const int c = (threadIdx.x & 63) * 4;
  const int row = m0 + r;
  if (row >= f.M) return;
  float4 a = *reinterpret_cast<const float4*>(f.acc + (static_cast<int64_t>(t) * 256 + r) * 256 + c);
  for (int sp = 1; sp < f.splits; ++sp) {
    const float4 b =
        *reinterpret_cast<const float4*>(f.acc + (static_cast<int64_t>(sp * f.tiles + t) * 256 + r) * 256 + c);
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
  }
  const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int col = n0 + c + e;
    if (col >= f.N) break;
    float v = av[e];
    if (f.R) v += f.r_f32 ? static_cast<const float*>(f.R)[row * f.ldr + col]
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(f.R)[row * f.ldr + col]);
    if (f.c_f32) static_cast<float*>(f.C)[row * f.ldc + col] = v;
    else static_cast<__nv_bfloat16*>(f.C)[row * f.ldc + col] = __float2bfloat16_rn(v);
  }
}

// ---------------------------------------------------------------------------
// host: tensor maps
// ---------------------------------------------------------------------------
// 2-D bf16 map: inner extent `inner` (contiguous), `outer` rows with row
// stride ld elements, box 64 x box_outer, 128-byte swizzle, zero fill.
kl_status make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, int64_t ld,
                   uint32_t box_outer) {
  auto fn = tensor_map_encoder();
  if (!fn) return set_error(KL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(KL_ERR_INVALID_ARG, "tensor map encode failed (%d): inner %llu outer %llu ld %lld",
                     static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
                     (long long)ld);
  return KL_OK;
}

// Output map of the plain-store epilogue: [M, N] with row stride ldc elements
// (bf16 or fp32), box 32 columns x 32 rows, the staging buffers' swizzle
// (64-byte for bf16 rows of 64 bytes, 128-byte for fp32 rows of 128 bytes).
bool make_map_c(CUtensorMap* m, void* ptr, int M, int N, int64_t ldc, bool f32) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * es};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major bf16 operand as a 3-D map: dims {64, K, MN/64} with strides
// {ld, 64} elements, box {64, 64, 2}, 128-byte swizzle. Needs MN % 64 == 0
// (every element addressed lies inside the MN x K operand); returns false if
// the encoder refuses the map (the caller then uses 2-D maps).
bool make_map_mn3(CUtensorMap* m, const void* ptr, uint64_t mn, uint64_t k, int64_t ld) {
  auto fn = tensor_map_encoder();
  if (!fn || mn % 64 != 0) return false;
  cuuint64_t dims[3] = {64, k, mn / 64};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// fp32 CUDA-core GEMM
// ---------------------------------------------------------------------------
constexpr int FT = 64;   // tile edge
constexpr int FK = 16;   // k step

__global__ void __launch_bounds__(256) gemm_f32_kernel(int M, int N, int nseg, GemmSpec spec) {
  pdl_enter();
  __shared__ float As[FK][FT + 1];
  __shared__ float Bs[FK][FT + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * FT, n0 = blockIdx.x * FT;
  float acc[4][4] = {};
  for (int s = 0; s < nseg; ++s) {
    const float* A = static_cast<const float*>(spec.A[s]);
    const float* B = static_cast<const float*>(spec.B[s]);
    const int K = spec.K[s];
    const int64_t lda = spec.lda[s], ldb = spec.ldb[s];
    for (int k0 = 0; k0 < K; k0 += FK) {
      for (int i = threadIdx.x; i < FK * FT; i += 256) {
        int kk, mm;
        if (spec.a_mn) { kk = i / FT; mm = i % FT; } else { mm = i / FK; kk = i % FK; }
        const int gm = m0 + mm, gk = k0 + kk;
        float a = 0.f;
        if (gm < M && gk < K) a = spec.a_mn ? A[gk * lda + gm] : A[gm * lda + gk];
        As[kk][mm] = a;
        int nn;
        if (spec.b_mn) { kk = i / FT; nn = i % FT; } else { nn = i / FK; kk = i % FK; }
        const int gn = n0 + nn;
        const int gk2 = k0 + kk;
        float b = 0.f;
        if (gn < N && gk2 < K) b = spec.b_mn ? B[gk2 * ldb + gn] : B[gn * ldb + gk2];
        Bs[kk][nn] = b;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < FK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j];
      if (spec.R) v += static_cast<const float*>(spec.R)[gm * spec.ldr + gn];
      static_cast<float*>(spec.C)[gm * spec.ldc + gn] = v;
    }
  }
}

}  // namespace

// Tile shape: pairs of CTAs (cta_group::2) on 256 x 256 tiles. A unit is one
// whole output tile (the full K range, so every output element is summed in
// one fixed order); only a launch's last round may cut tiles along K, into
// per-range scratch slices summed in range order (gemm_tail_finalize_kernel).
// Long-K problems rely on the heaviest-first order and on the lighter
// problems of the same launch to even out the CTA pairs' shares.
constexpr int GEMM_CL = 2;
constexpr int TILE_M = 256;

// Scheduler counters: one pair per launch slot, reused round-robin; each launch
// re-arms its pair when its last CTA exits.
constexpr int SCHED_SLOTS = 64;
__device__ unsigned int g_gemm_sched[SCHED_SLOTS][2];

unsigned int* sched_slot_ptr() {
  static unsigned int* base[64] = {};
  static std::atomic<unsigned> seq{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!base[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gemm_sched) != cudaSuccess) return nullptr;
    base[dev] = static_cast<unsigned int*>(ptr);
  }
  return base[dev] + 2 * (seq.fetch_add(1) % SCHED_SLOTS);
}

// Clusters of the pair kernel that fit on the device at once (queried once per
// device; the persistent grid is sized to it).
int max_gemm_clusters(int dev, const cudaLaunchConfig_t& cfg_in) {
  static int cached[64] = {};
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = cfg_in;
  cfg.gridDim = dim3(GEMM_CL * (num_sms() / GEMM_CL));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tcp_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = num_sms() / GEMM_CL;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

kl_status gemm_bf16(const GemmSpec* specs_in, int nspec, cudaStream_t st, const char* label) {
  if (nspec < 1 || nspec > GEMM_MAX_PROB) return set_error(KL_ERR_INVALID_ARG, "gemm: %d problems", nspec);
  if (gemm_skinny_fits(specs_in, nspec)) return gemm_skinny(specs_in, nspec, st, label);
  // Heavy units first: order the problems by k-blocks per unit, descending.
  int order[GEMM_MAX_PROB];
  int kbt[GEMM_MAX_PROB];
  for (int i = 0; i < nspec; ++i) {
    const GemmSpec& s = specs_in[i];
    int kb = 0;
    for (int g = 0; g < s.nseg && g < GEMM_MAX_SEG; ++g) kb += (s.K[g] + BK - 1) / BK;
    kbt[i] = kb;
    order[i] = i;
  }
  for (int a = 1; a < nspec; ++a)
    for (int b = a; b > 0 && kbt[order[b]] > kbt[order[b - 1]]; --b) {
      const int t = order[b];
      order[b] = order[b - 1];
      order[b - 1] = t;
    }
  GemmParams p;  // built on the host, passed by value into the launch
  memset(&p, 0, sizeof(p));
  int units = 0, tm = 0;
  double flops = 0.0, bytes = 0.0;
  for (int i = 0; i < nspec; ++i) {
    const int oi = order[i];
    const GemmSpec& s = specs_in[oi];
    if (s.M < 1 || s.N < 1 || s.nseg < 1 || s.nseg > GEMM_MAX_SEG || !s.C)
      return set_error(KL_ERR_INVALID_ARG, "gemm: bad problem %d (M %d N %d nseg %d)", oi, s.M, s.N, s.nseg);
    if (s.c_dtype != KL_BF16 && s.c_dtype != KL_F32)
      return set_error(KL_ERR_INVALID_ARG, "gemm: bad output dtype");
    const bool glu = s.epi == GEMM_EPI_SWIGLU;
    if (s.epi != GEMM_EPI_STORE) {
      const bool pairs_ok = s.epi != GEMM_EPI_SWIGLU || (s.B2 && aligned16(s.B2) && !s.b_mn && s.C2 && s.C3);
      const bool bwd_ok = s.epi != GEMM_EPI_SWIGLU_BWD || (s.X1 && s.X2 && s.C2);
      const bool dot_ok = s.epi != GEMM_EPI_ROWDOT || (s.X1 && s.dot_out && s.dot_S > 0 && s.M % s.dot_S == 0 &&
                                                       s.N % 128 == 0);
      const bool rope_ok = s.epi != GEMM_EPI_ROPE || (s.rope_cs && s.rope_S > 0 && s.N % 128 == 0 &&
                                                      aligned16(s.C) && s.ldc % 8 == 0);
      if (s.epi > GEMM_EPI_ROPE || s.c_dtype != KL_BF16 || s.R || s.nseg != 1 || !pairs_ok ||
          !bwd_ok || !dot_ok || !rope_ok)
        return set_error(KL_ERR_INVALID_ARG, "gemm: problem %d: bad epilogue variant %d", oi, s.epi);
    }
    if (tm + (glu ? 2 : s.nseg) > GEMM_MAX_PROB * GEMM_MAX_SEG)
      return set_error(KL_ERR_INVALID_ARG, "gemm: too many operand maps in one launch");
    GemmProb& pr = p.prob[i];
    pr.M = s.M;
    pr.N = s.N;
    pr.nseg = s.nseg;
    pr.a_mn = s.a_mn;
    pr.b_mn = s.b_mn;
    pr.tmap_base = tm;
    pr.epi = s.epi;
    pr.n_step = glu ? 128 : BN;
    pr.nmaps = glu ? 2 : s.nseg;
    pr.C2 = s.C2;
    pr.C3 = s.C3;
    pr.X1 = s.X1;
    pr.X2 = s.X2;
    pr.dot_out = s.dot_out;
    pr.dot_S = s.dot_S;
    pr.rope_cs = s.rope_cs;
    pr.rope_S = s.rope_S;
    double ksum = 0.0;
    for (int g = 0; g < s.nseg; ++g) {
      if (!s.A[g] || !s.B[g] || s.K[g] < 1)
        return set_error(KL_ERR_INVALID_ARG, "gemm: problem %d segment %d: null operand or K < 1", oi, g);
      if (!aligned16(s.A[g]) || !aligned16(s.B[g]) || (s.lda[g] % 8) || (s.ldb[g] % 8))
        return set_error(KL_ERR_INVALID_ARG,
                         "gemm: bf16 operands need 16-byte aligned bases and row strides that are multiples of 8");
      // A: 128-row boxes in both forms; B: each CTA of a pair stages 128 rows
      if (!s.a_mn) KL_TRY(make_map(&p.tmA[tm + g], s.A[g], s.K[g], s.M, s.lda[g], 128));
      else KL_TRY(make_map(&p.tmA[tm + g], s.A[g], s.M, s.K[g], s.lda[g], 64));
      if (!s.b_mn)
        KL_TRY(make_map(&p.tmB[tm + g], s.B[g], s.K[g], s.N, s.ldb[g], 128));
      else KL_TRY(make_map(&p.tmB[tm + g], s.B[g], s.N, s.K[g], s.ldb[g], 64));
      pr.kb[g] = (s.K[g] + BK - 1) / BK;
      pr.kb_total += pr.kb[g];
      ksum += s.K[g];
    }
    if (glu) {
      // leader stages gate rows, follower up rows, of the same 128 outputs
      if (s.ldb[0] % 8) return set_error(KL_ERR_INVALID_ARG, "gemm: up weights row stride");
      KL_TRY(make_map(&p.tmB[tm + 1], s.B2, s.K[0], s.N, s.ldb[0], 128));
      p.tmA[tm + 1] = p.tmA[tm];
    }
    // MN-major operands: one 3-D copy per half instead of two 2-D copies
    {
      CUtensorMap a3[GEMM_MAX_SEG], b3[GEMM_MAX_SEG];
      bool ok_a = s.a_mn != 0, ok_b = s.b_mn != 0;
      for (int g = 0; g < s.nseg; ++g) {
        if (ok_a) ok_a = make_map_mn3(&a3[g], s.A[g], s.M, s.K[g], s.lda[g]);
        if (ok_b) ok_b = make_map_mn3(&b3[g], s.B[g], s.N, s.K[g], s.ldb[g]);
      }
      for (int g = 0; ok_a && g < s.nseg; ++g) p.tmA[tm + g] = a3[g];
      for (int g = 0; ok_b && g < s.nseg; ++g) p.tmB[tm + g] = b3[g];
      pr.a3d = ok_a;
      pr.b3d = ok_b;
    }
    tm += pr.nmaps;
    pr.m_tiles = (s.M + TILE_M - 1) / TILE_M;
    pr.n_tiles = (s.N + pr.n_step - 1) / pr.n_step;
    // keep the smaller operand resident in L2: walk its dimension fastest
    pr.n_fast = s.N < s.M ? 1 : 0;
    pr.unit_begin = units;
    units += pr.m_tiles * pr.n_tiles;
    pr.C = s.C;
    pr.ldc = s.ldc;
    pr.c_f32 = s.c_dtype == KL_F32;
    pr.R = s.R;
    pr.ldr = s.ldr;
    pr.r_f32 = s.r_dtype == KL_F32;
    // outputs leave through shared memory and TMA stores: C (with any addend added
    // first), and C2, C3 of the SwiGLU variants
    {
      const bool f32 = s.c_dtype == KL_F32;
      const bool two = s.epi == GEMM_EPI_SWIGLU || s.epi == GEMM_EPI_SWIGLU_BWD;
      const bool three = s.epi == GEMM_EPI_SWIGLU;
      bool ok = aligned16(s.C) && (s.ldc * dtype_size(s.c_dtype)) % 16 == 0 &&
                (!two || aligned16(s.C2)) && (!three || aligned16(s.C3)) &&
                make_map_c(&p.tmC[i][0], s.C, s.M, s.N, s.ldc, f32);
      if (ok && two) ok = make_map_c(&p.tmC[i][1], s.C2, s.M, s.N, s.ldc, false);
      if (ok && three) ok = make_map_c(&p.tmC[i][2], s.C3, s.M, s.N, s.ldc, false);
      pr.tma_c = ok ? 1 : 0;
    }
    {
      const size_t ce = dtype_size(s.c_dtype), re = dtype_size(s.r_dtype);
      pr.vec_ok = aligned16(s.C) && (s.ldc * ce) % 16 == 0 &&
                  (!s.R || (aligned16(s.R) && (s.ldr * re) % 16 == 0)) &&
                  (!s.C2 || aligned16(s.C2)) && (!s.C3 || aligned16(s.C3)) && (!s.X1 || aligned16(s.X1)) &&
                  (!s.X2 || aligned16(s.X2));
    }
    const double nmul = glu ? 2.0 : 1.0;   // SwiGLU: a gate and an up product
    const double extra = glu ? 2.0 : s.epi == GEMM_EPI_SWIGLU_BWD ? 3.0 : s.epi == GEMM_EPI_ROWDOT ? 1.0 : 0.0;
    flops += 2.0 * s.M * s.N * nmul * ksum;
    bytes += 2.0 * (s.M + nmul * s.N) * ksum + static_cast<double>(s.M) * s.N * dtype_size(s.c_dtype) * (1.0 + extra) +
             (s.R ? static_cast<double>(s.M) * s.N * dtype_size(s.r_dtype) : 0.0);
  }
  static uint64_t attr_done = 0;  // one bit per device ordinal
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(gemm_bf16_tcp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM2_BYTES)));
    attr_done |= uint64_t(1) << dev;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = GEMM_CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_enter
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(PAIR_THREADS);
  cfg.dynamicSmemBytes = SMEM2_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int cap = max_gemm_clusters(dev, cfg);
  // Last round: if the units leave some CTA pairs idle in the last round (or
  // in the only one: a skinny problem such as a decode step's projections),
  // split the last problem's last tiles along K so that the round's work
  // spreads over every pair (each K range stored to its own slice of tail_ws,
  // the slices summed in split order below).
  int tail_prob = -1;
  {
    const int lp = nspec - 1;
    GemmProb& pr = p.prob[lp];
    const GemmSpec& s = specs_in[order[lp]];
    const int tiles = pr.m_tiles * pr.n_tiles;
    const int rem = units % cap;
    if (rem > 0 && s.tail_ws && pr.epi == GEMM_EPI_STORE && rem <= tiles &&
        pr.n_step == 256 && (reinterpret_cast<uintptr_t>(s.tail_ws) & 15u) == 0) {
      int ts = cap / rem;
      const int max_ts = pr.kb_total / 8;            // at least 8 k-blocks per piece
      if (ts > max_ts) ts = max_ts;
      const size_t need = static_cast<size_t>(ts) * rem * 256 * 256 * 4;   // ts * rem <= cap slices
      if (ts >= 2 && need <= s.tail_ws_bytes) {
        pr.whole_tiles = tiles - rem;
        pr.tail_tiles = rem;
        pr.tail_splits = ts;
        pr.tail_acc = s.tail_ws;
        units += rem * (ts - 1);
        tail_prob = lp;
      }
    }
  }
  p.nprob = nspec;
  p.total_units = units;
  p.sched = sched_slot_ptr();
  if (!p.sched) return set_error(KL_ERR_CUDA, "gemm: scheduler counters unavailable");
  p.err = device_error_word();
  {
    ProfScope ps(label, st, flops, bytes);
    const int clusters = units < cap ? units : cap;
    cfg.gridDim = dim3(GEMM_CL * clusters);
    cfg.numAttrs = 2;   // the occupancy query above used the cluster attribute alone
    KL_CUDA(cudaLaunchKernelEx(&cfg, gemm_bf16_tcp_kernel, p));
  }
  KL_CUDA(cudaGetLastError());
  if (tail_prob >= 0) {
    const GemmProb& pr = p.prob[tail_prob];
    const GemmSpec& s = specs_in[order[tail_prob]];
    TailFin f;
    f.M = pr.M; f.N = pr.N; f.m_tiles = pr.m_tiles; f.n_tiles = pr.n_tiles; f.n_fast = pr.n_fast;
    f.whole = pr.whole_tiles; f.tiles = pr.tail_tiles; f.splits = pr.tail_splits; f.acc = pr.tail_acc;
    f.C = s.C; f.ldc = s.ldc; f.c_f32 = s.c_dtype == KL_F32;
    f.R = s.R; f.ldr = s.ldr; f.r_f32 = s.r_dtype == KL_F32;
    const double n = static_cast<double>(pr.tail_tiles) * 256 * 256;
    ProfScope ps("gemm_tail_finalize", st, 0.0,
                 n * (4.0 * pr.tail_splits + dtype_size(s.c_dtype) + (s.R ? dtype_size(s.r_dtype) : 0)));
    launch_pdl(gemm_tail_finalize_kernel, dim3(pr.tail_tiles, 64), 256, 0, st, f);
    KL_CUDA(cudaGetLastError());
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

size_t gemm_tail_ws_bytes() { return align_up(static_cast<size_t>(num_sms() / GEMM_CL) * 256 * 256 * 4, 256); }

kl_status gemm_f32(const GemmSpec& s, cudaStream_t st, const char* label) {
  if (s.M < 1 || s.N < 1 || s.nseg < 1 || s.nseg > GEMM_MAX_SEG || !s.C)
    return set_error(KL_ERR_INVALID_ARG, "gemm f32: bad problem");
  if (s.c_dtype != KL_F32 || (s.R && s.r_dtype != KL_F32))
    return set_error(KL_ERR_UNSUPPORTED, "gemm f32: output and addend must be fp32");
  for (int g = 0; g < s.nseg; ++g)
    if (!s.A[g] || !s.B[g] || s.K[g] < 1) return set_error(KL_ERR_INVALID_ARG, "gemm f32: bad segment");
  dim3 grid((s.N + FT - 1) / FT, (s.M + FT - 1) / FT);
  double ksum = 0.0;
  for (int g = 0; g < s.nseg; ++g) ksum += s.K[g];
  ProfScope ps(label, st, 2.0 * s.M * s.N * ksum, 4.0 * ((s.M + s.N) * ksum + 1.0 * s.M * s.N));
  launch_pdl(gemm_f32_kernel, grid, 256, 0, st, s.M, s.N, s.nseg, s);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
