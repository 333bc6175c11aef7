// Causal grouped-query scaled-dot-product attention, forward and backward
// ("From-scratch GPU LLM training", capability list: scaled-dot-product
// attention gradient kernel; "KYNETRA FOUNDRY", tiled-attention paragraph:
// query tiles stream over key/value tiles with a running max and running
// sum, the score matrix never reaches HBM, the backward recomputes the tiles;
// grouped-query paragraph: one key/value head per contiguous query-head group).
//
// bf16 path (d = 128): tiled kernels on the tensor cores (mma.sync m16n8k16,
// fp32 accumulation, softmax statistics in fp32, exp2 with the log2(e)
// factor folded into the scale).
//   forward   CTA = 64 query rows of one head (4 warps x 16 rows), K/V tiles
//             of 64 keys double-buffered with cp.async; saves lse.
//   backward  CTA = 64 keys of one query head; loops over the query tiles at
//             or after the diagonal; recomputes P from lse; dK and dV stay in
//             registers and are added into fp32 accumulators of the shared
//             key/value head; dQ is added tile by tile into an fp32
//             accumulator. D = rowsum(dO * O) is a separate pass.
// fp32 path: one warp per (row, head), plain loops, any head dim <= 256.
#include <math.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ===========================================================================
// fp32 path
// ===========================================================================
__global__ void __launch_bounds__(256) attn_fwd_f32_kernel(int B, int S, int Hq, int Hkv, int d,
                                                           const float* __restrict__ q,
                                                           const float* __restrict__ k,
                                                           const float* __restrict__ v,
                                                           float* __restrict__ o,
                                                           float* __restrict__ lse, float scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (gw >= static_cast<int64_t>(B) * S * Hq) return;
  const int t = static_cast<int>(gw / Hq), h = static_cast<int>(gw % Hq);
  const int b = t / S, s = t % S, j = h * Hkv / Hq;
  const float* qr = q + (static_cast<int64_t>(t) * Hq + h) * d;
  float qv[8], acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    qv[i] = c < d ? qr[c] : 0.f;
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int key = 0; key <= s; ++key) {
    const int64_t kt = static_cast<int64_t>(b) * S + key;
    const float* kr = k + (kt * Hkv + j) * d;
    const float* vr = v + (kt * Hkv + j) * d;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < d) dot = fmaf(qv[i], kr[c], dot);
    }
    dot = warp_sum(dot) * scale;
    const float mn = fmaxf(m, dot);
    const float corr = expf(m - mn), p = expf(dot - mn);
    l = l * corr + p;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < d) acc[i] = acc[i] * corr + p * vr[c];
    }
    m = mn;
  }
  float* orow = o + (static_cast<int64_t>(t) * Hq + h) * d;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    if (c < d) orow[c] = acc[i] / l;
  }
  if (lane == 0) lse[(static_cast<int64_t>(b) * Hq + h) * S + s] = m + logf(l);
}

// dq for one (row, head) per warp; also writes D = rowsum(dO * O).
__global__ void __launch_bounds__(256) attn_bwd_dq_f32_kernel(
    int B, int S, int Hq, int Hkv, int d, const float* __restrict__ q, const float* __restrict__ k,
    const float* __restrict__ v, const float* __restrict__ o, const float* __restrict__ lse,
    const float* __restrict__ dout, float* __restrict__ Dd, float* __restrict__ dq, float scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (gw >= static_cast<int64_t>(B) * S * Hq) return;
  const int t = static_cast<int>(gw / Hq), h = static_cast<int>(gw % Hq);
  const int b = t / S, s = t % S, j = h * Hkv / Hq;
  const int64_t ro = (static_cast<int64_t>(t) * Hq + h) * d;
  float qv[8], dov[8], acc[8];
  float Dv = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    qv[i] = c < d ? q[ro + c] : 0.f;
    dov[i] = c < d ? dout[ro + c] : 0.f;
    if (c < d) Dv = fmaf(dov[i], o[ro + c], Dv);
    acc[i] = 0.f;
  }
  Dv = warp_sum(Dv);
  const int64_t li = (static_cast<int64_t>(b) * Hq + h) * S + s;
  if (lane == 0) Dd[li] = Dv;
  const float L = lse[li];
  for (int key = 0; key <= s; ++key) {
    const int64_t kt = static_cast<int64_t>(b) * S + key;
    const float* kr = k + (kt * Hkv + j) * d;
    const float* vr = v + (kt * Hkv + j) * d;
    float dot = 0.f, dp = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < d) {
        dot = fmaf(qv[i], kr[c], dot);
        dp = fmaf(dov[i], vr[c], dp);
      }
    }
    dot = warp_sum(dot);
    dp = warp_sum(dp);
    const float p = expf(dot * scale - L);
    const float ds = p * (dp - Dv) * scale;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < d) acc[i] = fmaf(ds, kr[c], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    if (c < d) dq[ro + c] = acc[i];
  }
}

// dk, dv for one (key row, kv head) per warp, summed over the query-head group.
__global__ void __launch_bounds__(256) attn_bwd_dkdv_f32_kernel(
    int B, int S, int Hq, int Hkv, int d, const float* __restrict__ q, const float* __restrict__ k,
    const float* __restrict__ v, const float* __restrict__ lse, const float* __restrict__ dout,
    const float* __restrict__ Dd, float* __restrict__ dk, float* __restrict__ dv, float scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (gw >= static_cast<int64_t>(B) * S * Hkv) return;
  const int kt = static_cast<int>(gw / Hkv), j = static_cast<int>(gw % Hkv);
  const int b = kt / S, key = kt % S;
  const int64_t ko = (static_cast<int64_t>(kt) * Hkv + j) * d;
  float kv[8], vv[8], adk[8], adv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    kv[i] = c < d ? k[ko + c] : 0.f;
    vv[i] = c < d ? v[ko + c] : 0.f;
    adk[i] = adv[i] = 0.f;
  }
  const int grp = Hq / Hkv;
  for (int h = j * grp; h < (j + 1) * grp; ++h) {
    for (int s = key; s < S; ++s) {
      const int64_t qt = static_cast<int64_t>(b) * S + s;
      const int64_t ro = (qt * Hq + h) * d;
      float dot = 0.f, dp = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        if (c < d) {
          dot = fmaf(q[ro + c], kv[i], dot);
          dp = fmaf(dout[ro + c], vv[i], dp);
        }
      }
      dot = warp_sum(dot);
      dp = warp_sum(dp);
      const int64_t li = (static_cast<int64_t>(b) * Hq + h) * S + s;
      const float p = expf(dot * scale - lse[li]);
      const float ds = p * (dp - Dd[li]) * scale;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        if (c < d) {
          adv[i] = fmaf(p, dout[ro + c], adv[i]);
          adk[i] = fmaf(ds, q[ro + c], adk[i]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = lane + 32 * i;
    if (c < d) {
      dk[ko + c] = adk[i];
      dv[ko + c] = adv[i];
    }
  }
}

// ===========================================================================
// bf16 tensor-core path (head dim 128)
// ===========================================================================
constexpr int HD = 128;      // head dim
constexpr int TB = 64;       // rows per tile (queries or keys)
constexpr int TILE_BYTES = TB * HD * 2;  // 16 KB, rows of 256 bytes

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                      uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                       uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c (0..15) of row r in a [rows][128] bf16 tile,
// XOR-swizzled so the 8 rows an ldmatrix reads hit 8 different bank groups.
__device__ __forceinline__ uint32_t sw(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 7)) << 4));
}
// Same for a [rows][64] bf16 tile (8 chunks per row).
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Load rows row0 .. row0+63 (valid below `rows`) of a [*, ld] bf16 matrix
// (columns col0 .. col0+127) into a swizzled tile; invalid rows read as 0.
__device__ __forceinline__ void load_tile(uint32_t sdst, const __nv_bfloat16* base, int64_t ld,
                                          int row0, int rows) {
  for (int i = threadIdx.x; i < TB * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const int gr = row0 + r;
    const bool ok = gr < rows;
    const __nv_bfloat16* src = base + static_cast<int64_t>(ok ? gr : 0) * ld + c * 8;
    cp_async16(sdst + sw(r, c), src, ok);
  }
}

__global__ void __launch_bounds__(128) fa_fwd_bf16_kernel(int S, int Hq, int Hkv,
                                                          const __nv_bfloat16* __restrict__ q,
                                                          const __nv_bfloat16* __restrict__ k,
                                                          const __nv_bfloat16* __restrict__ v,
                                                          __nv_bfloat16* __restrict__ o,
                                                          float* __restrict__ lse,
                                                          float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + TILE_BYTES;          // K tiles: sK0 + buf * 2 * TILE_BYTES
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = gridDim.x - 1 - blockIdx.x;     // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int j = h * Hkv / Hq;
  const int q0 = qb * TB;
  const int64_t ldq = static_cast<int64_t>(Hq) * HD, ldk = static_cast<int64_t>(Hkv) * HD;
  const __nv_bfloat16* qbase = q + static_cast<int64_t>(b) * S * ldq + h * HD;
  const __nv_bfloat16* kbase = k + static_cast<int64_t>(b) * S * ldk + j * HD;
  const __nv_bfloat16* vbase = v + static_cast<int64_t>(b) * S * ldk + j * HD;
  auto sK = [&](int buf) { return sK0 + buf * 2 * TILE_BYTES; };
  auto sV = [&](int buf) { return sK0 + buf * 2 * TILE_BYTES + TILE_BYTES; };

  const int kb_end = (min(q0 + TB, S) + TB - 1) / TB;
  load_tile(sQ, qbase, ldq, q0, S);
  load_tile(sK(0), kbase, ldk, 0, S);
  load_tile(sV(0), vbase, ldk, 0, S);
  cp_commit();

  uint32_t qf[8][4];
  float oacc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int row_a = q0 + warp * 16 + (lane >> 2);  // rows held by this thread: row_a, row_a + 8

  for (int kb = 0; kb < kb_end; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < kb_end) {
      load_tile(sK(buf ^ 1), kbase, ldk, (kb + 1) * TB, S);
      load_tile(sV(buf ^ 1), vbase, ldk, (kb + 1) * TB, S);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ldsm4(sQ + sw(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1],
              qf[kk][2], qf[kk][3]);
    }
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm4(sK(buf) + sw(np * 16 + ((lane >> 4) << 3) + (lane & 7), kk * 2 + ((lane >> 3) & 1)),
              b0, b1, b2, b3);
        mma16816(s[2 * np], qf[kk], b0, b1);
        mma16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // scale, causal mask, online softmax (base 2)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb * TB + nt * 8 + 2 * (lane & 3) + (e & 1);
        const int row = row_a + ((e >> 1) << 3);
        float val = s[nt][e] * scale_log2;
        if (key > row || key >= S) val = -INFINITY;
        s[nt][e] = val;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // A row can only be fully masked here if it lies past the sequence end.
    const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = exp2f(m0 - base0), a1 = exp2f(m1 - base1);
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base0);
      s[nt][1] = exp2f(s[nt][1] - base0);
      s[nt][2] = exp2f(s[nt][2] - base1);
      s[nt][3] = exp2f(s[nt][3] - base1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * a0 + rs0;
    l1 = l1 * a1 + rs1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      oacc[nt][0] *= a0;
      oacc[nt][1] *= a0;
      oacc[nt][2] *= a1;
      oacc[nt][3] *= a1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm4t(sV(buf) + sw(kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7), dp * 2 + (lane >> 4)),
               b0, b1, b2, b3);
        mma16816(oacc[2 * dp], pa, b0, b1);
        mma16816(oacc[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int r0 = row_a, r1 = row_a + 8;
  __nv_bfloat16* obase = o + static_cast<int64_t>(b) * S * ldq + h * HD;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int col = nt * 8 + 2 * (lane & 3);
    if (r0 < S)
      *reinterpret_cast<uint32_t*>(obase + r0 * ldq + col) =
          pack_bf16x2(oacc[nt][0] * inv0, oacc[nt][1] * inv0);
    if (r1 < S)
      *reinterpret_cast<uint32_t*>(obase + r1 * ldq + col) =
          pack_bf16x2(oacc[nt][2] * inv1, oacc[nt][3] * inv1);
  }
  if ((lane & 3) == 0) {
    float* lrow = lse + (static_cast<int64_t>(b) * Hq + h) * S;
    if (r0 < S) lrow[r0] = (m0 + log2f(l0)) * LN2;
    if (r1 < S) lrow[r1] = (m1 + log2f(l1)) * LN2;
  }
}

// D[b,h,s] = sum_c dO[t,h,c] * O[t,h,c] (fp32), one warp per (token, head).
__global__ void __launch_bounds__(256) attn_bwd_pre_bf16_kernel(int B, int S, int Hq,
                                                                const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dout,
                                                                float* __restrict__ Dd) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (gw >= static_cast<int64_t>(B) * S * Hq) return;
  const int t = static_cast<int>(gw / Hq), h = static_cast<int>(gw % Hq);
  const int64_t off = (static_cast<int64_t>(t) * Hq + h) * HD + lane * 4;
  const uint2 a = *reinterpret_cast<const uint2*>(o + off);
  const uint2 c = *reinterpret_cast<const uint2*>(dout + off);
  const float2 a0 = unpack_bf16x2(a.x), a1 = unpack_bf16x2(a.y);
  const float2 c0 = unpack_bf16x2(c.x), c1 = unpack_bf16x2(c.y);
  float acc = a0.x * c0.x + a0.y * c0.y + a1.x * c1.x + a1.y * c1.y;
  acc = warp_sum(acc);
  if (lane == 0) Dd[(static_cast<int64_t>(t / S) * Hq + h) * S + t % S] = acc;
}

__device__ __forceinline__ void red_add2(float* p, float a, float b) {
  atomicAdd(p, a);
  atomicAdd(p + 1, b);
}

// Backward, one CTA per (64-key tile, query head, batch).
__global__ void __launch_bounds__(128) fa_bwd_bf16_kernel(
    int S, int Hq, int Hkv, const __nv_bfloat16* __restrict__ q,
    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
    const float* __restrict__ Dd, float* __restrict__ dq_acc, float* __restrict__ dk_acc,
    float* __restrict__ dv_acc, float scale_log2, float scale) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + TILE_BYTES;
  const uint32_t sQ0 = sV + TILE_BYTES;            // per buffer: Q tile then dO tile
  const uint32_t sdS = sQ0 + 4 * TILE_BYTES;       // [64 keys][64 queries] bf16, 8 KB
  float* sStat = reinterpret_cast<float*>(smem + 6 * TILE_BYTES + 8192);  // [2][2][64]: lse2, D
  auto sQ = [&](int buf) { return sQ0 + buf * 2 * TILE_BYTES; };
  auto sdO = [&](int buf) { return sQ0 + buf * 2 * TILE_BYTES + TILE_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x;                       // key tiles near the start see most queries
  const int h = blockIdx.y, b = blockIdx.z;
  const int j = h * Hkv / Hq;
  const int k0 = kb * TB;
  const int64_t ldq = static_cast<int64_t>(Hq) * HD, ldk = static_cast<int64_t>(Hkv) * HD;
  const __nv_bfloat16* qbase = q + static_cast<int64_t>(b) * S * ldq + h * HD;
  const __nv_bfloat16* dobase = dout + static_cast<int64_t>(b) * S * ldq + h * HD;
  const __nv_bfloat16* kbase = k + static_cast<int64_t>(b) * S * ldk + j * HD;
  const __nv_bfloat16* vbase = v + static_cast<int64_t>(b) * S * ldk + j * HD;
  const float* lrow = lse + (static_cast<int64_t>(b) * Hq + h) * S;
  const float* drow = Dd + (static_cast<int64_t>(b) * Hq + h) * S;

  const int nqb = (S + TB - 1) / TB;
  auto load_q_tile = [&](int qb, int buf) {
    load_tile(sQ(buf), qbase, ldq, qb * TB, S);
    load_tile(sdO(buf), dobase, ldq, qb * TB, S);
    for (int i = threadIdx.x; i < TB; i += 128) {
      const int qr = qb * TB + i;
      sStat[buf * 128 + i] = qr < S ? lrow[qr] * LOG2E : 0.f;
      sStat[buf * 128 + 64 + i] = qr < S ? drow[qr] : 0.f;
    }
  };
  load_tile(sK, kbase, ldk, k0, S);
  load_tile(sV, vbase, ldk, k0, S);
  load_q_tile(kb, 0);
  cp_commit();

  float dk[16][4], dv[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;
  const int key_a = k0 + warp * 16 + (lane >> 2);  // keys held: key_a, key_a + 8

  for (int qb = kb; qb < nqb; ++qb) {
    const int buf = (qb - kb) & 1;
    if (qb + 1 < nqb) {
      load_q_tile(qb + 1, buf ^ 1);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const float* slse = sStat + buf * 128;
    const float* sD = sStat + buf * 128 + 64;

    // S^T = K_w Q^T and dP^T = V_w dO^T (16 keys x 64 queries per warp)
    float st[8][4], dpt[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t ka[4], va[4];
      ldsm4(sK + sw(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
      ldsm4(sV + sw(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int rr = np * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int cc = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm4(sQ(buf) + sw(rr, cc), b0, b1, b2, b3);
        mma16816(st[2 * np], ka, b0, b1);
        mma16816(st[2 * np + 1], ka, b2, b3);
        ldsm4(sdO(buf) + sw(rr, cc), b0, b1, b2, b3);
        mma16816(dpt[2 * np], va, b0, b1);
        mma16816(dpt[2 * np + 1], va, b2, b3);
      }
    }
    // P^T and dS^T (fp32), masked: key <= query < S
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ql = nt * 8 + 2 * (lane & 3) + (e & 1);
        const int qrow = qb * TB + ql;
        const int key = key_a + ((e >> 1) << 3);
        float p = exp2f(st[nt][e] * scale_log2 - slse[ql]);
        if (key > qrow || qrow >= S) p = 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - sD[ql]);
      }
    }
    // dV += P^T dO ; dK += dS^T Q   (k = query)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      sa[0] = pack_bf16x2(dpt[2 * kk][0], dpt[2 * kk][1]);
      sa[1] = pack_bf16x2(dpt[2 * kk][2], dpt[2 * kk][3]);
      sa[2] = pack_bf16x2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      sa[3] = pack_bf16x2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
      // dS^T tile to shared memory for the dQ product: row = key, col = query
      {
        const int kr = warp * 16 + (lane >> 2);
        const int qc0 = kk * 16 + 2 * (lane & 3);
        uint8_t* base = smem + 6 * TILE_BYTES;
        *reinterpret_cast<uint32_t*>(base + sw64(kr, qc0 >> 3) + (qc0 & 7) * 2) = sa[0];
        *reinterpret_cast<uint32_t*>(base + sw64(kr + 8, qc0 >> 3) + (qc0 & 7) * 2) = sa[1];
        *reinterpret_cast<uint32_t*>(base + sw64(kr, (qc0 + 8) >> 3) + (qc0 & 7) * 2) = sa[2];
        *reinterpret_cast<uint32_t*>(base + sw64(kr + 8, (qc0 + 8) >> 3) + (qc0 & 7) * 2) = sa[3];
      }
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int rr = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int cc = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm4t(sdO(buf) + sw(rr, cc), b0, b1, b2, b3);
        mma16816(dv[2 * dp], pa, b0, b1);
        mma16816(dv[2 * dp + 1], pa, b2, b3);
        ldsm4t(sQ(buf) + sw(rr, cc), b0, b1, b2, b3);
        mma16816(dk[2 * dp], sa, b0, b1);
        mma16816(dk[2 * dp + 1], sa, b2, b3);
      }
    }
    __syncthreads();
    // dQ[q, :] += sum_key dS[q, key] K[key, :]: warp w takes queries 16w..16w+15,
    // two halves of the head dim to bound registers.
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float dq[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int mat = lane >> 3;
        const int krow = kk * 16 + ((mat >> 1) << 3) + (lane & 7);
        const int qcol_chunk = (warp * 16 + ((mat & 1) << 3)) >> 3;
        uint32_t a[4];
        ldsm4t(sdS + sw64(krow, qcol_chunk), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          const int rr = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int cc = half * 8 + dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm4t(sK + sw(rr, cc), b0, b1, b2, b3);
          mma16816(dq[2 * dp], a, b0, b1);
          mma16816(dq[2 * dp + 1], a, b2, b3);
        }
      }
      const int qr0 = qb * TB + warp * 16 + (lane >> 2);
      const int qr1 = qr0 + 8;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = half * 64 + nt * 8 + 2 * (lane & 3);
        if (qr0 < S)
          red_add2(dq_acc + (static_cast<int64_t>(b) * S + qr0) * ldq + h * HD + col,
                   dq[nt][0] * scale, dq[nt][1] * scale);
        if (qr1 < S)
          red_add2(dq_acc + (static_cast<int64_t>(b) * S + qr1) * ldq + h * HD + col,
                   dq[nt][2] * scale, dq[nt][3] * scale);
      }
    }
    __syncthreads();
  }
  // dK (scaled), dV into the shared key/value head's fp32 accumulators
  const int kr0 = key_a, kr1 = key_a + 8;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int col = nt * 8 + 2 * (lane & 3);
    if (kr0 < S) {
      float* pk = dk_acc + (static_cast<int64_t>(b) * S + kr0) * ldk + j * HD + col;
      float* pv = dv_acc + (static_cast<int64_t>(b) * S + kr0) * ldk + j * HD + col;
      red_add2(pk, dk[nt][0] * scale, dk[nt][1] * scale);
      red_add2(pv, dv[nt][0], dv[nt][1]);
    }
    if (kr1 < S) {
      float* pk = dk_acc + (static_cast<int64_t>(b) * S + kr1) * ldk + j * HD + col;
      float* pv = dv_acc + (static_cast<int64_t>(b) * S + kr1) * ldk + j * HD + col;
      red_add2(pk, dk[nt][2] * scale, dk[nt][3] * scale);
      red_add2(pv, dv[nt][2], dv[nt][3]);
    }
  }
}

constexpr size_t FWD_SMEM = 5 * TILE_BYTES;
constexpr size_t BWD_SMEM = 6 * TILE_BYTES + 8192 + 4 * 64 * sizeof(float);

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kl_status set_smem_attrs() {
  static uint64_t done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(fa_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(FWD_SMEM)));
    KL_CUDA(cudaFuncSetAttribute(fa_bwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(BWD_SMEM)));
    done |= uint64_t(1) << dev;
  }
  return KL_OK;
}

kl_status check_args(int B, int S, int Hq, int Hkv, int d, int dtype) {
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv)
    return set_error(KL_ERR_INVALID_ARG, "attention: bad shape B %d S %d Hq %d Hkv %d d %d", B, S,
                     Hq, Hkv, d);
  if (dtype == KL_BF16 && d != HD)
    return set_error(KL_ERR_UNSUPPORTED, "attention: bf16 path needs head dim 128 (got %d)", d);
  if (dtype == KL_F32 && d > 256)
    return set_error(KL_ERR_UNSUPPORTED, "attention: fp32 path needs head dim <= 256");
  if (dtype != KL_BF16 && dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "attention: bad dtype");
  return KL_OK;
}

}  // namespace

kl_status attention_fwd(int B, int S, int Hq, int Hkv, int d, int dtype, const void* q,
                        const void* k, const void* v, void* o, float* lse, cudaStream_t st) {
  KL_TRY(check_args(B, S, Hq, Hkv, d, dtype));
  if (!q || !k || !v || !o || !lse) return set_error(KL_ERR_INVALID_ARG, "attention_fwd: null pointer");
  const float scale = 1.0f / sqrtf(static_cast<float>(d));
  const double causal_pairs = 0.5 * static_cast<double>(S) * (S + 1);
  ProfScope ps(dtype == KL_F32 ? "attn_fwd_f32" : "attn_fwd_bf16", st, 4.0 * B * Hq * d * causal_pairs,
               dtype_size(dtype) * (2.0 * B * S * Hq * d + 2.0 * B * S * Hkv * d) + 4.0 * B * Hq * S);
  if (dtype == KL_F32) {
    const int64_t rows = static_cast<int64_t>(B) * S * Hq;
    attn_fwd_f32_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
        B, S, Hq, Hkv, d, (const float*)q, (const float*)k, (const float*)v, (float*)o, lse, scale);
  } else {
    if (!al16(q) || !al16(k) || !al16(v) || !al16(o))
      return set_error(KL_ERR_INVALID_ARG, "attention_fwd: bf16 buffers must be 16-byte aligned");
    KL_TRY(attention_fwd_tc(B, S, Hq, Hkv, q, k, v, o, lse, st));
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

size_t attention_bwd_ws(int B, int S, int Hq, int Hkv, int d) {
  const size_t T = static_cast<size_t>(B) * S;
  return align_up(static_cast<size_t>(B) * Hq * S * 4, 256) + align_up(T * Hq * d * 4, 256) +
         2 * align_up(T * Hkv * d * 4, 256);
}

kl_status attention_bwd_accum(int B, int S, int Hq, int Hkv, int d, int dtype, const void* q,
                              const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* ws, size_t ws_bytes, float** dq_acc,
                              float** dk_acc, float** dv_acc, cudaStream_t st,
                              bool d_ready, void* dq_out, const float2* rope_cs) {
  KL_TRY(check_args(B, S, Hq, Hkv, d, dtype));
  if (!q || !k || !v || !o || !lse || !dout)
    return set_error(KL_ERR_INVALID_ARG, "attention_bwd: null pointer");
  if (!ws || ws_bytes < attention_bwd_ws(B, S, Hq, Hkv, d))
    return set_error(KL_ERR_NO_MEMORY, "attention_bwd: workspace too small");
  const size_t T = static_cast<size_t>(B) * S;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* Dd = reinterpret_cast<float*>(w);
  w += align_up(static_cast<size_t>(B) * Hq * S * 4, 256);
  float* dq = reinterpret_cast<float*>(w);
  w += align_up(T * Hq * d * 4, 256);
  float* dk = reinterpret_cast<float*>(w);
  w += align_up(T * Hkv * d * 4, 256);
  float* dv = reinterpret_cast<float*>(w);
  *dq_acc = dq;
  *dk_acc = dk;
  *dv_acc = dv;
  const float scale = 1.0f / sqrtf(static_cast<float>(d));
  const double causal_pairs = 0.5 * static_cast<double>(S) * (S + 1);
  const double bwd_flops = 10.0 * B * Hq * d * causal_pairs;
  if (dtype == KL_F32) {
    ProfScope ps("attn_bwd_f32", st, bwd_flops, 0.0);
    const int64_t rows = static_cast<int64_t>(T) * Hq;
    attn_bwd_dq_f32_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
        B, S, Hq, Hkv, d, (const float*)q, (const float*)k, (const float*)v, (const float*)o, lse,
        (const float*)dout, Dd, dq, scale);
    KL_CUDA(cudaGetLastError());
    const int64_t krows = static_cast<int64_t>(T) * Hkv;
    attn_bwd_dkdv_f32_kernel<<<static_cast<unsigned>((krows + 7) / 8), 256, 0, st>>>(
        B, S, Hq, Hkv, d, (const float*)q, (const float*)k, (const float*)v, lse,
        (const float*)dout, Dd, dk, dv, scale);
  } else {
    if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || !al16(dout))
      return set_error(KL_ERR_INVALID_ARG, "attention_bwd: bf16 buffers must be 16-byte aligned");
    KL_TRY(set_smem_attrs());
    KL_CUDA(cudaMemsetAsync(dk, 0, T * Hkv * d * 4, st));
    KL_CUDA(cudaMemsetAsync(dv, 0, T * Hkv * d * 4, st));
    const int64_t rows = static_cast<int64_t>(T) * Hq;
    if (!d_ready) {
      ProfScope ps("attn_bwd_pre_bf16", st, 0.0, 4.0 * T * Hq * d + 4.0 * T * Hq);
      attn_bwd_pre_bf16_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
          B, S, Hq, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, Dd);
      KL_CUDA(cudaGetLastError());
    }
    if (dq_out && !al16(dq_out)) return set_error(KL_ERR_INVALID_ARG, "attention_bwd: dq not 16-byte aligned");
    KL_TRY(attention_bwd_tc(B, S, Hq, Hkv, q, k, v, dout, lse, Dd, dq, dk, dv, st, dq_out, rope_cs));
    if (dq_out) *dq_acc = nullptr;
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
