// Normalisation, rotary and activation kernels of the layer ("From-scratch
// GPU LLM training", capability list: RMSNorm, SiLU / SwiGLU and RoPE
// gradient kernels; "KYNETRA FOUNDRY", pre-norm decoder and rotary
// paragraphs). All of them are HBM-bound: 128-bit loads and stores where the
// widths allow, fp32 arithmetic, warp-shuffle row reductions.
#include <math.h>

#include <atomic>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void decode(const uint4& a, float (&f)[8]) {
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
  }
  static __device__ __forceinline__ void load(const float* p, float (&f)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&f)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void decode(const uint4& a, float (&f)[8]) {
    const float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y), x2 = unpack_bf16x2(a.z),
                 x3 = unpack_bf16x2(a.w);
    f[0] = x0.x; f[1] = x0.y; f[2] = x1.x; f[3] = x1.y;
    f[4] = x2.x; f[5] = x2.y; f[6] = x3.x; f[7] = x3.y;
  }
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&f)[8]) {
    uint4 a = *reinterpret_cast<const uint4*>(p);
    float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y), x2 = unpack_bf16x2(a.z),
           x3 = unpack_bf16x2(a.w);
    f[0] = x0.x; f[1] = x0.y; f[2] = x1.x; f[3] = x1.y;
    f[4] = x2.x; f[5] = x2.y; f[6] = x3.x; f[7] = x3.y;
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&f)[8]) {
    uint4 o;
    o.x = pack_bf16x2(f[0], f[1]);
    o.y = pack_bf16x2(f[2], f[3]);
    o.z = pack_bf16x2(f[4], f[5]);
    o.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(p) = o;
  }
};

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// RoPE. Plane i pairs element i with element i + d/2 and turns it by the
// angle s * base^(-2i/d). The angle is reduced exactly in fixed point, as a
// phase accumulator does: plane i's rate in turns per position,
// base^(-2i/d) / (2 pi), is formed on the host in fp64 and passed as a 64-bit
// binary fraction of a turn; on the device s times that rate, taken modulo
// 2^64 by the integer multiply, is the position's angle in turns modulo one,
// and its top 32 bits read as a signed integer give the remainder in
// [-pi, pi) for the fp32 sincosf. No fp64 arithmetic runs on the device; the
// angle error is ~1e-11 rad from the rate plus 2^-32 of a turn from the
// truncation, below the fp32 rounding of the remainder itself.
// ---------------------------------------------------------------------------
constexpr int ROPE_MAX_HALF = 128;
struct RopeFreq {
  uint64_t turn[ROPE_MAX_HALF];   // plane i's rate, turns per position, in units of 2^-64 turn
};

RopeFreq rope_freq(int d, float base) {
  RopeFreq f;
  for (int i = 0; i < ROPE_MAX_HALF; ++i) {
    const double rate = i < d / 2 ? pow(static_cast<double>(base), -2.0 * i / d) / 6.283185307179586 : 0.0;
    f.turn[i] = static_cast<uint64_t>(ldexp(rate, 64));   // rate < 1/(2 pi): fits in 64 bits
  }
  return f;
}

__device__ __forceinline__ void rope_cos_sin(int s, uint64_t turn, float dir, float* c, float* sn) {
  const uint64_t phase = static_cast<uint64_t>(s) * turn;            // turns mod 1, in 2^-64 units
  const int32_t hi = static_cast<int32_t>(static_cast<uint32_t>(phase >> 32));
  const float r = static_cast<float>(hi) * 1.46291807926715968e-09f;  // 2 pi / 2^32
  float sf, cf;
  sincosf(r, &sf, &cf);
  *c = cf;
  *sn = dir * sf;
}

// ---------------------------------------------------------------------------
// RMSNorm forward: one warp per row.
// ---------------------------------------------------------------------------
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(int rows, int width,
                                                          const T* __restrict__ x,
                                                          const T* __restrict__ gamma, float eps,
                                                          T* __restrict__ h,
                                                          float* __restrict__ rstd) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= rows) return;
  const T* xr = x + static_cast<int64_t>(row) * width;
  T* hr = h + static_cast<int64_t>(row) * width;
  constexpr int V = Vec<T>::N;
  float ss = 0.f;
  if (VEC) {
    for (int j = lane * V; j < width; j += 32 * V) {
      float f[8];
      Vec<T>::load(xr + j, f);
#pragma unroll
      for (int e = 0; e < V; ++e) ss = fmaf(f[e], f[e], ss);
    }
  } else {
    for (int j = lane; j < width; j += 32) {
      const float f = ld_f(xr + j);
      ss = fmaf(f, f, ss);
    }
  }
  ss = warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / static_cast<float>(width) + eps);
  if (lane == 0) rstd[row] = r;
  if (VEC) {
    for (int j = lane * V; j < width; j += 32 * V) {
      float f[8], g[8];
      Vec<T>::load(xr + j, f);
      Vec<T>::load(gamma + j, g);
#pragma unroll
      for (int e = 0; e < V; ++e) f[e] = g[e] * (f[e] * r);
      Vec<T>::store(hr + j, f);
    }
  } else {
    for (int j = lane; j < width; j += 32) st_f(hr + j, ld_f(gamma + j) * (ld_f(xr + j) * r));
  }
}

// RMSNorm forward, row form: one 128-thread CTA per row, the row held in
// registers as raw 16-byte vectors (NC per thread), so x is read from HBM
// once; sum of squares by warp shuffles plus one barrier.
constexpr int RF_THREADS = 128, RF_MAXC = 8;

// With a table (cs non-null), the CTA of row s < S also writes the rotary
// (cos, sin) row of position s, [S][half], while its loads are in flight.
template <typename T, int NC>
__global__ void __launch_bounds__(RF_THREADS) rmsnorm_fwd_row_kernel(int width, const T* __restrict__ x,
                                                                     const T* __restrict__ gamma, float eps,
                                                                     T* __restrict__ h,
                                                                     float* __restrict__ rstd, int S,
                                                                     int half, const RopeFreq f,
                                                                     float2* __restrict__ cs) {
  pdl_enter();
  __shared__ float red[RF_THREADS / 32];
  constexpr int V = Vec<T>::N;
  const int row = blockIdx.x, tid = threadIdx.x;
  const int chunks = width / V;
  const int64_t off = static_cast<int64_t>(row) * width;
  uint4 raw[NC], graw[NC];   // the row and the gains, both in flight before the reduction
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * RF_THREADS;
    if (c < chunks) {
      raw[j] = *reinterpret_cast<const uint4*>(x + off + c * V);
      graw[j] = *reinterpret_cast<const uint4*>(gamma + c * V);
    }
  }
  if (cs && row < S) {
    for (int i = tid; i < half; i += RF_THREADS) {
      float c, sn;
      rope_cos_sin(row, f.turn[i], 1.0f, &c, &sn);
      cs[static_cast<int64_t>(row) * half + i] = make_float2(c, sn);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    if (tid + j * RF_THREADS < chunks) {
      float f[8];
      Vec<T>::decode(raw[j], f);
#pragma unroll
      for (int e = 0; e < V; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < RF_THREADS / 32; ++w) tot += red[w];
  const float r = 1.0f / sqrtf(tot / static_cast<float>(width) + eps);
  if (tid == 0) rstd[row] = r;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * RF_THREADS;
    if (c < chunks) {
      float f[8], g[8];
      Vec<T>::decode(raw[j], f);
      Vec<T>::decode(graw[j], g);
#pragma unroll
      for (int e = 0; e < V; ++e) f[e] = g[e] * (f[e] * r);
      Vec<T>::store(h + off + c * V, f);
    }
  }
}

// ---------------------------------------------------------------------------
// RMSNorm backward, any width: one CTA per row at a time, thread t owning
// columns t, t + 256, ... . The gain gradient of a column is summed in shared
// memory by its owning thread alone, in row order (no atomics, so the partial
// rows and the gain gradient are the same on every run), and written as one
// partial row per CTA, reduced afterwards in CTA order.
//   n = x*rstd, dn = dh*gamma, dx = resid + rstd*(dn - n*mean(dn*n)),
//   dgamma += dh*n.
// ---------------------------------------------------------------------------
template <typename T, typename TD>
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(
    int rows, int width, const TD* __restrict__ dh, const T* __restrict__ x,
    const T* __restrict__ gamma, const float* __restrict__ rstd, const T* __restrict__ resid,
    T* __restrict__ dx, float* __restrict__ partial) {
  pdl_enter();
  extern __shared__ float sacc[];
  __shared__ float red[2][8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int j = tid; j < width; j += 256) sacc[j] = 0.f;
  const float inv_w = 1.0f / static_cast<float>(width);
  int buf = 0;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int64_t off = static_cast<int64_t>(row) * width;
    const float r = rstd[row];
    float dot = 0.f;
    for (int j = tid; j < width; j += 256) {
      const float n = ld_f(x + off + j) * r;
      dot = fmaf(ld_f(dh + off + j) * ld_f(gamma + j), n, dot);
    }
    dot = warp_sum(dot);
    if (lane == 0) red[buf][warp] = dot;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[buf][w];
    tot *= inv_w;
    buf ^= 1;   // the next row's partial sums go to the other buffer: one barrier per row
    for (int j = tid; j < width; j += 256) {
      const float n = ld_f(x + off + j) * r;
      const float g = ld_f(dh + off + j);
      float v = r * (g * ld_f(gamma + j) - n * tot);
      if (resid) v += ld_f(resid + off + j);
      st_f(dx + off + j, v);
      sacc[j] += g * n;
    }
  }
  for (int j = tid; j < width; j += 256)
    partial[static_cast<int64_t>(blockIdx.x) * width + j] = sacc[j];
}

// RMSNorm backward, row-parallel form: one CTA covers a whole row (256
// threads x 4-element chunks, up to 8 chunks each, so width <= 8192), keeps
// its columns' gains and gain-gradient partial sums in registers across all
// rows it visits, and reduces the row dot product with one barrier.
constexpr int RB_MAXC = 8;

__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p);
  const float2 x0 = unpack_bf16x2(a.x), x1 = unpack_bf16x2(a.y);
  v[0] = x0.x; v[1] = x0.y; v[2] = x1.x; v[3] = x1.y;
}
__device__ __forceinline__ void store4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 o;
  o.x = pack_bf16x2(v[0], v[1]);
  o.y = pack_bf16x2(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = o;
}

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_bwd_rows_kernel(
    int rows, int width, const float* __restrict__ dh, const T* __restrict__ x,
    const T* __restrict__ gamma, const float* __restrict__ rstd, const T* __restrict__ resid,
    T* __restrict__ dx, float* __restrict__ partial) {
  pdl_enter();
  __shared__ float red[2][8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nchunk = width >> 2;
  float g[RB_MAXC][4], acc[RB_MAXC][4];
#pragma unroll
  for (int k = 0; k < RB_MAXC; ++k) {
    const int c = tid + 256 * k;
#pragma unroll
    for (int e = 0; e < 4; ++e) g[k][e] = acc[k][e] = 0.f;
    if (c < nchunk) load4(gamma + 4 * c, g[k]);
  }
  const float inv_w = 1.0f / static_cast<float>(width);
  int buf = 0;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int64_t off = static_cast<int64_t>(row) * width;
    const float r = rstd[row];
    float dv[RB_MAXC][4], xv[RB_MAXC][4];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < RB_MAXC; ++k) {
      const int c = tid + 256 * k;
      if (c < nchunk) {
        load4(dh + off + 4 * c, dv[k]);
        load4(x + off + 4 * c, xv[k]);
#pragma unroll
        for (int e = 0; e < 4; ++e) dot = fmaf(dv[k][e] * g[k][e], xv[k][e], dot);
      }
    }
    dot = warp_sum(dot);
    if (lane == 0) red[buf][warp] = dot;
    __syncthreads();
    dot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) dot += red[buf][w];
    dot *= r * inv_w;
    buf ^= 1;
#pragma unroll
    for (int k = 0; k < RB_MAXC; ++k) {
      const int c = tid + 256 * k;
      if (c < nchunk) {
        float o[4], rv[4] = {0.f, 0.f, 0.f, 0.f};
        if (resid) load4(resid + off + 4 * c, rv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float n = xv[k][e] * r;
          o[e] = r * (dv[k][e] * g[k][e] - n * dot) + rv[e];
          acc[k][e] = fmaf(dv[k][e], n, acc[k][e]);
        }
        store4(dx + off + 4 * c, o);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < RB_MAXC; ++k) {
    const int c = tid + 256 * k;
    if (c < nchunk) store4(partial + static_cast<int64_t>(blockIdx.x) * width + 4 * c, acc[k]);
  }
}

// RMSNorm backward for bf16 activations with an fp32 incoming gradient, row
// form with 8-element chunks: one 256-thread CTA per row at a time, two CTAs
// resident per SM. Every load of a row (dh, x and the residual gradient) is
// issued before the row's dot-product barrier; gains stay in registers as
// packed bf16 and the gain-gradient partial sums as fp32 across the CTA's rows.
constexpr int RW_THREADS = 256, RW_MAXC = 4;

// Grid-wide barrier of a cooperative launch (every CTA resident): one arrival
// counter and one generation word per slot in static device memory; the last
// CTA to arrive re-arms the counter and moves the generation on. The wait is
// bounded: past the limit it records KL_DEVERR_TIMEOUT and goes on.
constexpr int RB_BAR_SLOTS = 16;
__device__ unsigned int g_rms_bar[RB_BAR_SLOTS][2];

__device__ __forceinline__ void grid_barrier(unsigned int* bar, unsigned int nblocks, uint32_t* err) {
  __threadfence();   // this thread's writes before the arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned int* gen = bar + 1;
    const unsigned int g0 = *gen;   // read before arriving: the last arrival moves it on after
    const unsigned int prev = atomicAdd(bar, 1u);
    if (prev == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = global_timer_ns();
      uint32_t k = 0;
      while (*gen == g0) {
        if ((++k & 255u) == 0 && global_timer_ns() - t0 > KL_WAIT_LIMIT_NS) {
          record_error(err, KL_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// With dgamma (a cooperative launch), after its partial row each CTA passes a
// grid barrier and then sums 32-column slices of dgamma over every CTA's
// partial row in CTA order (the column-sum step in the same launch).
template <int NC>
__global__ void __launch_bounds__(RW_THREADS, 2) rmsnorm_bwd_row8_kernel(
    int rows, int width, const float* __restrict__ dh, const __nv_bfloat16* __restrict__ x,
    const __nv_bfloat16* __restrict__ gamma, const float* __restrict__ rstd,
    const __nv_bfloat16* __restrict__ resid, __nv_bfloat16* __restrict__ dx,
    float* __restrict__ partial, float* __restrict__ dgamma, unsigned int* __restrict__ bar,
    uint32_t* __restrict__ err) {
  pdl_enter();
  using T = __nv_bfloat16;
  __shared__ float red[2][RW_THREADS / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunks = width >> 3;
  uint4 graw[NC];
  float acc[NC][8];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * RW_THREADS;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    if (c < chunks) graw[j] = *reinterpret_cast<const uint4*>(gamma + 8 * c);
  }
  const float inv_w = 1.0f / static_cast<float>(width);
  int buf = 0;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int64_t off = static_cast<int64_t>(row) * width;
    float4 d0[NC], d1[NC];
    uint4 xraw[NC], rraw[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = tid + j * RW_THREADS;
      if (c < chunks) {
        d0[j] = *reinterpret_cast<const float4*>(dh + off + 8 * c);
        d1[j] = *reinterpret_cast<const float4*>(dh + off + 8 * c + 4);
        xraw[j] = *reinterpret_cast<const uint4*>(x + off + 8 * c);
        rraw[j] = resid ? *reinterpret_cast<const uint4*>(resid + off + 8 * c) : make_uint4(0, 0, 0, 0);
      }
    }
    const float r = rstd[row];
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (tid + j * RW_THREADS < chunks) {
        float xv[8], g[8];
        Vec<T>::decode(xraw[j], xv);
        Vec<T>::decode(graw[j], g);
        const float dv[8] = {d0[j].x, d0[j].y, d0[j].z, d0[j].w, d1[j].x, d1[j].y, d1[j].z, d1[j].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(dv[e] * g[e], xv[e], dot);
      }
    }
    dot = warp_sum(dot);
    if (lane == 0) red[buf][warp] = dot;
    __syncthreads();
    dot = 0.f;
#pragma unroll
    for (int w = 0; w < RW_THREADS / 32; ++w) dot += red[buf][w];
    dot *= r * inv_w;
    buf ^= 1;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = tid + j * RW_THREADS;
      if (c < chunks) {
        float xv[8], g[8], rv[8], o[8];
        Vec<T>::decode(xraw[j], xv);
        Vec<T>::decode(graw[j], g);
        Vec<T>::decode(rraw[j], rv);
        const float dv[8] = {d0[j].x, d0[j].y, d0[j].z, d0[j].w, d1[j].x, d1[j].y, d1[j].z, d1[j].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float n = xv[e] * r;
          o[e] = r * (dv[e] * g[e] - n * dot) + rv[e];
          acc[j][e] = fmaf(dv[e], n, acc[j][e]);
        }
        Vec<T>::store(dx + off + 8 * c, o);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * RW_THREADS;
    if (c < chunks) {
      float* p = partial + static_cast<int64_t>(blockIdx.x) * width + 8 * c;
      *reinterpret_cast<float4*>(p) = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
      *reinterpret_cast<float4*>(p + 4) = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
    }
  }
  if (!dgamma) return;
  grid_barrier(bar, gridDim.x, err);
  // dgamma: 32 columns per CTA (8 float4 lanes), the partial rows split over 32
  // row groups, then a fixed tree over the groups (deterministic)
  __shared__ float4 cred[32][8];
  const int cg = tid & 7, rg = tid >> 3;
  const int nrows = gridDim.x;
  for (int cb = blockIdx.x; cb * 32 < width; cb += gridDim.x) {
    const int c = cb * 32 + cg * 4;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < width) {
      for (int r2 = rg; r2 < nrows; r2 += 32) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(partial + static_cast<int64_t>(r2) * width + c));
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
    }
    cred[rg][cg] = sum;
    __syncthreads();
    for (int k = 16; k > 0; k >>= 1) {
      if (rg < k) {
        const float4 o = cred[rg + k][cg];
        float4& m = cred[rg][cg];
        m.x += o.x; m.y += o.y; m.z += o.z; m.w += o.w;
      }
      __syncthreads();
    }
    if (rg == 0 && c < width) *reinterpret_cast<float4*>(dgamma + c) = cred[0][cg];
    __syncthreads();
  }
}

// out[c] = sum over the partial rows, width a multiple of 4: a CTA takes 32
// columns (8 float4 lanes) and splits the rows over 32 groups, then a fixed
// tree over the groups (deterministic).
__global__ void __launch_bounds__(256) column_sum4_kernel(int nrows, int width,
                                                          const float* __restrict__ partial,
                                                          float* __restrict__ out) {
  pdl_enter();
  __shared__ float4 red[32][8];
  const int cg = threadIdx.x & 7, rg = threadIdx.x >> 3;
  const int c = blockIdx.x * 32 + cg * 4;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < width) {
#pragma unroll 4
    for (int r = rg; r < nrows; r += 32) {
      const float4 v = *reinterpret_cast<const float4*>(partial + static_cast<int64_t>(r) * width + c);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
  }
  red[rg][cg] = s;
  __syncthreads();
  for (int k = 16; k > 0; k >>= 1) {
    if (rg < k) {
      const float4 o = red[rg + k][cg];
      float4& m = red[rg][cg];
      m.x += o.x; m.y += o.y; m.z += o.z; m.w += o.w;
    }
    __syncthreads();
  }
  if (rg == 0 && c < width) *reinterpret_cast<float4*>(out + c) = red[0][cg];
}

// out[c] = sum over the partial rows (fixed order: deterministic).
__global__ void __launch_bounds__(256) column_sum_kernel(int nrows, int width,
                                                         const float* __restrict__ partial,
                                                         float* __restrict__ out) {
  pdl_enter();
  __shared__ float red[4][64];
  const int c = blockIdx.x * 64 + (threadIdx.x & 63);
  const int grp = threadIdx.x >> 6;
  float s = 0.f;
  if (c < width)
    for (int r = grp; r < nrows; r += 4) s += partial[static_cast<int64_t>(r) * width + c];
  red[grp][threadIdx.x & 63] = s;
  __syncthreads();
  if (grp == 0 && c < width) out[c] = (red[0][threadIdx.x] + red[1][threadIdx.x]) + (red[2][threadIdx.x] + red[3][threadIdx.x]);
}

int rmsnorm_bwd_grid(int rows) {
  const int want = rows;
  const int cap = 2 * num_sms();
  return want < cap ? want : cap;
}

// cos in cs[0, half), dir*sin in cs[half, d); the caller synchronises.
__device__ __forceinline__ void rope_table(int s, int d, const RopeFreq& f, float dir, float* cs) {
  const int half = d / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) rope_cos_sin(s, f.turn[i], dir, &cs[i], &cs[half + i]);
}

// The (cos, sin) table of every position and plane: consumed by the fused
// rotary epilogues of the q/k projection and of the attention dQ kernel.
__global__ void rope_cs_kernel(int S, int half, RopeFreq f, float2* __restrict__ cs) {
  pdl_enter();
  const int64_t n = static_cast<int64_t>(S) * half;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(idx / half), i = static_cast<int>(idx - static_cast<int64_t>(s) * half);
    float c, sn;
    rope_cos_sin(s, f.turn[i], 1.0f, &c, &sn);
    cs[idx] = make_float2(c, sn);
  }
}

template <typename T>
__global__ void rope_kernel(int S, int heads, int d, RopeFreq f, T* __restrict__ x, float dir) {
  pdl_enter();
  __shared__ float cs[2 * ROPE_MAX_HALF];
  const int t = blockIdx.x;
  rope_table(t % S, d, f, dir, cs);
  __syncthreads();
  const int half = d / 2;
  T* row = x + static_cast<int64_t>(t) * heads * d;
  for (int idx = threadIdx.x; idx < heads * half; idx += blockDim.x) {
    const int hh = idx / half, i = idx - hh * half;
    T* p = row + hh * d;
    const float a = ld_f(p + i), b = ld_f(p + half + i);
    const float c = cs[i], sn = cs[half + i];
    st_f(p + i, a * c - b * sn);
    st_f(p + half + i, a * sn + b * c);
  }
}

// Forward (dir = +1) or backward (dir = -1) rotation of q [T, hq, d] and k
// [T, hk, d] in place, one CTA per token. A work item is V consecutive planes
// of one head (elements i0 .. i0+V-1 and their partners at +d/2); each thread
// issues the loads of all its items before the angle table is formed, so the
// table's arithmetic overlaps the memory latency.
constexpr int RQ_THREADS = 128, RQ_ITEMS = 5;

template <typename T>
__global__ void __launch_bounds__(RQ_THREADS) rope_qk_kernel(int S, int hq, int hk, int d, RopeFreq f,
                                                             T* __restrict__ q, T* __restrict__ k,
                                                             float dir) {
  pdl_enter();
  __shared__ float cs[2 * ROPE_MAX_HALF];
  const int t = blockIdx.x;
  const int half = d / 2;
  constexpr int V = Vec<T>::N;
  const int groups = half / V;
  const int items = (hq + hk) * groups;
  for (int base = 0; base < items; base += RQ_THREADS * RQ_ITEMS) {
    uint4 ra[RQ_ITEMS], rb[RQ_ITEMS];
#pragma unroll
    for (int j = 0; j < RQ_ITEMS; ++j) {
      const int idx = base + threadIdx.x + j * RQ_THREADS;
      if (idx < items) {
        const int h = idx / groups, i0 = (idx - h * groups) * V;
        const T* p = h < hq ? q + (static_cast<int64_t>(t) * hq + h) * d
                            : k + (static_cast<int64_t>(t) * hk + (h - hq)) * d;
        ra[j] = *reinterpret_cast<const uint4*>(p + i0);
        rb[j] = *reinterpret_cast<const uint4*>(p + half + i0);
      }
    }
    if (base == 0) {
      rope_table(t % S, d, f, dir, cs);
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < RQ_ITEMS; ++j) {
      const int idx = base + threadIdx.x + j * RQ_THREADS;
      if (idx < items) {
        const int h = idx / groups, i0 = (idx - h * groups) * V;
        T* p = h < hq ? q + (static_cast<int64_t>(t) * hq + h) * d
                      : k + (static_cast<int64_t>(t) * hk + (h - hq)) * d;
        float a[8], b[8];
        Vec<T>::decode(ra[j], a);
        Vec<T>::decode(rb[j], b);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float c = cs[i0 + e], sn = cs[half + i0 + e];
          const float x = a[e], y = b[e];
          a[e] = x * c - y * sn;
          b[e] = x * sn + y * c;
        }
        Vec<T>::store(p + i0, a);
        Vec<T>::store(p + half + i0, b);
      }
    }
  }
}

// Attention-backward epilogue: fp32 accumulators -> dq, dk turned back by
// -angle, dv converted; one CTA per token. Items are 4-wide: a rotation item
// reads planes i0..i0+3 and their partners, a dv item reads 4 elements; all
// of a thread's loads are issued before the table is formed.
constexpr int RC_THREADS = 256, RC_ITEMS = 6;

template <typename T>
__global__ void __launch_bounds__(RC_THREADS) rope_bwd_convert_kernel(
    int S, int hq, int hk, int d, RopeFreq f, const float* __restrict__ dq_acc,
    const float* __restrict__ dk_acc, const float* __restrict__ dv_acc, T* __restrict__ dq,
    T* __restrict__ dk, T* __restrict__ dv) {
  pdl_enter();
  __shared__ float cs[2 * ROPE_MAX_HALF];
  const int t = blockIdx.x;
  const int half = d / 2;
  const int groups = half / 4;
  const int rot_items = (hq + hk) * groups;
  const int items = rot_items + hk * (d / 4);
  for (int base = 0; base < items; base += RC_THREADS * RC_ITEMS) {
    float4 ra[RC_ITEMS], rb[RC_ITEMS];
#pragma unroll
    for (int j = 0; j < RC_ITEMS; ++j) {
      const int idx = base + threadIdx.x + j * RC_THREADS;
      if (idx < rot_items) {
        const int h = idx / groups, i0 = (idx - h * groups) * 4;
        const float* src = h < hq ? dq_acc + (static_cast<int64_t>(t) * hq + h) * d
                                  : dk_acc + (static_cast<int64_t>(t) * hk + (h - hq)) * d;
        ra[j] = *reinterpret_cast<const float4*>(src + i0);
        rb[j] = *reinterpret_cast<const float4*>(src + half + i0);
      } else if (idx < items) {
        const int64_t o = static_cast<int64_t>(t) * hk * d + static_cast<int64_t>(idx - rot_items) * 4;
        ra[j] = *reinterpret_cast<const float4*>(dv_acc + o);
      }
    }
    if (base == 0) {
      rope_table(t % S, d, f, -1.0f, cs);
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < RC_ITEMS; ++j) {
      const int idx = base + threadIdx.x + j * RC_THREADS;
      if (idx < rot_items) {
        const int h = idx / groups, i0 = (idx - h * groups) * 4;
        T* dst = h < hq ? dq + (static_cast<int64_t>(t) * hq + h) * d
                        : dk + (static_cast<int64_t>(t) * hk + (h - hq)) * d;
        float a[4] = {ra[j].x, ra[j].y, ra[j].z, ra[j].w};
        float b[4] = {rb[j].x, rb[j].y, rb[j].z, rb[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float c = cs[i0 + e], sn = cs[half + i0 + e];
          const float x = a[e], y = b[e];
          a[e] = x * c - y * sn;
          b[e] = x * sn + y * c;
        }
        store4(dst + i0, a);
        store4(dst + half + i0, b);
      } else if (idx < items) {
        const int64_t o = static_cast<int64_t>(t) * hk * d + static_cast<int64_t>(idx - rot_items) * 4;
        const float a[4] = {ra[j].x, ra[j].y, ra[j].z, ra[j].w};
        store4(dv + o, a);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// q / k heads with the options: an optional RMSNorm over each head's d
// features (gain g[d]) followed by the rotary turn, planes (i, i+d/2) or
// interleaved (2i, 2i+1). One warp per (token, head) row; lane l owns planes
// l, l+32, ... (d/2 <= 128, so at most 4 planes per lane). Each element is read
// and written by the same lane only, so input and output may be one buffer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void plane_idx(int i, int d, int inter, int& ia, int& ib) {
  ia = inter ? 2 * i : i;
  ib = inter ? 2 * i + 1 : i + d / 2;
}
__device__ __forceinline__ float2 plane_cs(int pos, int i, int half, const RopeFreq& f, const float2* tab) {
  if (tab) return tab[static_cast<int64_t>(pos) * half + i];
  float c, sn;
  rope_cos_sin(pos, f.turn[i], 1.0f, &c, &sn);
  return make_float2(c, sn);
}

template <typename T>
__global__ void __launch_bounds__(256) qk_rope_fwd_kernel(int rows, int heads, int S, int d, const T* pre,
                                                          const T* __restrict__ gamma, float eps, int norm, int inter,
                                                          RopeFreq f, const float2* __restrict__ tab,
                                                          T* out, float* __restrict__ rstd,
                                                          const int32_t* __restrict__ pos_off) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= rows) return;
  // position of the row's token: its index in the sequence, plus the sequence's
  // offset when the tokens continue a cached prefix
  const int tok = row / heads;
  const int pos = tok % S + (pos_off ? pos_off[tok / S] : 0), half = d / 2;
  const T* x = pre + static_cast<int64_t>(row) * d;
  T* y = out + static_cast<int64_t>(row) * d;
  float r = 1.0f;
  if (norm) {
    float ss = 0.f;
    for (int j = lane; j < d; j += 32) {
      const float v = ld_f(x + j);
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    if (lane == 0) rstd[row] = r;
  }
  for (int i = lane; i < half; i += 32) {
    int ia, ib;
    plane_idx(i, d, inter, ia, ib);
    float a = ld_f(x + ia) * r, b = ld_f(x + ib) * r;
    if (norm) {
      a *= ld_f(gamma + ia);
      b *= ld_f(gamma + ib);
    }
    const float2 cs = plane_cs(pos, i, half, f, tab);
    st_f(y + ia, a * cs.x - b * cs.y);
    st_f(y + ib, a * cs.y + b * cs.x);
  }
}

// A step over a paged key/value cache, in one launch: every new token's q
// heads rotated (after the optional per-head norm) into q_out, its k heads
// rotated the same way straight into their cache slots, and its v heads copied
// to theirs. Token i of sequence b sits at position ctx[b] + i; its slot is
// block table[b][pos / bs], row pos % bs. One warp per (token, head) row, the
// q heads first; a position past its table row or a table entry outside the
// pool is skipped and recorded (KL_DEVERR_PAGE), a negative position skipped.
__global__ void __launch_bounds__(256) paged_qkv_rope_kernel(
    int T, int n_new, int Hq, int Hkv, int d, const __nv_bfloat16* __restrict__ q_pre,
    const __nv_bfloat16* __restrict__ k_pre, const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ gq,
    const __nv_bfloat16* __restrict__ gk, float eps, int norm, int inter, RopeFreq f, const int32_t* __restrict__ table,
    const int32_t* __restrict__ ctx, int bs, int max_blocks, int n_blocks, __nv_bfloat16* __restrict__ q_out,
    __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool, uint32_t* err) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = Hq + Hkv;
  const int row = blockIdx.x * 8 + warp;
  if (row >= T * heads) return;
  const int tok = row / heads, hh = row - tok * heads;
  const int b = tok / n_new, pos = ctx[b] + (tok - b * n_new), half = d / 2;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  const __nv_bfloat16* g;
  if (hh < Hq) {
    x = q_pre + (static_cast<int64_t>(tok) * Hq + hh) * d;
    y = q_out + (static_cast<int64_t>(tok) * Hq + hh) * d;
    g = gq;
  } else {
    const int h = hh - Hq;
    if (pos < 0) return;
    const int lb = pos / bs;
    const int blk = lb < max_blocks ? table[b * max_blocks + lb] : -1;
    if (blk < 0 || blk >= n_blocks) {
      if (lane == 0) record_error(err, KL_DEVERR_PAGE);
      return;
    }
    const int64_t dst = ((static_cast<int64_t>(blk) * bs + (pos - lb * bs)) * Hkv + h) * d;
    const int64_t src = (static_cast<int64_t>(tok) * Hkv + h) * d;
    x = k_pre + src;
    y = k_pool + dst;
    g = gk;
    for (int j = lane * 4; j < d; j += 128)   // the value row, unchanged
      *reinterpret_cast<uint2*>(v_pool + dst + j) = *reinterpret_cast<const uint2*>(v + src + j);
  }
  float r = 1.0f;
  if (norm) {
    float ss = 0.f;
    for (int j = lane; j < d; j += 32) {
      const float vv = ld_f(x + j);
      ss = fmaf(vv, vv, ss);
    }
    ss = warp_sum(ss);
    r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  }
  for (int i = lane; i < half; i += 32) {
    int ia, ib;
    plane_idx(i, d, inter, ia, ib);
    float a = ld_f(x + ia) * r, bb = ld_f(x + ib) * r;
    if (norm) {
      a *= ld_f(g + ia);
      bb *= ld_f(g + ib);
    }
    const float2 cs = plane_cs(pos, i, half, f, nullptr);
    st_f(y + ia, a * cs.x - bb * cs.y);
    st_f(y + ib, a * cs.y + bb * cs.x);
  }
}

// Backward: dy (gradient after the rotation, element type TD, scaled by
// dy_scale) turned back, then the RMSNorm backward
//   n = x r, dn = dy g, dx = r (dn - n mean(dn n)),  dg += dy n
// (without the norm dx = dy). Gain gradients: per-CTA partial rows
// partial[blockIdx.x][d], summed afterwards in a fixed order.
constexpr int QK_MAXP = 4;   // planes per lane (d/2 <= 128)

template <typename T, typename TD>
__global__ void __launch_bounds__(256) qk_rope_bwd_kernel(int rows, int heads, int S, int d, const TD* dyr,
                                                          float dy_scale, const T* __restrict__ pre,
                                                          const T* __restrict__ gamma, const float* __restrict__ rstd,
                                                          int norm, int inter, RopeFreq f,
                                                          const float2* __restrict__ tab, T* dx,
                                                          float* __restrict__ partial) {
  pdl_enter();
  __shared__ float sacc[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = d / 2;
  float acc_a[QK_MAXP], acc_b[QK_MAXP];
#pragma unroll
  for (int t = 0; t < QK_MAXP; ++t) acc_a[t] = acc_b[t] = 0.f;
  for (int row = blockIdx.x * 8 + warp; row < rows; row += gridDim.x * 8) {
    const int pos = (row / heads) % S;
    const int64_t o = static_cast<int64_t>(row) * d;
    float da[QK_MAXP], db[QK_MAXP], na[QK_MAXP], nb[QK_MAXP];
    const float r = norm ? rstd[row] : 1.0f;
    float dot = 0.f;
#pragma unroll
    for (int t = 0; t < QK_MAXP; ++t) {
      const int i = lane + 32 * t;
      da[t] = db[t] = na[t] = nb[t] = 0.f;
      if (i < half) {
        int ia, ib;
        plane_idx(i, d, inter, ia, ib);
        const float ya = ld_f(dyr + o + ia) * dy_scale, yb = ld_f(dyr + o + ib) * dy_scale;
        const float2 cs = plane_cs(pos, i, half, f, tab);
        da[t] = ya * cs.x + yb * cs.y;       // turned back by -angle
        db[t] = yb * cs.x - ya * cs.y;
        if (norm) {
          na[t] = ld_f(pre + o + ia) * r;
          nb[t] = ld_f(pre + o + ib) * r;
          dot = fmaf(da[t] * ld_f(gamma + ia), na[t], dot);
          dot = fmaf(db[t] * ld_f(gamma + ib), nb[t], dot);
        }
      }
    }
    if (norm) dot = warp_sum(dot) / static_cast<float>(d);
#pragma unroll
    for (int t = 0; t < QK_MAXP; ++t) {
      const int i = lane + 32 * t;
      if (i < half) {
        int ia, ib;
        plane_idx(i, d, inter, ia, ib);
        if (norm) {
          const float ga = ld_f(gamma + ia), gb = ld_f(gamma + ib);
          st_f(dx + o + ia, r * (da[t] * ga - na[t] * dot));
          st_f(dx + o + ib, r * (db[t] * gb - nb[t] * dot));
          acc_a[t] = fmaf(da[t], na[t], acc_a[t]);
          acc_b[t] = fmaf(db[t], nb[t], acc_b[t]);
        } else {
          st_f(dx + o + ia, da[t]);
          st_f(dx + o + ib, db[t]);
        }
      }
    }
  }
  if (!norm) return;
  // gain-gradient partial of this CTA: warps' rows summed in a fixed order
#pragma unroll
  for (int t = 0; t < QK_MAXP; ++t) {
    const int i = lane + 32 * t;
    if (i < half) {
      int ia, ib;
      plane_idx(i, d, inter, ia, ib);
      sacc[warp][ia] = acc_a[t];
      sacc[warp][ib] = acc_b[t];
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < 8; ++w) v += sacc[w][j];
    partial[static_cast<int64_t>(blockIdx.x) * d + j] = v;
  }
}

template <typename T>
__global__ void convert_kernel(int64_t n, const float* __restrict__ src, T* __restrict__ dst) {
  pdl_enter();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    st_f(dst + i, src[i]);
}

// ---------------------------------------------------------------------------
// SwiGLU: m = silu(g) * u; dg = dm*u*s*(1 + g*(1-s)), du = dm*g*s, s = sigmoid(g).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + expf(-g)); }

template <typename T, bool VEC>
__global__ void swiglu_fwd_kernel(int64_t n, const T* __restrict__ g, const T* __restrict__ u,
                                  T* __restrict__ m) {
  pdl_enter();
  constexpr int V = Vec<T>::N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (VEC) {
    for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * V; i < n;
         i += stride * V) {
      float a[8], b[8];
      Vec<T>::load(g + i, a);
      Vec<T>::load(u + i, b);
#pragma unroll
      for (int e = 0; e < V; ++e) a[e] = a[e] * sigmoidf_(a[e]) * b[e];
      Vec<T>::store(m + i, a);
    }
  } else {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
      const float a = ld_f(g + i);
      st_f(m + i, a * sigmoidf_(a) * ld_f(u + i));
    }
  }
}

template <typename T, bool VEC>
__global__ void swiglu_bwd_kernel(int64_t n, const T* __restrict__ dm, const T* __restrict__ g,
                                  const T* __restrict__ u, T* __restrict__ dg,
                                  T* __restrict__ du) {
  pdl_enter();
  constexpr int V = Vec<T>::N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (VEC) {
    for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * V; i < n;
         i += stride * V) {
      float a[8], b[8], c[8], o1[8], o2[8];
      Vec<T>::load(dm + i, c);
      Vec<T>::load(g + i, a);
      Vec<T>::load(u + i, b);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float s = sigmoidf_(a[e]);
        o1[e] = c[e] * b[e] * s * (1.0f + a[e] * (1.0f - s));
        o2[e] = c[e] * a[e] * s;
      }
      Vec<T>::store(dg + i, o1);
      Vec<T>::store(du + i, o2);
    }
  } else {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
      const float a = ld_f(g + i), b = ld_f(u + i), c = ld_f(dm + i);
      const float s = sigmoidf_(a);
      st_f(dg + i, c * b * s * (1.0f + a * (1.0f - s)));
      st_f(du + i, c * a * s);
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ew_grid(int64_t work_items) {
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  int64_t g = (work_items + 255) / 256;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

kl_status rmsnorm_fwd(int rows, int width, int dtype, const void* x, const void* gamma, float eps,
                      void* h, float* rstd, cudaStream_t st, int rope_S, int rope_d, float rope_base,
                      float2* rope_cs) {
  if (rows < 1 || width < 1 || !x || !gamma || !h || !rstd)
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_fwd: bad arguments");
  if (dtype != KL_BF16 && dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "rmsnorm_fwd: bad dtype %d", dtype);
  const int grid = (rows + 7) / 8;
  const int V = dtype == KL_BF16 ? 8 : 4;
  const bool vec = width % V == 0 && al16(x) && al16(gamma) && al16(h);
  const int nc = (width / V + RF_THREADS - 1) / RF_THREADS;
  const bool row_form = vec && nc <= RF_MAXC;
  // the rotary table rides with the row form (one CTA per row); otherwise its own launch
  const bool tab = rope_cs && row_form && rope_S <= rows && rope_d >= 2 && (rope_d & 1) == 0 &&
                   rope_d / 2 <= ROPE_MAX_HALF;
  if (rope_cs && !tab) KL_TRY(rope_cs_table(rope_S, rope_d, rope_base, rope_cs, st));
  const int rhalf = tab ? rope_d / 2 : 0;
  const RopeFreq f = rope_freq(tab ? rope_d : 2, rope_base);
  float2* cs = tab ? rope_cs : nullptr;
  ProfScope ps("rmsnorm_fwd", st, 0.0,
               2.0 * rows * width * dtype_size(dtype) + 4.0 * rows + 1.0 * width * dtype_size(dtype) +
                   8.0 * rope_S * rhalf);
  if (row_form) {
    if (dtype == KL_BF16) {
      using T = __nv_bfloat16;
      switch (nc) {
#define KL_RF_CASE(N) case N: launch_pdl(rmsnorm_fwd_row_kernel<T, N>, rows, RF_THREADS, 0, st, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd, rope_S, rhalf, f, cs); break;
        KL_RF_CASE(1) KL_RF_CASE(2) KL_RF_CASE(3) KL_RF_CASE(4) KL_RF_CASE(5) KL_RF_CASE(6) KL_RF_CASE(7) KL_RF_CASE(8)
#undef KL_RF_CASE
      }
    } else {
      using T = float;
      switch (nc) {
#define KL_RF_CASE(N) case N: launch_pdl(rmsnorm_fwd_row_kernel<T, N>, rows, RF_THREADS, 0, st, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd, rope_S, rhalf, f, cs); break;
        KL_RF_CASE(1) KL_RF_CASE(2) KL_RF_CASE(3) KL_RF_CASE(4) KL_RF_CASE(5) KL_RF_CASE(6) KL_RF_CASE(7) KL_RF_CASE(8)
#undef KL_RF_CASE
      }
    }
  } else if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    if (vec) launch_pdl(rmsnorm_fwd_kernel<T, true>, grid, 256, 0, st, rows, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd);
    else launch_pdl(rmsnorm_fwd_kernel<T, false>, grid, 256, 0, st, rows, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd);
  } else {
    if (vec) launch_pdl(rmsnorm_fwd_kernel<float, true>, grid, 256, 0, st, rows, width, (const float*)x, (const float*)gamma, eps, (float*)h, rstd);
    else launch_pdl(rmsnorm_fwd_kernel<float, false>, grid, 256, 0, st, rows, width, (const float*)x, (const float*)gamma, eps, (float*)h, rstd);
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

size_t rmsnorm_bwd_ws(int rows, int width) {
  return align_up(static_cast<size_t>(rmsnorm_bwd_grid(rows)) * width * sizeof(float), 256);
}

// The grid-barrier slot of the next fused RMSNorm backward (round-robin, so
// launches on different streams that overlap use different slots).
unsigned int* rms_bar_slot() {
  static unsigned int* base[64] = {};
  static std::atomic<unsigned> seq{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!base[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_rms_bar) != cudaSuccess) return nullptr;
    base[dev] = static_cast<unsigned int*>(ptr);
  }
  return base[dev] + 2 * (seq.fetch_add(1) % RB_BAR_SLOTS);
}

// Cooperative launch (every CTA resident at once, as the grid barrier needs),
// with programmatic stream serialization where the driver takes both.
template <typename... KArgs, typename... Args>
kl_status launch_coop(void (*kern)(KArgs...), int grid, cudaStream_t st, Args&&... args) {
  static bool with_pdl = true;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(RW_THREADS);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = with_pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e != cudaSuccess && with_pdl) {
    (void)cudaGetLastError();
    with_pdl = false;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  }
  if (e != cudaSuccess) return cuda_check(e, "rmsnorm_bwd cooperative launch");
  return KL_OK;
}

kl_status rms_bar_reset() {
  void* ptr = nullptr;
  KL_CUDA(cudaGetSymbolAddress(&ptr, g_rms_bar));
  KL_CUDA(cudaMemset(ptr, 0, sizeof(g_rms_bar)));
  return KL_OK;
}

kl_status rms_bar_abandon() {
  // one arrival counted in every slot, the barrier never completed (generations kept)
  unsigned int h[RB_BAR_SLOTS][2];
  KL_CUDA(cudaMemcpyFromSymbol(h, g_rms_bar, sizeof(h)));
  for (int s = 0; s < RB_BAR_SLOTS; ++s) h[s][0] = 1u;
  KL_CUDA(cudaMemcpyToSymbol(g_rms_bar, h, sizeof(h)));
  return KL_OK;
}

kl_status rmsnorm_bwd(int rows, int width, int dtype, const void* dh, int dh_dtype, const void* x,
                      const void* gamma, const float* rstd, const void* resid, void* dx,
                      float* dgamma, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (rows < 1 || width < 1 || !dh || !x || !gamma || !rstd || !dx || !dgamma)
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_bwd: bad arguments");
  if (width * sizeof(float) > 48 * 1024)
    return set_error(KL_ERR_UNSUPPORTED, "rmsnorm_bwd: width %d above 12288", width);
  if (!ws || ws_bytes < rmsnorm_bwd_ws(rows, width))
    return set_error(KL_ERR_NO_MEMORY, "rmsnorm_bwd: workspace too small");
  if (dtype != KL_BF16 && dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "rmsnorm_bwd: bad dtype %d", dtype);
  if (dtype == KL_F32 && dh_dtype != KL_F32)
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_bwd: fp32 mode needs fp32 dh");
  const int grid = rmsnorm_bwd_grid(rows);
  float* partial = static_cast<float*>(ws);
  const size_t es = dtype_size(dtype);
  const bool aligned = al16(dh) && al16(x) && al16(dx) && al16(gamma) && (!resid || al16(resid));
  // bf16 row form: fp32 dh, width a multiple of 8 up to 8192
  const int nc8 = (width / 8 + RW_THREADS - 1) / RW_THREADS;
  const bool row8_form = dtype == KL_BF16 && dh_dtype == KL_F32 && width % 8 == 0 && nc8 <= RW_MAXC && aligned;
  // generic row form: fp32 dh, width a multiple of 4 up to 8192, 16-byte aligned rows
  const bool rows_form = dh_dtype == KL_F32 && width % 4 == 0 && width <= 256 * 4 * RB_MAXC && aligned &&
                         (width * es) % 16 == 0;
  bool fused = false;
  {
    ProfScope ps("rmsnorm_bwd", st, 0.0,
                 1.0 * rows * width * (dtype_size(dh_dtype) + (resid ? 3.0 : 2.0) * es) + 4.0 * rows +
                     4.0 * grid * width);
    const size_t sm = width * sizeof(float);
    if (dtype == KL_BF16) {
      using T = __nv_bfloat16;
      if (row8_form) {
        // one cooperative launch: rows, partial dgamma rows, a grid barrier, the column sums
        fused = width % 4 == 0 && al16(dgamma);
        unsigned int* bar = fused ? rms_bar_slot() : nullptr;
        if (fused && !bar) fused = false;
        void (*kern)(int, int, const float*, const T*, const T*, const float*, const T*, T*, float*, float*,
                     unsigned int*, uint32_t*) = nullptr;
        switch (nc8) {
          case 1: kern = rmsnorm_bwd_row8_kernel<1>; break;
          case 2: kern = rmsnorm_bwd_row8_kernel<2>; break;
          case 3: kern = rmsnorm_bwd_row8_kernel<3>; break;
          default: kern = rmsnorm_bwd_row8_kernel<4>; break;
        }
        if (fused) {
          KL_TRY(launch_coop(kern, grid, st, rows, width, (const float*)dh, (const T*)x, (const T*)gamma, rstd,
                             (const T*)resid, (T*)dx, partial, dgamma, bar, device_error_word()));
        } else {
          launch_pdl(kern, grid, RW_THREADS, 0, st, rows, width, (const float*)dh, (const T*)x, (const T*)gamma, rstd,
                     (const T*)resid, (T*)dx, partial, static_cast<float*>(nullptr), static_cast<unsigned int*>(nullptr),
                     device_error_word());
        }
      } else if (rows_form)
        launch_pdl(rmsnorm_bwd_rows_kernel<T>, grid, 256, 0, st, rows, width, (const float*)dh, (const T*)x, (const T*)gamma, rstd, (const T*)resid, (T*)dx, partial);
      else if (dh_dtype == KL_F32)
        launch_pdl(rmsnorm_bwd_kernel<T, float>, grid, 256, sm, st, rows, width, (const float*)dh, (const T*)x, (const T*)gamma, rstd, (const T*)resid, (T*)dx, partial);
      else
        launch_pdl(rmsnorm_bwd_kernel<T, T>, grid, 256, sm, st, rows, width, (const T*)dh, (const T*)x, (const T*)gamma, rstd, (const T*)resid, (T*)dx, partial);
    } else {
      if (rows_form)
        launch_pdl(rmsnorm_bwd_rows_kernel<float>, grid, 256, 0, st, rows, width, (const float*)dh, (const float*)x, (const float*)gamma, rstd, (const float*)resid, (float*)dx, partial);
      else
        launch_pdl(rmsnorm_bwd_kernel<float, float>, grid, 256, sm, st, rows, width, (const float*)dh, (const float*)x, (const float*)gamma, rstd, (const float*)resid, (float*)dx, partial);
    }
  }
  KL_CUDA(cudaGetLastError());
  if (fused) return KL_OK;   // the column sums ran in the same launch
  ProfScope ps2("rmsnorm_bwd_colsum", st, 0.0, 4.0 * grid * width + 4.0 * width);
  if (width % 4 == 0 && al16(dgamma))
    launch_pdl(column_sum4_kernel, (width + 31) / 32, 256, 0, st, grid, width, partial, dgamma);
  else
    launch_pdl(column_sum_kernel, (width + 63) / 64, 256, 0, st, grid, width, partial, dgamma);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status rope_qk(int B, int S, int hq, int hk, int d, float base, int dtype, void* q, void* k,
                  int direction, cudaStream_t st) {
  if (B < 1 || S < 1 || hq < 0 || hk < 0 || hq + hk < 1 || d < 2 || (d & 1) || !q ||
      (hk > 0 && !k) || (direction != 1 && direction != -1))
    return set_error(KL_ERR_INVALID_ARG, "rope: bad arguments");
  if (dtype != KL_BF16 && dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "rope: bad dtype");
  if (d / 2 > ROPE_MAX_HALF) return set_error(KL_ERR_UNSUPPORTED, "rope: head dim %d above %d", d, 2 * ROPE_MAX_HALF);
  const int T = B * S;
  const float dir = static_cast<float>(direction);
  const RopeFreq f = rope_freq(d, base);
  const int V = dtype == KL_BF16 ? 8 : 4;
  const bool vec = (d / 2) % V == 0 && al16(q) && (hk == 0 || al16(k));
  ProfScope ps("rope", st, 0.0, 2.0 * T * (hq + hk) * d * dtype_size(dtype));
  if (vec) {
    if (dtype == KL_BF16)
      launch_pdl(rope_qk_kernel<__nv_bfloat16>, T, RQ_THREADS, 0, st, S, hq, hk, d, f, (__nv_bfloat16*)q, (__nv_bfloat16*)k, dir);
    else
      launch_pdl(rope_qk_kernel<float>, T, RQ_THREADS, 0, st, S, hq, hk, d, f, (float*)q, (float*)k, dir);
  } else {
    for (int w = 0; w < 2; ++w) {
      void* x = w == 0 ? q : k;
      const int heads = w == 0 ? hq : hk;
      if (heads == 0) continue;
      if (dtype == KL_BF16) launch_pdl(rope_kernel<__nv_bfloat16>, T, 128, 0, st, S, heads, d, f, (__nv_bfloat16*)x, dir);
      else launch_pdl(rope_kernel<float>, T, 128, 0, st, S, heads, d, f, (float*)x, dir);
    }
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status rope_cs_table(int S, int d, float base, float2* cs, cudaStream_t st) {
  if (S < 1 || d < 2 || (d & 1) || d / 2 > ROPE_MAX_HALF || !cs)
    return set_error(KL_ERR_INVALID_ARG, "rope table: bad arguments");
  const RopeFreq f = rope_freq(d, base);
  const int64_t n = static_cast<int64_t>(S) * (d / 2);
  ProfScope ps("rope_table", st, 0.0, 8.0 * n);
  launch_pdl(rope_cs_kernel, ew_grid(n), 256, 0, st, S, d / 2, f, cs);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status rope(int B, int S, int heads, int d, float base, int dtype, void* x, int direction,
               cudaStream_t st) {
  return rope_qk(B, S, heads, 0, d, base, dtype, x, nullptr, direction, st);
}

kl_status rope_bwd_convert(int B, int S, int hq, int hk, int d, float base, int dtype,
                           const float* dq_acc, const float* dk_acc, const float* dv_acc, void* dq,
                           void* dk, void* dv, cudaStream_t st) {
  if (d % 8) return set_error(KL_ERR_UNSUPPORTED, "rope backward: head dim %d not a multiple of 8", d);
  if (d / 2 > ROPE_MAX_HALF) return set_error(KL_ERR_UNSUPPORTED, "rope backward: head dim %d above %d", d, 2 * ROPE_MAX_HALF);
  const int T = B * S;
  const RopeFreq f = rope_freq(d, base);
  ProfScope ps("rope_bwd_convert", st, 0.0, 1.0 * T * (hq + 2 * hk) * d * (4 + dtype_size(dtype)));
  if (dtype == KL_BF16)
    launch_pdl(rope_bwd_convert_kernel<__nv_bfloat16>, T, RC_THREADS, 0, st, S, hq, hk, d, f, dq_acc, dk_acc, dv_acc,
                                                                     (__nv_bfloat16*)dq, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv);
  else
    launch_pdl(rope_bwd_convert_kernel<float>, T, RC_THREADS, 0, st, S, hq, hk, d, f, dq_acc, dk_acc, dv_acc, (float*)dq,
                                                             (float*)dk, (float*)dv);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

int qk_bwd_grid(int rows) {
  const int want = (rows + 7) / 8, cap = 2 * num_sms();
  return want < cap ? want : cap;
}

size_t qk_rope_bwd_ws(int rows, int d) { return align_up(static_cast<size_t>(qk_bwd_grid(rows)) * d * 4, 256); }

kl_status qk_rope_fwd(int T, int heads, int S, int d, int dtype, const void* pre, const void* gamma, float eps,
                      int norm, int inter, float base, const float2* tab, void* out, float* rstd, cudaStream_t st,
                      const int32_t* pos_off) {
  if (T < 1 || heads < 1 || d < 2 || (d & 1) || d / 2 > ROPE_MAX_HALF || !pre || !out || (norm && (!gamma || !rstd)) ||
      (pos_off && tab))
    return set_error(KL_ERR_INVALID_ARG, "q/k rotary: bad arguments");
  const int rows = T * heads;
  const RopeFreq f = rope_freq(d, base);
  ProfScope ps("qk_rope_fwd", st, 0.0, 2.0 * rows * d * dtype_size(dtype));
  const int grid = (rows + 7) / 8;
  if (dtype == KL_BF16)
    launch_pdl(qk_rope_fwd_kernel<__nv_bfloat16>, grid, 256, 0, st, rows, heads, S, d, (const __nv_bfloat16*)pre,
                                                           (const __nv_bfloat16*)gamma, eps, norm, inter, f, tab,
                                                           (__nv_bfloat16*)out, rstd, pos_off);
  else
    launch_pdl(qk_rope_fwd_kernel<float>, grid, 256, 0, st, rows, heads, S, d, (const float*)pre, (const float*)gamma, eps,
                                                   norm, inter, f, tab, (float*)out, rstd, pos_off);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status paged_qkv_rope(const kl_paged_cfg& pc, int Hq, int Hkv, int d, const void* q_pre, const void* k_pre,
                         const void* v, const void* gamma_q, const void* gamma_k, float eps, int norm, int inter,
                         float base, const int32_t* table, const int32_t* ctx, void* q_out, void* k_pool, void* v_pool,
                         cudaStream_t st) {
  if (d != 128 || !q_pre || !k_pre || !v || !table || !ctx || !q_out || !k_pool || !v_pool ||
      (norm && (!gamma_q || !gamma_k)))
    return set_error(KL_ERR_INVALID_ARG, "paged q/k/v rotation: bad arguments");
  const int T = pc.B * pc.n_new, rows = T * (Hq + Hkv);
  const RopeFreq f = rope_freq(d, base);
  ProfScope ps("paged_qkv_rope", st, 0.0, 2.0 * 2 * T * (Hq + 2 * Hkv) * d);
  launch_pdl(paged_qkv_rope_kernel, (rows + 7) / 8, 256, 0, st, T, pc.n_new, Hq, Hkv, d,
             static_cast<const __nv_bfloat16*>(q_pre), static_cast<const __nv_bfloat16*>(k_pre),
             static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(gamma_q),
             static_cast<const __nv_bfloat16*>(gamma_k), eps, norm, inter, f, table, ctx, pc.block_size,
             pc.max_blocks, pc.n_blocks, static_cast<__nv_bfloat16*>(q_out), static_cast<__nv_bfloat16*>(k_pool),
             static_cast<__nv_bfloat16*>(v_pool), device_error_word());
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status qk_rope_bwd(int T, int heads, int S, int d, int dtype, const void* dyr, int dy_dtype, const void* pre,
                      const void* gamma, const float* rstd, int norm, int inter, float base, const float2* tab,
                      void* dx, float* dgamma, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (T < 1 || heads < 1 || d < 2 || (d & 1) || d / 2 > ROPE_MAX_HALF || d > 256 || !dyr || !dx ||
      (norm && (!pre || !gamma || !rstd || !dgamma)))
    return set_error(KL_ERR_INVALID_ARG, "q/k rotary backward: bad arguments");
  const int rows = T * heads;
  if (norm && (!ws || ws_bytes < qk_rope_bwd_ws(rows, d)))
    return set_error(KL_ERR_NO_MEMORY, "q/k rotary backward: workspace too small");
  const RopeFreq f = rope_freq(d, base);
  const int grid = qk_bwd_grid(rows);
  float* partial = static_cast<float*>(ws);
  {
    ProfScope ps("qk_rope_bwd", st, 0.0, 1.0 * rows * d * (dtype_size(dy_dtype) + (norm ? 2.0 : 1.0) * dtype_size(dtype)));
#define KL_QKB(T_, TD_)                                                                                         \
  launch_pdl(qk_rope_bwd_kernel<T_, TD_>, grid, 256, 0, st, rows, heads, S, d, (const TD_*)dyr, 1.0f, (const T_*)pre,  \
                                                    (const T_*)gamma, rstd, norm, inter, f, tab, (T_*)dx, partial)
    if (dtype == KL_BF16) {
      if (dy_dtype == KL_BF16) KL_QKB(__nv_bfloat16, __nv_bfloat16);
      else KL_QKB(__nv_bfloat16, float);
    } else {
      KL_QKB(float, float);
    }
#undef KL_QKB
  }
  KL_CUDA(cudaGetLastError());
  if (norm) {
    ProfScope ps2("qk_rope_bwd_colsum", st, 0.0, 4.0 * grid * d);
    launch_pdl(column_sum_kernel, (d + 63) / 64, 256, 0, st, grid, d, partial, dgamma);
    KL_CUDA(cudaGetLastError());
  }
  return KL_OK;
}

kl_status convert_f32(int64_t n, int dtype, const float* src, void* dst, cudaStream_t st) {
  ProfScope ps("convert_f32", st, 0.0, 1.0 * n * (4 + dtype_size(dtype)));
  if (dtype == KL_BF16) launch_pdl(convert_kernel<__nv_bfloat16>, ew_grid(n), 256, 0, st, n, src, (__nv_bfloat16*)dst);
  else launch_pdl(convert_kernel<float>, ew_grid(n), 256, 0, st, n, src, (float*)dst);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status swiglu_fwd(int64_t n, int dtype, const void* g, const void* u, void* m, cudaStream_t st) {
  if (n < 1 || !g || !u || !m) return set_error(KL_ERR_INVALID_ARG, "swiglu_fwd: bad arguments");
  ProfScope ps("swiglu_fwd", st, 0.0, 3.0 * n * dtype_size(dtype));
  if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    if (n % 8 == 0 && al16(g) && al16(u) && al16(m))
      launch_pdl(swiglu_fwd_kernel<T, true>, ew_grid(n / 8), 256, 0, st, n, (const T*)g, (const T*)u, (T*)m);
    else
      launch_pdl(swiglu_fwd_kernel<T, false>, ew_grid(n), 256, 0, st, n, (const T*)g, (const T*)u, (T*)m);
  } else if (dtype == KL_F32) {
    if (n % 4 == 0 && al16(g) && al16(u) && al16(m))
      launch_pdl(swiglu_fwd_kernel<float, true>, ew_grid(n / 4), 256, 0, st, n, (const float*)g, (const float*)u, (float*)m);
    else
      launch_pdl(swiglu_fwd_kernel<float, false>, ew_grid(n), 256, 0, st, n, (const float*)g, (const float*)u, (float*)m);
  } else {
    return set_error(KL_ERR_INVALID_ARG, "swiglu_fwd: bad dtype");
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status swiglu_bwd(int64_t n, int dtype, const void* dm, const void* g, const void* u, void* dg,
                     void* du, cudaStream_t st) {
  if (n < 1 || !dm || !g || !u || !dg || !du) return set_error(KL_ERR_INVALID_ARG, "swiglu_bwd: bad arguments");
  ProfScope ps("swiglu_bwd", st, 0.0, 5.0 * n * dtype_size(dtype));
  if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    if (n % 8 == 0 && al16(dm) && al16(g) && al16(u) && al16(dg) && al16(du))
      launch_pdl(swiglu_bwd_kernel<T, true>, ew_grid(n / 8), 256, 0, st, n, (const T*)dm, (const T*)g, (const T*)u, (T*)dg, (T*)du);
    else
      launch_pdl(swiglu_bwd_kernel<T, false>, ew_grid(n), 256, 0, st, n, (const T*)dm, (const T*)g, (const T*)u, (T*)dg, (T*)du);
  } else if (dtype == KL_F32) {
    if (n % 4 == 0 && al16(dm) && al16(g) && al16(u) && al16(dg) && al16(du))
      launch_pdl(swiglu_bwd_kernel<float, true>, ew_grid(n / 4), 256, 0, st, n, (const float*)dm, (const float*)g, (const float*)u, (float*)dg, (float*)du);
    else
      launch_pdl(swiglu_bwd_kernel<float, false>, ew_grid(n), 256, 0, st, n, (const float*)dm, (const float*)g, (const float*)u, (float*)dg, (float*)du);
  } else {
    return set_error(KL_ERR_INVALID_ARG, "swiglu_bwd: bad dtype");
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
