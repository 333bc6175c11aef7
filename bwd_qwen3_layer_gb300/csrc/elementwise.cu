// Normalisation, rotary and activation kernels of the layer ("From-scratch
// GPU LLM training", capability list: RMSNorm, SiLU / SwiGLU and RoPE
// gradient kernels; "KYNETRA FOUNDRY", pre-norm decoder and rotary
// paragraphs). All of them are HBM-bound: 128-bit loads and stores where the
// widths allow, fp32 arithmetic, warp-shuffle row reductions.
#include <math.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
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
// RMSNorm forward: one warp per row.
// ---------------------------------------------------------------------------
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(int rows, int width,
                                                          const T* __restrict__ x,
                                                          const T* __restrict__ gamma, float eps,
                                                          T* __restrict__ h,
                                                          float* __restrict__ rstd) {
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

// ---------------------------------------------------------------------------
// RMSNorm backward: one warp per row; the gain gradient is accumulated per
// CTA in shared memory and written as a partial row, reduced afterwards.
//   n = x*rstd, dn = dh*gamma, dx = resid + rstd*(dn - n*mean(dn*n)),
//   dgamma += dh*n.
// ---------------------------------------------------------------------------
template <typename T, typename TD>
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(
    int rows, int width, const TD* __restrict__ dh, const T* __restrict__ x,
    const T* __restrict__ gamma, const float* __restrict__ rstd, const T* __restrict__ resid,
    T* __restrict__ dx, float* __restrict__ partial) {
  extern __shared__ float sacc[];
  for (int j = threadIdx.x; j < width; j += blockDim.x) sacc[j] = 0.f;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_w = 1.0f / static_cast<float>(width);
  for (int row = blockIdx.x * 8 + warp; row < rows; row += gridDim.x * 8) {
    const int64_t off = static_cast<int64_t>(row) * width;
    const float r = rstd[row];
    float dot = 0.f;
    for (int j = lane; j < width; j += 32) {
      const float n = ld_f(x + off + j) * r;
      const float g = ld_f(dh + off + j);
      dot = fmaf(g * ld_f(gamma + j), n, dot);
    }
    dot = warp_sum(dot) * inv_w;
    for (int j = lane; j < width; j += 32) {
      const float n = ld_f(x + off + j) * r;
      const float g = ld_f(dh + off + j);
      const float dn = g * ld_f(gamma + j);
      float v = r * (dn - n * dot);
      if (resid) v += ld_f(resid + off + j);
      st_f(dx + off + j, v);
      atomicAdd(&sacc[j], g * n);
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < width; j += blockDim.x)
    partial[static_cast<int64_t>(blockIdx.x) * width + j] = sacc[j];
}

__global__ void column_sum_kernel(int nrows, int width, const float* __restrict__ partial,
                                  float* __restrict__ out) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= width) return;
  float s = 0.f;
  for (int r = 0; r < nrows; ++r) s += partial[static_cast<int64_t>(r) * width + j];
  out[j] = s;
}

int rmsnorm_bwd_grid(int rows) {
  const int want = (rows + 7) / 8;
  const int cap = 2 * num_sms();
  return want < cap ? want : cap;
}

// ---------------------------------------------------------------------------
// RoPE: one CTA per token. The plane angles s * base^(-2i/d) are formed and
// reduced in fp64 (exact enough at any position), cos/sin rounded to fp32
// and kept in shared memory; every head of the token then uses them.
// Plane i pairs element i with element i + d/2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rope_table(int s, int d, float base, float dir, float* cs) {
  const int half = d / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double inv = pow(static_cast<double>(base), -2.0 * i / d);
    double sn, c;
    sincos(static_cast<double>(s) * inv, &sn, &c);
    cs[i] = static_cast<float>(c);
    cs[half + i] = dir * static_cast<float>(sn);
  }
  __syncthreads();
}

template <typename T>
__global__ void rope_kernel(int S, int heads, int d, float base, T* __restrict__ x, float dir) {
  extern __shared__ float cs[];
  const int t = blockIdx.x;
  rope_table(t % S, d, base, dir, cs);
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

template <typename T>
__global__ void rope_bwd_f32_kernel(int S, int heads, int d, float base,
                                    const float* __restrict__ src, T* __restrict__ dst) {
  extern __shared__ float cs[];
  const int t = blockIdx.x;
  rope_table(t % S, d, base, -1.0f, cs);
  const int half = d / 2;
  const int64_t off = static_cast<int64_t>(t) * heads * d;
  for (int idx = threadIdx.x; idx < heads * half; idx += blockDim.x) {
    const int hh = idx / half, i = idx - hh * half;
    const float a = src[off + hh * d + i], b = src[off + hh * d + half + i];
    const float c = cs[i], sn = cs[half + i];
    st_f(dst + off + hh * d + i, a * c - b * sn);
    st_f(dst + off + hh * d + half + i, a * sn + b * c);
  }
}

template <typename T>
__global__ void convert_kernel(int64_t n, const float* __restrict__ src, T* __restrict__ dst) {
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
                      void* h, float* rstd, cudaStream_t st) {
  if (rows < 1 || width < 1 || !x || !gamma || !h || !rstd)
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_fwd: bad arguments");
  const int grid = (rows + 7) / 8;
  ProfScope ps("rmsnorm_fwd", st, 0.0,
               2.0 * rows * width * dtype_size(dtype) + 4.0 * rows + 1.0 * width * dtype_size(dtype));
  if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    const bool vec = width % 8 == 0 && al16(x) && al16(gamma) && al16(h);
    if (vec) rmsnorm_fwd_kernel<T, true><<<grid, 256, 0, st>>>(rows, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd);
    else rmsnorm_fwd_kernel<T, false><<<grid, 256, 0, st>>>(rows, width, (const T*)x, (const T*)gamma, eps, (T*)h, rstd);
  } else if (dtype == KL_F32) {
    const bool vec = width % 4 == 0 && al16(x) && al16(gamma) && al16(h);
    if (vec) rmsnorm_fwd_kernel<float, true><<<grid, 256, 0, st>>>(rows, width, (const float*)x, (const float*)gamma, eps, (float*)h, rstd);
    else rmsnorm_fwd_kernel<float, false><<<grid, 256, 0, st>>>(rows, width, (const float*)x, (const float*)gamma, eps, (float*)h, rstd);
  } else {
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_fwd: bad dtype %d", dtype);
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

size_t rmsnorm_bwd_ws(int rows, int width) {
  return align_up(static_cast<size_t>(rmsnorm_bwd_grid(rows)) * width * sizeof(float), 256);
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
  const int grid = rmsnorm_bwd_grid(rows);
  float* partial = static_cast<float*>(ws);
  const size_t sm = width * sizeof(float);
  {
  ProfScope ps("rmsnorm_bwd", st, 0.0,
               1.0 * rows * width * (dtype_size(dh_dtype) + (resid ? 3.0 : 2.0) * dtype_size(dtype)) +
                   4.0 * rows + 4.0 * grid * width);
  if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    if (dh_dtype == KL_F32)
      rmsnorm_bwd_kernel<T, float><<<grid, 256, sm, st>>>(rows, width, (const float*)dh, (const T*)x, (const T*)gamma, rstd, (const T*)resid, (T*)dx, partial);
    else
      rmsnorm_bwd_kernel<T, T><<<grid, 256, sm, st>>>(rows, width, (const T*)dh, (const T*)x, (const T*)gamma, rstd, (const T*)resid, (T*)dx, partial);
  } else if (dtype == KL_F32) {
    if (dh_dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "rmsnorm_bwd: fp32 mode needs fp32 dh");
    rmsnorm_bwd_kernel<float, float><<<grid, 256, sm, st>>>(rows, width, (const float*)dh, (const float*)x, (const float*)gamma, rstd, (const float*)resid, (float*)dx, partial);
  } else {
    return set_error(KL_ERR_INVALID_ARG, "rmsnorm_bwd: bad dtype %d", dtype);
  }
  }
  KL_CUDA(cudaGetLastError());
  ProfScope ps2("rmsnorm_bwd_colsum", st, 0.0, 4.0 * grid * width + 4.0 * width);
  column_sum_kernel<<<(width + 255) / 256, 256, 0, st>>>(grid, width, partial, dgamma);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status rope(int B, int S, int heads, int d, float base, int dtype, void* x, int direction,
               cudaStream_t st) {
  if (B < 1 || S < 1 || heads < 1 || d < 2 || (d & 1) || !x || (direction != 1 && direction != -1))
    return set_error(KL_ERR_INVALID_ARG, "rope: bad arguments");
  const int T = B * S;
  const size_t sm = d * sizeof(float);
  const float dir = static_cast<float>(direction);
  ProfScope ps("rope", st, 0.0, 2.0 * T * heads * d * dtype_size(dtype));
  if (dtype == KL_BF16) rope_kernel<__nv_bfloat16><<<T, 128, sm, st>>>(S, heads, d, base, (__nv_bfloat16*)x, dir);
  else if (dtype == KL_F32) rope_kernel<float><<<T, 128, sm, st>>>(S, heads, d, base, (float*)x, dir);
  else return set_error(KL_ERR_INVALID_ARG, "rope: bad dtype");
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status rope_bwd_from_f32(int B, int S, int heads, int d, float base, int dtype,
                            const float* src, void* dst, cudaStream_t st) {
  const int T = B * S;
  const size_t sm = d * sizeof(float);
  ProfScope ps("rope_bwd_f32", st, 0.0, 1.0 * T * heads * d * (4 + dtype_size(dtype)));
  if (dtype == KL_BF16) rope_bwd_f32_kernel<__nv_bfloat16><<<T, 128, sm, st>>>(S, heads, d, base, src, (__nv_bfloat16*)dst);
  else rope_bwd_f32_kernel<float><<<T, 128, sm, st>>>(S, heads, d, base, src, (float*)dst);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status convert_f32(int64_t n, int dtype, const float* src, void* dst, cudaStream_t st) {
  ProfScope ps("convert_f32", st, 0.0, 1.0 * n * (4 + dtype_size(dtype)));
  if (dtype == KL_BF16) convert_kernel<__nv_bfloat16><<<ew_grid(n), 256, 0, st>>>(n, src, (__nv_bfloat16*)dst);
  else convert_kernel<float><<<ew_grid(n), 256, 0, st>>>(n, src, (float*)dst);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status swiglu_fwd(int64_t n, int dtype, const void* g, const void* u, void* m, cudaStream_t st) {
  if (n < 1 || !g || !u || !m) return set_error(KL_ERR_INVALID_ARG, "swiglu_fwd: bad arguments");
  ProfScope ps("swiglu_fwd", st, 0.0, 3.0 * n * dtype_size(dtype));
  if (dtype == KL_BF16) {
    using T = __nv_bfloat16;
    if (n % 8 == 0 && al16(g) && al16(u) && al16(m))
      swiglu_fwd_kernel<T, true><<<ew_grid(n / 8), 256, 0, st>>>(n, (const T*)g, (const T*)u, (T*)m);
    else
      swiglu_fwd_kernel<T, false><<<ew_grid(n), 256, 0, st>>>(n, (const T*)g, (const T*)u, (T*)m);
  } else if (dtype == KL_F32) {
    if (n % 4 == 0 && al16(g) && al16(u) && al16(m))
      swiglu_fwd_kernel<float, true><<<ew_grid(n / 4), 256, 0, st>>>(n, (const float*)g, (const float*)u, (float*)m);
    else
      swiglu_fwd_kernel<float, false><<<ew_grid(n), 256, 0, st>>>(n, (const float*)g, (const float*)u, (float*)m);
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
      swiglu_bwd_kernel<T, true><<<ew_grid(n / 8), 256, 0, st>>>(n, (const T*)dm, (const T*)g, (const T*)u, (T*)dg, (T*)du);
    else
      swiglu_bwd_kernel<T, false><<<ew_grid(n), 256, 0, st>>>(n, (const T*)dm, (const T*)g, (const T*)u, (T*)dg, (T*)du);
  } else if (dtype == KL_F32) {
    if (n % 4 == 0 && al16(dm) && al16(g) && al16(u) && al16(dg) && al16(du))
      swiglu_bwd_kernel<float, true><<<ew_grid(n / 4), 256, 0, st>>>(n, (const float*)dm, (const float*)g, (const float*)u, (float*)dg, (float*)du);
    else
      swiglu_bwd_kernel<float, false><<<ew_grid(n), 256, 0, st>>>(n, (const float*)dm, (const float*)g, (const float*)u, (float*)dg, (float*)du);
  } else {
    return set_error(KL_ERR_INVALID_ARG, "swiglu_bwd: bad dtype");
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
