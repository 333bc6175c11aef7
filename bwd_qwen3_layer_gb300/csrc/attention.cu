// Causal grouped-query scaled-dot-product attention, forward and backward
// ("From-scratch GPU LLM training", capability list: scaled-dot-product
// attention gradient kernel; "KYNETRA FOUNDRY", tiled-attention paragraph:
// query tiles stream over key/value tiles with a running max and running
// sum, the score matrix never reaches HBM, the backward recomputes the tiles;
// grouped-query paragraph: one key/value head per contiguous query-head group).
//
// bf16 path (d = 128): the tcgen05 kernels of attention_tc.cu (forward; dK/dV
// and dQ backward kernels); this file holds their host entry points, the
// workspace layout (D, fp32 dQ/dK/dV accumulators) and the D = rowsum(dO * O)
// pre-pass used when the caller has not produced D already.
// fp32 path: one warp per (row, head), plain loops, any head dim <= 256.
#include <math.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {


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
  pdl_enter();
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
  pdl_enter();
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
  pdl_enter();
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
// bf16: the D pre-pass (the tcgen05 kernels are in attention_tc.cu)
// ===========================================================================
constexpr int HD = 128;      // head dim
// D[b,h,s] = sum_c dO[t,h,c] * O[t,h,c] (fp32), one warp per (token, head).
__global__ void __launch_bounds__(256) attn_bwd_pre_bf16_kernel(int B, int S, int Hq,
                                                                const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dout,
                                                                float* __restrict__ Dd) {
  pdl_enter();
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

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
    launch_pdl(attn_fwd_f32_kernel, static_cast<unsigned>((rows + 7) / 8), 256, 0, st,
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
                              bool d_ready, void* dq_out, const float2* rope_cs, void* dk_out,
                              void* dv_out) {
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
    launch_pdl(attn_bwd_dq_f32_kernel, static_cast<unsigned>((rows + 7) / 8), 256, 0, st,
        B, S, Hq, Hkv, d, (const float*)q, (const float*)k, (const float*)v, (const float*)o, lse,
        (const float*)dout, Dd, dq, scale);
    KL_CUDA(cudaGetLastError());
    const int64_t krows = static_cast<int64_t>(T) * Hkv;
    launch_pdl(attn_bwd_dkdv_f32_kernel, static_cast<unsigned>((krows + 7) / 8), 256, 0, st,
        B, S, Hq, Hkv, d, (const float*)q, (const float*)k, (const float*)v, lse,
        (const float*)dout, Dd, dk, dv, scale);
  } else {
    if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || !al16(dout))
      return set_error(KL_ERR_INVALID_ARG, "attention_bwd: bf16 buffers must be 16-byte aligned");
    if (!dq_out || !dk_out || !dv_out) return set_error(KL_ERR_INVALID_ARG, "attention_bwd: null output");
    const int64_t rows = static_cast<int64_t>(T) * Hq;
    if (!d_ready) {
      ProfScope ps("attn_bwd_pre_bf16", st, 0.0, 4.0 * T * Hq * d + 4.0 * T * Hq);
      launch_pdl(attn_bwd_pre_bf16_kernel, static_cast<unsigned>((rows + 7) / 8), 256, 0, st,
          B, S, Hq, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, Dd);
      KL_CUDA(cudaGetLastError());
    }
    if (!al16(dq_out)) return set_error(KL_ERR_INVALID_ARG, "attention_bwd: dq not 16-byte aligned");
    KL_TRY(attention_bwd_tc(B, S, Hq, Hkv, q, k, v, dout, lse, Dd, nullptr, dq_out, dk_out, dv_out, rope_cs, st));
    *dq_acc = *dk_acc = *dv_acc = nullptr;
  }
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl
