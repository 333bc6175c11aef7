// Forward path with a paged key/value cache ("From-scratch GPU LLM training",
// "What is built": a GPU forward path with a paged key-value cache; "KYNETRA
// FOUNDRY", paged-KV paragraph: each sequence's cache is cut into fixed-size
// token blocks living anywhere in a global pool, a per-sequence block table
// maps logical positions to physical blocks, and attention gathers keys and
// values through it).
//
// Layout: a pool is [n_blocks][block_size][Hkv * d]; token position p of
// sequence b lives in block table[b][p / block_size], slot p % block_size. A
// step feeds n_new tokens to each of B sequences; sequence b already holds
// ctx[b] tokens, new token i sits at absolute position ctx[b] + i.
//
//   paged_kv_write_kernel  one warp per (new token, kv head): its key and value
//                          rows into their slots.
//   paged_attn_kernel      decode attention, HBM-bound: one CTA per (kv head,
//                          sequence, context split) takes all query rows of the
//                          head group (G heads x n_new tokens, at most 64),
//                          gathers 64-token K/V tiles through the block table
//                          into a cp.async double buffer, and keeps a base-2
//                          online softmax per row (warp = rows, lane = 2 keys
//                          for the scores and 4 of the 128 dims for P V).
//   paged_combine_kernel   merges the splits' (max, sum, O) when the context
//                          is split (few sequences).
#include <math.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int PA_THREADS = 256;
constexpr int PA_KT = 64;       // keys per tile
constexpr int PA_D = 128;       // head dim
constexpr int PA_RMAX = 64;     // query rows per CTA
constexpr int PA_RPW = PA_RMAX / (PA_THREADS / 32);   // rows per warp at most
constexpr float PA_LN2 = 0.6931471805599453f;
constexpr float PA_LOG2E = 1.4426950408889634f;

struct PagedParams {
  const __nv_bfloat16* q;     // [B*n_new, Hq*d]
  const __nv_bfloat16* kp;    // [n_blocks][bs][Hkv*d]
  const __nv_bfloat16* vp;
  const int32_t* table;       // [B][max_blocks]
  const int32_t* ctx;         // [B]
  __nv_bfloat16* o;           // [B*n_new, Hq*d] (one split)
  float* lse;                 // [B, Hq, n_new] natural log, or null (one split)
  float* part_o;              // [nsplit][B*n_new][Hq][d] unnormalised (several splits)
  float* part_ml;             // [nsplit][B*n_new][Hq][2] (max in log2 units, sum)
  int B, n_new, Hq, Hkv, bs, max_blocks, n_blocks, nsplit, tiles_per_split;
  float scale_log2;           // log2(e) / sqrt(d)
  uint32_t* err;              // device error word: a position past the table or a block outside the pool
};

// The physical block of position pos of sequence b, or -1 (and the error bit)
// if the position is past the table or the table entry outside the pool.
__device__ __forceinline__ int pa_block(const int32_t* table, int b, int pos, int bs, int max_blocks, int n_blocks,
                                        uint32_t* err) {
  const int lb = pos / bs;
  const int blk = lb < max_blocks ? table[b * max_blocks + lb] : -1;
  if (blk < 0 || blk >= n_blocks) {
    record_error(err, KL_DEVERR_PAGE);
    return -1;
  }
  return blk;
}

__device__ __forceinline__ void pa_cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;   // zero-fill when the token is outside the context
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void pa_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void pa_cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void pa_unpack8(const uint4& a, float (&f)[8]) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ float pa_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float pa_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256) paged_kv_write_kernel(int rows, int n_new, int Hkv, int bs, int max_blocks,
                                                             int n_blocks, uint32_t* err,
                                                             const __nv_bfloat16* __restrict__ k_new,
                                                             const __nv_bfloat16* __restrict__ v_new,
                                                             const int32_t* __restrict__ table,
                                                             const int32_t* __restrict__ ctx,
                                                             __nv_bfloat16* __restrict__ kp,
                                                             __nv_bfloat16* __restrict__ vp) {
  pdl_enter();
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= rows * Hkv) return;
  const int t = w / Hkv, g = w - t * Hkv;          // new token row, kv head
  const int b = t / n_new, pos = ctx[b] + (t - b * n_new);
  const int blk = pos >= 0 ? pa_block(table, b, pos, bs, max_blocks, n_blocks, err) : -1;
  if (blk < 0) return;
  const int64_t dst = ((static_cast<int64_t>(blk) * bs + pos % bs) * Hkv + g) * PA_D + lane * 4;
  const int64_t src = (static_cast<int64_t>(t) * Hkv + g) * PA_D + lane * 4;
  *reinterpret_cast<uint2*>(kp + dst) = *reinterpret_cast<const uint2*>(k_new + src);
  *reinterpret_cast<uint2*>(vp + dst) = *reinterpret_cast<const uint2*>(v_new + src);
}

__global__ void __launch_bounds__(PA_THREADS) paged_attn_kernel(const __grid_constant__ PagedParams p) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t pa_smem[];
  const int G = p.Hq / p.Hkv, R = G * p.n_new;
  __nv_bfloat16* kt = reinterpret_cast<__nv_bfloat16*>(pa_smem);            // [2][KT][D]
  __nv_bfloat16* vt = kt + 2 * PA_KT * PA_D;                                 // [2][KT][D]
  float* qs = reinterpret_cast<float*>(pa_smem + 4 * PA_KT * PA_D * 2);      // [R][D], pre-scaled
  const int g = blockIdx.x, b = blockIdx.y, sp = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ctxb = max(0, p.ctx[b]);
  const int L = ctxb + p.n_new;                                              // keys of this sequence
  const int ntiles = (L + PA_KT - 1) / PA_KT;
  const int t0 = sp * p.tiles_per_split;
  const int t1 = min(ntiles, t0 + p.tiles_per_split);
  const int nrow = (R - warp + 7) / 8;         // this warp's rows: r = warp + 8 k, k < nrow

  // tile t: key positions t*KT .. t*KT + KT - 1 (those < L), gathered through the table
  auto load_tile = [&](int t, int buf) {
    for (int e = threadIdx.x; e < PA_KT * 16; e += PA_THREADS) {
      const int j = e >> 4, ch = e & 15;
      const int pos = t * PA_KT + j;
      int blk = pos < L ? pa_block(p.table, b, pos, p.bs, p.max_blocks, p.n_blocks, p.err) : -1;
      const bool ok = blk >= 0;
      if (!ok) blk = 0;   // zero-filled from a valid address
      const int64_t row = (static_cast<int64_t>(blk) * p.bs + (ok ? pos % p.bs : 0)) * p.Hkv + g;
      pa_cp_async16(smem_u32(kt + (buf * PA_KT + j) * PA_D + ch * 8), p.kp + row * PA_D + ch * 8, ok);
      pa_cp_async16(smem_u32(vt + (buf * PA_KT + j) * PA_D + ch * 8), p.vp + row * PA_D + ch * 8, ok);
    }
    pa_cp_commit();
  };
  if (t0 < t1) load_tile(t0, 0);
  // query rows r = i * G + gg (token i, head g*G + gg), scaled by log2(e)/sqrt(d)
  for (int e = threadIdx.x; e < R * (PA_D / 8); e += PA_THREADS) {
    const int r = e / (PA_D / 8), c = e % (PA_D / 8);
    const int i = r / G, gg = r - i * G;
    float f[8];
    pa_unpack8(*reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b * p.n_new + i) * p.Hq + g * G + gg) *
                                                         PA_D + c * 8), f);
#pragma unroll
    for (int x = 0; x < 8; ++x) qs[r * PA_D + c * 8 + x] = f[x] * p.scale_log2;
  }

  float m_r[PA_RPW], l_r[PA_RPW], acc[PA_RPW][4];
#pragma unroll
  for (int k = 0; k < PA_RPW; ++k) {
    m_r[k] = -INFINITY;
    l_r[k] = 0.f;
    acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
  }
  for (int t = t0; t < t1; ++t) {
    const int buf = (t - t0) & 1;
    __syncthreads();                            // every warp is done with the other buffer
    if (t + 1 < t1) {
      load_tile(t + 1, buf ^ 1);
      pa_cp_wait<1>();
    } else {
      pa_cp_wait<0>();
    }
    __syncthreads();                            // tile t (and the query rows) visible to all
    const __nv_bfloat16* kb = kt + buf * PA_KT * PA_D;
    const __nv_bfloat16* vb = vt + buf * PA_KT * PA_D;
    // scores of keys lane and lane + 32 for this warp's rows; 16-byte chunks
    // visited in a lane-rotated order so the lanes spread over the banks
    float s[PA_RPW][2];
#pragma unroll
    for (int k = 0; k < PA_RPW; ++k) s[k][0] = s[k][1] = 0.f;
#pragma unroll 4
    for (int c = 0; c < PA_D / 8; ++c) {
      const int ch = (c + lane) & (PA_D / 8 - 1);
      float k0[8], k1[8];
      pa_unpack8(*reinterpret_cast<const uint4*>(kb + lane * PA_D + ch * 8), k0);
      pa_unpack8(*reinterpret_cast<const uint4*>(kb + (lane + 32) * PA_D + ch * 8), k1);
#pragma unroll
      for (int k = 0; k < PA_RPW; ++k) {
        if (k < nrow) {
          const float* qr = qs + (warp + 8 * k) * PA_D + ch * 8;
          const float4 qa = *reinterpret_cast<const float4*>(qr);
          const float4 qb = *reinterpret_cast<const float4*>(qr + 4);
          const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            s[k][0] = fmaf(qv[x], k0[x], s[k][0]);
            s[k][1] = fmaf(qv[x], k1[x], s[k][1]);
          }
        }
      }
    }
    // causal limit by absolute position, online softmax (base 2)
    float pr[PA_RPW][2];
#pragma unroll
    for (int k = 0; k < PA_RPW; ++k) {
      pr[k][0] = pr[k][1] = 0.f;
      if (k < nrow) {
        const int r = warp + 8 * k, qp = ctxb + r / G;
        const int kp0 = t * PA_KT + lane;
        const float a0 = kp0 <= qp ? s[k][0] : -INFINITY;
        const float a1 = kp0 + 32 <= qp ? s[k][1] : -INFINITY;
        const float mt = pa_warp_max(fmaxf(a0, a1));
        const float mn = fmaxf(m_r[k], mt);
        if (mn > -INFINITY) {                   // else nothing of this row is visible yet
          const float alpha = exp2f(m_r[k] - mn);
          pr[k][0] = exp2f(a0 - mn);
          pr[k][1] = exp2f(a1 - mn);
          l_r[k] = l_r[k] * alpha + pa_warp_sum(pr[k][0] + pr[k][1]);
#pragma unroll
          for (int x = 0; x < 4; ++x) acc[k][x] *= alpha;
          m_r[k] = mn;
        }
      }
    }
    // O += P V: lane owns dims 4*lane .. 4*lane + 3
    const int nkeys = min(PA_KT, L - t * PA_KT);
    for (int j = 0; j < nkeys; ++j) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vb + j * PA_D + lane * 4);
      const float v0 = __uint_as_float(vv.x << 16), v1 = __uint_as_float(vv.x & 0xFFFF0000u);
      const float v2 = __uint_as_float(vv.y << 16), v3 = __uint_as_float(vv.y & 0xFFFF0000u);
#pragma unroll
      for (int k = 0; k < PA_RPW; ++k) {
        if (k < nrow) {
          const float pj = __shfl_sync(0xffffffffu, j < 32 ? pr[k][0] : pr[k][1], j & 31);
          acc[k][0] = fmaf(pj, v0, acc[k][0]);
          acc[k][1] = fmaf(pj, v1, acc[k][1]);
          acc[k][2] = fmaf(pj, v2, acc[k][2]);
          acc[k][3] = fmaf(pj, v3, acc[k][3]);
        }
      }
    }
  }
  // results: the row's normalised output and lse, or this split's partial
#pragma unroll
  for (int k = 0; k < PA_RPW; ++k) {
    if (k < nrow) {
      const int r = warp + 8 * k, i = r / G, head = g * G + (r - i * G);
      const int64_t row = static_cast<int64_t>(b) * p.n_new + i;
      if (p.nsplit == 1) {
        const float inv = l_r[k] > 0.f ? 1.f / l_r[k] : 0.f;
        uint2 w;
        w.x = pack_bf16x2(acc[k][0] * inv, acc[k][1] * inv);
        w.y = pack_bf16x2(acc[k][2] * inv, acc[k][3] * inv);
        *reinterpret_cast<uint2*>(p.o + (row * p.Hq + head) * PA_D + lane * 4) = w;
        if (p.lse && lane == 0)
          p.lse[(static_cast<int64_t>(b) * p.Hq + head) * p.n_new + i] = (m_r[k] + log2f(l_r[k])) * PA_LN2;
      } else {
        const int64_t pr_off = ((static_cast<int64_t>(sp) * p.B * p.n_new + row) * p.Hq + head);
        *reinterpret_cast<float4*>(p.part_o + pr_off * PA_D + lane * 4) =
            make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
        if (lane == 0) {
          p.part_ml[pr_off * 2] = m_r[k];
          p.part_ml[pr_off * 2 + 1] = l_r[k];
        }
      }
    }
  }
}

// One warp per (new token, query head): O = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
__global__ void __launch_bounds__(256) paged_combine_kernel(int rows, int Hq, int nsplit, int n_new,
                                                            const float* __restrict__ part_o,
                                                            const float* __restrict__ part_ml,
                                                            __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  pdl_enter();
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= rows * Hq) return;
  const int64_t stride = static_cast<int64_t>(rows) * Hq;   // one split's rows x heads
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[(s * stride + w) * 2]);
  float Lsum = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (M > -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ms = part_ml[(s * stride + w) * 2];
      if (!(ms > -INFINITY)) continue;
      const float f = exp2f(ms - M);
      Lsum += part_ml[(s * stride + w) * 2 + 1] * f;
      const float4 v = *reinterpret_cast<const float4*>(part_o + (s * stride + w) * PA_D + lane * 4);
      a0 = fmaf(v.x, f, a0);
      a1 = fmaf(v.y, f, a1);
      a2 = fmaf(v.z, f, a2);
      a3 = fmaf(v.w, f, a3);
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  uint2 wv;
  wv.x = pack_bf16x2(a0 * inv, a1 * inv);
  wv.y = pack_bf16x2(a2 * inv, a3 * inv);
  *reinterpret_cast<uint2*>(o + static_cast<int64_t>(w) * PA_D + lane * 4) = wv;
  if (lse && lane == 0) {
    const int t = w / Hq, h = w - t * Hq, b = t / n_new, i = t - b * n_new;
    lse[(static_cast<int64_t>(b) * Hq + h) * n_new + i] = (M + log2f(Lsum)) * PA_LN2;
  }
}

}  // namespace

namespace {

struct PagedSplit {
  int nsplit, tiles_per_split;
};

// Context splits: enough CTAs for two per SM when the sequences alone do not
// give them, each split a whole number of 64-token tiles.
PagedSplit paged_split(const kl_paged_cfg& pc, int Hkv) {
  const int max_tiles = (pc.max_blocks * pc.block_size + PA_KT - 1) / PA_KT;
  const int want = 2 * num_sms();
  int ns = (want + Hkv * pc.B - 1) / (Hkv * pc.B);
  ns = ns < 1 ? 1 : (ns > max_tiles ? max_tiles : ns);
  const int tps = (max_tiles + ns - 1) / ns;
  return {(max_tiles + tps - 1) / tps, tps};
}

constexpr size_t PA_SMEM_MAX = 4 * PA_KT * PA_D * 2 + PA_RMAX * PA_D * 4;

}  // namespace

kl_status paged_check(const kl_paged_cfg* pc, int Hq, int Hkv, int d, int dtype) {
  if (!pc) return set_error(KL_ERR_INVALID_ARG, "paged: null configuration");
  if (pc->B < 1 || pc->n_new < 1 || pc->block_size < 1 || pc->max_blocks < 1 || pc->n_blocks < 1)
    return set_error(KL_ERR_INVALID_ARG, "paged: bad sizes (B %d, n_new %d, block %d, table %d, pool %d)", pc->B,
                     pc->n_new, pc->block_size, pc->max_blocks, pc->n_blocks);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return set_error(KL_ERR_INVALID_ARG, "paged: bad head counts %d / %d", Hq, Hkv);
  if (d != PA_D || dtype != KL_BF16)
    return set_error(KL_ERR_UNSUPPORTED, "paged: bf16 with head dim 128 only (got dtype %d, d %d)", dtype, d);
  if ((Hq / Hkv) * pc->n_new > PA_RMAX)
    return set_error(KL_ERR_UNSUPPORTED, "paged: %d query heads per kv head x %d new tokens above %d rows",
                     Hq / Hkv, pc->n_new, PA_RMAX);
  return KL_OK;
}

size_t paged_attention_ws(const kl_paged_cfg& pc, int Hq, int Hkv) {
  const PagedSplit sp = paged_split(pc, Hkv);
  if (sp.nsplit <= 1) return 0;
  const size_t rows = static_cast<size_t>(sp.nsplit) * pc.B * pc.n_new * Hq;
  return align_up(rows * PA_D * 4, 256) + align_up(rows * 2 * 4, 256);
}

kl_status paged_kv_write(const kl_paged_cfg& pc, int Hkv, const void* k_new, const void* v_new, const int32_t* table,
                         const int32_t* ctx, void* kp, void* vp, cudaStream_t st) {
  if (!k_new || !v_new || !table || !ctx || !kp || !vp) return set_error(KL_ERR_INVALID_ARG, "paged write: null pointer");
  const int rows = pc.B * pc.n_new;
  ProfScope ps("paged_kv_write", st, 0.0, 2.0 * 2 * rows * Hkv * PA_D * 2);
  launch_pdl(paged_kv_write_kernel, (rows * Hkv + 7) / 8, 256, 0, st, rows, pc.n_new, Hkv, pc.block_size,
             pc.max_blocks, pc.n_blocks, device_error_word(), static_cast<const __nv_bfloat16*>(k_new),
             static_cast<const __nv_bfloat16*>(v_new), table, ctx, static_cast<__nv_bfloat16*>(kp),
             static_cast<__nv_bfloat16*>(vp));
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status paged_attention(const kl_paged_cfg& pc, int Hq, int Hkv, const void* q, const void* kp, const void* vp,
                          const int32_t* table, const int32_t* ctx, void* o, float* lse, void* ws, size_t ws_bytes,
                          cudaStream_t st) {
  if (!q || !kp || !vp || !table || !ctx || !o) return set_error(KL_ERR_INVALID_ARG, "paged attention: null pointer");
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kp) | reinterpret_cast<uintptr_t>(vp) |
        reinterpret_cast<uintptr_t>(o)) & 15u) != 0)
    return set_error(KL_ERR_INVALID_ARG, "paged attention: q, pools and o must be 16-byte aligned");
  const PagedSplit sp = paged_split(pc, Hkv);
  const size_t need = paged_attention_ws(pc, Hq, Hkv);
  if (need && (!ws || ws_bytes < need)) return set_error(KL_ERR_NO_MEMORY, "paged attention: workspace too small");
  static uint64_t attr_done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(paged_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PA_SMEM_MAX)));
    attr_done |= uint64_t(1) << dev;
  }
  PagedParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kp = static_cast<const __nv_bfloat16*>(kp);
  p.vp = static_cast<const __nv_bfloat16*>(vp);
  p.table = table;
  p.ctx = ctx;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const size_t rows = static_cast<size_t>(sp.nsplit) * pc.B * pc.n_new * Hq;
  p.part_o = sp.nsplit > 1 ? static_cast<float*>(ws) : nullptr;
  p.part_ml = sp.nsplit > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align_up(rows * PA_D * 4, 256))
                            : nullptr;
  p.B = pc.B;
  p.n_new = pc.n_new;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.bs = pc.block_size;
  p.max_blocks = pc.max_blocks;
  p.n_blocks = pc.n_blocks;
  p.nsplit = sp.nsplit;
  p.tiles_per_split = sp.tiles_per_split;
  p.scale_log2 = PA_LOG2E / sqrtf(static_cast<float>(PA_D));
  p.err = device_error_word();
  const size_t smem = 4 * PA_KT * PA_D * 2 + static_cast<size_t>(Hq / Hkv) * pc.n_new * PA_D * 4;
  {
    // HBM bytes: the keys and values of the contexts (at most the tables' extent) read once,
    // the queries read and the outputs written once; flops: 4 d per (query, key) pair
    const double kv = 2.0 * pc.B * Hkv * static_cast<double>(pc.max_blocks) * pc.block_size * PA_D * 2;
    ProfScope ps("paged_attention", st, 0.0, kv + 2.0 * pc.B * pc.n_new * Hq * PA_D * 2);
    launch_pdl(paged_attn_kernel, dim3(Hkv, pc.B, sp.nsplit), PA_THREADS, smem, st, p);
  }
  KL_CUDA(cudaGetLastError());
  if (sp.nsplit > 1) {
    const int r = pc.B * pc.n_new;
    ProfScope ps("paged_combine", st, 0.0, 4.0 * rows * (PA_D + 2) + 2.0 * r * Hq * PA_D);
    launch_pdl(paged_combine_kernel, (r * Hq + 7) / 8, 256, 0, st, r, Hq, sp.nsplit, pc.n_new, p.part_o, p.part_ml,
               p.o, lse);
    KL_CUDA(cudaGetLastError());
  }
  return KL_OK;
}

}  // namespace kl
