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
//   paged_attn_kernel      decode attention, HBM-bound: the keys and values of
//                          each (sequence, kv head) are read once for all its
//                          query rows (G heads x n_new tokens, 16 per item);
//                          persistent CTAs take equal runs of 64-key tiles,
//                          gather them through the block table by cp.async
//                          into a 3-stage ring and do Q K^T and P V on the
//                          tensor cores (warp-level m16n8k16: the rows are too
//                          few for a tcgen05 tile; the bound is HBM either way).
//   paged_combine_kernel   merges the pieces of items that two or more CTAs
//                          shared.
#include <math.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int PA_THREADS = 128;    // four warps
constexpr int PA_WARPS = PA_THREADS / 32;
constexpr int PA_KT = 64;          // keys per tile, 16 per warp
constexpr int PA_D = 128;          // head dim
constexpr int PA_RMAX = 64;        // query rows per kv head (G heads x n_new tokens)
constexpr int PA_MR = 16;          // query rows per work item: one m16 MMA tile
constexpr int PA_NST = 3;          // cp.async pipeline stages
constexpr int PA_TILE_BYTES = PA_KT * PA_D * 2;       // the K (or V) rows of one tile
constexpr int PA_STAGE_BYTES = 2 * PA_TILE_BYTES;
constexpr int PA_OB_STRIDE = PA_D + 4;                // fp32 words per row of the warp-combine buffer
constexpr size_t PA_SMEM = static_cast<size_t>(PA_NST) * PA_STAGE_BYTES + PA_MR * PA_OB_STRIDE * 4 +
                           PA_WARPS * PA_MR * 2 * 4;
constexpr float PA_LN2 = 0.6931471805599453f;
constexpr float PA_LOG2E = 1.4426950408889634f;

struct PagedParams {
  const __nv_bfloat16* q;     // [B*n_new, Hq*d]
  const __nv_bfloat16* kp;    // [n_blocks][bs][Hkv*d]
  const __nv_bfloat16* vp;
  const int32_t* table;       // [B][max_blocks]
  const int32_t* ctx;         // [B]
  __nv_bfloat16* o;           // [B*n_new, Hq*d]
  float* lse;                 // [B, Hq, n_new] natural log, or null
  float* part_o;              // [items][maxp][16][d] unnormalised pieces of split items
  float* part_ml;             // [items][maxp][16][2] (max in log2 units, sum)
  int B, n_new, Hq, Hkv, bs, max_blocks, n_blocks;
  int G, R, RG;               // query heads per kv head, rows per kv head (G n_new), groups of 16 rows
  int T;                      // tiles per item (the table's extent in 64-key tiles)
  int P;                      // tiles per CTA
  int W;                      // items x T
  int maxp;                   // pieces per item at most
  float scale_log2;           // log2(e) / sqrt(d)
  uint32_t* err;              // device error word: a position past the table or a block outside the pool
};

__device__ __forceinline__ void pa_cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;   // zero-fill when the token is outside the context
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void pa_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void pa_cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// four 8x8 b16 matrices; lanes 8m .. 8m+7 address the rows of matrix m
__device__ __forceinline__ void pa_ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void pa_ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// d += a (16x16 bf16, row) * b (16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void pa_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// byte offset of 16-byte chunk ch of key row j in a [64][128] bf16 tile; the
// chunk index is XORed with j mod 8 so that eight consecutive rows of one chunk
// column fall in different banks (ldmatrix reads them together)
__device__ __forceinline__ uint32_t pa_swz(int j, int ch) { return j * (PA_D * 2) + ((ch ^ (j & 7)) << 4); }

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

// Work is cut into items (sequence b, kv head g, group rg of 16 query rows)
// and each item into T tiles of 64 key positions; the W = items x T tiles, in
// item-major order, are dealt out in equal runs of P to persistent CTAs. A CTA
// walks its run through a 3-stage cp.async ring: every thread copies 16 of the
// tile's 256-byte K and V rows' chunks, the rows found through the block table
// one tile ahead. Warp w takes keys 16w .. 16w+15 of each tile: S = Q K^T and
// O += P V by m16n8k16 MMAs (query rows as M, fragments from ldmatrix), an
// online base-2 softmax per row. Where the run leaves an item (or ends), the
// four warps' (max, sum, O) are merged in shared memory in warp order and the
// CTA writes either the final row (it held the whole item) or a piece that
// paged_combine_kernel merges.
__device__ __forceinline__ int pa_first_cta(long long i, int T, int P) { return static_cast<int>(i * T / P); }
__device__ __forceinline__ int pa_last_cta(long long i, int T, int P) { return static_cast<int>(((i + 1) * T - 1) / P); }

__global__ void __launch_bounds__(PA_THREADS, 2) paged_attn_kernel(const __grid_constant__ PagedParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t pa_smem[];
  float* obuf = reinterpret_cast<float*>(pa_smem + PA_NST * PA_STAGE_BYTES);   // [16][PA_OB_STRIDE]
  float* mlbuf = obuf + PA_MR * PA_OB_STRIDE;                                   // [warp][16][2]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;      // fragment row (and row + 8), column pair
  const int u0 = blockIdx.x * p.P;
  const int u1 = min(p.W, u0 + p.P);
  if (u0 >= u1) return;

  // Table lookup of tile u for this lane: lanes l and l + 16 resolve key
  // 2 warp + (l & 1) + 8 ((l >> 1) & 7) to its pool row (block * bs + slot) * Hkv + g,
  // or -1 past the context. `live` says whether the tile holds any key at all.
  auto resolve = [&](int u, int& row, bool& live) {
    const int i = u / p.T, tile = u - i * p.T;
    const int bg = i / p.RG, b = bg / p.Hkv, g = bg - b * p.Hkv;
    const int L = max(0, p.ctx[b]) + p.n_new;
    live = tile * PA_KT < L;
    const int pos = tile * PA_KT + 2 * warp + (lane & 1) + 8 * ((lane >> 1) & 7);
    row = -1;
    if (pos < L) {
      const int lb = pos / p.bs;
      const int blk = lb < p.max_blocks ? p.table[b * p.max_blocks + lb] : -1;
      if (blk < 0 || blk >= p.n_blocks)
        record_error(p.err, KL_DEVERR_PAGE);
      else
        row = ((blk * p.bs) + (pos - lb * p.bs)) * p.Hkv + g;
    }
  };
  // copies of one tile: thread tid moves chunk tid & 15 of keys (tid >> 4) + 8k, k < 8
  auto issue = [&](int stage, int row) {
    const uint32_t kb = smem_u32(pa_smem + stage * PA_STAGE_BYTES);
    const int ch = tid & 15;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = __shfl_sync(0xffffffffu, row, (lane >> 4) | (k << 1));
      const uint32_t off = pa_swz((tid >> 4) + 8 * k, ch);
      const size_t src = static_cast<size_t>(r < 0 ? 0 : r) * PA_D + ch * 8;
      pa_cp_async16(kb + off, p.kp + src, r >= 0);
      pa_cp_async16(kb + PA_TILE_BYTES + off, p.vp + src, r >= 0);
    }
  };

  int nrow = -1;
  bool nlive = false;
#pragma unroll
  for (int k = 0; k < PA_NST - 1; ++k) {
    if (u0 + k < u1) {
      resolve(u0 + k, nrow, nlive);
      if (nlive) issue(k, nrow);
    }
    pa_cp_commit();
  }
  if (u0 + PA_NST - 1 < u1) resolve(u0 + PA_NST - 1, nrow, nlive);

  // the current item's state
  int cur = -1, b = 0, g = 0, rg = 0, ctxb = 0, L = 0;
  int qpos[2];
  uint32_t qa[8][4];
  float o[16][4], mrow[2], lrow[2];

  auto start = [&](int i) {
    cur = i;
    rg = i % p.RG;
    const int bg = i / p.RG;
    b = bg / p.Hkv;
    g = bg - b * p.Hkv;
    ctxb = max(0, p.ctx[b]);
    L = ctxb + p.n_new;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rg * PA_MR + gq + 8 * h;
      qpos[h] = ctxb + min(r, p.R - 1) / p.G;   // padding rows copy the last real row's limit
      const __nv_bfloat16* qr = nullptr;
      if (r < p.R) {
        const int it = r / p.G, head = g * p.G + (r - it * p.G);
        qr = p.q + (static_cast<int64_t>(b * p.n_new + it) * p.Hq + head) * PA_D + 2 * tq;
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][h] = qr ? *reinterpret_cast<const uint32_t*>(qr + 16 * ks) : 0u;
        qa[ks][h + 2] = qr ? *reinterpret_cast<const uint32_t*>(qr + 16 * ks + 8) : 0u;
      }
      mrow[h] = -INFINITY;
      lrow[h] = 0.f;
    }
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  };

  auto finish = [&]() {
    __syncthreads();                            // the previous merge is done with obuf / mlbuf
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
      lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
      if (tq == 0) {
        mlbuf[(warp * PA_MR + gq + 8 * h) * 2] = mrow[h];
        mlbuf[(warp * PA_MR + gq + 8 * h) * 2 + 1] = lrow[h];
      }
    }
    __syncthreads();
    float M[2], f[2], Lt[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = gq + 8 * h;
      M[h] = -INFINITY;
#pragma unroll
      for (int w = 0; w < PA_WARPS; ++w) M[h] = fmaxf(M[h], mlbuf[(w * PA_MR + rr) * 2]);
      Lt[h] = 0.f;
#pragma unroll
      for (int w = 0; w < PA_WARPS; ++w) {
        const float mw = mlbuf[(w * PA_MR + rr) * 2];
        if (mw > -INFINITY) Lt[h] += mlbuf[(w * PA_MR + rr) * 2 + 1] * exp2f(mw - M[h]);
      }
      f[h] = mrow[h] > -INFINITY ? exp2f(mrow[h] - M[h]) : 0.f;
    }
    // the warps' rows summed into obuf in warp order (a fixed order: reproducible)
#pragma unroll 1
    for (int w = 0; w < PA_WARPS - 1; ++w) {
      if (warp == w) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float* ob = obuf + (gq + 8 * h) * PA_OB_STRIDE + 2 * tq;
#pragma unroll
          for (int dn = 0; dn < 16; ++dn) {
            float2 v = make_float2(o[dn][2 * h] * f[h], o[dn][2 * h + 1] * f[h]);
            if (w > 0) {
              const float2 a = *reinterpret_cast<const float2*>(ob + 8 * dn);
              v.x += a.x;
              v.y += a.y;
            }
            *reinterpret_cast<float2*>(ob + 8 * dn) = v;
          }
        }
      }
      __syncthreads();
    }
    if (warp != PA_WARPS - 1) return;
    const int first = pa_first_cta(cur, p.T, p.P), last = pa_last_cta(cur, p.T, p.P);
    const bool whole = first == last;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = gq + 8 * h, r = rg * PA_MR + rr;
      if (r >= p.R) continue;
      const float* ob = obuf + rr * PA_OB_STRIDE + 2 * tq;
      if (whole) {
        const int it = r / p.G, head = g * p.G + (r - it * p.G);
        const float inv = Lt[h] > 0.f ? 1.f / Lt[h] : 0.f;
        __nv_bfloat16* orow = p.o + (static_cast<int64_t>(b * p.n_new + it) * p.Hq + head) * PA_D + 2 * tq;
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
          const float2 a = *reinterpret_cast<const float2*>(ob + 8 * dn);
          *reinterpret_cast<uint32_t*>(orow + 8 * dn) =
              pack_bf16x2((a.x + o[dn][2 * h] * f[h]) * inv, (a.y + o[dn][2 * h + 1] * f[h]) * inv);
        }
        if (p.lse && tq == 0)
          p.lse[(static_cast<int64_t>(b) * p.Hq + head) * p.n_new + it] = (M[h] + log2f(Lt[h])) * PA_LN2;
      } else {
        const int64_t pc = (static_cast<int64_t>(cur) * p.maxp + (blockIdx.x - first)) * PA_MR + rr;
        float* po = p.part_o + pc * PA_D + 2 * tq;
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
          const float2 a = *reinterpret_cast<const float2*>(ob + 8 * dn);
          *reinterpret_cast<float2*>(po + 8 * dn) = make_float2(a.x + o[dn][2 * h] * f[h], a.y + o[dn][2 * h + 1] * f[h]);
        }
        if (tq == 0) {
          p.part_ml[pc * 2] = M[h];
          p.part_ml[pc * 2 + 1] = Lt[h];
        }
      }
    }
  };

  for (int u = u0; u < u1; ++u) {
    const int stage = (u - u0) % PA_NST;
    pa_cp_wait<PA_NST - 2>();
    __syncthreads();                            // tile u landed for every thread; tile u-1's stage is free
    {
      const int un = u + PA_NST - 1;
      if (un < u1 && nlive) issue((stage + PA_NST - 1) % PA_NST, nrow);
      pa_cp_commit();
      if (un + 1 < u1) resolve(un + 1, nrow, nlive);
    }
    const int i = u / p.T, tile = u - i * p.T;
    if (i != cur) {
      if (cur >= 0) finish();
      start(i);
    }
    if (tile * PA_KT >= L) continue;            // past this sequence's context

    const uint32_t kb = smem_u32(pa_smem + stage * PA_STAGE_BYTES), vb = kb + PA_TILE_BYTES;
    const int lm = lane >> 3, lr = lane & 7;    // ldmatrix: matrix and row this lane addresses
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {            // S = Q K^T over dims 16 ks .. 16 ks + 15
      uint32_t kf[4];
      pa_ldsm4(kb + pa_swz(16 * warp + 8 * (lm >> 1) + lr, 2 * ks + (lm & 1)), kf);
      pa_mma(sc[0], qa[ks], kf[0], kf[1]);
      pa_mma(sc[1], qa[ks], kf[2], kf[3]);
    }
    // causal limit by absolute position; online softmax in base 2
    const int key0 = tile * PA_KT + 16 * warp + 2 * tq;
    uint32_t pa[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          v[2 * nt + e] = key0 + 8 * nt + e <= qpos[h] ? sc[nt][2 * h + e] * p.scale_log2 : -INFINITY;
      float mt = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float mn = fmaxf(mrow[h], mt);
      const float mu = mn > -INFINITY ? mn : 0.f;
      const float alpha = exp2f(mrow[h] - mu);
#pragma unroll
      for (int x = 0; x < 4; ++x) v[x] = exp2f(v[x] - mu);
      lrow[h] = lrow[h] * alpha + ((v[0] + v[1]) + (v[2] + v[3]));
      mrow[h] = mn;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        o[dn][2 * h] *= alpha;
        o[dn][2 * h + 1] *= alpha;
      }
      pa[h] = pack_bf16x2(v[0], v[1]);          // keys 2tq, 2tq+1 of the warp's first 8
      pa[h + 2] = pack_bf16x2(v[2], v[3]);      // and of its second 8
    }
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {            // O += P V over dims 16 dp .. 16 dp + 15
      uint32_t vf[4];
      pa_ldsm4_t(vb + pa_swz(16 * warp + 8 * (lm & 1) + lr, 2 * dp + (lm >> 1)), vf);
      pa_mma(o[2 * dp], pa, vf[0], vf[1]);
      pa_mma(o[2 * dp + 1], pa, vf[2], vf[3]);
    }
  }
  finish();
}

// One warp per (item, row of its 16): O = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M)
// over the item's pieces; items held whole by one CTA were written by it.
__global__ void __launch_bounds__(256) paged_combine_kernel(const __grid_constant__ PagedParams p, int items) {
  pdl_enter();
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= items * PA_MR) return;
  const int i = w / PA_MR, rr = w - i * PA_MR;
  const int rg = i % p.RG, bg = i / p.RG, b = bg / p.Hkv, g = bg - b * p.Hkv;
  const int r = rg * PA_MR + rr;
  if (r >= p.R) return;
  const int first = pa_first_cta(i, p.T, p.P), np = pa_last_cta(i, p.T, p.P) - first + 1;
  if (np == 1) return;
  const int64_t base = static_cast<int64_t>(i) * p.maxp * PA_MR + rr;
  float M = -INFINITY;
  for (int s = 0; s < np; ++s) M = fmaxf(M, p.part_ml[(base + s * PA_MR) * 2]);
  float Lsum = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (M > -INFINITY) {
    for (int s = 0; s < np; ++s) {
      const int64_t pc = base + s * PA_MR;
      const float ms = p.part_ml[pc * 2];
      if (!(ms > -INFINITY)) continue;
      const float f = exp2f(ms - M);
      Lsum += p.part_ml[pc * 2 + 1] * f;
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + pc * PA_D + lane * 4);
      a0 = fmaf(v.x, f, a0);
      a1 = fmaf(v.y, f, a1);
      a2 = fmaf(v.z, f, a2);
      a3 = fmaf(v.w, f, a3);
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int it = r / p.G, head = g * p.G + (r - it * p.G);
  uint2 wv;
  wv.x = pack_bf16x2(a0 * inv, a1 * inv);
  wv.y = pack_bf16x2(a2 * inv, a3 * inv);
  *reinterpret_cast<uint2*>(p.o + (static_cast<int64_t>(b * p.n_new + it) * p.Hq + head) * PA_D + lane * 4) = wv;
  if (p.lse && lane == 0) p.lse[(static_cast<int64_t>(b) * p.Hq + head) * p.n_new + it] = (M + log2f(Lsum)) * PA_LN2;
}

}  // namespace

namespace {

// How the (item, tile) units are dealt to CTAs: two resident CTAs per SM, each
// a run of P consecutive tiles; an item cut by a run boundary leaves pieces.
struct PagedPlan {
  int G, R, RG, items, T, W, P, grid, maxp;
  bool split;   // some item is cut: pieces and the combine kernel
};

PagedPlan paged_plan(const kl_paged_cfg& pc, int Hq, int Hkv) {
  PagedPlan pl;
  pl.G = Hq / Hkv;
  pl.R = pl.G * pc.n_new;
  pl.RG = (pl.R + PA_MR - 1) / PA_MR;
  pl.items = pc.B * Hkv * pl.RG;
  pl.T = (pc.max_blocks * pc.block_size + PA_KT - 1) / PA_KT;
  pl.W = pl.items * pl.T;
  const int slots = 2 * num_sms();
  pl.P = (pl.W + slots - 1) / slots;
  pl.grid = (pl.W + pl.P - 1) / pl.P;
  pl.maxp = (pl.T - 1) / pl.P + 2;
  pl.split = pl.grid > 1 && pl.P % pl.T != 0;
  return pl;
}

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
  const double rows = static_cast<double>(pc->n_blocks) * pc->block_size * Hkv;
  const double units = static_cast<double>(pc->B) * Hkv * (((Hq / Hkv) * pc->n_new + PA_MR - 1) / PA_MR) *
                       (static_cast<double>(pc->max_blocks) * pc->block_size / PA_KT + 1);
  if (rows >= 2147483647.0 || units >= 2147483647.0)
    return set_error(KL_ERR_UNSUPPORTED, "paged: pool rows (%.0f) or work units (%.0f) beyond 32-bit indexing", rows,
                     units);
  return KL_OK;

}

size_t paged_attention_ws(const kl_paged_cfg& pc, int Hq, int Hkv) {
  const PagedPlan pl = paged_plan(pc, Hq, Hkv);
  if (!pl.split) return 0;
  const size_t pieces = static_cast<size_t>(pl.items) * pl.maxp * PA_MR;
  return align_up(pieces * PA_D * 4, 256) + align_up(pieces * 2 * 4, 256);
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
  const PagedPlan pl = paged_plan(pc, Hq, Hkv);
  const size_t need = paged_attention_ws(pc, Hq, Hkv);
  if (need && (!ws || ws_bytes < need)) return set_error(KL_ERR_NO_MEMORY, "paged attention: workspace too small");
  static uint64_t attr_done = 0;
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !(attr_done >> dev & 1u)) {
    KL_CUDA(cudaFuncSetAttribute(paged_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PA_SMEM)));
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
  const size_t pieces = static_cast<size_t>(pl.items) * pl.maxp * PA_MR;
  p.part_o = pl.split ? static_cast<float*>(ws) : nullptr;
  p.part_ml = pl.split ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align_up(pieces * PA_D * 4, 256))
                       : nullptr;
  p.B = pc.B;
  p.n_new = pc.n_new;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.bs = pc.block_size;
  p.max_blocks = pc.max_blocks;
  p.n_blocks = pc.n_blocks;
  p.G = pl.G;
  p.R = pl.R;
  p.RG = pl.RG;
  p.T = pl.T;
  p.P = pl.P;
  p.W = pl.W;
  p.maxp = pl.maxp;
  p.scale_log2 = PA_LOG2E / sqrtf(static_cast<float>(PA_D));
  p.err = device_error_word();
  {
    // HBM bytes: the keys and values of the contexts (at most the tables' extent) read once per
    // group of 16 query rows, the queries read and the outputs written once
    const double kv = 2.0 * pc.B * Hkv * pl.RG * static_cast<double>(pc.max_blocks) * pc.block_size * PA_D * 2;
    ProfScope ps("paged_attention", st, 0.0, kv + 2.0 * pc.B * pc.n_new * Hq * PA_D * 2);
    launch_pdl(paged_attn_kernel, pl.grid, PA_THREADS, PA_SMEM, st, p);
  }
  KL_CUDA(cudaGetLastError());
  if (pl.split) {
    ProfScope ps("paged_combine", st, 0.0, 4.0 * pieces * (PA_D + 2) + 2.0 * pc.B * pc.n_new * Hq * PA_D);
    launch_pdl(paged_combine_kernel, (pl.items * PA_MR + 7) / 8, 256, 0, st, p, pl.items);
    KL_CUDA(cudaGetLastError());
  }
  return KL_OK;
}

}  // namespace kl
