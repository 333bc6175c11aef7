// Softmax cross-entropy + argmax + dlogits in a single launch ("From-scratch
// GPU LLM training", capability list: GPU lm-head, softmax cross-entropy and
// argmax fused in a single launch).
//
// One row of fp32 logits per 8-CTA thread-block cluster. Each CTA copies its
// eighth of the row (the vocabulary tile) into shared memory once, reduces
// max / lowest argmax over it, then replaces each logit by e = exp(z - tile
// max) and sums them, publishes the three numbers in shared memory and reads
// its seven peers' through distributed shared memory to form the row's
// logsumexp and argmax. It then writes dlogits = (e exp(tile max - lse) -
// onehot) / N for its tile from shared memory: one exp per logit, the row read
// from HBM exactly once and dlogits written once. The mean loss is reduced in
// a fixed order by the last cluster to finish (deterministic).
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include <mutex>

#include "internal.h"
#include "kl_common.cuh"

namespace cg = cooperative_groups;

namespace kl {
namespace {

// CTAs per row (cluster size) and threads per CTA. Measured on the 4096 x
// 151936 workload: 8 x 256 beats 8 x 512 / 384 / 128 and 16 x 256 (two CTAs
// of ~76 KB shared memory per SM either way).
constexpr int CLUSTER = 8;
constexpr int THREADS = 256;
constexpr int NWARP = THREADS / 32;

struct Part {
  float m;
  float s;
  int idx;
};

__device__ __forceinline__ void better(float& m, int& i, float m2, int i2) {
  if (m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

template <bool VEC>
__global__ void __launch_bounds__(THREADS)
    ce_argmax_kernel(int N, int V, int slice, const float* __restrict__ z,
                     const int32_t* __restrict__ targets, float* __restrict__ loss_rows,
                     int32_t* __restrict__ argmax, void* __restrict__ dz, int dz_f32, float invN,
                     unsigned int* __restrict__ counter, float* __restrict__ loss,
                     uint32_t* __restrict__ err) {
  pdl_enter();
  extern __shared__ __align__(16) float sz[];
  __shared__ float red_m[NWARP];
  __shared__ float red_s[NWARP];
  __shared__ int red_i[NWARP];
  __shared__ Part part;
  __shared__ int is_last;
  __shared__ __align__(8) uint64_t load_bar;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int n = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = rank * slice;
  const int len = max(0, min(V, c0 + slice) - c0);
  const float* zr = z + static_cast<int64_t>(n) * V + c0;

  // 1. copy the tile to shared memory; running max and lowest argmax
  float m = -INFINITY;
  int mi = INT_MAX;
  if (VEC) {
    // One bulk asynchronous copy of the whole tile (16-byte aligned, length a
    // multiple of 16 bytes), completed on an mbarrier: the row is in flight at
    // once instead of one vector per thread.
    const uint32_t bar = smem_u32(&load_bar);
    if (threadIdx.x == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      if (len > 0) {
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(len) * 4u);
        bulk_copy_g2s(smem_u32(sz), zr, static_cast<uint32_t>(len) * 4u, bar);
      } else {
        mbar_arrive(bar);
      }
    }
    mbar_wait(bar, 0, err);
    for (int i = threadIdx.x * 4; i < len; i += THREADS * 4) {
      const float4 a = *reinterpret_cast<const float4*>(sz + i);
      better(m, mi, a.x, c0 + i);
      better(m, mi, a.y, c0 + i + 1);
      better(m, mi, a.z, c0 + i + 2);
      better(m, mi, a.w, c0 + i + 3);
    }
  } else {
    for (int i = threadIdx.x; i < len; i += THREADS) {
      const float a = zr[i];
      sz[i] = a;
      better(m, mi, a, c0 + i);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, mi, o);
    better(m, mi, m2, i2);
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_i[warp] = mi;
  }
  __syncthreads();
  float tm = red_m[0];
  int ti = red_i[0];
  for (int w = 1; w < NWARP; ++w) better(tm, ti, red_m[w], red_i[w]);
  // 2. e = exp(z - tile max), kept in place (vector form), and its sum
  float s = 0.f;
  if (len > 0) {
    if (VEC) {
      for (int i = threadIdx.x * 4; i < len; i += THREADS * 4) {
        float4 a = *reinterpret_cast<const float4*>(sz + i);
        a.x = expf(a.x - tm);
        a.y = expf(a.y - tm);
        a.z = expf(a.z - tm);
        a.w = expf(a.w - tm);
        s += (a.x + a.y) + (a.z + a.w);
        *reinterpret_cast<float4*>(sz + i) = a;
      }
    } else {
      for (int i = threadIdx.x; i < len; i += THREADS) s += expf(sz[i] - tm);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red_s[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float ts = 0.f;
    for (int w = 0; w < NWARP; ++w) ts += red_s[w];
    part.m = tm;
    part.s = ts;
    part.idx = ti;
  }
  cluster.sync();
  // 3. combine the eight tiles (every CTA does it; fixed rank order)
  float M = -INFINITY;
  int I = INT_MAX;
  Part ps[CLUSTER];
#pragma unroll
  for (int r = 0; r < CLUSTER; ++r) {
    ps[r] = *cluster.map_shared_rank(&part, r);
    better(M, I, ps[r].m, ps[r].idx);
  }
  float tot = 0.f;
#pragma unroll
  for (int r = 0; r < CLUSTER; ++r)
    if (ps[r].s > 0.f) tot += ps[r].s * expf(ps[r].m - M);
  const float lse = M + logf(tot);
  int t = targets[n];
  const bool t_ok = t >= 0 && t < V;
  if (!t_ok) {
    if (threadIdx.x == 0 && rank == 0) record_error(err, KL_DEVERR_TARGET);
    t = -1;
  }
  // 4. dlogits for this tile
  if (dz_f32) {
    float* out = static_cast<float*>(dz) + static_cast<int64_t>(n) * V + c0;
    const float sc = len > 0 && tm > -INFINITY ? expf(tm - lse) : 0.f;
    for (int i = threadIdx.x; i < len; i += THREADS) {
      float p = VEC ? sz[i] * sc : expf(sz[i] - lse);
      if (c0 + i == t) p -= 1.f;
      out[i] = p * invN;
    }
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(dz) + static_cast<int64_t>(n) * V + c0;
    if (VEC) {
      const float sc = len > 0 && tm > -INFINITY ? expf(tm - lse) : 0.f;   // the tile holds exp(z - tm)
      for (int i = threadIdx.x * 4; i < len; i += THREADS * 4) {
        const float4 a = *reinterpret_cast<const float4*>(sz + i);
        float p0 = a.x * sc, p1 = a.y * sc, p2 = a.z * sc, p3 = a.w * sc;
        const int d = t - (c0 + i);
        if (d == 0) p0 -= 1.f;
        if (d == 1) p1 -= 1.f;
        if (d == 2) p2 -= 1.f;
        if (d == 3) p3 -= 1.f;
        uint2 o;
        o.x = pack_bf16x2(p0 * invN, p1 * invN);
        o.y = pack_bf16x2(p2 * invN, p3 * invN);
        *reinterpret_cast<uint2*>(out + i) = o;
      }
    } else {
      for (int i = threadIdx.x; i < len; i += THREADS) {
        float p = expf(sz[i] - lse);
        if (c0 + i == t) p -= 1.f;
        out[i] = __float2bfloat16_rn(p * invN);
      }
    }
  }
  // 5. per-row loss and argmax; the last row to finish reduces the mean
  if (rank == 0 && threadIdx.x == 0) {
    const float zt = t_ok ? z[static_cast<int64_t>(n) * V + t] : lse;
    loss_rows[n] = lse - zt;
    argmax[n] = I;
    __threadfence();
    const unsigned prev = atomicAdd(counter, 1u);
    is_last = prev == static_cast<unsigned>(N - 1);
  }
  cluster.sync();  // peers may still read this CTA's `part`
  if (rank != 0) return;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  float acc = 0.f;
  for (int i = threadIdx.x; i < N; i += THREADS) acc += __ldcg(loss_rows + i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) red_s[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot2 = 0.f;
    for (int w = 0; w < NWARP; ++w) tot2 += red_s[w];
    *loss = tot2 * invN;
    *counter = 0u;
  }
}

}  // namespace

size_t ce_ws(int N) { return align_up(static_cast<size_t>(N) * 4, 256) + 256; }

kl_status ce_argmax(int N, int V, const float* z, const int32_t* targets, float* loss,
                    int32_t* argmax, void* dz, int dz_dtype, void* ws, size_t ws_bytes,
                    cudaStream_t st) {
  if (N < 1 || V < 1 || !z || !targets || !loss || !argmax || !dz)
    return set_error(KL_ERR_INVALID_ARG, "ce_argmax: bad arguments");
  if (N > 65535) return set_error(KL_ERR_UNSUPPORTED, "ce_argmax: N above 65535");
  if (!ws || ws_bytes < ce_ws(N)) return set_error(KL_ERR_NO_MEMORY, "ce_argmax: workspace too small");
  const bool vec = V % 4 == 0 && (reinterpret_cast<uintptr_t>(z) & 15u) == 0 &&
                   (dz_dtype == KL_F32 || (reinterpret_cast<uintptr_t>(dz) & 7u) == 0);
  int slice = (V + CLUSTER - 1) / CLUSTER;
  slice = (slice + 3) / 4 * 4;
  const size_t smem = static_cast<size_t>(slice) * sizeof(float);
  if (smem > 200 * 1024) return set_error(KL_ERR_UNSUPPORTED, "ce_argmax: vocabulary %d too large", V);
  float* loss_rows = static_cast<float*>(ws);
  unsigned int* counter =
      reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + align_up(static_cast<size_t>(N) * 4, 256));
  KL_CUDA(cudaMemsetAsync(counter, 0, sizeof(unsigned int), st));
  dim3 grid(CLUSTER, N);
  ProfScope ps("ce_argmax", st, 0.0, static_cast<double>(N) * V * (4 + dtype_size(dz_dtype)) + 12.0 * N);
  const float invN = 1.0f / static_cast<float>(N);
  const int f32 = dz_dtype == KL_F32;
  auto launch = [&](auto kernel) -> kl_status {
    KL_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_enter
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    KL_CUDA(cudaLaunchKernelEx(&cfg, kernel, N, V, slice, z, targets, loss_rows, argmax, dz, f32, invN, counter, loss,
                               device_error_word()));
    return KL_OK;
  };
  if (vec) KL_TRY(launch(ce_argmax_kernel<true>));
  else KL_TRY(launch(ce_argmax_kernel<false>));
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

}  // namespace kl

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot hand the library a workspace: a host application whose
// device memory is owned by its own pool and forbids raw cudaMalloc, a plugin
// with no allocator hook, or a latency-bound loop where cudaMalloc's implicit
// device synchronisation is not acceptable. For them the cross-entropy step
// can run on scratch that is compiled into the library instead: a static
// device array sized for KL_CE_NOALLOC_MAX_ROWS rows (about 256 KB), present
// on every device that loads libkl until the process exits.
//
// The array's device address is looked up once per device, on the first call
// made with that device current (cudaGetSymbolAddress); make that first call
// before any stream capture. All calls share the one array and each leaves
// its contents behind: the completion counter is cleared before every launch,
// and calls whose kernels may run at the same time on the GPU (different
// streams without ordering between them) race on it and must not be issued.
// ---------------------------------------------------------------------------
// Per-row losses (rows 0 .. KL_CE_NOALLOC_MAX_ROWS-1), then the completion
// counter at the next 256-byte boundary: the layout ce_argmax() expects.
static __device__ __align__(256) float g_ce_noalloc_scratch[KL_CE_NOALLOC_MAX_ROWS + 1 + 64];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};   // device address of the array, per device ordinal
}  // namespace

extern "C" kl_status kl_ce_argmax_noalloc(int32_t N, int32_t V, const float* z,
                                          const int32_t* targets, float* loss, int32_t* argmax,
                                          void* dlogits, int32_t dz_dtype, void* stream) {
  using namespace kl;
  if (N < 1 || N > KL_CE_NOALLOC_MAX_ROWS)
    return set_error(KL_ERR_UNSUPPORTED,
                     "kl_ce_argmax_noalloc: N = %d rows is outside [1, %d], the size of the static scratch",
                     N, KL_CE_NOALLOC_MAX_ROWS);
  if (dz_dtype != KL_F32 && dz_dtype != KL_BF16)
    return set_error(KL_ERR_INVALID_ARG, "kl_ce_argmax_noalloc: bad dlogits dtype");
  int dev = 0;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(KL_ERR_UNSUPPORTED, "kl_ce_argmax_noalloc: device %d", dev);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_ce_noalloc_scratch);
      if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(static CE scratch)");
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  const size_t bytes = sizeof(g_ce_noalloc_scratch);
  return ce_argmax(N, V, z, targets, loss, argmax, dlogits, dz_dtype, scratch, bytes,
                   static_cast<cudaStream_t>(stream));
}

