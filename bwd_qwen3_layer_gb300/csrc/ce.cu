// Softmax cross-entropy + argmax + dlogits in a single launch ("From-scratch
// GPU LLM training", capability list: GPU lm-head, softmax cross-entropy and
// argmax fused in a single launch).
//
// One row of fp32 logits per 8-CTA thread-block cluster, each CTA a slice of
// the vocabulary. Pass 1 reads the slice once and keeps per-thread running
// summaries (maximum, sum of exponentials against it, lowest argmax); the
// summaries merge across the warp, the CTA and the cluster (distributed shared
// memory, rank order) into the row's logsumexp and argmax. Pass 2 reads the
// slice again from L2 and writes dlogits = (softmax - onehot) / N once. The
// mean loss is reduced in a fixed order by the last cluster to finish
// (deterministic).
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>
#include <stdlib.h>

#include <mutex>

#include "internal.h"
#include "kl_common.cuh"

namespace cg = cooperative_groups;

namespace kl {
namespace {

// CTAs per row (cluster size, a template parameter: 8 portable, 16 with the
// non-portable opt-in) and threads per CTA.
constexpr int THREADS = 256;
constexpr int NWARP = THREADS / 32;
constexpr float LOG2E = 1.4426950408889634f;

// Pass 1 marks the logits it reads for keeping in L2 (evict-last), pass 2
// reads them for the last time (evict-first), so the ~150 rows in flight stay
// in L2 between the passes; dlogits are written evict-first.
struct f8 {
  float v[8];
};
// 32-byte loads (Blackwell's 256-bit form, which carries the L2 priority)
__device__ __forceinline__ f8 ld_keep(const float* p) {
  f8 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_last.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]), "=f"(r.v[6]),
                 "=f"(r.v[7])
               : "l"(p));
  return r;
}
__device__ __forceinline__ f8 ld_last(const float* p) {
  f8 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]), "=f"(r.v[6]),
                 "=f"(r.v[7])
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 2^x by the hardware approximation (about 2 ulp; 0 for -inf).
__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Part {
  float m;
  float s;
  int idx;
};

// (m, s, idx) summarises a set of logits: its maximum m, the sum s of
// exp(z - m) over it, and the lowest index attaining m. Merging two summaries
// is exact up to the rescaling's rounding.
__device__ __forceinline__ void merge(float& m, float& s, int& i, float m2, float s2, int i2) {
  if (m2 > m) {
    s = (m > -INFINITY ? s * ex2a((m - m2) * LOG2E) : 0.f) + s2;
    m = m2;
    i = i2;
  } else {
    if (m2 > -INFINITY) s += s2 * ex2a((m2 - m) * LOG2E);
    if (m2 == m && i2 < i) i = i2;
  }
}

// Adds eight logits a[0..7] at indices j0 .. j0 + 7 (increasing, after every
// index already summarised by this thread, so a tie never moves the argmax)
// to the running summary (m, s, idx), with mL = m log2 e kept alongside: one
// max of the eight, a rescale only when it exceeds the running max, then
// eight exponentials into the sum.
__device__ __forceinline__ void add_logits8(float& m, float& mL, float& s, int& i, const float (&a)[8], int j0) {
  float cm = fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
  if (cm > m) {
    s = m > -INFINITY ? s * ex2a(mL - cm * LOG2E) : 0.f;
    m = cm;
    mL = cm * LOG2E;
    int k = 7;
#pragma unroll
    for (int e = 6; e >= 0; --e)
      if (a[e] == cm) k = e;
    i = j0 + k;
  }
  if (m > -INFINITY) {
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) t += ex2a(fmaf(a[e], LOG2E, -mL));
    s += t;
  }
}

// Adds logit z at index j to the running summary (m, s, idx).
__device__ __forceinline__ void add_logit(float& m, float& s, int& i, float z, int j) {
  if (z > m) {
    s = (m > -INFINITY ? s * ex2a((m - z) * LOG2E) : 0.f) + 1.f;
    m = z;
    i = j;
  } else if (z > -INFINITY) {
    s += ex2a((z - m) * LOG2E);
    if (z == m && j < i) i = j;
  }
}

// One row of logits per cluster of CLUSTER CTAs; CTA r takes the r-th slice
// of the vocabulary. Pass 1 streams the slice once from HBM into per-thread
// running summaries (maximum, sum of exponentials against it, lowest argmax),
// merged across the warp, the CTA and (through distributed shared memory, in
// rank order) the cluster into the row's logsumexp and argmax. Pass 2 reads
// the slice again, from L2 (the rows in flight fit there), and writes
// dlogits = (softmax - onehot) / N. No tile is held in shared memory, so eight
// CTAs fit on an SM and keep enough loads in flight to stream at HBM rate.
template <int CLUSTER, bool VEC>
__global__ void __launch_bounds__(THREADS)
    ce_argmax_kernel(int N, int V, int slice, const float* __restrict__ z,
                     const int32_t* __restrict__ targets, float* __restrict__ loss_rows,
                     int32_t* __restrict__ argmax, void* __restrict__ dz, int dz_f32, float invN,
                     unsigned int* __restrict__ counter, float* __restrict__ loss,
                     uint32_t* __restrict__ err) {
  pdl_enter();
  __shared__ float red_m[NWARP];
  __shared__ float red_s[NWARP];
  __shared__ int red_i[NWARP];
  __shared__ Part part;
  __shared__ int is_last;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int n = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = rank * slice;
  const int len = max(0, min(V, c0 + slice) - c0);
  const float* zr = z + static_cast<int64_t>(n) * V + c0;

  // 1. running summary of this thread's logits (32-byte loads, two in flight)
  float m = -INFINITY, s = 0.f;
  int mi = INT_MAX;
  if (VEC) {
    constexpr int U = 2;
    float mL = -INFINITY;
    int i = threadIdx.x * 8;
    for (; i + (U - 1) * THREADS * 8 < len; i += U * THREADS * 8) {
      f8 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] = ld_keep(zr + i + u * THREADS * 8);
#pragma unroll
      for (int u = 0; u < U; ++u) add_logits8(m, mL, s, mi, a[u].v, c0 + i + u * THREADS * 8);
    }
    for (; i < len; i += THREADS * 8) {
      const f8 a = ld_keep(zr + i);
      add_logits8(m, mL, s, mi, a.v, c0 + i);
    }
  } else {
    for (int i = threadIdx.x; i < len; i += THREADS) add_logit(m, s, mi, zr[i], c0 + i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, mi, o);
    merge(m, s, mi, m2, s2, i2);
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = s;
    red_i[warp] = mi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tm = red_m[0], ts = red_s[0];
    int ti = red_i[0];
    for (int w = 1; w < NWARP; ++w) merge(tm, ts, ti, red_m[w], red_s[w], red_i[w]);
    part.m = tm;
    part.s = ts;
    part.idx = ti;
  }
  cluster.sync();
  // 2. the row's summary from the CLUSTER slices (every CTA, fixed rank order)
  float M = -INFINITY, tot = 0.f;
  int I = INT_MAX;
#pragma unroll
  for (int r = 0; r < CLUSTER; ++r) {
    const Part q = *cluster.map_shared_rank(&part, r);
    merge(M, tot, I, q.m, q.s, q.idx);
  }
  const float lse = M + logf(tot);
  const float lsel = lse * LOG2E;
  int t = targets[n];
  const bool t_ok = t >= 0 && t < V;
  if (!t_ok) {
    if (threadIdx.x == 0 && rank == 0) record_error(err, KL_DEVERR_TARGET);
    t = -1;
  }
  // 3. dlogits for this slice (the logits again, now from L2)
  if (dz_f32) {
    float* out = static_cast<float*>(dz) + static_cast<int64_t>(n) * V + c0;
    for (int i = threadIdx.x; i < len; i += THREADS) {
      float p = ex2a(fmaf(zr[i], LOG2E, -lsel));
      if (c0 + i == t) p -= 1.f;
      out[i] = p * invN;
    }
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(dz) + static_cast<int64_t>(n) * V + c0;
    if (VEC) {
      // softmax / N = 2^(z log2 e - lse log2 e + log2(1/N)): the 1/N rides in the exponent
      const float off = -lsel + log2f(invN);
#pragma unroll 2
      for (int i = threadIdx.x * 8; i < len; i += THREADS * 8) {
        const f8 a = ld_last(zr + i);
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = ex2a(fmaf(a.v[e], LOG2E, off));
        const int d = t - (c0 + i);
        if (d >= 0 && d < 8) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e == d) p[e] -= invN;
        }
        uint4 o;
        o.x = pack_bf16x2(p[0], p[1]);
        o.y = pack_bf16x2(p[2], p[3]);
        o.z = pack_bf16x2(p[4], p[5]);
        o.w = pack_bf16x2(p[6], p[7]);
        st_stream(out + i, o);
      }
    } else {
      for (int i = threadIdx.x; i < len; i += THREADS) {
        float p = ex2a(fmaf(zr[i], LOG2E, -lsel));
        if (c0 + i == t) p -= 1.f;
        out[i] = __float2bfloat16_rn(p * invN);
      }
    }
  }
  // 4. per-row loss and argmax; the last row to finish reduces the mean
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

// CTAs per row. Tuning override: KL_CE_CLUSTER = 8 or 16.
int ce_cluster_size(int V) {
  (void)V;
  if (const char* e = getenv("KL_CE_CLUSTER")) {
    const int v = atoi(e);
    if (v == 8 || v == 16) return v;
  }
  return 8;
}

kl_status ce_argmax(int N, int V, const float* z, const int32_t* targets, float* loss,
                    int32_t* argmax, void* dz, int dz_dtype, void* ws, size_t ws_bytes,
                    cudaStream_t st) {
  if (N < 1 || V < 1 || !z || !targets || !loss || !argmax || !dz)
    return set_error(KL_ERR_INVALID_ARG, "ce_argmax: bad arguments");
  if (N > 65535) return set_error(KL_ERR_UNSUPPORTED, "ce_argmax: N above 65535");
  if (!ws || ws_bytes < ce_ws(N)) return set_error(KL_ERR_NO_MEMORY, "ce_argmax: workspace too small");
  {
    // dlogits must not overlap the logits: a row's loss reads its target logit
    // after the other CTAs of the row have written their dlogits slices
    const uintptr_t z0 = reinterpret_cast<uintptr_t>(z), d0 = reinterpret_cast<uintptr_t>(dz);
    const uintptr_t nv = static_cast<uintptr_t>(N) * static_cast<uintptr_t>(V);
    if (z0 < d0 + nv * dtype_size(dz_dtype) && d0 < z0 + nv * 4)
      return set_error(KL_ERR_INVALID_ARG, "ce_argmax: dlogits overlaps the logits");
  }
  // the vector path: 32-byte logit loads, 16-byte bf16 dlogit stores
  const bool vec = V % 8 == 0 && (reinterpret_cast<uintptr_t>(z) & 31u) == 0 &&
                   (dz_dtype == KL_F32 || (reinterpret_cast<uintptr_t>(dz) & 15u) == 0);
  const int CL = ce_cluster_size(V);
  int slice = (V + CL - 1) / CL;
  slice = (slice + 7) / 8 * 8;
  float* loss_rows = static_cast<float*>(ws);
  unsigned int* counter =
      reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + align_up(static_cast<size_t>(N) * 4, 256));
  KL_CUDA(cudaMemsetAsync(counter, 0, sizeof(unsigned int), st));
  dim3 grid(CL, N);
  ProfScope ps("ce_argmax", st, 0.0, static_cast<double>(N) * V * (4 + dtype_size(dz_dtype)) + 12.0 * N);
  const float invN = 1.0f / static_cast<float>(N);
  const int f32 = dz_dtype == KL_F32;
  auto launch = [&](auto kernel) -> kl_status {
    if (CL > 8) KL_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_enter
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    KL_CUDA(cudaLaunchKernelEx(&cfg, kernel, N, V, slice, z, targets, loss_rows, argmax, dz, f32, invN, counter, loss,
                               device_error_word()));
    return KL_OK;
  };
  if (CL == 16) {
    if (vec) KL_TRY(launch(ce_argmax_kernel<16, true>));
    else KL_TRY(launch(ce_argmax_kernel<16, false>));
  } else {
    if (vec) KL_TRY(launch(ce_argmax_kernel<8, true>));
    else KL_TRY(launch(ce_argmax_kernel<8, false>));
  }
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

