// Host-side declarations shared by the translation units of libkl.
#pragma once

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <utility>
#include <stddef.h>
#include <stdint.h>

#include "kl.h"

namespace kl {

// ---------------------------------------------------------------------------
// GEMM: C[M,N] = sum over segments s of op(A_s) op(B_s)^T (+ R)
// ---------------------------------------------------------------------------
constexpr int GEMM_MAX_SEG = 3;
constexpr int GEMM_MAX_PROB = 4;

struct GemmSpec {
  int M = 0, N = 0;
  int nseg = 1;
  const void* A[GEMM_MAX_SEG] = {};
  int64_t lda[GEMM_MAX_SEG] = {};
  const void* B[GEMM_MAX_SEG] = {};
  int64_t ldb[GEMM_MAX_SEG] = {};
  int K[GEMM_MAX_SEG] = {};
  int a_mn = 0;  // 0: A is [M,K] (K contiguous); 1: A stored [K,M]
  int b_mn = 0;  // 0: B is [N,K]; 1: B stored [K,N]
  void* C = nullptr;
  int64_t ldc = 0;
  int c_dtype = KL_BF16;
  const void* R = nullptr;  // optional addend, [M,N] with row stride ldr
  int64_t ldr = 0;
  int r_dtype = KL_BF16;
  // Epilogue variant (bf16 operands and outputs, one segment, no addend, no K
  // split); every extra tensor is [M, N] with row stride ldc:
  //   GEMM_EPI_SWIGLU      B = gate weights, B2 = up weights ([N, K] both):
  //                        C = g, C2 = u, C3 = m = silu(g) * u, m formed from
  //                        the fp32 accumulators.
  //   GEMM_EPI_SWIGLU_BWD  the product is dm; X1 = g, X2 = u;
  //                        C = dg = dm u s (1 + g (1 - s)), C2 = du = dm g s,
  //                        s = sigmoid(g).
  //   GEMM_EPI_ROWDOT      C = the product (bf16, as usual); X1 = O; and
  //                        dot_out[(b * N/128 + h) * dot_S + t] = sum over the
  //                        128 columns of head h of bf16(C) * O for token row
  //                        b * dot_S + t (N a multiple of 128).
  // Optional compact fp32 scratch for the last round of the launch: when the
  // launch's work leaves its last round of CTA pairs partly idle, the last
  // tiles of the last problem (in execution order) are split along K,
  // accumulated here ([tiles][256][256] fp32) and finished after the launch
  // (residual added, converted). Plain-store problems only.
  float* tail_ws = nullptr;
  size_t tail_ws_bytes = 0;
  // B (and B2) are constant weights that no kernel of this library launched
  // before the GEMM writes: the few-rows kernel may then start copying them
  // before it waits for its predecessor on the stream.
  int b_const = 0;
  int epi = 0;
  const void* B2 = nullptr;
  void* C2 = nullptr;
  void* C3 = nullptr;
  const void* X1 = nullptr;
  const void* X2 = nullptr;
  float* dot_out = nullptr;
  int dot_S = 0;
  // GEMM_EPI_ROPE: columns are heads of 128; the pair (i, i + 64) of each head
  // is turned by the angle of token row % rope_S, cos/sin from rope_cs[pos][64].
  const float2* rope_cs = nullptr;
  int rope_S = 0;
};
// Bytes of tail_ws that let every launch split its last round (at most one
// 256 x 256 fp32 tile per CTA pair of the device).
size_t gemm_tail_ws_bytes();

// The driver's cuTensorMapEncodeTiled (looked up once through the runtime), or
// null if the driver has none; every TMA tensor map of the library is made with it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
constexpr int GEMM_EPI_STORE = 0;
constexpr int GEMM_EPI_SWIGLU = 1;
constexpr int GEMM_EPI_SWIGLU_BWD = 2;
constexpr int GEMM_EPI_ROWDOT = 3;
constexpr int GEMM_EPI_ROPE = 4;

// bf16 operands on the tcgen05 tensor cores; up to GEMM_MAX_PROB independent
// problems share one persistent launch.
kl_status gemm_bf16(const GemmSpec* specs, int nspec, cudaStream_t st, const char* label = "gemm");
// Few-row GEMMs (every problem M <= 128, K-major operands, plain store or
// SwiGLU): the weights stream once over one CTA per SM. gemm_bf16 routes here
// when gemm_skinny_fits (it also needs the problems' tail_ws as scratch).
bool gemm_skinny_fits(const GemmSpec* specs, int nspec);
kl_status gemm_skinny(const GemmSpec* specs, int nspec, cudaStream_t st, const char* label);
// Zeroes the few-rows GEMM's arrival counters on the current device
// (synchronous; used after a launch reported a timeout).
kl_status skinny_cnt_reset();
// Zeroes the fused RMSNorm backward's grid-barrier counters on the current
// device (synchronous; used after a launch reported a timeout).
kl_status rms_bar_reset();
// Test hooks (synchronous): leave every few-rows arrival counter, and every
// RMSNorm grid-barrier arrival counter, as a launch that gave up on a wait can
// leave it (one arrival counted, never completed).
kl_status skinny_cnt_abandon();
kl_status rms_bar_abandon();
// fp32 operands on CUDA cores (one problem).
kl_status gemm_f32(const GemmSpec& spec, cudaStream_t st, const char* label = "gemm_f32");

// ---------------------------------------------------------------------------
// elementwise / normalisation kernels (elementwise.cu)
// ---------------------------------------------------------------------------
// With rope_cs, also writes the rotary (cos, sin) table [rope_S][rope_d / 2] of
// base rope_base (in the same launch when the rows take the row form).
kl_status rmsnorm_fwd(int rows, int width, int dtype, const void* x, const void* gamma, float eps,
                      void* h, float* rstd, cudaStream_t st, int rope_S = 0, int rope_d = 0,
                      float rope_base = 0.f, float2* rope_cs = nullptr);
size_t rmsnorm_bwd_ws(int rows, int width);
kl_status rmsnorm_bwd(int rows, int width, int dtype, const void* dh, int dh_dtype, const void* x,
                      const void* gamma, const float* rstd, const void* resid, void* dx,
                      float* dgamma, void* ws, size_t ws_bytes, cudaStream_t st);
kl_status rope(int B, int S, int heads, int d, float base, int dtype, void* x, int direction,
               cudaStream_t st);
// q / k heads with the layer options: rows [T*heads, d] of `pre` -> optional
// RMSNorm over each row (gain gamma[d], rstd[row] saved) -> rotary turn, planes
// (i, i+d/2) or interleaved (2i, 2i+1); cos/sin from tab ([S][d/2]) or formed.
kl_status qk_rope_fwd(int T, int heads, int S, int d, int dtype, const void* pre, const void* gamma, float eps,
                      int norm, int inter, float base, const float2* tab, void* out, float* rstd, cudaStream_t st,
                      const int32_t* pos_off = nullptr);
// Its backward: dyr (gradient after the rotation, dy_dtype) -> dx (dtype);
// with the norm also dgamma (fp32 [d], overwritten). Workspace: qk_rope_bwd_ws.
size_t qk_rope_bwd_ws(int rows, int d);
kl_status qk_rope_bwd(int T, int heads, int S, int d, int dtype, const void* dyr, int dy_dtype, const void* pre,
                      const void* gamma, const float* rstd, int norm, int inter, float base, const float2* tab,
                      void* dx, float* dgamma, void* ws, size_t ws_bytes, cudaStream_t st);
// cs[s * d/2 + i] = (cos, sin) of the angle s * base^(-2i/d), s < S (d/2 <= 128).
kl_status rope_cs_table(int S, int d, float base, float2* cs, cudaStream_t st);
// q [T, hq, d] and k [T, hk, d] rotated in place in one launch (hk may be 0).
kl_status rope_qk(int B, int S, int hq, int hk, int d, float base, int dtype, void* q, void* k,
                  int direction, cudaStream_t st);
// Attention-backward epilogue: fp32 accumulators of dq and dk rotated back by
// the negative angle, dv converted, into dtype outputs (d a multiple of 8).
kl_status rope_bwd_convert(int B, int S, int hq, int hk, int d, float base, int dtype,
                           const float* dq_acc, const float* dk_acc, const float* dv_acc, void* dq,
                           void* dk, void* dv, cudaStream_t st);
kl_status convert_f32(int64_t n, int dtype, const float* src, void* dst, cudaStream_t st);

// paged.cu: the forward path with a paged key/value cache (bf16, d = 128)
kl_status paged_check(const kl_paged_cfg* pc, int Hq, int Hkv, int d, int dtype);
size_t paged_attention_ws(const kl_paged_cfg& pc, int Hq, int Hkv);
// One launch for a paged step's rotations and cache writes: q rotated into
// q_out, k rotated into its cache slots, v copied into its (bf16, d = 128).
kl_status paged_qkv_rope(const kl_paged_cfg& pc, int Hq, int Hkv, int d, const void* q_pre, const void* k_pre,
                         const void* v, const void* gamma_q, const void* gamma_k, float eps, int norm, int inter,
                         float base, const int32_t* table, const int32_t* ctx, void* q_out, void* k_pool, void* v_pool,
                         cudaStream_t st);
kl_status paged_kv_write(const kl_paged_cfg& pc, int Hkv, const void* k_new, const void* v_new, const int32_t* table,
                         const int32_t* ctx, void* kp, void* vp, cudaStream_t st);
kl_status paged_attention(const kl_paged_cfg& pc, int Hq, int Hkv, const void* q, const void* kp, const void* vp,
                          const int32_t* table, const int32_t* ctx, void* o, float* lse, void* ws, size_t ws_bytes,
                          cudaStream_t st);
kl_status swiglu_fwd(int64_t n, int dtype, const void* g, const void* u, void* m, cudaStream_t st);
kl_status swiglu_bwd(int64_t n, int dtype, const void* dm, const void* g, const void* u, void* dg,
                     void* du, cudaStream_t st);

// ---------------------------------------------------------------------------
// attention (attention.cu)
// ---------------------------------------------------------------------------
kl_status attention_fwd(int B, int S, int Hq, int Hkv, int d, int dtype, const void* q,
                        const void* k, const void* v, void* o, float* lse, cudaStream_t st);
// bf16, head dim 128, on the tcgen05 tensor cores (attention_tc.cu).
kl_status attention_fwd_tc(int B, int S, int Hq, int Hkv, const void* q, const void* k, const void* v,
                           void* o, float* lse, cudaStream_t st);
// Backward on the tcgen05 tensor cores. dK and dV (summed over each kv head's
// query heads) are written once as bf16 into dk_out / dv_out; dQ as bf16 into
// dq_out or, when that is null, as fp32 into dq_acc. With rope_cs ([S][64]
// cos/sin) dQ (bf16) and dK leave turned back by the rotary angle.
kl_status attention_bwd_tc(int B, int S, int Hq, int Hkv, const void* q, const void* k, const void* v,
                           const void* dout, const float* lse, const float* Dd, float* dq_acc, void* dq_out,
                           void* dk_out, void* dv_out, const float2* rope_cs, cudaStream_t st);
// CTAs (a cluster) that share one kv head's key tile in the dK/dV kernel.
int attention_dkdv_split(int B, int S, int Hq, int Hkv, int sms);
size_t attention_bwd_ws(int B, int S, int Hq, int Hkv, int d);
// fp32: dQ, dK, dV as fp32 accumulators [T, H*d] inside ws (*dq_acc, *dk_acc,
// *dv_acc); the caller converts them (with the rotary backward) afterwards.
// bf16 (tensor cores): dK and dV go straight to dk_out / dv_out as bf16 and dQ
// to dq_out (required), dQ and dK turned back by the rotary angles of rope_cs
// ([S][d/2] cos/sin) when that is given; the three accumulator pointers are
// null. The workspace starts with D = rowsum(dO * O) as fp32 [B, Hq, S];
// d_ready (bf16) means the caller has already written it there
// (attention_bwd_d_rows).
inline float* attention_bwd_d_rows(void* ws) { return static_cast<float*>(ws); }
kl_status attention_bwd_accum(int B, int S, int Hq, int Hkv, int d, int dtype, const void* q,
                              const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* ws, size_t ws_bytes, float** dq_acc,
                              float** dk_acc, float** dv_acc, cudaStream_t st,
                              bool d_ready = false, void* dq_out = nullptr,
                              const float2* rope_cs = nullptr, void* dk_out = nullptr,
                              void* dv_out = nullptr);

// ---------------------------------------------------------------------------
// cross entropy (ce.cu)
// ---------------------------------------------------------------------------
size_t ce_ws(int N);
kl_status ce_argmax(int N, int V, const float* z, const int32_t* targets, float* loss,
                    int32_t* argmax, void* dz, int dz_dtype, void* ws, size_t ws_bytes,
                    cudaStream_t st);

// Launches `kern` on `st` with programmatic stream serialization: the grid may
// be scheduled while the stream's previous kernel drains; the kernel itself
// waits for that kernel's completion first thing (pdl_enter). Arguments are
// converted to the kernel's parameter types. Launch errors are also left for
// cudaGetLastError.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Whether the launch profiler is on (kl_profile_enable): launches that would
// overlap on two streams then run one after the other, so that each one's
// event-timed duration is its own.
bool profiling_on();

// Counts a kernel launch and, while profiling is on, brackets it with CUDA
// events on `st` (construct immediately before the launch; the destructor
// records the stop event right after it). `flops` and `bytes` are the
// launch's algorithmic work.
class ProfScope {
 public:
  ProfScope(const char* name, cudaStream_t st, double flops, double bytes);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  cudaStream_t st_;
  int ev_;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t dtype_size(int dt) { return dt == KL_F32 ? 4 : 2; }

}  // namespace kl
