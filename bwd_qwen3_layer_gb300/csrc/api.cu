// C ABI of libkl (declared in include/kl.h): argument checks, status
// plumbing, buffer carving and the layer / lm-head orchestration. Every step
// runs in the kernels of gemm.cu, elementwise.cu, attention.cu and ce.cu on
// the caller's stream; nothing here synchronises except kl_device_status.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {

static thread_local char g_last_error[512] = "";

kl_status set_error(kl_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

kl_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaErrorMemoryAllocation)
    return set_error(KL_ERR_NO_MEMORY, "%s: %s", what, cudaGetErrorString(e));
  return set_error(KL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One 32-bit error word per device, in static device memory (no allocation).
__device__ uint32_t g_device_error_word;

uint32_t* device_error_word() {
  static uint32_t* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

int num_sms() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kl_status run_gemms(int dtype, GemmSpec* specs, int n, cudaStream_t st, const char* label) {
  if (dtype == KL_BF16) return gemm_bf16(specs, n, st, label);
  for (int i = 0; i < n; ++i) KL_TRY(gemm_f32(specs[i], st, label));
  return KL_OK;
}

// C[M,N] = A[M,K] B[N,K]^T with both operands K-major (a forward projection).
GemmSpec proj(int M, int N, int K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
              int64_t ldc, int c_dtype, const void* R = nullptr, int r_dtype = KL_BF16) {
  GemmSpec s;
  s.M = M; s.N = N; s.nseg = 1;
  s.A[0] = A; s.lda[0] = lda; s.B[0] = B; s.ldb[0] = ldb; s.K[0] = K;
  s.a_mn = 0; s.b_mn = 0;
  s.C = C; s.ldc = ldc; s.c_dtype = c_dtype;
  s.R = R; s.ldr = ldc; s.r_dtype = r_dtype;
  s.b_const = 1;   // every caller passes a layer weight as B
  return s;
}

// dW[M=out, N=in] = dY[T,out]^T X[T,in]: both operands MN-major, K = T.
GemmSpec wgrad(int out, int in, int T, const void* dY, const void* X, void* dW, int dw_dtype) {
  GemmSpec s;
  s.M = out; s.N = in; s.nseg = 1;
  s.A[0] = dY; s.lda[0] = out; s.B[0] = X; s.ldb[0] = in; s.K[0] = T;
  s.a_mn = 1; s.b_mn = 1;
  s.C = dW; s.ldc = in; s.c_dtype = dw_dtype;
  return s;
}

// dX[T, in] = dY[T, out] W[out, in]: A K-major, B MN-major, K = out.
GemmSpec dgrad(int T, int in, int out, const void* dY, const void* W, void* dX, int dx_dtype) {
  GemmSpec s;
  s.M = T; s.N = in; s.nseg = 1;
  s.A[0] = dY; s.lda[0] = out; s.B[0] = W; s.ldb[0] = in; s.K[0] = out;
  s.a_mn = 0; s.b_mn = 1;
  s.C = dX; s.ldc = in; s.c_dtype = dx_dtype;
  return s;
}

struct Dims {
  int B, S, T, H, Hq, Hkv, d, I, Dq, Dkv;
  int dt;
  size_t es;
  int qk_norm, inter;   // layer options: per-head q/k RMSNorm, interleaved rotary planes
};

kl_status check_cfg(const kl_layer_cfg* c, Dims* o) {
  if (!c) return set_error(KL_ERR_INVALID_ARG, "null cfg");
  if (c->B < 1 || c->S < 1 || c->H < 1 || c->Hq < 1 || c->Hkv < 1 || c->d < 8 || c->I < 1 ||
      (c->d % 8) || c->Hq % c->Hkv || c->eps < 0.f || !(c->rope_base > 0.f))
    return set_error(KL_ERR_INVALID_ARG, "bad layer cfg (B %d S %d H %d Hq %d Hkv %d d %d I %d)",
                     c->B, c->S, c->H, c->Hq, c->Hkv, c->d, c->I);
  if (c->dtype != KL_BF16 && c->dtype != KL_F32)
    return set_error(KL_ERR_INVALID_ARG, "bad dtype %d", c->dtype);
  const int64_t T = static_cast<int64_t>(c->B) * c->S;
  if (T > (1 << 24)) return set_error(KL_ERR_UNSUPPORTED, "too many tokens");
  if (c->dtype == KL_BF16) {
    if (c->d != 128) return set_error(KL_ERR_UNSUPPORTED, "bf16 layer needs head dim 128");
    if (c->H % 8 || c->I % 8)
      return set_error(KL_ERR_UNSUPPORTED, "bf16 layer needs H and I multiples of 8");
  } else if (c->d > 256) {
    return set_error(KL_ERR_UNSUPPORTED, "fp32 layer needs head dim <= 256");
  }
  if (c->H * 4 > 48 * 1024) return set_error(KL_ERR_UNSUPPORTED, "hidden width above 12288");
  if ((c->qk_norm != 0 && c->qk_norm != 1) || (c->rope_interleaved != 0 && c->rope_interleaved != 1))
    return set_error(KL_ERR_INVALID_ARG, "qk_norm and rope_interleaved are 0 or 1");
  o->B = c->B; o->S = c->S; o->T = static_cast<int>(T); o->H = c->H; o->Hq = c->Hq;
  o->Hkv = c->Hkv; o->d = c->d; o->I = c->I; o->Dq = c->Hq * c->d; o->Dkv = c->Hkv * c->d;
  o->dt = c->dtype;
  o->es = dtype_size(c->dtype);
  o->qk_norm = c->qk_norm;
  o->inter = c->rope_interleaved;
  return KL_OK;
}

// Carves consecutive 256-byte aligned pieces out of one buffer.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += align_up(bytes, 256);
    return p;
  }
};

// The rotary (cos, sin) table [S][d/2] used by the fused q/k projection, dQ and dK epilogues.
size_t rope_table_bytes(const Dims& D) { return align_up(static_cast<size_t>(D.S) * (D.d / 2) * 8, 256); }

void carve_saved(const Dims& D, Carver& c, kl_layer_saved* s) {
  const size_t T = D.T, es = D.es;
  s->h1 = c.take(T * D.H * es);
  s->rstd1 = static_cast<float*>(c.take(T * 4));
  s->q = c.take(T * D.Dq * es);
  s->k = c.take(T * D.Dkv * es);
  s->v = c.take(T * D.Dkv * es);
  s->o = c.take(T * D.Dq * es);
  s->lse = static_cast<float*>(c.take(static_cast<size_t>(D.B) * D.Hq * D.S * 4));
  s->x2 = c.take(T * D.H * es);
  s->h2 = c.take(T * D.H * es);
  s->rstd2 = static_cast<float*>(c.take(T * 4));
  s->g = c.take(T * D.I * es);
  s->u = c.take(T * D.I * es);
  s->m = c.take(T * D.I * es);
  if (D.qk_norm) {
    s->q_pre = c.take(T * D.Dq * es);
    s->k_pre = c.take(T * D.Dkv * es);
    s->rstd_q = static_cast<float*>(c.take(T * D.Hq * 4));
    s->rstd_k = static_cast<float*>(c.take(T * D.Hkv * 4));
  } else {
    s->q_pre = s->k_pre = nullptr;
    s->rstd_q = s->rstd_k = nullptr;
  }
  s->rope = D.dt == KL_BF16 ? static_cast<float*>(c.take(rope_table_bytes(D))) : nullptr;
}

struct BwdWs {
  void *dm, *dg, *du, *dx2, *dO, *dq, *dk, *dv;
  float *dh2, *dh1;
  void* att;
  size_t att_bytes;
  void* norm;
  size_t norm_bytes;
  void* tail;             // fp32 scratch balancing the GEMM launches' last rounds (bf16)
  size_t tail_bytes;
  void *qk_q, *qk_k;      // gain-gradient partials of the per-head q / k norms (qk_norm)
  size_t qk_q_bytes, qk_k_bytes;
};

void carve_bwd(const Dims& D, Carver& c, BwdWs* w) {
  const size_t T = D.T, es = D.es;
  w->dm = c.take(T * D.I * es);
  w->dg = c.take(T * D.I * es);
  w->du = c.take(T * D.I * es);
  w->dh2 = static_cast<float*>(c.take(T * D.H * 4));
  w->dx2 = c.take(T * D.H * es);
  w->dO = c.take(T * D.Dq * es);
  w->dq = c.take(T * D.Dq * es);
  w->dk = c.take(T * D.Dkv * es);
  w->dv = c.take(T * D.Dkv * es);
  w->dh1 = static_cast<float*>(c.take(T * D.H * 4));
  w->att_bytes = attention_bwd_ws(D.B, D.S, D.Hq, D.Hkv, D.d);
  w->att = c.take(w->att_bytes);
  w->norm_bytes = rmsnorm_bwd_ws(D.T, D.H);
  w->norm = c.take(w->norm_bytes);
  w->tail_bytes = D.dt == KL_BF16 ? gemm_tail_ws_bytes() : 0;
  w->tail = w->tail_bytes ? c.take(w->tail_bytes) : nullptr;
  w->qk_q_bytes = D.qk_norm ? qk_rope_bwd_ws(D.T * D.Hq, D.d) : 0;
  w->qk_k_bytes = D.qk_norm ? qk_rope_bwd_ws(D.T * D.Hkv, D.d) : 0;
  w->qk_q = D.qk_norm ? c.take(w->qk_q_bytes) : nullptr;
  w->qk_k = D.qk_norm ? c.take(w->qk_k_bytes) : nullptr;
}

// Workspace of the paged-cache layer forward: the step's activations (T = B *
// n_new rows), the attention split partials and the GEMMs' last-round scratch.
struct PagedWs {
  void *h1, *q_pre, *k_pre, *v, *q, *k, *o, *x2, *h2, *g, *u, *m;
  float *rstd1, *rstd2, *rstd_q, *rstd_k;
  void* att;
  size_t att_bytes;
  void* tail;
  size_t tail_bytes;
};

void carve_paged(const Dims& D, const kl_paged_cfg& pc, Carver& c, PagedWs* w) {
  const size_t T = D.T, es = D.es;
  w->h1 = c.take(T * D.H * es);
  w->rstd1 = static_cast<float*>(c.take(T * 4));
  w->q_pre = c.take(T * D.Dq * es);
  w->k_pre = c.take(T * D.Dkv * es);
  w->v = c.take(T * D.Dkv * es);
  w->q = c.take(T * D.Dq * es);
  w->k = c.take(T * D.Dkv * es);
  w->rstd_q = static_cast<float*>(c.take(T * D.Hq * 4));
  w->rstd_k = static_cast<float*>(c.take(T * D.Hkv * 4));
  w->o = c.take(T * D.Dq * es);
  w->x2 = c.take(T * D.H * es);
  w->h2 = c.take(T * D.H * es);
  w->rstd2 = static_cast<float*>(c.take(T * 4));
  w->g = c.take(T * D.I * es);
  w->u = c.take(T * D.I * es);
  w->m = c.take(T * D.I * es);
  w->att_bytes = paged_attention_ws(pc, D.Hq, D.Hkv);
  w->att = w->att_bytes ? c.take(w->att_bytes) : nullptr;
  w->tail_bytes = gemm_tail_ws_bytes();
  w->tail = c.take(w->tail_bytes);
}

kl_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
  for (const void* p : ptrs) {
    if (!p) return set_error(KL_ERR_INVALID_ARG, "%s: null pointer", what);
    if (!al16(p)) return set_error(KL_ERR_INVALID_ARG, "%s: pointer not 16-byte aligned", what);
  }
  return KL_OK;
}

}  // namespace
}  // namespace kl

using namespace kl;

extern "C" {

const char* kl_version(void) { return "kl 0.1 (sm_103a)"; }

const char* kl_status_str(kl_status s) {
  switch (s) {
    case KL_OK: return "ok";
    case KL_ERR_INVALID_ARG: return "invalid argument";
    case KL_ERR_UNSUPPORTED: return "unsupported";
    case KL_ERR_CUDA: return "cuda error";
    case KL_ERR_TIMEOUT: return "timeout";
    case KL_ERR_NO_MEMORY: return "no memory";
    case KL_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

const char* kl_last_error(void) { return g_last_error; }

kl_status kl_device_status(void* stream, uint32_t* bits) {
  KL_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  uint32_t v = 0;
  KL_CUDA(cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof(v)));
  const uint32_t zero = 0;
  KL_CUDA(cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero)));
  if (bits) *bits = v;
  if (v & KL_DEVERR_TIMEOUT) {
    // a few-rows GEMM or a fused RMSNorm backward that gave up may have left arrival counts behind
    kl_status rs = skinny_cnt_reset();
    if (rs == KL_OK) rs = rms_bar_reset();
    if (rs != KL_OK) return rs;
    return set_error(KL_ERR_TIMEOUT, "a kernel wait timed out (bits 0x%x)", v);
  }
  if (v) return set_error(KL_ERR_DEVICE, "a kernel rejected its input (bits 0x%x)", v);
  return KL_OK;
}

kl_status kl_test_abandon_counters(void) {
  KL_CUDA(cudaDeviceSynchronize());
  KL_TRY(skinny_cnt_abandon());
  KL_TRY(rms_bar_abandon());
  uint32_t v = 0;
  KL_CUDA(cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof(v)));
  v |= KL_DEVERR_TIMEOUT;
  KL_CUDA(cudaMemcpyToSymbol(g_device_error_word, &v, sizeof(v)));
  return KL_OK;
}

size_t kl_layer_saved_bytes(const kl_layer_cfg* cfg) {
  Dims D;
  if (check_cfg(cfg, &D) != KL_OK) return 0;
  Carver c(nullptr);
  kl_layer_saved s;
  carve_saved(D, c, &s);
  return c.off;
}

kl_status kl_layer_saved_carve(const kl_layer_cfg* cfg, void* base, size_t bytes,
                               kl_layer_saved* out) {
  Dims D;
  KL_TRY(check_cfg(cfg, &D));
  if (!base || !out) return set_error(KL_ERR_INVALID_ARG, "saved_carve: null pointer");
  if (reinterpret_cast<uintptr_t>(base) & 255u)
    return set_error(KL_ERR_INVALID_ARG, "saved_carve: base not 256-byte aligned");
  Carver c(base);
  kl_layer_saved s;
  memset(&s, 0, sizeof(s));
  carve_saved(D, c, &s);
  if (c.off > bytes) return set_error(KL_ERR_NO_MEMORY, "saved_carve: need %zu bytes", c.off);
  *out = s;
  return KL_OK;
}

size_t kl_layer_fwd_workspace_bytes(const kl_layer_cfg* cfg) {
  Dims D;
  if (check_cfg(cfg, &D) != KL_OK) return 0;
  return D.dt == KL_BF16 ? gemm_tail_ws_bytes() : 256;
}

size_t kl_layer_bwd_workspace_bytes(const kl_layer_cfg* cfg) {
  Dims D;
  if (check_cfg(cfg, &D) != KL_OK) return 0;
  Carver c(nullptr);
  BwdWs w;
  carve_bwd(D, c, &w);
  return c.off;
}

// Gives every spec of a launch the fp32 scratch that balances its last round.
void with_tail(GemmSpec* g, int n, void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return;
  for (int i = 0; i < n; ++i) {
    g[i].tail_ws = static_cast<float*>(ws);
    g[i].tail_ws_bytes = bytes;
  }
}

kl_status kl_layer_forward(const kl_layer_cfg* cfg, const kl_layer_weights* w, const void* X,
                           void* Y, kl_layer_saved* s, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  KL_TRY(check_cfg(cfg, &D));
  if (!w || !s) return set_error(KL_ERR_INVALID_ARG, "layer_forward: null weights or saved");
  KL_TRY(check_ptrs({w->gamma1, w->wq, w->wk, w->wv, w->wo, w->gamma2, w->wg, w->wu, w->wd}, "layer_forward weights"));
  KL_TRY(check_ptrs({X, Y, s->h1, s->rstd1, s->q, s->k, s->v, s->o, s->lse, s->x2, s->h2, s->rstd2,
                     s->g, s->u, s->m}, "layer_forward buffers"));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = D.T, H = D.H, I = D.I, dt = D.dt;
  if (D.qk_norm) {
    KL_TRY(check_ptrs({w->gamma_q, w->gamma_k}, "layer_forward q/k norm gains"));
    KL_TRY(check_ptrs({s->q_pre, s->k_pre, s->rstd_q, s->rstd_k}, "layer_forward q/k norm buffers"));
  }
  // bf16: the rotary table is written with the first norm into the saved set (the
  // rotation fused into the q/k projection's epilogue when neither layer option is
  // on; the backward reads the same table); with the workspace, the projections'
  // last round of tiles is split along K
  const bool bf = dt == KL_BF16;
  if (bf && !s->rope) return set_error(KL_ERR_INVALID_ARG, "layer_forward: saved rotary table missing");
  const bool fused = bf && ws && ws_bytes >= kl_layer_fwd_workspace_bytes(cfg) &&
                     (reinterpret_cast<uintptr_t>(ws) & 255u) == 0;
  const bool options = D.qk_norm || D.inter;
  const size_t tail_bytes = fused ? gemm_tail_ws_bytes() : 0;
  float2* rope_tab = bf ? reinterpret_cast<float2*>(s->rope) : nullptr;
  s->x = X;
  KL_TRY(rmsnorm_fwd(T, H, dt, X, w->gamma1, cfg->eps, s->h1, s->rstd1, st, D.S, D.d, cfg->rope_base, rope_tab));
  {
    // with the q/k norm the projections land in q_pre / k_pre first
    void* qdst = D.qk_norm ? s->q_pre : s->q;
    void* kdst = D.qk_norm ? s->k_pre : s->k;
    GemmSpec g[3] = {proj(T, D.Dq, H, s->h1, H, w->wq, H, qdst, D.Dq, dt),
                     proj(T, D.Dkv, H, s->h1, H, w->wk, H, kdst, D.Dkv, dt),
                     proj(T, D.Dkv, H, s->h1, H, w->wv, H, s->v, D.Dkv, dt)};
    if (fused) with_tail(g, 3, ws, tail_bytes);
    for (int i = 0; i < 2 && bf && !options; ++i) {   // q and k leave the epilogue rotated
      g[i].epi = GEMM_EPI_ROPE;
      g[i].rope_cs = rope_tab;
      g[i].rope_S = D.S;
    }
    KL_TRY(run_gemms(dt, g, 3, st, "gemm.fwd_qkv"));
  }
  if (options) {
    // optional per-head norm, then the rotation (pairs of either layout)
    const void* qsrc = D.qk_norm ? s->q_pre : s->q;
    const void* ksrc = D.qk_norm ? s->k_pre : s->k;
    KL_TRY(qk_rope_fwd(T, D.Hq, D.S, D.d, dt, qsrc, w->gamma_q, cfg->eps, D.qk_norm, D.inter, cfg->rope_base,
                       rope_tab, s->q, s->rstd_q, st));
    KL_TRY(qk_rope_fwd(T, D.Hkv, D.S, D.d, dt, ksrc, w->gamma_k, cfg->eps, D.qk_norm, D.inter, cfg->rope_base,
                       rope_tab, s->k, s->rstd_k, st));
  } else if (!bf) {
    KL_TRY(rope_qk(D.B, D.S, D.Hq, D.Hkv, D.d, cfg->rope_base, dt, s->q, s->k, 1, st));
  }
  KL_TRY(attention_fwd(D.B, D.S, D.Hq, D.Hkv, D.d, dt, s->q, s->k, s->v, s->o, s->lse, st));
  {
    GemmSpec g = proj(T, H, D.Dq, s->o, D.Dq, w->wo, D.Dq, s->x2, H, dt, X, dt);
    if (fused) with_tail(&g, 1, ws, tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.fwd_o"));
  }
  KL_TRY(rmsnorm_fwd(T, H, dt, s->x2, w->gamma2, cfg->eps, s->h2, s->rstd2, st));
  if (dt == KL_BF16) {
    // g and u of the same 128 columns in one tile; m = silu(g) u in the epilogue
    GemmSpec g = proj(T, I, H, s->h2, H, w->wg, H, s->g, I, dt);
    g.epi = GEMM_EPI_SWIGLU;
    g.B2 = w->wu;
    g.C2 = s->u;
    g.C3 = s->m;
    if (fused) with_tail(&g, 1, ws, tail_bytes);   // scratch of the few-rows kernel
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.fwd_gateup"));
  } else {
    GemmSpec g[2] = {proj(T, I, H, s->h2, H, w->wg, H, s->g, I, dt),
                     proj(T, I, H, s->h2, H, w->wu, H, s->u, I, dt)};
    KL_TRY(run_gemms(dt, g, 2, st, "gemm.fwd_gateup"));
    KL_TRY(swiglu_fwd(static_cast<int64_t>(T) * I, dt, s->g, s->u, s->m, st));
  }
  {
    GemmSpec g = proj(T, H, I, s->m, I, w->wd, I, Y, H, dt, s->x2, dt);
    if (fused) with_tail(&g, 1, ws, tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.fwd_down"));
  }
  return KL_OK;
}

kl_status kl_layer_backward(const kl_layer_cfg* cfg, const kl_layer_weights* w,
                            const kl_layer_saved* s, const void* dY, void* dX,
                            const kl_layer_grads* gr, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  KL_TRY(check_cfg(cfg, &D));
  if (!w || !s || !gr) return set_error(KL_ERR_INVALID_ARG, "layer_backward: null struct");
  KL_TRY(check_ptrs({w->gamma1, w->wq, w->wk, w->wv, w->wo, w->gamma2, w->wg, w->wu, w->wd}, "layer_backward weights"));
  KL_TRY(check_ptrs({s->x, s->h1, s->rstd1, s->q, s->k, s->v, s->o, s->lse, s->x2, s->h2,
                     s->rstd2, s->g, s->u, s->m}, "layer_backward saved"));
  KL_TRY(check_ptrs({dY, dX, gr->gamma1, gr->wq, gr->wk, gr->wv, gr->wo, gr->gamma2, gr->wg,
                     gr->wu, gr->wd}, "layer_backward outputs"));
  if (gr->dtype != KL_F32 && gr->dtype != KL_BF16)
    return set_error(KL_ERR_INVALID_ARG, "layer_backward: bad gradient dtype");
  if (D.qk_norm) {
    KL_TRY(check_ptrs({w->gamma_q, w->gamma_k, gr->gamma_q, gr->gamma_k}, "layer_backward q/k norm gains"));
    KL_TRY(check_ptrs({s->q_pre, s->k_pre, s->rstd_q, s->rstd_k}, "layer_backward q/k norm saved"));
  }
  if (D.dt == KL_F32 && gr->dtype != KL_F32)
    return set_error(KL_ERR_UNSUPPORTED, "layer_backward: fp32 layer needs fp32 gradients");
  const size_t need = kl_layer_bwd_workspace_bytes(cfg);
  if (!ws || ws_bytes < need) return set_error(KL_ERR_NO_MEMORY, "layer_backward: workspace needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return set_error(KL_ERR_INVALID_ARG, "layer_backward: workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  BwdWs b;
  carve_bwd(D, c, &b);
  const int T = D.T, H = D.H, I = D.I, dt = D.dt, gdt = gr->dtype;

  // MLP: dm = dY Wd (bf16: dg, du formed from it in the epilogue), dWd = dY^T m
  {
    GemmSpec g[2] = {dgrad(T, I, H, dY, w->wd, b.dm, dt), wgrad(H, I, T, dY, s->m, gr->wd, gdt)};
    if (dt == KL_BF16) {
      g[0].epi = GEMM_EPI_SWIGLU_BWD;
      g[0].C = b.dg;
      g[0].C2 = b.du;
      g[0].X1 = s->g;
      g[0].X2 = s->u;
    }
    with_tail(g, 2, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, g, 2, st, "gemm.bwd_down"));
  }
  if (dt != KL_BF16) KL_TRY(swiglu_bwd(static_cast<int64_t>(T) * I, dt, b.dm, s->g, s->u, b.dg, b.du, st));
  {
    GemmSpec dh = dgrad(T, H, I, b.dg, w->wg, b.dh2, KL_F32);
    dh.nseg = 2;
    dh.A[1] = b.du; dh.lda[1] = I; dh.B[1] = w->wu; dh.ldb[1] = H; dh.K[1] = I;
    GemmSpec g[3] = {dh, wgrad(I, H, T, b.dg, s->h2, gr->wg, gdt),
                     wgrad(I, H, T, b.du, s->h2, gr->wu, gdt)};
    with_tail(g, 3, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, g, 3, st, "gemm.bwd_gateup"));
  }
  KL_TRY(rmsnorm_bwd(T, H, dt, b.dh2, KL_F32, s->x2, w->gamma2, s->rstd2, dY, b.dx2,
                     static_cast<float*>(gr->gamma2), b.norm, b.norm_bytes, st));
  // attention block: dO = dx2 Wo (bf16: D = rowsum(dO * O) per head from the
  // epilogue, straight into the attention workspace), dWo = dx2^T o
  const bool d_ready = dt == KL_BF16;
  {
    GemmSpec g[2] = {dgrad(T, D.Dq, H, b.dx2, w->wo, b.dO, dt),
                     wgrad(H, D.Dq, T, b.dx2, s->o, gr->wo, gdt)};
    if (d_ready) {
      g[0].epi = GEMM_EPI_ROWDOT;
      g[0].X1 = s->o;
      g[0].dot_out = attention_bwd_d_rows(b.att);
      g[0].dot_S = D.S;
    }
    with_tail(g, 2, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, g, 2, st, "gemm.bwd_o"));
  }
  float *dq_acc = nullptr, *dk_acc = nullptr, *dv_acc = nullptr;
  const float2* rope = reinterpret_cast<const float2*>(s->rope);   // bf16: the forward's table
  if (dt == KL_BF16 && !rope) return set_error(KL_ERR_INVALID_ARG, "layer_backward: saved rotary table missing");
  if (!D.qk_norm && !D.inter) {
    // bf16: dQ leaves the attention kernel rotated back and converted; dK, dV (summed
    // over each kv head's query heads) are finished below
    KL_TRY(attention_bwd_accum(D.B, D.S, D.Hq, D.Hkv, D.d, dt, s->q, s->k, s->v, s->o, s->lse, b.dO,
                               b.att, b.att_bytes, &dq_acc, &dk_acc, &dv_acc, st, d_ready,
                               rope ? b.dq : nullptr, rope, b.dk, b.dv));
    if (dk_acc)   // fp32: the accumulators are rotated back and stored here
      KL_TRY(rope_bwd_convert(D.B, D.S, dq_acc ? D.Hq : 0, D.Hkv, D.d, cfg->rope_base, dt, dq_acc, dk_acc, dv_acc,
                              b.dq, b.dk, b.dv, st));
  } else {
    // layer options: dQ (bf16, still rotated, in b.dq) or its fp32 accumulator, then the
    // rotation back and the per-head norm backward for q and k; dV converted
    KL_TRY(attention_bwd_accum(D.B, D.S, D.Hq, D.Hkv, D.d, dt, s->q, s->k, s->v, s->o, s->lse, b.dO,
                               b.att, b.att_bytes, &dq_acc, &dk_acc, &dv_acc, st, d_ready,
                               dt == KL_BF16 ? b.dq : nullptr, nullptr, b.dk, b.dv));
    // bf16: dQ and dK (still rotated) are read from and rewritten in place in b.dq, b.dk
    const void* dqr = dq_acc ? static_cast<const void*>(dq_acc) : b.dq;
    KL_TRY(qk_rope_bwd(T, D.Hq, D.S, D.d, dt, dqr, dq_acc ? KL_F32 : KL_BF16, s->q_pre, w->gamma_q, s->rstd_q,
                       D.qk_norm, D.inter, cfg->rope_base, rope, b.dq, static_cast<float*>(gr->gamma_q), b.qk_q,
                       b.qk_q_bytes, st));
    const void* dkr = dk_acc ? static_cast<const void*>(dk_acc) : b.dk;
    KL_TRY(qk_rope_bwd(T, D.Hkv, D.S, D.d, dt, dkr, dk_acc ? KL_F32 : KL_BF16, s->k_pre, w->gamma_k, s->rstd_k,
                       D.qk_norm, D.inter, cfg->rope_base, rope, b.dk, static_cast<float*>(gr->gamma_k), b.qk_k,
                       b.qk_k_bytes, st));
    if (dv_acc) KL_TRY(convert_f32(static_cast<int64_t>(T) * D.Dkv, dt, dv_acc, b.dv, st));
  }
  {
    GemmSpec dh = dgrad(T, H, D.Dq, b.dq, w->wq, b.dh1, KL_F32);
    dh.nseg = 3;
    dh.A[1] = b.dk; dh.lda[1] = D.Dkv; dh.B[1] = w->wk; dh.ldb[1] = H; dh.K[1] = D.Dkv;
    dh.A[2] = b.dv; dh.lda[2] = D.Dkv; dh.B[2] = w->wv; dh.ldb[2] = H; dh.K[2] = D.Dkv;
    GemmSpec g[4] = {dh, wgrad(D.Dq, H, T, b.dq, s->h1, gr->wq, gdt),
                     wgrad(D.Dkv, H, T, b.dk, s->h1, gr->wk, gdt),
                     wgrad(D.Dkv, H, T, b.dv, s->h1, gr->wv, gdt)};
    with_tail(g, 4, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, g, 4, st, "gemm.bwd_qkv"));
  }
  KL_TRY(rmsnorm_bwd(T, H, dt, b.dh1, KL_F32, s->x, w->gamma1, s->rstd1, b.dx2, dX,
                     static_cast<float*>(gr->gamma1), b.norm, b.norm_bytes, st));
  return KL_OK;
}

// ---------------------------------------------------------------------------
// lm-head
// ---------------------------------------------------------------------------
static kl_status check_lm(const kl_lmhead_cfg* c) {
  if (!c || c->N < 1 || c->H < 1 || c->V < 1)
    return set_error(KL_ERR_INVALID_ARG, "bad lm-head cfg");
  if ((c->dtype != KL_BF16 && c->dtype != KL_F32) || (c->dw_dtype != KL_BF16 && c->dw_dtype != KL_F32))
    return set_error(KL_ERR_INVALID_ARG, "bad lm-head dtype");
  if (c->dtype == KL_F32 && c->dw_dtype != KL_F32)
    return set_error(KL_ERR_UNSUPPORTED, "fp32 lm-head needs fp32 dW");
  if (c->dtype == KL_BF16 && (c->H % 8 || c->V % 8))
    return set_error(KL_ERR_UNSUPPORTED, "bf16 lm-head needs H and V multiples of 8");
  return KL_OK;
}

size_t kl_lmhead_workspace_bytes(const kl_lmhead_cfg* c) {
  if (check_lm(c) != KL_OK) return 0;
  const size_t NV = static_cast<size_t>(c->N) * c->V;
  return align_up(NV * 4, 256) + align_up(NV * dtype_size(c->dtype), 256) + ce_ws(c->N) +
         (c->dtype == KL_BF16 ? gemm_tail_ws_bytes() : 0);
}

kl_status kl_lmhead_ce_argmax(const kl_lmhead_cfg* c, const void* X, const void* W,
                              const int32_t* targets, float* loss, int32_t* argmax, void* dlogits,
                              void* dX, void* dW, void* ws, size_t ws_bytes, void* stream) {
  KL_TRY(check_lm(c));
  KL_TRY(check_ptrs({X, W, dX, dW}, "lmhead"));
  if (!targets || !loss || !argmax) return set_error(KL_ERR_INVALID_ARG, "lmhead: null pointer");
  if (dlogits && !al16(dlogits)) return set_error(KL_ERR_INVALID_ARG, "lmhead: dlogits not aligned");
  const size_t need = kl_lmhead_workspace_bytes(c);
  if (!ws || ws_bytes < need) return set_error(KL_ERR_NO_MEMORY, "lmhead: workspace needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return set_error(KL_ERR_INVALID_ARG, "lmhead: workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = c->N, H = c->H, V = c->V, dt = c->dtype;
  const size_t NV = static_cast<size_t>(N) * V;
  Carver cv(ws);
  float* z = static_cast<float*>(cv.take(NV * 4));
  void* dz_ws = cv.take(NV * dtype_size(dt));
  void* ce = cv.take(ce_ws(N));
  const size_t tail_bytes = dt == KL_BF16 ? gemm_tail_ws_bytes() : 0;
  void* tail = tail_bytes ? cv.take(tail_bytes) : nullptr;
  void* dz = dlogits ? dlogits : dz_ws;
  {
    GemmSpec g = proj(N, V, H, X, H, W, H, z, V, KL_F32);
    with_tail(&g, 1, tail, tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.lm_logits"));
  }
  KL_TRY(ce_argmax(N, V, z, targets, loss, argmax, dz, dt, ce, ce_ws(N), st));
  {
    GemmSpec g[2] = {dgrad(N, H, V, dz, W, dX, dt), wgrad(V, H, N, dz, X, dW, c->dw_dtype)};
    with_tail(g, 2, tail, tail_bytes);
    KL_TRY(run_gemms(dt, g, 2, st, "gemm.lm_bwd"));
  }
  return KL_OK;
}

size_t kl_ce_workspace_bytes(int32_t N) { return N > 0 ? ce_ws(N) : 0; }

kl_status kl_ce_argmax(int32_t N, int32_t V, const float* z, const int32_t* targets, float* loss,
                       int32_t* argmax, void* dlogits, int32_t dz_dtype, void* ws, size_t ws_bytes,
                       void* stream) {
  if (dz_dtype != KL_F32 && dz_dtype != KL_BF16) return set_error(KL_ERR_INVALID_ARG, "ce: bad dtype");
  return ce_argmax(N, V, z, targets, loss, argmax, dlogits, dz_dtype, ws, ws_bytes,
                   static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// individual kernels
// ---------------------------------------------------------------------------
kl_status kl_gemm(int32_t M, int32_t N, int32_t K, int32_t dtype, const void* A, int64_t lda,
                  int32_t a_mn_major, const void* B, int64_t ldb, int32_t b_mn_major, void* C,
                  int64_t ldc, int32_t c_dtype, const void* R, int64_t ldr, int32_t r_dtype,
                  void* stream) {
  return kl_gemm_ex(M, N, K, dtype, A, lda, a_mn_major, B, ldb, b_mn_major, C, ldc, c_dtype, R, ldr, r_dtype,
                    nullptr, 0, stream);
}

size_t kl_gemm_scratch_bytes(void) { return gemm_tail_ws_bytes(); }

kl_status kl_gemm_ex(int32_t M, int32_t N, int32_t K, int32_t dtype, const void* A, int64_t lda,
                     int32_t a_mn_major, const void* B, int64_t ldb, int32_t b_mn_major, void* C,
                     int64_t ldc, int32_t c_dtype, const void* R, int64_t ldr, int32_t r_dtype, void* ws,
                     size_t ws_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !B || !C) return set_error(KL_ERR_INVALID_ARG, "gemm: bad arguments");
  if ((dtype != KL_F32 && dtype != KL_BF16) || (c_dtype != KL_F32 && c_dtype != KL_BF16) ||
      (R && r_dtype != KL_F32 && r_dtype != KL_BF16))
    return set_error(KL_ERR_INVALID_ARG, "gemm: bad dtype");
  const int64_t a_rows_min = a_mn_major ? M : K, b_rows_min = b_mn_major ? N : K;
  if (lda < a_rows_min || ldb < b_rows_min || ldc < N || (R && ldr < N))
    return set_error(KL_ERR_INVALID_ARG, "gemm: leading dimension too small");
  GemmSpec s;
  s.M = M; s.N = N; s.nseg = 1;
  s.A[0] = A; s.lda[0] = lda; s.B[0] = B; s.ldb[0] = ldb; s.K[0] = K;
  s.a_mn = a_mn_major ? 1 : 0; s.b_mn = b_mn_major ? 1 : 0;
  s.C = C; s.ldc = ldc; s.c_dtype = c_dtype;
  s.R = R; s.ldr = ldr; s.r_dtype = r_dtype;
  if (ws_bytes >= gemm_tail_ws_bytes()) with_tail(&s, 1, ws, ws_bytes);
  return run_gemms(dtype, &s, 1, static_cast<cudaStream_t>(stream), "gemm");
}

kl_status kl_rmsnorm_fwd(int32_t rows, int32_t width, int32_t dtype, const void* x,
                         const void* gamma, float eps, void* h, float* rstd, void* stream) {
  return rmsnorm_fwd(rows, width, dtype, x, gamma, eps, h, rstd, static_cast<cudaStream_t>(stream));
}

size_t kl_rmsnorm_bwd_ws_bytes(int32_t rows, int32_t width) {
  return rows > 0 && width > 0 ? rmsnorm_bwd_ws(rows, width) : 0;
}

kl_status kl_rmsnorm_bwd(int32_t rows, int32_t width, int32_t dtype, const void* dh,
                         int32_t dh_dtype, const void* x, const void* gamma, const float* rstd,
                         const void* resid, void* dx, float* dgamma, void* ws, size_t ws_bytes,
                         void* stream) {
  return rmsnorm_bwd(rows, width, dtype, dh, dh_dtype, x, gamma, rstd, resid, dx, dgamma, ws,
                     ws_bytes, static_cast<cudaStream_t>(stream));
}

kl_status kl_rope(int32_t B, int32_t S, int32_t heads, int32_t d, float base, int32_t dtype,
                  void* x, int32_t direction, void* stream) {
  return rope(B, S, heads, d, base, dtype, x, direction, static_cast<cudaStream_t>(stream));
}

kl_status kl_swiglu_fwd(int64_t n, int32_t dtype, const void* g, const void* u, void* m,
                        void* stream) {
  return swiglu_fwd(n, dtype, g, u, m, static_cast<cudaStream_t>(stream));
}

kl_status kl_swiglu_bwd(int64_t n, int32_t dtype, const void* dm, const void* g, const void* u,
                        void* dg, void* du, void* stream) {
  return swiglu_bwd(n, dtype, dm, g, u, dg, du, static_cast<cudaStream_t>(stream));
}

kl_status kl_attention_fwd(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d,
                           int32_t dtype, const void* q, const void* k, const void* v, void* o,
                           float* lse, void* stream) {
  return attention_fwd(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, static_cast<cudaStream_t>(stream));
}

size_t kl_attention_bwd_ws_bytes(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d) {
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1) return 0;
  return attention_bwd_ws(B, S, Hq, Hkv, d);
}

kl_status kl_attention_bwd(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d,
                           int32_t dtype, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* ws, size_t ws_bytes, void* stream) {
  if (!dq || !dk || !dv) return set_error(KL_ERR_INVALID_ARG, "attention_bwd: null output");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float *dq_acc = nullptr, *dk_acc = nullptr, *dv_acc = nullptr;
  const bool bf = dtype == KL_BF16;
  KL_TRY(attention_bwd_accum(B, S, Hq, Hkv, d, dtype, q, k, v, o, lse, dout, ws, ws_bytes, &dq_acc,
                             &dk_acc, &dv_acc, st, false, bf ? dq : nullptr, nullptr, bf ? dk : nullptr,
                             bf ? dv : nullptr));
  const int64_t T = static_cast<int64_t>(B) * S;
  if (dq_acc) KL_TRY(convert_f32(T * Hq * d, dtype, dq_acc, dq, st));
  if (dk_acc) KL_TRY(convert_f32(T * Hkv * d, dtype, dk_acc, dk, st));
  if (dv_acc) KL_TRY(convert_f32(T * Hkv * d, dtype, dv_acc, dv, st));
  return KL_OK;
}

size_t kl_paged_attention_ws_bytes(const kl_paged_cfg* pc, int32_t Hq, int32_t Hkv, int32_t d) {
  if (paged_check(pc, Hq, Hkv, d, KL_BF16) != KL_OK) return 0;
  return paged_attention_ws(*pc, Hq, Hkv);
}

kl_status kl_paged_kv_write(const kl_paged_cfg* pc, int32_t Hkv, int32_t d, int32_t dtype, const void* k_new,
                            const void* v_new, const int32_t* table, const int32_t* ctx, void* k_pool, void* v_pool,
                            void* stream) {
  KL_TRY(paged_check(pc, Hkv, Hkv, d, dtype));
  return paged_kv_write(*pc, Hkv, k_new, v_new, table, ctx, k_pool, v_pool, static_cast<cudaStream_t>(stream));
}

kl_status kl_paged_attention(const kl_paged_cfg* pc, int32_t Hq, int32_t Hkv, int32_t d, int32_t dtype,
                             const void* q, const void* k_pool, const void* v_pool, const int32_t* table,
                             const int32_t* ctx, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  KL_TRY(paged_check(pc, Hq, Hkv, d, dtype));
  return paged_attention(*pc, Hq, Hkv, q, k_pool, v_pool, table, ctx, o, lse, ws, ws_bytes,
                         static_cast<cudaStream_t>(stream));
}

size_t kl_layer_forward_paged_ws_bytes(const kl_layer_cfg* cfg, const kl_paged_cfg* pc) {
  Dims D;
  if (check_cfg(cfg, &D) != KL_OK || paged_check(pc, D.Hq, D.Hkv, D.d, D.dt) != KL_OK) return 0;
  if (cfg->B != pc->B || cfg->S != pc->n_new) return 0;
  Carver c(nullptr);
  PagedWs w;
  carve_paged(D, *pc, c, &w);
  return c.off;
}

kl_status kl_layer_forward_paged(const kl_layer_cfg* cfg, const kl_paged_cfg* pc, const kl_layer_weights* w,
                                 const void* X, void* Y, void* k_pool, void* v_pool, const int32_t* table,
                                 const int32_t* ctx, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  KL_TRY(check_cfg(cfg, &D));
  KL_TRY(paged_check(pc, D.Hq, D.Hkv, D.d, D.dt));
  if (cfg->B != pc->B || cfg->S != pc->n_new)
    return set_error(KL_ERR_INVALID_ARG, "layer_forward_paged: cfg B, S must be the step's B, n_new");
  if (!w) return set_error(KL_ERR_INVALID_ARG, "layer_forward_paged: null weights");
  KL_TRY(check_ptrs({w->gamma1, w->wq, w->wk, w->wv, w->wo, w->gamma2, w->wg, w->wu, w->wd},
                    "layer_forward_paged weights"));
  if (D.qk_norm) KL_TRY(check_ptrs({w->gamma_q, w->gamma_k}, "layer_forward_paged q/k norm gains"));
  KL_TRY(check_ptrs({X, Y, k_pool, v_pool, table, ctx}, "layer_forward_paged buffers"));
  const size_t need = kl_layer_forward_paged_ws_bytes(cfg, pc);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return set_error(KL_ERR_NO_MEMORY, "layer_forward_paged: workspace too small or not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carver c(ws);
  PagedWs b;
  carve_paged(D, *pc, c, &b);
  const int T = D.T, H = D.H, I = D.I, dt = D.dt;
  KL_TRY(rmsnorm_fwd(T, H, dt, X, w->gamma1, cfg->eps, b.h1, b.rstd1, st));
  {
    GemmSpec g[3] = {proj(T, D.Dq, H, b.h1, H, w->wq, H, b.q_pre, D.Dq, dt),
                     proj(T, D.Dkv, H, b.h1, H, w->wk, H, b.k_pre, D.Dkv, dt),
                     proj(T, D.Dkv, H, b.h1, H, w->wv, H, b.v, D.Dkv, dt)};
    with_tail(g, 3, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, g, 3, st, "gemm.paged_qkv"));
  }
  // optional per-head norm, the rotation at the tokens' absolute positions ctx[b] + i, and the new keys
  // and values written into their cache slots: one launch
  KL_TRY(paged_qkv_rope(*pc, D.Hq, D.Hkv, D.d, b.q_pre, b.k_pre, b.v, w->gamma_q, w->gamma_k, cfg->eps, D.qk_norm,
                        D.inter, cfg->rope_base, table, ctx, b.q, k_pool, v_pool, st));
  KL_TRY(paged_attention(*pc, D.Hq, D.Hkv, b.q, k_pool, v_pool, table, ctx, b.o, nullptr, b.att, b.att_bytes, st));
  {
    GemmSpec g = proj(T, H, D.Dq, b.o, D.Dq, w->wo, D.Dq, b.x2, H, dt, X, dt);
    with_tail(&g, 1, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.paged_o"));
  }
  KL_TRY(rmsnorm_fwd(T, H, dt, b.x2, w->gamma2, cfg->eps, b.h2, b.rstd2, st));
  {
    GemmSpec g = proj(T, I, H, b.h2, H, w->wg, H, b.g, I, dt);
    g.epi = GEMM_EPI_SWIGLU;
    g.B2 = w->wu;
    g.C2 = b.u;
    g.C3 = b.m;
    with_tail(&g, 1, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.paged_gateup"));
  }
  {
    GemmSpec g = proj(T, H, I, b.m, I, w->wd, I, Y, H, dt, b.x2, dt);
    with_tail(&g, 1, b.tail, b.tail_bytes);
    KL_TRY(run_gemms(dt, &g, 1, st, "gemm.paged_down"));
  }
  return KL_OK;
}

}  // extern "C"

