// Layer-streaming driver ("From-scratch GPU LLM training", capability list:
// the full-depth model runs holding one layer's weights at a time, lossless
// against the bulk forward; the end-to-end smoke trains under gradient
// clipping).
//
// Weights of the decoder layers stay in host memory. Two device weight slots
// hold the layer being computed and the next one, uploaded on a separate copy
// stream while the current layer runs (events order the slot reuse). One
// training step: forward through every layer saving its activations, lm-head
// cross-entropy on the last hidden state, backward in reverse (the last two
// layers are still resident; earlier ones are uploaded again), then the global
// L2 norm of every weight gradient (deterministic two-stage reduction in
// fp64) and the clip coefficient min(1, max_norm / (norm + 1e-6)), applied to
// every gradient where it was delivered. Gradients bound for device memory are
// computed in place and scaled in place; gradients bound for pinned host memory
// are computed into device buffers kept for the whole step, then written out
// already scaled by one kernel through the destination's device-visible
// address (the clip needs every gradient before any can be final).
//
// If the caller's layer weights are already device memory the driver runs in
// "bulk" mode: no slots, no uploads, the same kernels in the same order. Its
// results are what the streamed mode is compared with.
//
// Modes. SAVE_ALL keeps every layer's saved activations from the forward to
// the backward. RECOMPUTE keeps only each layer's input (the previous layer's
// output) and runs the layer's forward again, into one shared saved set, right
// before its backward, with the weights already resident for the backward (the
// last layer's set is still intact after the forward and is not recomputed);
// the price is one more layer forward per layer but the last. FORWARD holds
// only what a forward needs: two weight slots, one layer's working set, two
// hidden buffers; device memory does not grow with depth.
#include <string.h>

#include <vector>

#include "internal.h"
#include "kl_common.cuh"

namespace kl {
namespace {

constexpr int SUMSQ_BLOCKS = 256;
constexpr int SUMSQ_THREADS = 256;
constexpr double CLIP_EPS = 1e-6;

struct GradRef {
  const float* src;
  float* dst;
  int64_t n;
  int64_t chunk_begin;   // first global 16384-element chunk of this tensor
};

constexpr int64_t SCALE_CHUNK = 16384;

// partial[b] = sum of squares of p over the elements block b owns (fixed
// assignment, fp32 within a thread over four interleaved accumulators, fp64
// across threads and blocks in a fixed order: deterministic).
__global__ void __launch_bounds__(SUMSQ_THREADS) sumsq_kernel(const float* __restrict__ p, int64_t n,
                                                              double* __restrict__ partial) {
  pdl_enter();
  __shared__ double red[SUMSQ_THREADS / 32];
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int64_t stride = static_cast<int64_t>(SUMSQ_BLOCKS) * SUMSQ_THREADS;
  const int64_t start = blockIdx.x * static_cast<int64_t>(SUMSQ_THREADS) + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
    const int64_t n4 = n >> 2;
    const float4* p4 = reinterpret_cast<const float4*>(p);
    for (int64_t i = start; i < n4; i += stride) {
      const float4 v = p4[i];
      a0 = fmaf(v.x, v.x, a0);
      a1 = fmaf(v.y, v.y, a1);
      a2 = fmaf(v.z, v.z, a2);
      a3 = fmaf(v.w, v.w, a3);
    }
    for (int64_t i = (n4 << 2) + start; i < n; i += stride) a0 = fmaf(p[i], p[i], a0);
  } else {
    for (int64_t i = start; i < n; i += stride) a0 = fmaf(p[i], p[i], a0);
  }
  double acc = (static_cast<double>(a0) + a1) + (static_cast<double>(a2) + a3);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < SUMSQ_THREADS / 32; ++w) t += red[w];
    partial[blockIdx.x] = t;
  }
}

// result = {loss, norm, coef}; partials [count][SUMSQ_BLOCKS] summed in order.
__global__ void clip_finalize_kernel(const double* __restrict__ partial, int count,
                                     const float* __restrict__ loss, float max_norm,
                                     float* __restrict__ result) {
  pdl_enter();
  __shared__ double red[SUMSQ_THREADS / 32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < count * SUMSQ_BLOCKS; i += blockDim.x) acc += partial[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < SUMSQ_THREADS / 32; ++w) t += red[w];
    const double norm = sqrt(t);
    double coef = static_cast<double>(max_norm) / (norm + CLIP_EPS);
    if (coef > 1.0) coef = 1.0;
    result[0] = *loss;
    result[1] = static_cast<float>(norm);
    result[2] = static_cast<float>(coef);
  }
}

// dst = src * coef for every listed gradient (in place when src == dst, where
// coef == 1 leaves nothing to do). The tensors are cut into chunks of
// SCALE_CHUNK elements numbered across all of them; blocks stride over chunks.
__global__ void __launch_bounds__(256) clip_scale_kernel(const GradRef* __restrict__ refs, int count,
                                                         int64_t total_chunks,
                                                         const float* __restrict__ result) {
  pdl_enter();
  const float coef = result[2];
  int r = 0;
  for (int64_t ch = blockIdx.x; ch < total_chunks; ch += gridDim.x) {
    while (r + 1 < count && ch >= refs[r + 1].chunk_begin) ++r;
    const float* src = refs[r].src;
    float* dst = refs[r].dst;
    if (src == dst && coef == 1.0f) continue;
    const int64_t lo = (ch - refs[r].chunk_begin) * SCALE_CHUNK;
    const int64_t hi = min(refs[r].n, lo + SCALE_CHUNK);
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0 && (lo & 3) == 0) {
      const int64_t n4 = (hi - lo) >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src + lo);
      float4* d4 = reinterpret_cast<float4*>(dst + lo);
      for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        float4 v = s4[i];
        v.x *= coef; v.y *= coef; v.z *= coef; v.w *= coef;
        d4[i] = v;
      }
      for (int64_t i = lo + (n4 << 2) + threadIdx.x; i < hi; i += blockDim.x) dst[i] = src[i] * coef;
    } else {
      for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) dst[i] = src[i] * coef;
    }
  }
}

size_t weight_elems(const kl_layer_cfg& c, int which) {
  const size_t H = c.H, Dq = static_cast<size_t>(c.Hq) * c.d, Dkv = static_cast<size_t>(c.Hkv) * c.d,
               I = c.I;
  switch (which) {
    case 0: return H;          // gamma1
    case 1: return Dq * H;     // wq
    case 2: return Dkv * H;    // wk
    case 3: return Dkv * H;    // wv
    case 4: return H * Dq;     // wo
    case 5: return H;          // gamma2
    case 6: return I * H;      // wg
    case 7: return I * H;      // wu
    case 8: return H * I;      // wd
    default: return static_cast<size_t>(c.d);   // gamma_q, gamma_k
  }
}

// Weight tensors of one layer: the nine of the pages' layer, plus the two
// per-head q/k norm gains with cfg.qk_norm.
int n_weights(const kl_layer_cfg& c) { return c.qk_norm ? 11 : 9; }

const void** wfield(kl_layer_weights& w, int i) {
  const void** f[11] = {&w.gamma1, &w.wq, &w.wk, &w.wv, &w.wo, &w.gamma2, &w.wg, &w.wu, &w.wd, &w.gamma_q, &w.gamma_k};
  return f[i];
}
void** gfield(kl_layer_grads& g, int i) {
  void** f[11] = {&g.gamma1, &g.wq, &g.wk, &g.wv, &g.wo, &g.gamma2, &g.wg, &g.wu, &g.wd, &g.gamma_q, &g.gamma_k};
  return f[i];
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Device-visible address of a destination buffer (device, managed, or
// page-locked host memory); nullptr if the GPU cannot reach it.
void* device_visible(void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

}  // namespace
}  // namespace kl

using namespace kl;

struct kl_stream {
  kl_stream_cfg cfg;
  int device = 0;
  bool bulk = false;
  int mode = KL_STREAM_SAVE_ALL;
  std::vector<kl_layer_weights> layers;  // as given (host, or device in bulk mode)
  const void* lm_host = nullptr;
  std::vector<void*> allocs;
  size_t device_bytes = 0;
  // streamed mode
  kl_layer_weights slot[2] = {};
  int slot_layer[2] = {-1, -1};
  cudaStream_t copy = nullptr;
  cudaEvent_t ev_loaded[2] = {}, ev_used[2] = {}, ev_lm = nullptr;
  const void* lm_w = nullptr;
  // activations and workspace
  std::vector<kl_layer_saved> saved;   // one per layer (SAVE_ALL) or one shared set
  std::vector<void*> hidden;   // output of layer l (two alternating buffers with FORWARD)
  void* dx[2] = {};
  void* ws = nullptr;          // layer workspace (the backward's, which the forward reuses)
  size_t ws_bytes = 0;
  void* lm_ws = nullptr;
  size_t lm_ws_bytes = 0;
  float* loss = nullptr;
  int32_t* argmax = nullptr;
  // gradients bound for host memory are kept here until the clip is known
  std::vector<kl_layer_grads> retain;   // allocated on first use
  float* dwlm_retain = nullptr;
  double* partials = nullptr;
  float* result = nullptr;
  GradRef* refs = nullptr;
  int max_refs = 0;

  void* alloc(size_t bytes, kl_status* st) {
    void* p = nullptr;
    if (*st != KL_OK) return nullptr;
    const cudaError_t e = cudaMalloc(&p, align_up(bytes, 256));
    if (e != cudaSuccess) {
      *st = cuda_check(e, "kl_stream: cudaMalloc");
      return nullptr;
    }
    allocs.push_back(p);
    device_bytes += align_up(bytes, 256);
    return p;
  }
  kl_layer_saved* saved_for(int l) { return &saved[mode == KL_STREAM_SAVE_ALL ? l : 0]; }
  void* hidden_of(int l) { return hidden[mode == KL_STREAM_FORWARD ? (l & 1) : l]; }

  void release() {
    for (void* p : allocs) cudaFree(p);
    allocs.clear();
    for (int i = 0; i < 2; ++i) {
      if (ev_loaded[i]) cudaEventDestroy(ev_loaded[i]);
      if (ev_used[i]) cudaEventDestroy(ev_used[i]);
    }
    if (ev_lm) cudaEventDestroy(ev_lm);
    if (copy) cudaStreamDestroy(copy);
  }
};

namespace {

kl_status upload_layer(kl_stream* s, int layer, int slot) {
  const kl_layer_cfg& c = s->cfg.layer;
  const size_t es = dtype_size(c.dtype);
  KL_CUDA(cudaStreamWaitEvent(s->copy, s->ev_used[slot], 0));
  for (int i = 0; i < n_weights(c); ++i)
    KL_CUDA(cudaMemcpyAsync(const_cast<void*>(*wfield(s->slot[slot], i)), *wfield(s->layers[layer], i),
                            weight_elems(c, i) * es, cudaMemcpyHostToDevice, s->copy));
  KL_CUDA(cudaEventRecord(s->ev_loaded[slot], s->copy));
  s->slot_layer[slot] = layer;
  return KL_OK;
}

// Makes `layer` resident (uploading into the slot not holding `keep` if
// needed) and returns its slot.
kl_status acquire(kl_stream* s, int layer, int keep_slot, int* slot_out) {
  for (int i = 0; i < 2; ++i)
    if (s->slot_layer[i] == layer) {
      *slot_out = i;
      return KL_OK;
    }
  const int v = keep_slot == 0 ? 1 : 0;
  KL_TRY(upload_layer(s, layer, v));
  *slot_out = v;
  return KL_OK;
}

kl_status sumsq(kl_stream* s, const float* p, int64_t n, int index, cudaStream_t st) {
  ProfScope ps("grad_sumsq", st, 0.0, 4.0 * n);
  launch_pdl(sumsq_kernel, SUMSQ_BLOCKS, SUMSQ_THREADS, 0, st, p, n, s->partials + static_cast<int64_t>(index) * SUMSQ_BLOCKS);
  KL_CUDA(cudaGetLastError());
  return KL_OK;
}

kl_status make_stream_events(kl_stream* s) {
  cudaError_t e = cudaStreamCreateWithFlags(&s->copy, cudaStreamNonBlocking);
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
    e = cudaEventCreateWithFlags(&s->ev_loaded[k], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->ev_used[k], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->ev_lm, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_check(e, "kl_stream_create: stream/event");
  return KL_OK;
}

// The weights of layer l for the compute stream: the caller's (bulk) or a
// slot, uploaded if it is not resident (never into keep_slot), the compute
// stream made to wait for the upload.
kl_status weights_for(kl_stream* s, int l, int keep_slot, int* slot, kl_layer_weights* w, cudaStream_t cs) {
  if (s->bulk) {
    *w = s->layers[l];
    *slot = -1;
    return KL_OK;
  }
  KL_TRY(acquire(s, l, keep_slot, slot));
  KL_CUDA(cudaStreamWaitEvent(cs, s->ev_loaded[*slot], 0));
  *w = s->slot[*slot];
  return KL_OK;
}

// Start of a pass: the slots' contents may be stale (weights change between
// calls), and nothing of this pass has used them yet.
kl_status begin_pass(kl_stream* s, cudaStream_t cs) {
  if (s->bulk) return KL_OK;
  s->slot_layer[0] = s->slot_layer[1] = -1;
  KL_CUDA(cudaEventRecord(s->ev_used[0], cs));
  KL_CUDA(cudaEventRecord(s->ev_used[1], cs));
  return KL_OK;
}

// One of `pieces` equal pieces of the lm-head weight's upload on the copy
// stream; the last piece records ev_lm.
kl_status upload_lm_piece(kl_stream* s, int piece, int pieces) {
  const size_t bytes = static_cast<size_t>(s->cfg.V) * s->cfg.layer.H * dtype_size(s->cfg.layer.dtype);
  const size_t lo = bytes * piece / pieces, hi = bytes * (piece + 1) / pieces;
  if (hi > lo)
    KL_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(const_cast<void*>(s->lm_w)) + lo,
                            static_cast<const uint8_t*>(s->lm_host) + lo, hi - lo, cudaMemcpyHostToDevice, s->copy));
  if (piece == pieces - 1) KL_CUDA(cudaEventRecord(s->ev_lm, s->copy));
  return KL_OK;
}

// Forward through every layer: layer l reads X (l = 0) or the previous
// layer's output, writes hidden_of(l) (`last` for the last layer when given),
// with layer l + 1's weights uploaded while layer l runs. With `with_lm` the
// lm-head weight's upload is cut into one piece per layer, each queued behind
// that layer's prefetch, so that no layer's weights wait for the whole head.
// *cur receives the slot holding the last layer.
kl_status forward_layers(kl_stream* s, const void* X, void* last, cudaStream_t cs, int* cur_out, bool with_lm) {
  const kl_layer_cfg& c = s->cfg.layer;
  const int L = s->cfg.n_layers;
  int cur = -1;
  for (int l = 0; l < L; ++l) {
    kl_layer_weights w;
    KL_TRY(weights_for(s, l, cur == 0 ? 1 : 0, &cur, &w, cs));
    if (!s->bulk && l + 1 < L) {
      int nxt;
      KL_TRY(acquire(s, l + 1, cur, &nxt));  // prefetch while layer l runs
    }
    if (!s->bulk && with_lm) KL_TRY(upload_lm_piece(s, l, L));
    const void* xin = l == 0 ? X : s->hidden_of(l - 1);
    void* out = (l == L - 1 && last) ? last : s->hidden_of(l);
    KL_TRY(kl_layer_forward(&c, &w, xin, out, s->saved_for(l), s->ws, s->ws_bytes, cs));
    if (!s->bulk) KL_CUDA(cudaEventRecord(s->ev_used[cur], cs));
  }
  *cur_out = cur;
  return KL_OK;
}

}  // namespace

extern "C" {

kl_status kl_stream_create(const kl_stream_cfg* cfg, const kl_layer_weights* host_layers,
                           const void* host_lm_head, kl_stream** out) {
  if (!cfg || !host_layers || !out) return set_error(KL_ERR_INVALID_ARG, "kl_stream_create: null argument");
  *out = nullptr;
  const int mode = cfg->mode;
  if (mode != KL_STREAM_SAVE_ALL && mode != KL_STREAM_RECOMPUTE && mode != KL_STREAM_FORWARD)
    return set_error(KL_ERR_INVALID_ARG, "kl_stream_create: bad mode %d", mode);
  const bool train = mode != KL_STREAM_FORWARD;
  if (train && !host_lm_head) return set_error(KL_ERR_INVALID_ARG, "kl_stream_create: null lm-head weight");
  if (cfg->n_layers < 1 || (train && cfg->V < 1))
    return set_error(KL_ERR_INVALID_ARG, "kl_stream_create: bad n_layers or V");
  const kl_layer_cfg& c = cfg->layer;
  const size_t saved_bytes = kl_layer_saved_bytes(&c);
  if (saved_bytes == 0) return KL_ERR_INVALID_ARG;  // message set by the size query's checks
  kl_lmhead_cfg lc = {c.B * c.S, c.H, train ? cfg->V : 1, c.dtype, KL_F32};
  const size_t lm_ws = train ? kl_lmhead_workspace_bytes(&lc) : 0;
  if (train && lm_ws == 0) return KL_ERR_UNSUPPORTED;
  for (int l = 0; l < cfg->n_layers; ++l)
    for (int i = 0; i < n_weights(c); ++i)
      if (!*wfield(const_cast<kl_layer_weights&>(host_layers[l]), i))
        return set_error(KL_ERR_INVALID_ARG, "kl_stream_create: layer %d weight %d is null", l, i);

  kl_stream* s = new kl_stream();
  s->cfg = *cfg;
  KL_CUDA(cudaGetDevice(&s->device));
  s->layers.assign(host_layers, host_layers + cfg->n_layers);
  s->lm_host = host_lm_head;
  s->mode = mode;
  s->bulk = is_device_ptr(host_layers[0].wq);
  kl_status st = KL_OK;
  const int L = cfg->n_layers;
  const size_t T = static_cast<size_t>(c.B) * c.S, es = dtype_size(c.dtype);
  if (!s->bulk) {
    for (int k = 0; k < 2; ++k)
      for (int i = 0; i < n_weights(c); ++i) *wfield(s->slot[k], i) = s->alloc(weight_elems(c, i) * es, &st);
    if (train) s->lm_w = s->alloc(static_cast<size_t>(cfg->V) * c.H * es, &st);
    if (st == KL_OK) st = make_stream_events(s);
  } else {
    if (train && !is_device_ptr(host_lm_head))
      st = set_error(KL_ERR_INVALID_ARG, "kl_stream_create: device layers need a device lm-head weight");
    s->lm_w = host_lm_head;
  }
  s->saved.resize(mode == KL_STREAM_SAVE_ALL ? L : 1);
  s->hidden.resize(mode == KL_STREAM_FORWARD ? 2 : L);
  for (size_t i = 0; i < s->saved.size() && st == KL_OK; ++i) {
    void* mem = s->alloc(saved_bytes, &st);
    if (st == KL_OK) st = kl_layer_saved_carve(&c, mem, saved_bytes, &s->saved[i]);
  }
  for (size_t i = 0; i < s->hidden.size(); ++i) s->hidden[i] = s->alloc(T * c.H * es, &st);
  s->ws_bytes = train ? kl_layer_bwd_workspace_bytes(&c) : kl_layer_fwd_workspace_bytes(&c);
  s->ws = s->alloc(s->ws_bytes, &st);
  if (train) {
    s->dx[0] = s->alloc(T * c.H * es, &st);
    s->dx[1] = s->alloc(T * c.H * es, &st);
    s->lm_ws_bytes = lm_ws;
    s->lm_ws = s->alloc(lm_ws, &st);
    s->loss = static_cast<float*>(s->alloc(sizeof(float), &st));
    s->argmax = static_cast<int32_t*>(s->alloc(T * sizeof(int32_t), &st));
    s->max_refs = n_weights(c) * L + 1;
    s->partials = static_cast<double*>(s->alloc(static_cast<size_t>(s->max_refs) * SUMSQ_BLOCKS * 8, &st));
    s->result = static_cast<float*>(s->alloc(4 * sizeof(float), &st));
    s->refs = static_cast<GradRef*>(s->alloc(static_cast<size_t>(s->max_refs) * sizeof(GradRef), &st));
  }
  if (st != KL_OK) {
    s->release();
    delete s;
    return st;
  }
  *out = s;
  return KL_OK;
}

kl_status kl_stream_run(kl_stream* s, const void* X, const int32_t* targets, float clip_max_norm,
                        const kl_layer_grads* grads, void* dW_lm, kl_stream_result* result,
                        void* stream) {
  if (!s || !X || !targets || !grads || !dW_lm || !result)
    return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: null argument");
  if (!(clip_max_norm > 0.f)) return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: clip_max_norm must be > 0");
  if (s->mode == KL_STREAM_FORWARD)
    return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: the driver was created forward-only");
  int dev = -1;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev != s->device) return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: created on device %d, current %d", s->device, dev);
  const kl_layer_cfg& c = s->cfg.layer;
  const int L = s->cfg.n_layers;
  const int T = c.B * c.S;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  // Where each gradient is computed (src) and where it must end up (dst).
  std::vector<kl_layer_grads> dst(grads, grads + L);
  std::vector<bool> on_device(L);
  bool any_host = false;
  for (int l = 0; l < L; ++l) {
    if (dst[l].dtype != KL_F32) return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: gradients must be fp32");
    bool dev_all = true;
    for (int i = 0; i < n_weights(c); ++i) {
      void* p = *gfield(dst[l], i);
      if (!p) return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: layer %d gradient %d is null", l, i);
      if (!device_visible(p))
        return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: layer %d gradient %d is not device-visible (pin it)", l, i);
      if (!is_device_ptr(p)) dev_all = false;
    }
    on_device[l] = dev_all;
    any_host = any_host || !dev_all;
  }
  void* dwlm_dev = device_visible(dW_lm);
  if (!dwlm_dev) return set_error(KL_ERR_INVALID_ARG, "kl_stream_run: dW_lm is not device-visible (pin it)");
  const bool dwlm_on_device = is_device_ptr(dW_lm);
  if ((any_host && s->retain.empty()) || (!dwlm_on_device && !s->dwlm_retain)) {
    kl_status st = KL_OK;
    if (any_host && s->retain.empty()) {
      s->retain.resize(L);
      for (int l = 0; l < L; ++l) {
        for (int i = 0; i < n_weights(c); ++i) *gfield(s->retain[l], i) = s->alloc(weight_elems(c, i) * 4, &st);
        s->retain[l].dtype = KL_F32;
      }
    }
    if (!dwlm_on_device && !s->dwlm_retain)
      s->dwlm_retain = static_cast<float*>(s->alloc(static_cast<size_t>(s->cfg.V) * c.H * 4, &st));
    if (st != KL_OK) return st;
  }
  std::vector<kl_layer_grads> src(L);
  std::vector<GradRef> refs;
  for (int l = 0; l < L; ++l) {
    src[l] = on_device[l] ? dst[l] : s->retain[l];
    for (int i = 0; i < n_weights(c); ++i)
      refs.push_back({static_cast<const float*>(*gfield(src[l], i)),
                      static_cast<float*>(device_visible(*gfield(dst[l], i))),
                      static_cast<int64_t>(weight_elems(c, i)), 0});
  }
  float* dwlm_src = dwlm_on_device ? static_cast<float*>(dW_lm) : s->dwlm_retain;
  refs.push_back({dwlm_src, static_cast<float*>(dwlm_dev), static_cast<int64_t>(s->cfg.V) * c.H, 0});
  int64_t total_chunks = 0;
  for (GradRef& r : refs) {
    r.chunk_begin = total_chunks;
    total_chunks += (r.n + SCALE_CHUNK - 1) / SCALE_CHUNK;
  }
  KL_CUDA(cudaMemcpyAsync(s->refs, refs.data(), refs.size() * sizeof(GradRef), cudaMemcpyHostToDevice, cs));

  KL_TRY(begin_pass(s, cs));

  // ---------------- forward (the lm-head weight uploaded alongside) ----------------
  int cur = -1;
  KL_TRY(forward_layers(s, X, nullptr, cs, &cur, true));
  // ---------------- lm-head ----------------
  if (!s->bulk) KL_CUDA(cudaStreamWaitEvent(cs, s->ev_lm, 0));
  kl_lmhead_cfg lc = {T, c.H, s->cfg.V, c.dtype, KL_F32};
  KL_TRY(kl_lmhead_ce_argmax(&lc, s->hidden[L - 1], s->lm_w, targets, s->loss, s->argmax, nullptr, s->dx[0],
                             dwlm_src, s->lm_ws, s->lm_ws_bytes, cs));
  KL_TRY(sumsq(s, dwlm_src, static_cast<int64_t>(s->cfg.V) * c.H, n_weights(c) * L, cs));
  // ---------------- backward ----------------
  int in = 0;
  for (int l = L - 1; l >= 0; --l) {
    kl_layer_weights w;
    KL_TRY(weights_for(s, l, cur, &cur, &w, cs));
    if (!s->bulk && l - 1 >= 0) {
      int nxt;
      KL_TRY(acquire(s, l - 1, cur, &nxt));
    }
    kl_layer_saved* sv = s->saved_for(l);
    if (s->mode == KL_STREAM_RECOMPUTE && l != L - 1)   // the layer's activations again, from its input
      KL_TRY(kl_layer_forward(&c, &w, l == 0 ? X : s->hidden[l - 1], s->hidden[l], sv, s->ws, s->ws_bytes, cs));
    KL_TRY(kl_layer_backward(&c, &w, sv, s->dx[in], s->dx[in ^ 1], &src[l], s->ws, s->ws_bytes, cs));
    in ^= 1;
    for (int i = 0; i < n_weights(c); ++i)
      KL_TRY(sumsq(s, static_cast<const float*>(*gfield(src[l], i)), static_cast<int64_t>(weight_elems(c, i)),
                   n_weights(c) * l + i, cs));
    if (!s->bulk) KL_CUDA(cudaEventRecord(s->ev_used[cur], cs));
  }
  // ---------------- global norm, clip, delivery ----------------
  {
    const int nref = n_weights(c) * L + 1;
    ProfScope ps("clip_finalize", cs, 0.0, 8.0 * nref * SUMSQ_BLOCKS);
    launch_pdl(clip_finalize_kernel, 1, SUMSQ_THREADS, 0, cs, s->partials, nref, s->loss, clip_max_norm, s->result);
  }
  KL_CUDA(cudaGetLastError());
  {
    double moved = 0.0;
    for (const GradRef& r : refs) moved += 8.0 * static_cast<double>(r.n);
    ProfScope ps("clip_scale", cs, 0.0, moved);
    launch_pdl(clip_scale_kernel, 8 * num_sms(), 256, 0, cs, s->refs, static_cast<int>(refs.size()), total_chunks,
                                                     s->result);
  }
  KL_CUDA(cudaGetLastError());
  float host_res[4] = {};
  KL_CUDA(cudaMemcpyAsync(host_res, s->result, 3 * sizeof(float), cudaMemcpyDeviceToHost, cs));
  KL_CUDA(cudaStreamSynchronize(cs));
  result->loss = host_res[0];
  result->total_norm = host_res[1];
  result->clip_coef = host_res[2];
  return KL_OK;
}

kl_status kl_stream_forward(kl_stream* s, const void* X, void* Y, void* stream) {
  if (!s || !X || !Y) return set_error(KL_ERR_INVALID_ARG, "kl_stream_forward: null argument");
  int dev = -1;
  KL_CUDA(cudaGetDevice(&dev));
  if (dev != s->device)
    return set_error(KL_ERR_INVALID_ARG, "kl_stream_forward: created on device %d, current %d", s->device, dev);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  KL_TRY(begin_pass(s, cs));
  int cur = -1;
  KL_TRY(forward_layers(s, X, Y, cs, &cur, false));
  KL_CUDA(cudaStreamSynchronize(cs));
  return KL_OK;
}

size_t kl_stream_device_bytes(const kl_stream* s) { return s ? s->device_bytes : 0; }

void kl_stream_destroy(kl_stream* s) {
  if (!s) return;
  cudaDeviceSynchronize();
  s->release();
  delete s;
}

}  // extern "C"
