/*
 * kl.h - C ABI of libkl: forward and backward of one Qwen3-style decoder layer
 * and the lm-head softmax cross-entropy with argmax, on one NVIDIA GB300
 * (sm_103a).
 *
 * What is computed follows the public pages on the subject:
 *   - "From-scratch GPU LLM training" (keilab.pages.dev/ai/gpu-llm and the
 *     markdown twin, section "What is built"): six gradient kernels (matrix
 *     multiply, RMSNorm, SiLU/SwiGLU, RoPE, softmax cross-entropy,
 *     scaled-dot-product attention); a GPU layer backward chaining them to 10
 *     tensors; a forward that saves activations for the backward; an lm-head
 *     softmax cross-entropy fused with argmax in a single launch; a
 *     layer-streaming driver that holds one layer's weights at a time.
 *   - "KYNETRA FOUNDRY" (hyperbridge-deck.pages.dev): pre-norm decoder wiring
 *     (RMSNorm -> causal self-attention -> SwiGLU FFN, each in a residual),
 *     grouped-query attention, rotary position embedding, tiled attention
 *     with an online softmax (an exact reordering of plain attention).
 *
 * Conventions for every entry point
 *   - Tensors are dense, row-major, token-major: T = B*S rows, token
 *     t = b*S + s sits at position s. Activations [T, width]; q [T, Hq*d];
 *     k, v [T, Hkv*d]; lse [B, Hq, S] fp32. Projection weights are stored
 *     [out, in] and applied as y = x W^T.
 *   - Rotary planes pair element i with element i + d/2; plane i turns by
 *     s * rope_base^(-2i/d). Query head h reads key/value head
 *     floor(h * Hkv / Hq). Attention scale 1/sqrt(d); causal mask keeps
 *     keys j <= i.
 *   - RMSNorm: h = gamma * x / sqrt(mean(x^2) + eps), statistics in fp32.
 *   - SwiGLU: m = silu(gate) * up.
 *   - dtype KL_BF16: weights and activations are bf16, every matrix product
 *     runs on the tensor cores with fp32 accumulation, normalisation and
 *     softmax statistics in fp32. dtype KL_F32: everything fp32, matrix
 *     products on CUDA cores (no TF32).
 *   - Pointers marked "device" must be device memory (or managed memory) of
 *     the current device, 16-byte aligned. The caller owns every buffer:
 *     outputs, saved activations and workspace. Sizes come from the *_bytes
 *     queries. Only kl_stream_* allocates, and frees in kl_stream_destroy.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously; no entry point synchronises
 *     the stream except where stated.
 *   - Errors: every call returns a kl_status and never aborts the process.
 *     On a non-KL_OK return kl_last_error() describes it (thread-local). A
 *     bad argument found on the host enqueues no work. Faults found inside a
 *     kernel (a target id out of range, a bounded wait that ran out) are
 *     recorded in a device error word and reported by kl_device_status().
 */
#ifndef KL_H_
#define KL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KL_API __attribute__((visibility("default")))
#else
#define KL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kl_status {
  KL_OK = 0,
  KL_ERR_INVALID_ARG = 1,  /* null pointer, misaligned buffer, bad size */
  KL_ERR_UNSUPPORTED = 2,  /* shape or dtype this build does not handle */
  KL_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  KL_ERR_TIMEOUT = 4,      /* a bounded wait inside a kernel ran out */
  KL_ERR_NO_MEMORY = 5,    /* workspace too small, or allocation failed */
  KL_ERR_DEVICE = 6        /* a kernel rejected its input (see kl_last_error) */
} kl_status;

typedef enum kl_dtype { KL_F32 = 0, KL_BF16 = 1 } kl_dtype;

/* Device error word bits, reported by kl_device_status(). */
#define KL_DEVERR_TIMEOUT 0x1u      /* a pipeline wait gave up */
#define KL_DEVERR_TARGET 0x2u       /* a CE target id was outside [0, V) */
#define KL_DEVERR_SMEM 0x4u         /* a kernel found its shared memory misaligned
                                       and returned without doing its work */
#define KL_DEVERR_PAGE 0x8u         /* a paged-cache position past its block-table row,
                                       or a table entry outside the pool (the access
                                       was skipped)                                   */

KL_API const char* kl_version(void);
KL_API const char* kl_status_str(kl_status s);
/* Message of the last failing call on this host thread ("" if none). */
KL_API const char* kl_last_error(void);
/* Synchronises `stream`, then reads and clears the current device's error
 * word. Returns KL_OK if it was zero, KL_ERR_TIMEOUT or KL_ERR_DEVICE if a
 * kernel recorded a fault; *bits (may be NULL) receives the raw word. */
KL_API kl_status kl_device_status(void* stream, uint32_t* bits);
/* Test hook for the recovery path above (no counterpart on the pages): waits
 * for the whole device, then leaves the arrival counters of the few-rows GEMM
 * and of the fused RMSNorm backward's grid barrier as a launch that gave up on
 * a wait can leave them (one arrival counted, never completed) and sets
 * KL_DEVERR_TIMEOUT in the error word, which is what such a launch does. The
 * next kl_device_status returns KL_ERR_TIMEOUT and zeroes those counters;
 * a launch of either kernel before that call reads the stale counts (wrong
 * results, no hang: neither kernel waits on these counters without a limit).
 * Returns KL_OK or KL_ERR_CUDA. */
KL_API kl_status kl_test_abandon_counters(void);

/* Launch profiler. Every kernel launch of the library is counted. While
 * profiling is on, each launch is also bracketed by CUDA events on its
 * stream and tagged with its algorithmic work (FLOPs for contractions,
 * minimal HBM bytes for the memory-bound kernels). kl_profile_enable(1)
 * clears earlier records; kl_profile_read synchronises on the last event and
 * aggregates per kernel name into out[0..max) (returns the entry count, or
 * -1 on a CUDA error). Not thread-safe across concurrent streams' timing. */
typedef struct kl_prof_entry {
  char name[48];
  int32_t launches;
  double ms;           /* summed event time                                */
  double flops;        /* summed algorithmic FLOPs                         */
  double bytes;        /* summed algorithmic HBM bytes                     */
} kl_prof_entry;
KL_API kl_status kl_profile_enable(int32_t on);
KL_API int32_t kl_profile_read(kl_prof_entry* out, int32_t max_entries);
KL_API uint64_t kl_launch_count(void);

/* ------------------------------------------------------------------------ */
/* Decoder layer ("From-scratch GPU LLM training", "What is built": forward  */
/* with saved activations; layer backward orchestrating the six kernels)    */
/* ------------------------------------------------------------------------ */

typedef struct kl_layer_cfg {
  int32_t B, S;        /* batch, sequence length; T = B*S tokens           */
  int32_t H;           /* hidden width                                      */
  int32_t Hq, Hkv, d;  /* query heads, key/value heads, head dim           */
  int32_t I;           /* SwiGLU intermediate width                        */
  float eps;           /* RMSNorm epsilon                                   */
  float rope_base;     /* rotary base                                       */
  int32_t dtype;       /* kl_dtype of weights, activations and arithmetic  */
  /* Options beyond the pages' layer (0 = off): */
  int32_t qk_norm;     /* 1: RMSNorm over each q and k head (gains gamma_q,
                          gamma_k of length d shared by the heads), before
                          the rotation, as in Qwen3 checkpoints              */
  int32_t rope_interleaved; /* 1: rotary planes (2i, 2i+1); 0: (i, i+d/2)   */
} kl_layer_cfg;

/* Device pointers, dtype = cfg.dtype. gamma1/gamma2: [H]. wq [Hq*d, H],
 * wk/wv [Hkv*d, H], wo [H, Hq*d], wg/wu [I, H], wd [H, I]; gamma_q/gamma_k
 * [d] (read only when cfg.qk_norm, may be NULL otherwise). */
typedef struct kl_layer_weights {
  const void *gamma1, *wq, *wk, *wv, *wo, *gamma2, *wg, *wu, *wd;
  const void *gamma_q, *gamma_k;
} kl_layer_weights;

/* Activations the forward saves for the backward (device, caller-owned).
 * Element type is cfg.dtype unless noted. The forward also records its
 * input X in `x`; X must stay alive and unchanged until the backward. */
typedef struct kl_layer_saved {
  const void* x;       /* [T,H] the forward's input (pointer recorded)     */
  void* h1;            /* [T,H] RMSNorm-1 output                           */
  float* rstd1;        /* [T]   1/sqrt(mean(x^2)+eps) of X                 */
  void* q;             /* [T,Hq*d]  query after RoPE                       */
  void* k;             /* [T,Hkv*d] key after RoPE                         */
  void* v;             /* [T,Hkv*d] value                                  */
  void* o;             /* [T,Hq*d]  attention output                       */
  float* lse;          /* [B,Hq,S]  softmax logsumexp (natural log)        */
  void* x2;            /* [T,H] residual stream after attention            */
  void* h2;            /* [T,H] RMSNorm-2 output                           */
  float* rstd2;        /* [T]                                              */
  void* g;             /* [T,I] gate projection                            */
  void* u;             /* [T,I] up projection                              */
  void* m;             /* [T,I] silu(g) * u                                */
  /* cfg.qk_norm only (NULL otherwise): */
  void* q_pre;         /* [T,Hq*d]  query projection before its norm        */
  void* k_pre;         /* [T,Hkv*d] key projection before its norm          */
  float* rstd_q;       /* [T,Hq]  per-head 1/sqrt(mean(q^2)+eps)            */
  float* rstd_k;       /* [T,Hkv]                                           */
  /* KL_BF16 only (NULL otherwise): the rotary (cos, sin) pairs [S][d/2] fp32,
   * written by the forward (with the first norm), read by the backward. */
  float* rope;
} kl_layer_saved;

/* Gradients written by the backward (device, caller-owned). Projection
 * gradients have element type `dtype` (KL_F32 or KL_BF16; KL_F32 only when
 * cfg.dtype is KL_F32 or for the streaming driver's clip); gain gradients
 * dgamma1/dgamma2 are always fp32 [H]. Each is overwritten, not added to. */
typedef struct kl_layer_grads {
  void *gamma1, *wq, *wk, *wv, *wo, *gamma2, *wg, *wu, *wd;
  int32_t dtype;
  void *gamma_q, *gamma_k;  /* fp32 [d], cfg.qk_norm only (may be NULL otherwise) */
} kl_layer_grads;

/* Bytes of one buffer holding every saved activation, and a carve of such a
 * buffer into a kl_layer_saved (base must be 256-byte aligned, device). */
KL_API size_t kl_layer_saved_bytes(const kl_layer_cfg* cfg);
KL_API kl_status kl_layer_saved_carve(const kl_layer_cfg* cfg, void* base, size_t bytes,
                               kl_layer_saved* out);
/* Workspace bytes of the forward and the backward (device, caller-owned,
 * 256-byte aligned; contents undefined between calls). The forward's
 * workspace is optional (ws may be NULL): with it, the projections' last
 * round of tiles is split along K over every CTA pair. */
KL_API size_t kl_layer_fwd_workspace_bytes(const kl_layer_cfg* cfg);
KL_API size_t kl_layer_bwd_workspace_bytes(const kl_layer_cfg* cfg);

/* Y = x2 + W_d(silu(W_g h2) * W_u h2), h2 = RMSNorm(x2; gamma2),
 * x2 = X + W_o Attn(RoPE(W_q h1), RoPE(W_k h1), W_v h1), h1 = RMSNorm(X; gamma1).
 * X, Y: [T,H] device, cfg.dtype. Fills *saved (its buffers caller-owned).
 * KL_BF16 needs d = 128, H, Hq*d, Hkv*d and I multiples of 64, Hq % Hkv = 0. */
KL_API kl_status kl_layer_forward(const kl_layer_cfg* cfg, const kl_layer_weights* w,
                           const void* X, void* Y, kl_layer_saved* saved,
                           void* ws, size_t ws_bytes, void* stream);

/* Backward of kl_layer_forward for upstream gradient dY [T,H]: writes dX
 * [T,H] (cfg.dtype) and all nine parameter gradients into *grads. */
KL_API kl_status kl_layer_backward(const kl_layer_cfg* cfg, const kl_layer_weights* w,
                            const kl_layer_saved* saved, const void* dY, void* dX,
                            const kl_layer_grads* grads, void* ws, size_t ws_bytes,
                            void* stream);

/* ------------------------------------------------------------------------ */
/* lm-head softmax cross-entropy + argmax ("From-scratch GPU LLM training",  */
/* capability list: softmax cross-entropy and argmax fused in one launch)    */
/* ------------------------------------------------------------------------ */

typedef struct kl_lmhead_cfg {
  int32_t N;        /* tokens                                               */
  int32_t H;        /* hidden width                                         */
  int32_t V;        /* vocabulary                                           */
  int32_t dtype;    /* kl_dtype of X, W, dX, dlogits                        */
  int32_t dw_dtype; /* kl_dtype of dW (KL_F32 allowed with KL_BF16 inputs)  */
} kl_lmhead_cfg;

KL_API size_t kl_lmhead_workspace_bytes(const kl_lmhead_cfg* cfg);

/* z = X W^T (fp32 logits, kept in workspace); per row lse, loss_n =
 * lse - z[target]; *loss = mean_n loss_n (device fp32 scalar); argmax[n] =
 * lowest index of the row maximum of the fp32 logits; dlogits = (softmax -
 * onehot)/N; dX = dlogits W; dW = dlogits^T X.
 * X [N,H], W [V,H], targets int32 [N] in [0,V), argmax int32 [N],
 * dlogits [N,V] (may be NULL: kept in workspace), dX [N,H], dW [V,H].
 * All device. */
KL_API kl_status kl_lmhead_ce_argmax(const kl_lmhead_cfg* cfg, const void* X, const void* W,
                              const int32_t* targets, float* loss, int32_t* argmax,
                              void* dlogits, void* dX, void* dW, void* ws,
                              size_t ws_bytes, void* stream);

/* The single-launch cross-entropy step alone, on given fp32 logits z [N,V]:
 * loss (device fp32 scalar, mean over rows), argmax int32 [N], dlogits [N,V]
 * of type dz_dtype, scaled by 1/N. Workspace: kl_ce_workspace_bytes(N).
 * dlogits must not overlap z (KL_ERR_INVALID_ARG): a row's loss reads its
 * target logit after the row's dlogits are written. */
KL_API size_t kl_ce_workspace_bytes(int32_t N);
KL_API kl_status kl_ce_argmax(int32_t N, int32_t V, const float* z, const int32_t* targets,
                       float* loss, int32_t* argmax, void* dlogits, int32_t dz_dtype,
                       void* ws, size_t ws_bytes, void* stream);

/* Allocation-free form of kl_ce_argmax. The pages have no counterpart: this
 * is a library addition for callers that cannot give the library device
 * memory -- an application whose device memory belongs to its own pool and
 * forbids raw cudaMalloc, a plugin without an allocator hook, or a loop that
 * cannot afford cudaMalloc's implicit device synchronisation. Same inputs,
 * outputs and results as kl_ce_argmax, but the per-row losses and the
 * completion counter live in a static device array compiled into libkl
 * (KL_CE_NOALLOC_MAX_ROWS + 65 floats, about 256 KB), which every device that
 * loads the library keeps until process exit. Calls no cudaMalloc/cudaFree.
 * The first call on each device (with that device current) looks up the
 * array's address; make that first call before any stream capture. Every call
 * shares the array and the counter is cleared before each launch, so calls
 * whose kernels may overlap on the GPU (unordered streams) race: do not issue
 * them. N above KL_CE_NOALLOC_MAX_ROWS returns KL_ERR_UNSUPPORTED. */
#define KL_CE_NOALLOC_MAX_ROWS 65535
KL_API kl_status kl_ce_argmax_noalloc(int32_t N, int32_t V, const float* z, const int32_t* targets,
                                      float* loss, int32_t* argmax, void* dlogits, int32_t dz_dtype,
                                      void* stream);

/* ------------------------------------------------------------------------ */
/* The individual gradient kernels (the pages' six), for callers composing   */
/* their own layers and for kernel-level tests. Same layouts as above.       */
/* ------------------------------------------------------------------------ */

/* C[M,N] = op(A) op(B)^T (+ R), fp32 accumulation.
 * a_mn_major = 0: A is [M,K] with row stride lda (K contiguous);
 *            = 1: A is stored [K,M] with row stride lda (M contiguous).
 * b_mn_major = 0: B is [N,K] row stride ldb; = 1: B is stored [K,N].
 * A, B have type `dtype`; C has c_dtype; R (may be NULL) has r_dtype, [M,N]
 * row stride ldr. KL_BF16 runs on the tensor cores and needs lda, ldb, K
 * multiples of 8; KL_F32 on CUDA cores. C must not overlap A or B (output
 * tiles are written while other tiles still read the operands); R may be C
 * itself (each element's addend is read before that element is written). */
KL_API kl_status kl_gemm(int32_t M, int32_t N, int32_t K, int32_t dtype,
                  const void* A, int64_t lda, int32_t a_mn_major,
                  const void* B, int64_t ldb, int32_t b_mn_major,
                  void* C, int64_t ldc, int32_t c_dtype,
                  const void* R, int64_t ldr, int32_t r_dtype, void* stream);
/* kl_gemm with an fp32 device scratch (ws, 256-byte aligned; ws_bytes of at
 * least kl_gemm_scratch_bytes(), else it is not used). With it a KL_BF16
 * product may (a) split its last round of tiles along K when that round would
 * leave CTA pairs idle, and (b) when M <= 128 with both operands K-major, run
 * on the few-rows kernel (the weights streamed once over one CTA per SM,
 * K-range pieces summed in a fixed order). Results are deterministic either
 * way. The scratch's content is not kept between calls. */
KL_API size_t kl_gemm_scratch_bytes(void);
KL_API kl_status kl_gemm_ex(int32_t M, int32_t N, int32_t K, int32_t dtype,
                  const void* A, int64_t lda, int32_t a_mn_major,
                  const void* B, int64_t ldb, int32_t b_mn_major,
                  void* C, int64_t ldc, int32_t c_dtype,
                  const void* R, int64_t ldr, int32_t r_dtype,
                  void* ws, size_t ws_bytes, void* stream);

/* h = gamma * x * rstd, rstd = 1/sqrt(mean(x^2)+eps); x,h [rows,width]. */
KL_API kl_status kl_rmsnorm_fwd(int32_t rows, int32_t width, int32_t dtype, const void* x,
                         const void* gamma, float eps, void* h, float* rstd, void* stream);
/* dx = resid + rstd*(dn - n*mean(dn*n)), dn = dh*gamma, n = x*rstd;
 * dgamma = sum_rows dh*n (fp32 [width]). dh has dh_dtype (fp32 or dtype);
 * resid (may be NULL) and dx have dtype. Workspace: kl_rmsnorm_bwd_ws_bytes. */
KL_API size_t kl_rmsnorm_bwd_ws_bytes(int32_t rows, int32_t width);
KL_API kl_status kl_rmsnorm_bwd(int32_t rows, int32_t width, int32_t dtype, const void* dh,
                         int32_t dh_dtype, const void* x, const void* gamma, const float* rstd,
                         const void* resid, void* dx, float* dgamma, void* ws, size_t ws_bytes,
                         void* stream);
/* In-place rotary embedding of x [B*S, heads, d]; direction +1 forward,
 * -1 backward (rotation by the negative angle). */
KL_API kl_status kl_rope(int32_t B, int32_t S, int32_t heads, int32_t d, float base, int32_t dtype,
                  void* x, int32_t direction, void* stream);
/* m = silu(g)*u; and its backward dg = dm*u*silu'(g), du = dm*silu(g). */
KL_API kl_status kl_swiglu_fwd(int64_t n, int32_t dtype, const void* g, const void* u, void* m,
                        void* stream);
KL_API kl_status kl_swiglu_bwd(int64_t n, int32_t dtype, const void* dm, const void* g, const void* u,
                        void* dg, void* du, void* stream);
/* Causal GQA attention: q [T,Hq*d], k/v [T,Hkv*d] -> o [T,Hq*d], lse fp32 [B,Hq,S]. */
KL_API kl_status kl_attention_fwd(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d,
                           int32_t dtype, const void* q, const void* k, const void* v, void* o,
                           float* lse, void* stream);
/* Backward: dq [T,Hq*d], dk/dv [T,Hkv*d] (dtype), recomputing the softmax
 * from lse. Workspace: kl_attention_bwd_ws_bytes. */
KL_API size_t kl_attention_bwd_ws_bytes(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d);
KL_API kl_status kl_attention_bwd(int32_t B, int32_t S, int32_t Hq, int32_t Hkv, int32_t d,
                           int32_t dtype, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, void* dq,
                           void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Layer streaming ("From-scratch GPU LLM training", capability list: the   */
/* full-depth model runs holding one layer's weights at a time, lossless    */
/* against the bulk forward; end-to-end smoke trains under gradient clip)   */
/* ------------------------------------------------------------------------ */

typedef struct kl_stream kl_stream;

/* What the driver keeps between a layer's forward and its backward. */
enum {
  KL_STREAM_SAVE_ALL = 0,   /* every layer's saved activations stay resident    */
  KL_STREAM_RECOMPUTE = 1,  /* only each layer's input stays resident; the layer's
                               forward is run again (same slot, same weights)
                               right before its backward. Device memory for
                               activations: one layer's saved set + T x H per
                               layer, independent of depth otherwise          */
  KL_STREAM_FORWARD = 2     /* forward only (kl_stream_forward): two weight
                               slots, one layer's working set and two hidden
                               buffers: device memory independent of depth;
                               no lm-head weight, kl_stream_run refused       */
};

typedef struct kl_stream_cfg {
  kl_layer_cfg layer;  /* dims of every layer; dtype must be KL_BF16 or F32 */
  int32_t n_layers;
  int32_t V;           /* lm-head vocabulary (ignored by KL_STREAM_FORWARD) */
  int32_t mode;        /* KL_STREAM_SAVE_ALL, _RECOMPUTE or _FORWARD         */
} kl_stream_cfg;

typedef struct kl_stream_result {
  float loss;          /* mean CE loss                                     */
  float total_norm;    /* global L2 norm of all weight gradients, unclipped */
  float clip_coef;     /* min(1, max_norm / (total_norm + 1e-6))            */
} kl_stream_result;

/* host_layers[n_layers]: HOST pointers (pinned or pageable) to each layer's
 * weights in cfg.layer.dtype (gamma_q/gamma_k too when cfg.layer.qk_norm,
 * else they are ignored); host_lm_head [V,H] host (may be null with
 * KL_STREAM_FORWARD). The driver keeps the pointers (no copy of the weights);
 * they must stay valid until destroy. Device-memory layer weights select the
 * bulk mode (no slots, no uploads, same kernels in the same order).
 * Allocates on the current device: two weight slots, the lm-head weight,
 * saved activations (per cfg->mode) and workspace. */
KL_API kl_status kl_stream_create(const kl_stream_cfg* cfg, const kl_layer_weights* host_layers,
                           const void* host_lm_head, kl_stream** out);
/* One training step: streams layer weights in (copy stream, double-buffered),
 * forward through every layer saving activations, lm-head CE on `targets`,
 * backward in reverse re-streaming the weights, global-norm clip of every
 * weight gradient at clip_max_norm. X [T,H] and targets [T] are device.
 * grads[n_layers] and dW_lm [V,H]: destination of the clipped gradients, fp32,
 * device memory or page-locked host memory (reached through its device-visible
 * address). Gradients for device destinations are computed and scaled in
 * place; gradients for host destinations are computed into device buffers the
 * driver allocates on first use (fp32, every layer's gradients) and written
 * out already clipped after the backward. *result is written before the call
 * returns; the call synchronises `stream`. */
KL_API kl_status kl_stream_run(kl_stream* s, const void* X, const int32_t* targets,
                        float clip_max_norm, const kl_layer_grads* grads, void* dW_lm,
                        kl_stream_result* result, void* stream);
/* Forward only, in any mode: X [T,H] device -> Y [T,H] device (cfg.layer.dtype),
 * the hidden state after the last layer, streaming every layer's weights as
 * kl_stream_run's forward does (the lm-head is not applied). Synchronises
 * `stream` before returning. X and Y must not overlap the driver's buffers. */
KL_API kl_status kl_stream_forward(kl_stream* s, const void* X, void* Y, void* stream);
/* Device bytes the driver allocated (weight slots + activations + workspace;
 * the retained gradient buffers once a run delivered to host memory). */
KL_API size_t kl_stream_device_bytes(const kl_stream* s);
KL_API void kl_stream_destroy(kl_stream* s);

/* ------------------------------------------------------------------------ */
/* Forward with a paged key/value cache ("From-scratch GPU LLM training",    */
/* "What is built": a GPU forward path with a paged key-value cache;         */
/* "KYNETRA FOUNDRY", paged-KV paragraph: fixed-size token blocks anywhere   */
/* in a global pool, a per-sequence block table mapping logical positions to */
/* physical blocks, keys and values gathered through it)                     */
/* ------------------------------------------------------------------------ */

/* A step feeds n_new new tokens to each of B sequences (n_new = 1: decode).
 * Sequence b already holds ctx[b] tokens in the cache, so its new token i
 * sits at absolute position ctx[b] + i: the rotary angle and the causal
 * limit use that position. A pool (one for keys, one for values, per layer)
 * is [n_blocks][block_size][Hkv * d] in the layer dtype; position p of
 * sequence b lives in block table[b * max_blocks + p / block_size], slot
 * p % block_size. The caller owns pools and tables and assigns the blocks.
 * This path is bf16 with head dim 128 and at most 64 query rows per kv head
 * and step ((Hq / Hkv) * n_new <= 64). A position past its table row or a
 * table entry outside [0, n_blocks) is skipped and reported by
 * kl_device_status (KL_DEVERR_PAGE). Pool rows (n_blocks * block_size * Hkv)
 * must stay below 2^31. */
typedef struct kl_paged_cfg {
  int32_t B;           /* sequences in the step                              */
  int32_t n_new;       /* new tokens per sequence                            */
  int32_t block_size;  /* tokens per cache block                             */
  int32_t max_blocks;  /* length of each block-table row                     */
  int32_t n_blocks;    /* blocks in each pool                                */
} kl_paged_cfg;

/* The new tokens' keys and values (k_new, v_new [B*n_new, Hkv*d] device,
 * rows b * n_new + i) into their cache slots. table [B*max_blocks] and ctx
 * [B] are device int32. */
KL_API kl_status kl_paged_kv_write(const kl_paged_cfg* pc, int32_t Hkv, int32_t d, int32_t dtype,
                                   const void* k_new, const void* v_new, const int32_t* table,
                                   const int32_t* ctx, void* k_pool, void* v_pool, void* stream);
/* Workspace for kl_paged_attention: the partial results of (sequence, kv
 * head) items whose keys are shared out between several CTAs; 0 when none is.
 * It depends on the device's SM count. */
KL_API size_t kl_paged_attention_ws_bytes(const kl_paged_cfg* pc, int32_t Hq, int32_t Hkv, int32_t d);
/* Causal GQA attention of the new queries q [B*n_new, Hq*d] (after the
 * rotation) over each sequence's cache, positions 0 .. ctx[b] + n_new - 1:
 * the new tokens' keys and values must already be written. Query i of
 * sequence b sees keys at positions <= ctx[b] + i; scale 1/sqrt(d); query
 * head h reads kv head floor(h * Hkv / Hq). o [B*n_new, Hq*d] device; lse
 * [B, Hq, n_new] fp32 device (natural log) or NULL. */
KL_API kl_status kl_paged_attention(const kl_paged_cfg* pc, int32_t Hq, int32_t Hkv, int32_t d, int32_t dtype,
                                    const void* q, const void* k_pool, const void* v_pool,
                                    const int32_t* table, const int32_t* ctx, void* o, float* lse,
                                    void* ws, size_t ws_bytes, void* stream);
/* Workspace for kl_layer_forward_paged. */
KL_API size_t kl_layer_forward_paged_ws_bytes(const kl_layer_cfg* cfg, const kl_paged_cfg* pc);
/* The layer forward of kl_layer_forward for the step's new tokens against a
 * paged cache: X, Y [B*n_new, H] device with cfg->B == pc->B and cfg->S ==
 * pc->n_new (so T = B*S rows, as everywhere); q and k are rotated at their
 * absolute positions, the new keys and values are written into the layer's
 * pools, then attention reads the cache. Nothing is saved for a backward. */
KL_API kl_status kl_layer_forward_paged(const kl_layer_cfg* cfg, const kl_paged_cfg* pc,
                                        const kl_layer_weights* w, const void* X, void* Y, void* k_pool,
                                        void* v_pool, const int32_t* table, const int32_t* ctx, void* ws,
                                        size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KL_H_ */
