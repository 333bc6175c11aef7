// Layer-streaming driver (placeholder until the streamed stack is wired).
#include "internal.h"
#include "kl_common.cuh"

using namespace kl;

struct kl_stream {
  int unused;
};

extern "C" {

kl_status kl_stream_create(const kl_stream_cfg* cfg, const kl_layer_weights* host_layers,
                           const void* host_lm_head, kl_stream** out) {
  (void)cfg; (void)host_layers; (void)host_lm_head;
  if (out) *out = nullptr;
  return set_error(KL_ERR_UNSUPPORTED, "layer streaming not built yet");
}

kl_status kl_stream_run(kl_stream* s, const void* X, const int32_t* targets, float clip_max_norm,
                        const kl_layer_grads* grads, void* dW_lm, kl_stream_result* result,
                        void* stream) {
  (void)s; (void)X; (void)targets; (void)clip_max_norm; (void)grads; (void)dW_lm; (void)result; (void)stream;
  return set_error(KL_ERR_UNSUPPORTED, "layer streaming not built yet");
}

size_t kl_stream_device_bytes(const kl_stream* s) { (void)s; return 0; }

void kl_stream_destroy(kl_stream* s) { (void)s; }

}
