// argus_window_prefill_attn: attention of a query chunk against one window of
// cached keys, folded into an fp32 accumulator by log2-sum-exp.
//
// "feat(kvcache): host-RAM KV tier for sparse-attention models", comment on
// "--kv-placement host": cached pages are staged into a 131,072-token device
// window, attended per window, and the windows folded by their log2-sum-exp
// into a float32 accumulator allocated up front.
#include "common.cuh"

using namespace argus;

extern "C" argus_status argus_window_prefill_attn(const argus_geom* g, int32_t n_q, const void* q,
                                                  const void* k, const void* v, int64_t kv_head_stride,
                                                  int64_t win_len, int64_t win_pos0, int64_t q_pos0,
                                                  float softmax_scale, float* acc_o, float* acc_lse2,
                                                  int32_t fold, void* stream) {
  (void)g; (void)n_q; (void)q; (void)k; (void)v; (void)kv_head_stride; (void)win_len;
  (void)win_pos0; (void)q_pos0; (void)softmax_scale; (void)acc_o; (void)acc_lse2; (void)fold;
  (void)stream;
  return fail(ARGUS_E_UNSUPPORTED, "window prefill: not implemented in this build");
}
