// A task processor for the tests of include/tg_custom.cuh: every token's
// score plus the entry of the row's state in its bucket (token mod S).
#include "tg_custom.cuh"

struct BucketBias {
  __device__ float operator()(float score, int token, const float* state, int S) const {
    return __fadd_rn(score, state[token % S]);
  }
};

extern "C" int task_select(const void* logits, int B, int V, const int32_t* hist_ids, const int64_t* hist_offsets,
                           const int32_t* prompt_lens, const void* cfg, const float* state, int S,
                           const float* uniforms, float* scores, int32_t* out_ids, float* out_logprobs,
                           void* stream) {
  return tg_custom::tg_select_custom(logits, B, V, hist_ids, hist_offsets, prompt_lens,
                                     static_cast<const tg_config*>(cfg), state, S, uniforms, scores, out_ids,
                                     out_logprobs, static_cast<tg_stream>(stream), BucketBias());
}

extern "C" int task_verify(const void* target, int B, int V, const int32_t* cand, int K, const void* cfg,
                           const float* state, int S, const float* uniforms, float* scores, int32_t* out_match,
                           int32_t* out_next, void* stream) {
  return tg_custom::tg_verify_custom(target, B, V, cand, K, static_cast<const tg_config*>(cfg), state, S, uniforms,
                                     scores, out_match, out_next, static_cast<tg_stream>(stream), BucketBias());
}
