/*
 * tg_custom.cuh -- a task's processor as a device function compiled by the
 * caller (Transmuter.Generation, section "Processors": a processor is a
 * per-row state made on the host before each step, plus a function of the
 * row's logits and that state run in the compiled selection; the task's
 * processors come after begin_suppress_tokens and before the temperature).
 *
 * Header-only: include it in a .cu file compiled with nvcc for sm_103a
 * (-I include -I logits_processing_token_gb300/csrc) and link libtg.
 *
 * The function is a functor
 *
 *     struct MyProcessor {
 *       __device__ float operator()(float score, int token, const float* state, int S) const;
 *     };
 *
 * giving token `token`'s new score from its score after the built-in
 * processors (repetition penalty .. begin_suppress_tokens) and the row's
 * state (S floats, the same shape every step; NULL when no state is given).
 * Its result is never taken below the filter value (-FLT_MAX).  It runs once
 * per token of every row that is not empty, forced rows included.  It may
 * read any of the row's state but only its own token's score: a processor
 * that needs the other scores of the row is not expressible here.
 *
 * tg_select_custom<Proc>(...) runs it in one kernel that writes every row's
 * final scores (after the temperature, when sampling) to `scores` (device
 * f32 [B, V], owned by the caller), then selects from them with
 * tg_config_selection(cfg): tg_select, or tg_select_logprobs when
 * out_logprobs is not NULL.  That is one more write and read of B x V x 4
 * bytes than tg_select's single pass.  Arguments as tg_select, plus:
 *  state   device f32 [B, S] row-major, or NULL with S = 0.
 *  scores  device f32 [B, V] scratch.
 * Errors: TG_ERR_INVALID_ARGUMENT for a bad argument or a config with the
 * sparse processor kinds (those run in tg_select_state), TG_ERR_CUDA.
 *
 * tg_verify_custom<Proc>(...) is assisted-generation verify (Assisted
 * Generation, steps 3-5) with the task processor at every one of the K+1
 * positions of each row: position j of row b is target row b (K+1) + j, with
 * state row b (K+1) + j (state: device f32 [B (K+1), S], or NULL with S = 0);
 * as in tg_verify, the history processors do not run per position.  Its
 * scores (then the temperature) go to `scores` (device f32 [B (K+1), V]) and
 * tg_verify selects from them with tg_config_selection(cfg).  Arguments as
 * tg_verify otherwise.
 */
#pragma once

#include <cuda_runtime.h>

#include "tg.h"
#include "tg_device.cuh"

namespace tg_custom {

constexpr int kThreads = tg::kThreads;

// HIST: the rows have histories and the built-in processors run (select);
// otherwise every row is a verify position and only the task's function runs.
template <int DT, class Proc, bool HIST>
__global__ void __launch_bounds__(kThreads) task_scores_kernel(const tg::DevCfg c, const void* logits, int B, int V,
                                                               const int32_t* hist, const int64_t* off,
                                                               const int32_t* plen, const float* state, int S,
                                                               float* scores, Proc proc) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int nwords = (V + 31) / 32;
  unsigned* H = reinterpret_cast<unsigned*>(smem_raw);
  unsigned* N = H + (nwords * 4 + 127) / 128 * 32;
  const int row = static_cast<int>(blockIdx.x);
  tg::RowMeta rm{};
  int zs[8];
  int nz = 0;
  if (HIST) {
    rm = tg::row_meta(c, hist, off, plen, row, B);
    if (rm.bad || rm.L == 0) return;   // the selection gives these rows -1
    tg::build_row_bitmaps(c, hist, rm, H, N, nwords);
    nz = rm.forced ? tg::forced_zeros(c, rm, zs) : 0;
  }
  const float* st = state ? state + static_cast<size_t>(row) * S : nullptr;
  const bool tempered = c.mode == tg::kSample && c.temp != 1.0f;
  const unsigned char* rowp = static_cast<const unsigned char*>(logits) + static_cast<size_t>(row) * V * (DT == tg::kF32 ? 4 : 2);
  float* out = scores + static_cast<size_t>(row) * V;
  for (int i = threadIdx.x; i < V; i += kThreads) {
    float s;
    if (HIST && rm.forced) {
      s = tg::kFilter;
      for (int q = 0; q < nz; ++q) s = zs[q] == i ? 0.0f : s;
    } else {
      const float x = DT == tg::kF32
                          ? __ldg(reinterpret_cast<const float*>(rowp) + i)
                          : __uint_as_float(static_cast<unsigned>(__ldg(reinterpret_cast<const unsigned short*>(rowp) + i)) << 16);
      s = HIST ? tg::process_elem(c, H, N, x, i, false) : x;
    }
    s = tg::clampf(proc(s, i, st, S));
    if (tempered) s = tg::clampf(__fdiv_rn(s, c.temp));
    out[i] = s;
  }
}

template <class Proc>
inline tg_status tg_select_custom(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                                  const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                                  const float* state, int32_t S, const float* uniforms, float* scores,
                                  int32_t* out_ids, float* out_logprobs, tg_stream stream, Proc proc = Proc()) {
  tg::DevCfg c;
  if (!cfg || tg_config_view(cfg, &c, sizeof(c)) != TG_OK) return TG_ERR_INVALID_ARGUMENT;
  if (c.nproc > 0 || B < 0 || V != c.V || S < 0 || (S > 0) != (state != nullptr)) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (!logits || !hist_offsets || !prompt_lens || !scores || !out_ids) return TG_ERR_INVALID_ARGUMENT;
  const int nwords = (V + 31) / 32;
  const int smem = 2 * ((nwords * 4 + 127) / 128 * 128);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto k = c.dtype == tg::kF32 ? task_scores_kernel<tg::kF32, Proc, true> : task_scores_kernel<tg::kBF16, Proc, true>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return TG_ERR_CUDA;
  k<<<B, kThreads, smem, s>>>(c, logits, B, V, hist_ids, hist_offsets, prompt_lens, state, S, scores, proc);
  if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
  const tg_config* sel = tg_config_selection(cfg);
  if (out_logprobs)
    return tg_select_logprobs(scores, B, V, hist_ids, hist_offsets, prompt_lens, sel, uniforms, out_ids, out_logprobs,
                              stream);
  return tg_select(scores, B, V, hist_ids, hist_offsets, prompt_lens, sel, uniforms, out_ids, stream);
}

template <class Proc>
inline tg_status tg_verify_custom(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids, int32_t K,
                                  const tg_config* cfg, const float* state, int32_t S, const float* uniforms,
                                  float* scores, int32_t* out_match, int32_t* out_next, tg_stream stream,
                                  Proc proc = Proc()) {
  tg::DevCfg c;
  if (!cfg || tg_config_view(cfg, &c, sizeof(c)) != TG_OK) return TG_ERR_INVALID_ARGUMENT;
  if (c.nproc > 0 || B < 0 || K < 1 || V != c.V || S < 0 || (S > 0) != (state != nullptr))
    return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (!target_logits || !cand_ids || !scores || !out_match || !out_next) return TG_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(B) * (K + 1) > 0x7fffffffLL) return TG_ERR_INVALID_ARGUMENT;
  const int rows = B * (K + 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto k = c.dtype == tg::kF32 ? task_scores_kernel<tg::kF32, Proc, false> : task_scores_kernel<tg::kBF16, Proc, false>;
  k<<<rows, kThreads, 0, s>>>(c, target_logits, rows, V, nullptr, nullptr, nullptr, state, S, scores, proc);
  if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
  return tg_verify(scores, B, V, cand_ids, K, tg_config_selection(cfg), uniforms, out_match, out_next, stream);
}

}  // namespace tg_custom
