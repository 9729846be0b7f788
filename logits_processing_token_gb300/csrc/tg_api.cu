// C ABI of libtg (declared in include/tg.h): argument checks, config
// creation and kernel launches.  Every check that can be made on the host is
// made here, before anything is enqueued.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/tg.h"
#include "tg_device.cuh"

struct LaunchPlan {
  int nstage = 0;
  int smem = 0;
  int blocks_per_sm = 0;
};

struct tg_config {
  tg::DevCfg dev;
  int device = 0;
  int nsm = 0;
  int V = 0;
  int dtype = 0;
  int mode = 0;
  int max_batch = 0;
  // greedy ids of a small batch over several CTAs per row: one key and one
  // count per row (tg::launch_split_greedy), in dmem, zero between calls
  unsigned long long* split_best = nullptr;
  unsigned* split_tick = nullptr;
  int nwords = 0;
  LaunchPlan sel, ver;
  int proc_smem = 0;
  int state_smem = 0;
  void* dmem = nullptr;
  // the config that selects from scores a task processor compiled by the
  // caller has already produced (include/tg_custom.cuh): f32, the same mode,
  // top_k and top_p, every processor and the temperature off
  tg_config* plain = nullptr;
};

namespace {

tg_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TG_OK;
  if (e == cudaErrorMemoryAllocation) return TG_ERR_OUT_OF_MEMORY;
  return TG_ERR_CUDA;
}

bool ids_in_range(const int32_t* p, int32_t n, int32_t V) {
  if (n < 0 || (n > 0 && !p)) return false;
  for (int32_t i = 0; i < n; ++i)
    if (p[i] < 0 || p[i] >= V) return false;
  return true;
}

std::vector<int> sorted_unique(std::initializer_list<std::pair<const int32_t*, int32_t>> lists) {
  std::vector<int> v;
  for (auto& l : lists)
    for (int32_t i = 0; i < l.second; ++i) v.push_back(l.first[i]);
  std::sort(v.begin(), v.end());
  v.erase(std::unique(v.begin(), v.end()), v.end());
  return v;
}

// The split greedy path: bytes of logits per CTA, and at most this many CTAs per row.
constexpr long long kSplitSliceBytes = 16 * 1024;
constexpr long long kSplitMaxSlices = 32;

// Pick the TMA ring depth.  One CTA per SM (512 threads at 128 registers
// fill the register file); three stages of 32 KB keep a row's stream fed, and
// a deeper ring measured slower (less L1 for the row-end reads, more of the
// next row prefetched while the row end runs); two when three do not fit.
tg_status plan_select(int dtype, bool verify, int nwords, LaunchPlan* out) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return from_cuda(e);
  const int base = tg::select_smem_bytes(0, nwords);
  const int ns = std::min(tg::kRingStages, (optin - base) / tg::kStageBytes);
  if (ns < 2) return TG_ERR_UNSUPPORTED;
  const int smem = tg::select_smem_bytes(ns, nwords);
  int occ = 0;
  e = tg::select_occupancy(dtype, verify, smem, &occ);
  if (e != cudaSuccess) return from_cuda(e);
  if (occ < 1) return TG_ERR_UNSUPPORTED;
  out->nstage = ns;
  out->smem = smem;
  out->blocks_per_sm = 1;
  return TG_OK;
}

tg_status check_device(const tg_config* cfg) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
  return dev == cfg->device ? TG_OK : TG_ERR_INVALID_ARGUMENT;
}

}  // namespace

extern "C" {

void tg_params_init(tg_params* p, int32_t vocab) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->vocab = vocab;
  p->logits_dtype = TG_DTYPE_F32;
  p->mode = TG_GREEDY;
  p->repetition_penalty = 1.0f;
  p->forced_bos_token_id = -1;
  p->temperature = 1.0f;
  p->top_p = 1.0f;
}

namespace {
tg_status config_create(const tg_params* p, tg_config** out, tg_stream stream, bool with_plain);
}

tg_status tg_config_create(const tg_params* p, tg_config** out, tg_stream stream) {
  return config_create(p, out, stream, true);
}

namespace {
tg_status config_create(const tg_params* p, tg_config** out, tg_stream stream, bool with_plain) {
  if (!p || !out) return TG_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  const int32_t V = p->vocab;
  if (V < 1) return TG_ERR_INVALID_ARGUMENT;
  if (V > TG_MAX_VOCAB) return TG_ERR_UNSUPPORTED;
  if (p->logits_dtype != TG_DTYPE_F32 && p->logits_dtype != TG_DTYPE_BF16) return TG_ERR_INVALID_ARGUMENT;
  if (p->mode != TG_GREEDY && p->mode != TG_SAMPLE) return TG_ERR_INVALID_ARGUMENT;
  if (!(p->repetition_penalty > 0.0f) || !std::isfinite(p->repetition_penalty)) return TG_ERR_INVALID_ARGUMENT;
  if (p->no_repeat_ngram_size < 0) return TG_ERR_INVALID_ARGUMENT;
  if (!ids_in_range(p->bad_words_ids, p->n_bad_words_ids, V)) return TG_ERR_INVALID_ARGUMENT;
  if (!ids_in_range(p->suppress_tokens, p->n_suppress_tokens, V)) return TG_ERR_INVALID_ARGUMENT;
  if (!ids_in_range(p->begin_suppress_tokens, p->n_begin_suppress_tokens, V)) return TG_ERR_INVALID_ARGUMENT;
  if (p->n_eos_token_ids > TG_MAX_EOS || !ids_in_range(p->eos_token_ids, p->n_eos_token_ids, V))
    return TG_ERR_INVALID_ARGUMENT;
  if (p->n_forced_eos_token_ids > TG_MAX_EOS ||
      !ids_in_range(p->forced_eos_token_ids, p->n_forced_eos_token_ids, V))
    return TG_ERR_INVALID_ARGUMENT;
  if (p->min_length < 0 || p->min_new_tokens < 0) return TG_ERR_INVALID_ARGUMENT;
  if (p->forced_bos_token_id < -1 || p->forced_bos_token_id >= V) return TG_ERR_INVALID_ARGUMENT;
  if (p->n_forced_eos_token_ids > 0 && p->max_new_tokens < 1) return TG_ERR_INVALID_ARGUMENT;
  if (p->max_new_tokens < 0) return TG_ERR_INVALID_ARGUMENT;
  if (!(p->temperature > 0.0f) || !std::isfinite(p->temperature)) return TG_ERR_INVALID_ARGUMENT;
  if (p->top_k < 0) return TG_ERR_INVALID_ARGUMENT;
  if (!(p->top_p > 0.0f && p->top_p <= 1.0f)) return TG_ERR_INVALID_ARGUMENT;
  if (p->max_batch < 0) return TG_ERR_INVALID_ARGUMENT;
  if (p->n_processors < 0 || p->n_processors > TG_MAX_PROCESSORS) return TG_ERR_INVALID_ARGUMENT;
  if (p->n_processors > 0) {
    if (!p->processor_kinds || !p->processor_sizes) return TG_ERR_INVALID_ARGUMENT;
    long long cols = 0;
    for (int32_t k = 0; k < p->n_processors; ++k) {
      if (p->processor_kinds[k] != TG_PROC_BIAS && p->processor_kinds[k] != TG_PROC_SET) return TG_ERR_INVALID_ARGUMENT;
      if (p->processor_sizes[k] < 1) return TG_ERR_INVALID_ARGUMENT;
      cols += p->processor_sizes[k];
    }
    if (cols > TG_MAX_STATE_COLS) return TG_ERR_INVALID_ARGUMENT;
  }
  if (p->n_bad_word_seqs < 0) return TG_ERR_INVALID_ARGUMENT;
  if (p->n_bad_word_seqs > 0) {
    if (!p->bad_word_seq_offsets || p->bad_word_seq_offsets[0] != 0) return TG_ERR_INVALID_ARGUMENT;
    for (int32_t s = 0; s < p->n_bad_word_seqs; ++s) {
      const int32_t n = p->bad_word_seq_offsets[s + 1] - p->bad_word_seq_offsets[s];
      if (n < 1 || n > TG_MAX_BAD_WORD_LEN) return TG_ERR_INVALID_ARGUMENT;
    }
    if (!ids_in_range(p->bad_word_seq_ids, p->bad_word_seq_offsets[p->n_bad_word_seqs], V))
      return TG_ERR_INVALID_ARGUMENT;
  }

  tg_config* cfg = new (std::nothrow) tg_config();
  if (!cfg) return TG_ERR_OUT_OF_MEMORY;
  tg_status st = TG_OK;
  cudaError_t e = cudaGetDevice(&cfg->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&cfg->nsm, cudaDevAttrMultiProcessorCount, cfg->device);
  if (e != cudaSuccess) { delete cfg; return from_cuda(e); }

  cfg->V = V;
  cfg->dtype = p->logits_dtype;
  cfg->mode = p->mode;
  cfg->max_batch = p->max_batch ? p->max_batch : 4096;
  cfg->nwords = (V + 31) / 32;

  // bad words of one token join the constant ban list; longer ones are kept
  // as words (ids, then offsets)
  std::vector<int> one_tok, seq_ids, seq_off{0};
  for (int32_t s = 0; s < p->n_bad_word_seqs; ++s) {
    const int32_t o0 = p->bad_word_seq_offsets[s], o1 = p->bad_word_seq_offsets[s + 1];
    if (o1 - o0 == 1) {
      one_tok.push_back(p->bad_word_seq_ids[o0]);
    } else {
      for (int32_t i = o0; i < o1; ++i) seq_ids.push_back(p->bad_word_seq_ids[i]);
      seq_off.push_back(static_cast<int>(seq_ids.size()));
    }
  }
  std::vector<int> ban = sorted_unique({{p->bad_words_ids, p->n_bad_words_ids}, {p->suppress_tokens, p->n_suppress_tokens},
                                        {one_tok.data(), static_cast<int32_t>(one_tok.size())}});
  std::vector<int> sup = sorted_unique({{p->suppress_tokens, p->n_suppress_tokens}});
  std::vector<int> bsup = sorted_unique({{p->begin_suppress_tokens, p->n_begin_suppress_tokens}});
  std::vector<int> feos = sorted_unique({{p->forced_eos_token_ids, p->n_forced_eos_token_ids}});

  // one allocation: [ban][sup][bsup][seq ids][seq offsets][tickets][status u32][pad][slow_rows u64]
  // [split keys u64 x max_batch][split counts u32 x max_batch]
  const size_t n_int = ban.size() + sup.size() + bsup.size() + seq_ids.size() + seq_off.size() +
                       static_cast<size_t>(cfg->max_batch) + 2;
  const size_t bytes = ((n_int * 4 + 15) / 16) * 16 + 16 + static_cast<size_t>(cfg->max_batch) * 12;
  e = cudaMalloc(&cfg->dmem, bytes);
  if (e != cudaSuccess) { delete cfg; return from_cuda(e); }
  std::vector<int> host(bytes / 4, 0);
  size_t o = 0;
  auto put = [&](const std::vector<int>& v) { size_t at = o; std::copy(v.begin(), v.end(), host.begin() + o); o += v.size(); return at; };
  size_t o_ban = put(ban), o_sup = put(sup), o_bsup = put(bsup), o_seq = put(seq_ids), o_soff = put(seq_off);
  size_t o_tick = o; o += cfg->max_batch;
  size_t o_status = o; o += 1;
  size_t o_slow = ((o * 4 + 15) / 16) * 16 / 4;
  const size_t o_sbest = o_slow + 2;                                        // 8-byte aligned
  const size_t o_stick = o_sbest + 2 * static_cast<size_t>(cfg->max_batch);
  e = cudaMemcpyAsync(cfg->dmem, host.data(), bytes, cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) { cudaFree(cfg->dmem); delete cfg; return from_cuda(e); }

  int* d = static_cast<int*>(cfg->dmem);
  tg::DevCfg& c = cfg->dev;
  std::memset(&c, 0, sizeof(c));
  c.V = V;
  c.dtype = p->logits_dtype;
  c.mode = p->mode;
  c.rho = p->repetition_penalty;
  c.ngram = p->no_repeat_ngram_size;
  c.ban_sorted = d + o_ban; c.n_ban = static_cast<int>(ban.size());
  c.sup_sorted = d + o_sup; c.n_sup = static_cast<int>(sup.size());
  c.bsup_sorted = d + o_bsup; c.n_bsup = static_cast<int>(bsup.size());
  c.seq_ids = d + o_seq; c.seq_off = d + o_soff; c.n_seq = static_cast<int>(seq_off.size()) - 1;
  c.renorm = p->renormalize_logits ? 1 : 0;
  c.n_eos = p->n_eos_token_ids;
  for (int i = 0; i < c.n_eos; ++i) c.eos[i] = p->eos_token_ids[i];
  c.min_length = p->min_length;
  c.min_new = p->min_new_tokens;
  c.bos = p->forced_bos_token_id;
  c.n_feos = static_cast<int>(feos.size());
  for (int i = 0; i < c.n_feos; ++i) c.feos[i] = feos[i];
  c.max_new = p->max_new_tokens;
  c.temp = p->temperature;
  c.top_k = p->top_k;
  c.top_p = p->top_p;
  c.nproc = p->n_processors;
  c.pcol[0] = 0;
  for (int k = 0; k < c.nproc; ++k) {
    c.pkind[k] = p->processor_kinds[k];
    c.pcol[k + 1] = c.pcol[k] + p->processor_sizes[k];
  }
  c.tickets = reinterpret_cast<unsigned*>(d + o_tick);
  c.status = reinterpret_cast<unsigned*>(d + o_status);
  c.slow_rows = reinterpret_cast<unsigned long long*>(d + o_slow);
  cfg->split_best = reinterpret_cast<unsigned long long*>(d + o_sbest);
  cfg->split_tick = reinterpret_cast<unsigned*>(d + o_stick);

  st = plan_select(c.dtype, false, cfg->nwords, &cfg->sel);
  if (st == TG_OK) st = plan_select(c.dtype, true, 0, &cfg->ver);
  cfg->proc_smem = tg::process_smem_bytes(cfg->nwords, c.pcol[c.nproc]);
  cfg->state_smem = tg::state_smem_bytes(cfg->nwords, c.pcol[c.nproc]);
  if (st == TG_OK && c.nproc > 0) {
    // the state kernels stage the state in shared memory: it must fit
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, cfg->device);
    if (e != cudaSuccess) st = from_cuda(e);
    else if (cfg->state_smem > optin || cfg->proc_smem > optin) st = TG_ERR_UNSUPPORTED;
  }
  if (st == TG_OK && with_plain) {
    tg_params q;
    tg_params_init(&q, V);
    q.mode = p->mode;
    q.top_k = p->top_k;
    q.top_p = p->top_p;
    q.max_batch = p->max_batch;
    st = config_create(&q, &cfg->plain, stream, false);
    if (st == TG_OK) {
      // its launches report in this config's status word and slow-row count
      cfg->plain->dev.status = cfg->dev.status;
      cfg->plain->dev.slow_rows = cfg->dev.slow_rows;
    }
  }
  if (st != TG_OK) {
    cudaFree(cfg->dmem);
    delete cfg;
    return st;
  }
  *out = cfg;
  return TG_OK;
}
}  // namespace

tg_status tg_config_destroy(tg_config* cfg) {
  if (!cfg) return TG_ERR_INVALID_ARGUMENT;
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t e2 = cudaFree(cfg->dmem);
  if (cfg->plain) {
    const tg_status s2 = tg_config_destroy(cfg->plain);
    if (e2 == cudaSuccess && s2 != TG_OK) e2 = cudaErrorUnknown;
  }
  delete cfg;
  return from_cuda(e != cudaSuccess ? e : e2);
}

tg_status tg_config_view(const tg_config* cfg, void* out, size_t size) {
  if (!cfg || !out || size != sizeof(tg::DevCfg)) return TG_ERR_INVALID_ARGUMENT;
  std::memcpy(out, &cfg->dev, sizeof(tg::DevCfg));
  return TG_OK;
}

const tg_config* tg_config_selection(const tg_config* cfg) { return cfg ? cfg->plain : nullptr; }

namespace {
// Greedy ids of a batch too small to fill the GPU: each of the rows over
// several CTAs of about kSplitSliceBytes, when every CTA fits in one wave.
bool split_plan(const tg_config* cfg, long long rows, int* nslice, int* slice_tok) {
  if (cfg->mode != TG_GREEDY || rows < 1 || rows > cfg->max_batch) return false;
  const long long rb = static_cast<long long>(cfg->V) * (cfg->dtype == TG_DTYPE_BF16 ? 2 : 4);
  const long long ns = std::min<long long>(kSplitMaxSlices, (rb + kSplitSliceBytes - 1) / kSplitSliceBytes);
  if (ns < 2 || rows * ns > cfg->nsm) return false;
  *slice_tok = static_cast<int>((cfg->V + ns - 1) / ns + 7) / 8 * 8;
  *nslice = (cfg->V + *slice_tok - 1) / *slice_tok;
  return true;
}

tg_status select_impl(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                      const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                      const float* uniforms, int32_t* out_ids, float* out_logprobs, tg_stream stream) {
  if (!cfg || B < 0 || V != cfg->V || cfg->dev.nproc > 0) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (!logits || !hist_offsets || !prompt_lens || !out_ids) return TG_ERR_INVALID_ARGUMENT;
  if (cfg->mode == TG_SAMPLE && !uniforms) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  // Log-probabilities come from the sampling kernel, which sums the row's
  // mass: a greedy config runs it with the warpers off and u = 0.
  tg::DevCfg dev = cfg->dev;
  if (out_logprobs && cfg->mode == TG_GREEDY) {
    dev.mode = tg::kSample;
    dev.temp = 1.0f;
    dev.top_k = 0;
    dev.top_p = 1.0f;
    uniforms = nullptr;
  }
  tg::SelArgs a{};
  a.logprobs = out_logprobs;
  a.logits = logits;
  a.nrows = B;
  a.nrows_total = B;
  a.V = V;
  a.hist = hist_ids;
  a.off = hist_offsets;
  a.plen = prompt_lens;
  a.uniforms = uniforms;
  a.out = out_ids;
  a.nstage = cfg->sel.nstage;
  a.nwords = cfg->nwords;
  int nslice = 0, slice_tok = 0;
  if (!out_logprobs && split_plan(cfg, B, &nslice, &slice_tok))
    return from_cuda(tg::launch_split_greedy(dev, a, nslice, slice_tok, cfg->split_best, cfg->split_tick, false,
                                             reinterpret_cast<cudaStream_t>(stream)));
  int grid = std::min<long long>(B, static_cast<long long>(cfg->sel.blocks_per_sm) * cfg->nsm);
  return from_cuda(tg::launch_select(dev, a, false, grid, cfg->sel.smem, reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

tg_status tg_select(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                    const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                    const float* uniforms, int32_t* out_ids, tg_stream stream) {
  return select_impl(logits, B, V, hist_ids, hist_offsets, prompt_lens, cfg, uniforms, out_ids, nullptr, stream);
}

tg_status tg_select_logprobs(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                             const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                             const float* uniforms, int32_t* out_ids, float* out_logprobs, tg_stream stream) {
  if (!out_logprobs && B > 0) return TG_ERR_INVALID_ARGUMENT;
  return select_impl(logits, B, V, hist_ids, hist_offsets, prompt_lens, cfg, uniforms, out_ids, out_logprobs,
                     stream);
}

tg_status tg_verify(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids, int32_t K,
                    const tg_config* cfg, const float* uniforms, int32_t* out_match, int32_t* out_next,
                    tg_stream stream) {
  if (!cfg || B < 0 || V != cfg->V || K < 1 || cfg->dev.nproc > 0) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (B > cfg->max_batch) return TG_ERR_INVALID_ARGUMENT;
  if (!target_logits || !cand_ids || !out_match || !out_next) return TG_ERR_INVALID_ARGUMENT;
  if (cfg->mode == TG_SAMPLE && !uniforms) return TG_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(B) * (K + 1) > 0x7fffffffLL) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  tg::SelArgs a{};
  a.logits = target_logits;
  a.nrows = B * (K + 1);
  a.nrows_total = a.nrows;
  a.V = V;
  a.uniforms = uniforms;
  a.out = out_next;
  a.cand = cand_ids;
  a.K = K;
  a.out_match = out_match;
  a.nstage = cfg->ver.nstage;
  a.nwords = 0;
  // this call's counts of finished positions start at zero
  cudaError_t e = cudaMemsetAsync(cfg->dev.tickets, 0, static_cast<size_t>(B) * sizeof(unsigned),
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  int nslice = 0, slice_tok = 0;
  if (split_plan(cfg, a.nrows, &nslice, &slice_tok))
    return from_cuda(tg::launch_split_greedy(cfg->dev, a, nslice, slice_tok, cfg->split_best, cfg->split_tick, true,
                                             reinterpret_cast<cudaStream_t>(stream)));
  int grid = std::min<long long>(a.nrows, static_cast<long long>(cfg->ver.blocks_per_sm) * cfg->nsm);
  return from_cuda(tg::launch_select(cfg->dev, a, true, grid, cfg->ver.smem, reinterpret_cast<cudaStream_t>(stream)));
}

tg_status tg_verify_history(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids, int32_t K,
                            const int32_t* hist_ids, const int64_t* hist_offsets, const int32_t* prompt_lens,
                            const tg_config* cfg, const float* uniforms, int32_t* out_match, int32_t* out_next,
                            tg_stream stream) {
  if (!cfg || B < 0 || V != cfg->V || K < 1 || cfg->dev.nproc > 0) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (B > cfg->max_batch) return TG_ERR_INVALID_ARGUMENT;
  if (!target_logits || !cand_ids || !out_match || !out_next || !hist_offsets || !prompt_lens)
    return TG_ERR_INVALID_ARGUMENT;
  if (cfg->mode == TG_SAMPLE && !uniforms) return TG_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(B) * (K + 1) > 0x7fffffffLL) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  tg::SelArgs a{};
  a.logits = target_logits;
  a.nrows = B * (K + 1);
  a.nrows_total = a.nrows;
  a.V = V;
  a.hist = hist_ids;
  a.off = hist_offsets;
  a.plen = prompt_lens;
  a.uniforms = uniforms;
  a.out = out_next;
  a.cand = cand_ids;
  a.K = K;
  a.out_match = out_match;
  a.vhist = 1;
  // the row bitmaps need the select kernel's shared-memory plan
  a.nstage = cfg->sel.nstage;
  a.nwords = cfg->nwords;
  // this call's counts of finished positions start at zero
  cudaError_t e = cudaMemsetAsync(cfg->dev.tickets, 0, static_cast<size_t>(B) * sizeof(unsigned),
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  int grid = std::min<long long>(a.nrows, static_cast<long long>(cfg->sel.blocks_per_sm) * cfg->nsm);
  return from_cuda(tg::launch_select(cfg->dev, a, true, grid, cfg->sel.smem, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
tg_status process_impl(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                       const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                       const int32_t* state_ids, const float* state_values, float* out_scores,
                       uint32_t* out_banbits, float* out_probs, tg_stream stream) {
  if (!cfg || B < 0 || V != cfg->V) return TG_ERR_INVALID_ARGUMENT;
  if ((cfg->dev.nproc > 0) != (state_ids != nullptr)) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (!logits || !hist_offsets || !prompt_lens || !out_scores) return TG_ERR_INVALID_ARGUMENT;
  if (state_ids && !state_values) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  tg::SelArgs a{};
  a.logits = logits;
  a.nrows = B;
  a.nrows_total = B;
  a.V = V;
  a.hist = hist_ids;
  a.off = hist_offsets;
  a.plen = prompt_lens;
  a.nwords = cfg->nwords;
  return from_cuda(tg::launch_process(cfg->dev, a, out_scores, out_banbits, out_probs, cfg->proc_smem,
                                      reinterpret_cast<cudaStream_t>(stream), state_ids, state_values));
}
}  // namespace

tg_status tg_process(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                     const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                     float* out_scores, uint32_t* out_banbits, float* out_probs, tg_stream stream) {
  return process_impl(logits, B, V, hist_ids, hist_offsets, prompt_lens, cfg, nullptr, nullptr, out_scores,
                      out_banbits, out_probs, stream);
}

tg_status tg_process_state(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                           const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                           const int32_t* state_ids, const float* state_values, float* out_scores,
                           uint32_t* out_banbits, float* out_probs, tg_stream stream) {
  if (!state_ids || !state_values) return TG_ERR_INVALID_ARGUMENT;
  return process_impl(logits, B, V, hist_ids, hist_offsets, prompt_lens, cfg, state_ids, state_values, out_scores,
                      out_banbits, out_probs, stream);
}

tg_status tg_select_state(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                          const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                          const int32_t* state_ids, const float* state_values, const float* uniforms,
                          int32_t* out_ids, float* out_logprobs, tg_stream stream) {
  if (!cfg || B < 0 || V != cfg->V || cfg->dev.nproc < 1) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (!logits || !hist_offsets || !prompt_lens || !out_ids || !state_ids || !state_values)
    return TG_ERR_INVALID_ARGUMENT;
  if (cfg->mode == TG_SAMPLE && !uniforms) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  // log-probabilities of a greedy config: the sampling kernel with the
  // warpers off and u = 0 (its first token is the argmax, lowest index)
  tg::DevCfg dev = cfg->dev;
  if (out_logprobs && cfg->mode == TG_GREEDY) {
    dev.mode = tg::kSample;
    dev.temp = 1.0f;
    dev.top_k = 0;
    dev.top_p = 1.0f;
    uniforms = nullptr;
  }
  tg::SelArgs a{};
  a.logprobs = out_logprobs;
  a.logits = logits;
  a.nrows = B;
  a.nrows_total = B;
  a.V = V;
  a.hist = hist_ids;
  a.off = hist_offsets;
  a.plen = prompt_lens;
  a.uniforms = uniforms;
  a.out = out_ids;
  a.nwords = cfg->nwords;
  a.st_ids = state_ids;
  a.st_vals = state_values;
  // select_kernel finishes the rows its one-pass path can (the state ids are
  // marked tokens there) and leaves the rest to state_kernel
  a.nstage = cfg->sel.nstage;
  const int grid_sel = static_cast<int>(std::min<long long>(B, static_cast<long long>(cfg->sel.blocks_per_sm) * cfg->nsm));
  cudaError_t e = tg::launch_select(dev, a, false, grid_sel, cfg->sel.smem, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  a.fixup = 1;
  const int grid = static_cast<int>(std::min<long long>(B, cfg->nsm));
  return from_cuda(tg::launch_state(dev, a, grid, cfg->state_smem, reinterpret_cast<cudaStream_t>(stream),
                                    state_ids, state_values));
}

tg_status tg_query_status(const tg_config* cfg, uint32_t* flags, uint64_t* slow_rows) {
  if (!cfg) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  unsigned f = 0;
  unsigned long long s = 0;
  cudaError_t e = cudaMemcpy(&f, cfg->dev.status, sizeof(f), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&s, cfg->dev.slow_rows, sizeof(s), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  if (flags) *flags = f;
  if (slow_rows) *slow_rows = s;
  return TG_OK;
}

tg_status tg_status_word(const tg_config* cfg, uint32_t* flags) {
  if (!flags) return TG_ERR_INVALID_ARGUMENT;
  return tg_query_status(cfg, flags, nullptr);
}

tg_status tg_clear_status(const tg_config* cfg) {
  if (!cfg) return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  cudaError_t e = cudaMemset(cfg->dev.status, 0, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(cfg->dev.slow_rows, 0, sizeof(unsigned long long));
  // tickets a launch left behind (one whose bounded wait ran out) start at zero again
  if (e == cudaSuccess) e = cudaMemset(cfg->dev.tickets, 0, static_cast<size_t>(cfg->max_batch) * sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(cfg->split_best, 0, static_cast<size_t>(cfg->max_batch) * 12);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return from_cuda(e);
}

int32_t tg_beam_keep(const tg_config* cfg, int32_t num_beams) {
  if (!cfg || num_beams < 1) return -1;
  const int per = std::max(2, 1 + cfg->dev.n_eos);
  return per * num_beams;
}

tg_status tg_beam_step(const void* logits, int32_t num_prompts, int32_t num_beams, int32_t V,
                       const float* beam_scores, const int32_t* hist_ids, const int64_t* hist_offsets,
                       const int32_t* prompt_lens, const tg_config* cfg, float* out_scores,
                       int32_t* out_tokens, int32_t* out_beams, tg_stream stream) {
  if (!cfg || num_prompts < 0 || num_beams < 1 || V != cfg->V || cfg->dev.nproc > 0) return TG_ERR_INVALID_ARGUMENT;
  if (num_beams > tg::kMaxClusterBeams) return TG_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(num_prompts) * num_beams;
  if (rows > 0x7fffffffLL) return TG_ERR_INVALID_ARGUMENT;
  if (rows == 0) return TG_OK;
  if (!logits || !beam_scores || !hist_offsets || !prompt_lens || !out_scores || !out_tokens || !out_beams)
    return TG_ERR_INVALID_ARGUMENT;
  tg_status st = check_device(cfg);
  if (st != TG_OK) return st;
  tg::BeamArgs a{};
  a.logits = logits;
  a.nrows = static_cast<int>(rows);
  a.nb = num_beams;
  a.V = V;
  a.keep = tg_beam_keep(cfg, num_beams);
  a.beam_scores = beam_scores;
  a.hist = hist_ids;
  a.off = hist_offsets;
  a.plen = prompt_lens;
  a.out_scores = out_scores;
  a.out_tokens = out_tokens;
  a.out_beams = out_beams;
  a.nwords = cfg->nwords;
  return from_cuda(tg::launch_beam(cfg->dev, a, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t tg_next_num_candidates(int32_t K, int32_t n_match, int32_t K_max) {
  int32_t K2 = n_match >= K ? K + 2 : K - 1;
  if (K_max < 1) K_max = 1;
  return K2 < 1 ? 1 : (K2 > K_max ? K_max : K2);
}

const char* tg_status_string(tg_status s) {
  switch (s) {
    case TG_OK: return "TG_OK";
    case TG_ERR_INVALID_ARGUMENT: return "TG_ERR_INVALID_ARGUMENT";
    case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
    case TG_ERR_CUDA: return "TG_ERR_CUDA";
    case TG_ERR_OUT_OF_MEMORY: return "TG_ERR_OUT_OF_MEMORY";
  }
  return "TG_UNKNOWN_STATUS";
}

}  // extern "C"
