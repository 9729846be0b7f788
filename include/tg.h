/*
 * tg.h -- C ABI of the GB300 token-selection library (libtg.so).
 *
 * One decode step of autoregressive generation ends with token selection:
 * the logits processors of transformers run over each row's scores in a fixed
 * order, then greedy argmax or a multinomial draw picks the row's next token.
 * The order and the length rules follow "Transmuter.Generation (transmuter
 * v2.0.0)": module intro (processor order), section "Lengths" (how a row's
 * length counts prompt and new tokens, and when min_length, min_new_tokens,
 * forced bos/eos and begin_suppress_tokens apply), section "Log-probabilities"
 * (f32 scores, the smallest finite f32 as the filter value) and section
 * "Batches" (ragged rows, empty rows give no token).  The verify step follows
 * "Assisted Generation: a new direction toward low-latency text generation",
 * section "Greedy decoding with assisted generation", steps 2-6.
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA device (or managed) memory of the device that
 *    was current when the config was created; that device must be current at
 *    every call.  The caller owns them; the library never frees or keeps
 *    them past the call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and the call returns without waiting.  Results are ready when the
 *    stream reaches that point.
 *  - Argument errors are found on the host and returned before anything is
 *    enqueued.  A failed launch returns TG_ERR_CUDA.  Bad values that only
 *    the device sees (history ids outside [0, V), inconsistent offsets) never
 *    fault: the kernel skips them and raises a bit in the config's status
 *    word (tg_query_status).
 *  - Calls that share a tg_config use its small device workspace (verify
 *    tickets, the per-row keys and counts of split greedy rows, status
 *    word); issue them in stream order (one stream, or events between
 *    streams).  Use one config per concurrent stream.
 *  - Scores: the filter value F is -FLT_MAX; no score goes below it.
 */
#ifndef TG_H_
#define TG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is a struct CUstream_st* */
typedef struct CUstream_st* tg_stream;

typedef enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARGUMENT = -1,
  TG_ERR_UNSUPPORTED = -2,
  TG_ERR_CUDA = -3,
  TG_ERR_OUT_OF_MEMORY = -4
} tg_status;

typedef enum { TG_DTYPE_F32 = 0, TG_DTYPE_BF16 = 1 } tg_dtype;
typedef enum { TG_GREEDY = 0, TG_SAMPLE = 1 } tg_mode;

/* Status-word bits (sticky until tg_clear_status). */
#define TG_FLAG_HISTORY_ID_OUT_OF_RANGE 0x1u /* a history id was < 0 or >= V; skipped */
#define TG_FLAG_BAD_ROW 0x2u                 /* offsets/prompt length inconsistent; row gave -1 */
#define TG_FLAG_SLOW_PATH 0x4u               /* a row needed the multi-pass exact path */
/* A bounded wait on a bulk copy ran out (about 1 s): the launch stopped
 * loading logits.  The rows it had not finished give -1 in out_ids /
 * out_next (log-probability NaN); in verify, their batch rows give
 * out_match = -1.  Every other output of the call is valid. */
#define TG_FLAG_TIMEOUT 0x8u
#define TG_FLAG_BAD_STATE 0x10u              /* a row's processor state broke its layout; dropped */

/* Largest vocabulary the kernels take. */
#define TG_MAX_VOCAB (1 << 18)
/* Longest list accepted for eos ids and forced eos ids. */
#define TG_MAX_BAD_WORD_LEN 16
#define TG_MAX_EOS 8
/* The task's processors: at most this many, owning at most this many state
 * columns in all. */
#define TG_MAX_PROCESSORS 8
#define TG_MAX_STATE_COLS 4096

/* Kinds of the task's processors (tg_params.processor_kinds). */
typedef enum {
  TG_PROC_BIAS = 0, /* s + v for each (id, v) of the row's state */
  TG_PROC_SET = 1   /* v for each (id, v) of the row's state */
} tg_proc_kind;

/*
 * Generation settings, named after transformers' generation_config fields.
 * Host pointers; tg_config_create copies what it needs.  tg_params_init
 * fills the "off" defaults.
 */
typedef struct tg_params {
  int32_t vocab;                /* V, 1 .. TG_MAX_VOCAB */
  tg_dtype logits_dtype;        /* element type of the logits rows */
  tg_mode mode;                 /* greedy argmax or multinomial draw */
  float repetition_penalty;     /* > 0; 1 = off */
  int32_t no_repeat_ngram_size; /* >= 0; 0 = off */
  const int32_t* bad_words_ids; /* single-token bad words, each in [0, V) */
  int32_t n_bad_words_ids;
  const int32_t* suppress_tokens; /* each in [0, V) */
  int32_t n_suppress_tokens;
  const int32_t* begin_suppress_tokens; /* each in [0, V) */
  int32_t n_begin_suppress_tokens;
  const int32_t* eos_token_ids; /* removed while min_length/min_new_tokens hold */
  int32_t n_eos_token_ids;      /* 0 .. TG_MAX_EOS */
  int32_t min_length;           /* >= 0; 0 = off */
  int32_t min_new_tokens;       /* >= 0; 0 = off; when > 0 it replaces min_length */
  int32_t forced_bos_token_id;  /* -1 = off, else in [0, V) */
  const int32_t* forced_eos_token_ids; /* forced at L == prompt + max_new_tokens - 1 */
  int32_t n_forced_eos_token_ids;      /* 0 = off .. TG_MAX_EOS */
  int32_t max_new_tokens;       /* > 0 when forced eos ids are given */
  float temperature;            /* > 0; 1 = off (sampling only) */
  int32_t top_k;                /* >= 0; 0 = off (sampling only) */
  float top_p;                  /* (0, 1]; 1 = off (sampling only) */
  int32_t max_batch;            /* largest B a tg_verify call may pass; 0 = 4096 */
  /* Bad words of one or more tokens, back to back: word i is
   * bad_word_seq_ids[bad_word_seq_offsets[i] .. bad_word_seq_offsets[i+1]),
   * n_bad_word_seqs + 1 offsets (0 first, non-decreasing), ids in [0, V), each
   * word at most TG_MAX_BAD_WORD_LEN ids.  A one-token word is always banned;
   * a longer one bans its last token when the row ends with the rest of it. */
  const int32_t* bad_word_seq_ids;
  const int32_t* bad_word_seq_offsets;
  int32_t n_bad_word_seqs;
  /* 0/1: renormalize_logits, a log-softmax of the scores after the processors
   * and before temperature.  Selection does not change under it (a per-row
   * shift); tg_process and tg_beam_step apply it. */
  int32_t renormalize_logits;
  /* The task's processors (Transmuter.Generation, section "Processors": a
   * per-row state made before the step, and a function of the row's scores
   * and that state; they run after begin_suppress_tokens and before
   * renormalize_logits and temperature, in list order).  Processor k has
   * kind processor_kinds[k] (tg_proc_kind) and owns processor_sizes[k] >= 1
   * consecutive columns of the state; S = the sum of the sizes.  A config
   * with processors is used through tg_select_state and tg_process_state
   * only; the other entry points that take a config refuse it. */
  const int32_t* processor_kinds;
  const int32_t* processor_sizes;
  int32_t n_processors; /* 0 .. TG_MAX_PROCESSORS; S <= TG_MAX_STATE_COLS */
} tg_params;

/* Opaque, immutable after creation; holds the constant masks on the device. */
typedef struct tg_config tg_config;

/* Fill *p with the defaults: every processor off, greedy, f32. */
void tg_params_init(tg_params* p, int32_t vocab);

/*
 * Validate *params and build a config on the current device: sorted
 * constant ban lists (bad words and suppress tokens), begin-suppress list,
 * status word and verify tickets.  The uploads are enqueued on `stream`
 * (NULL: the default stream) and the call waits for that stream before it
 * returns, so the config is ready for any later call.  Errors:
 * TG_ERR_INVALID_ARGUMENT (a field out of range), TG_ERR_UNSUPPORTED
 * (V > TG_MAX_VOCAB), TG_ERR_OUT_OF_MEMORY, TG_ERR_CUDA.
 */
tg_status tg_config_create(const tg_params* params, tg_config** out, tg_stream stream);

/* Free the config's device memory (synchronises the device first). */
tg_status tg_config_destroy(tg_config* cfg);

/*
 * For include/tg_custom.cuh (a task processor compiled by the caller):
 * tg_config_view copies the config's device settings (a tg::DevCfg of
 * `size` bytes: TG_ERR_INVALID_ARGUMENT when the size differs) to *out;
 * tg_config_selection returns the config, owned by cfg, that selects from
 * scores that already went through every processor and the temperature:
 * f32 rows, cfg's mode, top_k and top_p, nothing else.  Its launches report
 * in cfg's status word.
 */
tg_status tg_config_view(const tg_config* cfg, void* out, size_t size);
const tg_config* tg_config_selection(const tg_config* cfg);

/*
 * tg_select -- process and select one token per row.
 *
 *  logits        device, [B, V] row-major, cfg's dtype (f32 or bf16), rows
 *                V elements apart.  16-byte aligned rows take the bulk-copy
 *                path; other layouts work at lower speed.
 *  B, V          batch rows (>= 0) and vocabulary (must equal cfg's vocab).
 *  hist_ids      device int32, every row's history back to back: prompt
 *                then new tokens (unpadded; may be NULL when all rows are
 *                empty).
 *  hist_offsets  device int64 [B+1]; row b's history is
 *                hist_ids[hist_offsets[b] .. hist_offsets[b+1]); its length
 *                L is the row length the processors count.
 *  prompt_lens   device int32 [B]; P for each row, 0 <= P <= L.
 *  cfg           from tg_config_create.
 *  uniforms      device f32 [B], each in [0, 1): the draw of row b.  May be
 *                NULL in greedy mode.
 *  out_ids       device int32 [B]; the selected id, or -1 for an empty row.
 *
 * Steps per row (processor order of the Transmuter.Generation module intro):
 * repetition_penalty, no_repeat_ngram_size, bad words, min_length /
 * min_new_tokens, forced bos, forced eos, suppress_tokens,
 * begin_suppress_tokens; then greedy argmax (lowest index among equal
 * maxima), or temperature, top_k, top_p and an inverse-CDF draw with
 * uniforms[b] over the kept tokens ordered by (score desc, index asc).
 * A greedy batch small enough that its rows, cut into slices of about 16 KB
 * of logits, fit one wave of CTAs is read with each row split over several
 * CTAs (same ids; B <= max_batch); plain greedy tg_verify likewise.
 */
tg_status tg_select(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                    const int64_t* hist_offsets, const int32_t* prompt_lens,
                    const tg_config* cfg, const float* uniforms, int32_t* out_ids,
                    tg_stream stream);

/*
 * tg_select_logprobs -- tg_select, plus the log-probability of each row's
 * token (Transmuter.Generation, section "Log-probabilities"): the
 * log-softmax, at the token, of the scores the step selects from.  For
 * greedy rows those are the processed scores; for sampled rows the
 * processed scores after temperature, with every token outside the kept
 * top_k / top_p set removed.
 *
 *  out_logprobs  device f32 [B]; NaN for an empty row.  Computed from the
 *                token's score and the kept set's 44-bit fixed-point mass
 *                (about 1e-7 relative); out_ids as tg_select gives them.
 *
 * Other arguments, layouts and errors as tg_select; out_logprobs must not be
 * NULL.  A greedy config runs the sampling kernel with temperature, top_k
 * and top_p off and u = 0 (the first token of the (score desc, index asc)
 * order is the argmax with the lowest index), so the row's mass is summed.
 */
tg_status tg_select_logprobs(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                             const int64_t* hist_offsets, const int32_t* prompt_lens,
                             const tg_config* cfg, const float* uniforms, int32_t* out_ids,
                             float* out_logprobs, tg_stream stream);

/*
 * tg_verify -- assisted-generation verification (Assisted Generation,
 * "Greedy decoding with assisted generation", steps 3-5).
 *
 *  target_logits device, [B, K+1, V] row-major in cfg's dtype: the target
 *                model's logits after the prefix and after each candidate.
 *  cand_ids      device int32 [B, K]: the assistant's candidates.
 *  K             candidates per row, >= 1.
 *  uniforms      device f32 [B, K+1] for sampling mode (NULL for greedy).
 *  out_match     device int32 [B]: n_b, the number of leading candidates
 *                equal to the target's selection.
 *  out_next      device int32 [B, K+1]: the target's tokens 0..n_b (the
 *                matches and the first divergent, or bonus, token); -1 after.
 *
 * Position j selects with cfg's mode and warpers (temperature, top_k,
 * top_p); history processors do not run per position.  B <= cfg's max_batch.
 * A batch row whose positions a timed-out launch left unfinished gives
 * out_match = -1 (TG_FLAG_TIMEOUT).  Calls on one config share its per-row
 * counts of finished positions (cleared on `stream` at the start of each
 * call): run them in stream order.
 */
tg_status tg_verify(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids,
                    int32_t K, const tg_config* cfg, const float* uniforms, int32_t* out_match,
                    int32_t* out_next, tg_stream stream);

/*
 * tg_process -- diagnostic, not tuned: the scores tg_select computes.
 * Same inputs as tg_select, plus:
 *  out_scores   device f32 [B, V]: scores after the processors (and after
 *               temperature in sampling mode); rows with L == 0 untouched.
 *  out_banbits  device uint32 [B, ceil(V/32)], or NULL: bit i of row b is set
 *               when a ban or force processor set token i to the filter value.
 *  out_probs    device f32 [B, V], or NULL: the distribution the draw uses
 *               (after top_k/top_p, renormalised; 0 outside the kept set);
 *               in greedy mode the softmax of out_scores.
 */
tg_status tg_process(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                     const int64_t* hist_offsets, const int32_t* prompt_lens,
                     const tg_config* cfg, float* out_scores, uint32_t* out_banbits,
                     float* out_probs, tg_stream stream);

/*
 * tg_set_wait_limit -- testing.  The select and verify kernels give up a
 * wait on a bulk copy of logits after about one second (TG_FLAG_TIMEOUT);
 * this sets that limit to `cycles` SM cycles on the current device, for the
 * launches that follow (0 restores the default).  The wait for copies still
 * in flight after such an error keeps the full limit, so no copy outlives
 * its CTA.  Not for use while other calls run.  Errors: TG_ERR_CUDA.
 */
tg_status tg_set_wait_limit(uint64_t cycles);

/* Largest B that tg_verify_noalloc takes. */
#define TG_NOALLOC_MAX_BATCH 1024

/*
 * tg_verify_noalloc -- tg_verify for callers that cannot allocate device
 * memory.  (An addition of this library; the pages have no counterpart.)
 *
 * Some callers may not call cudaMalloc: a serving engine that gives all of
 * HBM to its KV-cache pool at start-up and forbids later allocations, or a
 * pipelined decode step where an allocation would synchronise the device.
 * They cannot create a tg_config either, so this entry point takes the
 * settings in *params by value (only vocab, logits_dtype, mode, temperature,
 * top_k and top_p are read; as in tg_verify, no history processor runs) and
 * keeps its per-row tickets in a fixed array in the library's own device
 * memory (TG_NOALLOC_MAX_BATCH + 4 words per device, held until the process
 * exits).  A call allocates nothing.
 *
 * Arguments, layouts and outputs are those of tg_verify.  Errors:
 * TG_ERR_UNSUPPORTED when B > TG_NOALLOC_MAX_BATCH or V > TG_MAX_VOCAB;
 * TG_ERR_INVALID_ARGUMENT for a bad setting or pointer; TG_ERR_CUDA when the
 * set-up or the launch fails.  Device-side status bits of this entry point
 * are not reported; a batch row that a timed-out launch left unfinished
 * gives out_match = -1 (and -1 in its unfinished out_next entries).
 *
 * The first call on a device does a one-time synchronous set-up on the
 * current device (it resolves the array's address and zeroes it); make that
 * first call before any stream capture.  Each call clears the tickets it
 * uses on `stream`.  All calls on a device share the one array: calls that
 * overlap on the GPU (different streams without ordering) race on it.
 */
tg_status tg_verify_noalloc(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids,
                            int32_t K, const tg_params* params, const float* uniforms, int32_t* out_match,
                            int32_t* out_next, tg_stream stream);

/*
 * tg_verify_history -- tg_verify with the whole processor chain at every
 * position: position j of row b sees the row's history (hist_ids,
 * hist_offsets, prompt_lens as tg_select, B rows) followed by its first j
 * candidates, as the target model did (Assisted Generation, "Greedy decoding
 * with assisted generation", step 2).  The length rules count that extended
 * history.  A row with an empty history is a padding row (out_next -1,
 * out_match 0).  The extended history must fit 8,192 ids: a longer one makes
 * the position a bad row (-1, status bit).  Other arguments and errors as
 * tg_verify.
 */
tg_status tg_verify_history(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids, int32_t K,
                            const int32_t* hist_ids, const int64_t* hist_offsets, const int32_t* prompt_lens,
                            const tg_config* cfg, const float* uniforms, int32_t* out_match, int32_t* out_next,
                            tg_stream stream);

/*
 * tg_select_state -- tg_select (or tg_select_logprobs) with the task's
 * processors of cfg (Transmuter.Generation, section "Processors").
 *
 *  state_ids     device int32 [B, S]: row b's state is state_ids[b*S ..
 *                b*S + S); processor k reads its own columns.  Within a
 *                processor's columns the ids in use come first, strictly
 *                ascending, each in [0, V), and the unused columns hold -1.
 *  state_values  device f32 [B, S]: the value of each (id) entry.  A "bias"
 *                entry (t, v) makes s[t] + v (an f32 add), a "set" entry
 *                makes v; either never goes below the filter value.
 *  out_logprobs  device f32 [B] or NULL: as tg_select_logprobs.
 *
 * The processors run on the scores after the processors of tg_select (also
 * on a forced row, whose other tokens hold the filter value) and before
 * temperature, top_k, top_p and the draw.  A row whose state breaks its
 * layout runs without the processors and raises TG_FLAG_BAD_STATE.  The
 * state ids join the one-pass path of tg_select as marked tokens; a row that
 * path cannot finish goes to a second kernel in the same stream (multi-pass,
 * counted in the slow-row count).  out_ids may hold -2 between the two
 * kernels, never after the call's work completes.  Other arguments, layouts
 * and errors as tg_select; a cfg without processors, or a NULL state
 * pointer, is TG_ERR_INVALID_ARGUMENT.
 */
tg_status tg_select_state(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                          const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                          const int32_t* state_ids, const float* state_values, const float* uniforms,
                          int32_t* out_ids, float* out_logprobs, tg_stream stream);

/*
 * tg_process_state -- tg_process with the task's processors: the scores
 * tg_select_state selects from (diagnostic, not tuned).  state_ids and
 * state_values as tg_select_state; out_banbits marks what the processors of
 * tg_select set to the filter value (the task's processors do not change
 * it).  Other arguments as tg_process.
 */
tg_status tg_process_state(const void* logits, int32_t B, int32_t V, const int32_t* hist_ids,
                           const int64_t* hist_offsets, const int32_t* prompt_lens, const tg_config* cfg,
                           const int32_t* state_ids, const float* state_values, float* out_scores,
                           uint32_t* out_banbits, float* out_probs, tg_stream stream);

/* Read (synchronously) the sticky status bits and the count of rows that took
 * the multi-pass exact path since the last clear. */
tg_status tg_query_status(const tg_config* cfg, uint32_t* flags, uint64_t* slow_rows);
tg_status tg_clear_status(const tg_config* cfg);
/* The status bits alone (synchronously): tg_query_status without the count. */
tg_status tg_status_word(const tg_config* cfg, uint32_t* flags);

/* Assisted Generation, step 6: the next candidate count.  K + 2 when
 * n_match == K (all candidates matched), else K - 1; bounded to [1, K_max]. */
int32_t tg_next_num_candidates(int32_t K, int32_t n_match, int32_t K_max);

/*
 * tg_beam_step -- the device part of one beam-search step
 * (Transmuter.Generation, module intro, the paragraphs on num_beams; the
 * host's part -- finished hypotheses, length penalty, stopping -- is the
 * caller's).
 *
 *  logits        device, [num_prompts * num_beams, V], cfg's dtype; prompt i
 *                owns rows i*num_beams .. i*num_beams + num_beams - 1.
 *  num_beams     1 .. 8 (one thread-block cluster per prompt).
 *  beam_scores   device f32 [num_prompts * num_beams]: each beam's running
 *                score (at the first step 0 for beam 0 and a very negative
 *                value for the others, so that only the first beam counts).
 *  hist_ids, hist_offsets, prompt_lens   each beam row's history, as tg_select.
 *  out_scores    device f32 [num_prompts, keep]; out_tokens, out_beams
 *                device int32 [num_prompts, keep]; keep = tg_beam_keep().
 *
 * Per row: the log-softmax of the logits (f32), the processors of tg_select
 * in their order (no temperature, top_k or top_p), plus the beam's score, in
 * f32 and never below the filter value.  Per prompt: the best keep of its
 * num_beams * V candidates in the order (score desc, beam * V + token asc).
 * An empty row gives no candidates; a prompt with fewer than keep gets
 * (filter value, -1, -1) in the remaining slots.  Errors as tg_select;
 * num_beams outside 1 .. 8 is TG_ERR_UNSUPPORTED.
 */
tg_status tg_beam_step(const void* logits, int32_t num_prompts, int32_t num_beams, int32_t V,
                       const float* beam_scores, const int32_t* hist_ids, const int64_t* hist_offsets,
                       const int32_t* prompt_lens, const tg_config* cfg, float* out_scores,
                       int32_t* out_tokens, int32_t* out_beams, tg_stream stream);

/* Candidates a prompt keeps per beam step: max(2, 1 + eos ids) * num_beams,
 * or -1 for a NULL config or num_beams < 1. */
int32_t tg_beam_keep(const tg_config* cfg, int32_t num_beams);

/* A static, human-readable name of a status code. */
const char* tg_status_string(tg_status s);

#ifdef __cplusplus
}
#endif
#endif /* TG_H_ */
