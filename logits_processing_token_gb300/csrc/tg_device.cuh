// Device-side building blocks of the token-selection kernels (sm_103a).
//
// Scores follow "Transmuter.Generation (transmuter v2.0.0)": f32 scores, the
// filter value is -FLT_MAX and no score goes below it (section
// Log-probabilities); row lengths and the conditional processors follow its
// section "Lengths"; the processor order follows its module intro.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace tg {

// Threads per CTA: 512 for every kernel of tg_kernels.cu; a translation unit
// may define TG_THREADS before including this header (tg_beam.cu: 256, two
// CTAs per SM).
#ifndef TG_THREADS
#define TG_THREADS 512
#endif
constexpr int kThreads = TG_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kStageBytes = 32768;          // one TMA bulk copy / sub-chunk of a row
constexpr int kRingStages = 3;              // TMA ring depth when it fits (else two)
constexpr int kCandCap = 4096;              // candidate slots of the one-pass path
constexpr float kFilter = -3.40282346638528859812e+38f;  // -FLT_MAX
constexpr float kLog2e = 1.44269504088896340736f;
constexpr int kFixShift = 44;               // fixed-point mass: weight * 2^44, weight <= 1
constexpr double kFixScale = 17592186044416.0;  // 2^44
constexpr unsigned long long kWaitLimitCycles = 2000000000ull;  // ~1 s bound on any wait

// Status bits (mirrors tg.h).
constexpr unsigned kFlagBadId = 0x1u;
constexpr unsigned kFlagBadRow = 0x2u;
constexpr unsigned kFlagSlow = 0x4u;
constexpr unsigned kFlagTimeout = 0x8u;
constexpr unsigned kFlagBadState = 0x10u;
constexpr int kMaxProcs = 8;           // the task's processors per config

enum { kGreedy = 0, kSample = 1 };
enum { kF32 = 0, kBF16 = 1 };

// Everything a kernel needs to know about the settings, passed by value.
struct DevCfg {
  int V;
  int dtype;
  int mode;
  float rho;                  // repetition penalty
  int ngram;                  // no_repeat_ngram_size
  const int* ban_sorted;      // bad words + suppress tokens, sorted, unique
  int n_ban;
  const int* sup_sorted;      // suppress tokens, sorted, unique
  int n_sup;
  const int* bsup_sorted;     // begin-suppress tokens, sorted, unique
  int n_bsup;
  const int* seq_ids;         // bad words of 2+ tokens, back to back
  const int* seq_off;         // n_seq + 1 offsets into seq_ids
  int n_seq;
  int renorm;                 // renormalize_logits
  int eos[8];
  int n_eos;
  int min_length;
  int min_new;
  int bos;                    // -1 = off
  int feos[8];                // forced eos ids, sorted, unique
  int n_feos;
  int max_new;
  float temp;
  int top_k;
  float top_p;
  unsigned* status;
  unsigned long long* slow_rows;
  unsigned* tickets;
  // The task's processors: kind (0 bias, 1 set) and state columns
  // [pcol[k], pcol[k+1]) of processor k; pcol[nproc] = S.
  int nproc;
  int pkind[kMaxProcs];
  int pcol[kMaxProcs + 1];
  // Set per row on a thread-local copy by the kernels that take a state:
  // prow routes process_elem through process_state_elem.
  bool prow;
  bool forced_row;              // a6/a7 active: the forced ids score 0, the rest F
  int nfz;                      // forced ids left after a8/a9
  int fz[8];
  const int* pst_ids;           // this row's state (S columns), or null when dropped
  const float* pst_vals;
  const unsigned* pbits;        // bitmap of this row's state ids (shared memory)
  bool sparse_row;              // forced row with a state: only the pbits tokens can score above F
  const float* sp_s;            // a sparse row's tokens above F: processed scores and ids (shared memory)
  const unsigned* sp_i;
  int sp_n;
};

struct SelArgs {
  const void* logits;
  int nrows;             // rows of this launch end here (exclusive)
  int row_begin;         // rows of this launch start here
  int nrows_total;       // B (select) or B*(K+1) (verify): rows of the whole call
  int V;
  const int32_t* hist;
  const int64_t* off;
  const int32_t* plen;
  const float* uniforms;
  int32_t* out;          // out_ids (select) or out_next (verify)
  const int32_t* cand;   // verify
  int K;
  int32_t* out_match;
  int vhist;             // verify: the processors run at every position, with the candidates as history
  float* logprobs;       // select: the token's log-probability per row, or null
  int nstage;
  int nwords;
  // the task's processors (tg_select_state): row b's state is st_ids/st_vals[b*S .. b*S+S)
  const int32_t* st_ids;
  const float* st_vals;
  int fixup;             // state_kernel: only rows select_kernel deferred (out == kDeferred)
};
// select_kernel with a state leaves this id for the rows it hands to state_kernel.
constexpr int kDeferred = -2;

// Launch helpers (tg_kernels.cu).
int select_smem_bytes(int nstage, int nwords);
int process_smem_bytes(int nwords, int S);
int state_smem_bytes(int nwords, int S);
cudaError_t launch_select(const DevCfg& c, const SelArgs& a, bool verify, int grid, int smem, cudaStream_t s);
// Greedy ids of rows [a.row_begin, a.nrows), each split over nslice CTAs of
// slice_tok tokens (a multiple of 8); best and tick: one key and one count per
// row, zero before the launch and left at zero after it (tg_kernels.cu).
// verify: the rows are a plain verify's positions (no processors), and the
// last position of each sequence writes its match (c.tickets zero before).
int split_greedy_smem(int nwords);
cudaError_t launch_split_greedy(const DevCfg& c, const SelArgs& a, int nslice, int slice_tok, unsigned long long* best,
                                unsigned* tick, bool verify, cudaStream_t s);
cudaError_t launch_process(const DevCfg& c, const SelArgs& a, float* scores, unsigned* banbits, float* probs,
                           int smem, cudaStream_t s, const int32_t* st_ids = nullptr, const float* st_vals = nullptr);
cudaError_t launch_state(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s,
                         const int32_t* st_ids, const float* st_vals);
cudaError_t select_occupancy(int dtype, bool verify, int smem, int* blocks_per_sm);

// Beam search, the device part of one step (tg_beam.cu).
constexpr int kMaxClusterBeams = 8;   // beams of a prompt: one CTA each, one cluster per prompt
struct BeamArgs {
  const void* logits;          // [P * nb, V]
  int nrows;                   // P * nb
  int nb;                      // beams per prompt
  int V;
  int keep;                    // candidates kept per prompt
  const float* beam_scores;    // [P * nb]
  const int32_t* hist;
  const int64_t* off;
  const int32_t* plen;
  float* out_scores;           // [P, keep]
  int32_t* out_tokens;
  int32_t* out_beams;
  int nwords;
};
int beam_smem_bytes(int nwords);
cudaError_t launch_beam(const DevCfg& c, const BeamArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
// Barrier over the kThreads "consumer" threads only (named barrier 1).  The
// select kernel adds one producer warp that never takes part.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// Order-preserving map f32 -> u32 (larger float -> larger key); -0 maps to +0.
__device__ __forceinline__ unsigned fkey(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(unsigned k) {
  unsigned u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ float clampf(float s) { return fmaxf(s, kFilter); }

__device__ __forceinline__ float bf16lo(unsigned p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16hi(unsigned p) { return __uint_as_float(p & 0xffff0000u); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Fast weight used only for the excluded mass: 2^(s*log2e - m*log2e).
__device__ __forceinline__ float wfast(float s, float c) { return ex2_approx(fmaf(s, kLog2e, -c)); }

// round(x * 2^44) for a finite x in [0, 2^19), ties to even: the value
// __float2ull_rn(x * 2^44) gives, computed with integer operations only (a
// 64-bit float-to-integer conversion is a slow instruction on this GPU).
__device__ __forceinline__ unsigned long long fix44(float x) {
  const unsigned b = __float_as_uint(x);
  const int e = static_cast<int>((b >> 23) & 0xffu);
  if (e == 0 || (b >> 31)) return 0ull;            // zero, subnormal (< 2^-126) or negative
  if (e >= 127 + 19) return 0x7fffffffffffffffull; // out of range (or inf/nan): saturate
  const unsigned long long mant = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u);
  const int sh = e - 127 - 23 + kFixShift;          // x * 2^44 = mant * 2^sh
  if (sh >= 0) return mant << sh;
  const int r = -sh;
  if (r > 24) return 0ull;                           // below one half
  const unsigned long long q = mant >> r;
  const unsigned long long rem = mant & ((1ull << r) - 1ull);
  const unsigned long long half = 1ull << (r - 1);
  return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

// Accurate weight exp(s - m) in fixed point (x 2^44).  s - m is formed
// exactly as hi + lo (TwoSum); exp(hi + lo) ~= exp(hi) * (1 + lo).
__device__ __forceinline__ unsigned long long wfix(float s, float m) {
  float a = s, b = -m;
  float hi = __fadd_rn(a, b);
  float bb = __fsub_rn(hi, a);
  float lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
  float e = expf(hi);
  float w = fmaf(e, lo, e);
  w = fminf(fmaxf(w, 0.0f), 1.0f);
  return fix44(w);
}

// Fast weight in fixed point: the one-pass path's weight, consistent with
// the excluded mass it accumulates with wfast (cc = m * log2e).
__device__ __forceinline__ unsigned long long wfix_fast(float s, float cc) {
  return fix44(wfast(s, cc));
}

// Weight functors for the radix engine.
struct WExact {
  float m;
  __device__ __forceinline__ unsigned long long operator()(float s) const { return wfix(s, m); }
};
struct WFast {
  float cc;
  __device__ __forceinline__ unsigned long long operator()(float s) const { return wfix_fast(s, cc); }
};

// Temperature, then the clamp at the filter value.  A patched slot holding
// -inf stays -inf (it is counted through its side-list entry instead).
__device__ __forceinline__ float temper(float v, float T) {
  float q = __fdiv_rn(v, T);
  return fmaxf(q, v == -INFINITY ? -INFINITY : kFilter);
}

__device__ __forceinline__ float penalize(float x, float rho) {
  float s = x < 0.0f ? __fmul_rn(x, rho) : __fdiv_rn(x, rho);
  return clampf(s);
}

// Binary search in a sorted int array (global memory, small).
__device__ __forceinline__ bool in_sorted(const int* a, int n, int t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    int v = __ldg(a + mid);
    if (v < t) lo = mid + 1; else hi = mid;
  }
  return lo < n && __ldg(a + lo) == t;
}

// ---------------------------------------------------------------------------
// block reductions (all threads must call)
// ---------------------------------------------------------------------------
struct RedScratch {
  float f[kWarps];
  double d[kWarps];
  unsigned u[kWarps];
  unsigned long long q[kWarps];
};

__device__ __forceinline__ float block_max(float v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  csync();
  if ((threadIdx.x & 31) == 0) r->f[threadIdx.x >> 5] = v;
  csync();
  float m = r->f[0];
  for (int i = 1; i < kWarps; ++i) m = fmaxf(m, r->f[i]);
  return m;
}
__device__ __forceinline__ float block_sum_f(float v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  csync();
  if ((threadIdx.x & 31) == 0) r->f[threadIdx.x >> 5] = v;
  csync();
  // pairwise over the 16 warp partials
  float a[kWarps];
#pragma unroll
  for (int i = 0; i < kWarps; ++i) a[i] = r->f[i];
#pragma unroll
  for (int w = kWarps / 2; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] += a[i + w];
  return a[0];
}
// Max of m and sum of e over the block in one exchange.
__device__ __forceinline__ void block_max_sum(float& m, float& e, RedScratch* r) {
  for (int o = 16; o; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    e += __shfl_xor_sync(0xffffffffu, e, o);
  }
  csync();
  if ((threadIdx.x & 31) == 0) { r->f[threadIdx.x >> 5] = m; r->u[threadIdx.x >> 5] = __float_as_uint(e); }
  csync();
  float a[kWarps];
  float mm = r->f[0];
#pragma unroll
  for (int i = 0; i < kWarps; ++i) { a[i] = __uint_as_float(r->u[i]); mm = fmaxf(mm, r->f[i]); }
#pragma unroll
  for (int w = kWarps / 2; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] += a[i + w];
  m = mm;
  e = a[0];
}
__device__ __forceinline__ double block_sum_d(double v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  csync();
  if ((threadIdx.x & 31) == 0) r->d[threadIdx.x >> 5] = v;
  csync();
  double s = 0.0;
  for (int i = 0; i < kWarps; ++i) s += r->d[i];
  return s;
}
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  csync();
  if ((threadIdx.x & 31) == 0) r->q[threadIdx.x >> 5] = v;
  csync();
  unsigned long long s = 0;
  for (int i = 0; i < kWarps; ++i) s += r->q[i];
  return s;
}
__device__ __forceinline__ unsigned block_min_u(unsigned v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  csync();
  if ((threadIdx.x & 31) == 0) r->u[threadIdx.x >> 5] = v;
  csync();
  unsigned m = r->u[0];
  for (int i = 1; i < kWarps; ++i) m = min(m, r->u[i]);
  return m;
}
__device__ __forceinline__ unsigned block_max_u(unsigned v, RedScratch* r) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  csync();
  if ((threadIdx.x & 31) == 0) r->u[threadIdx.x >> 5] = v;
  csync();
  unsigned m = r->u[0];
  for (int i = 1; i < kWarps; ++i) m = max(m, r->u[i]);
  return m;
}

// ---------------------------------------------------------------------------
// Row metadata: the "Lengths" rules evaluated once per row
// ---------------------------------------------------------------------------
struct RowMeta {
  long long h0;     // first history id
  int L, P;
  int Lb;           // the first Lb ids are hist[h0 ..]; the other L - Lb are ext[0 ..]
  const int32_t* ext;
  bool bad;         // inconsistent offsets / prompt length
  bool eos_off;     // a5: eos ids removed
  bool forced;      // a6 or a7 active
  bool forced_eos;  // a7 active (it runs after a6 and overrides it)
  bool bsup;        // a9: begin-suppress active
};

__device__ __forceinline__ void row_meta_rules(const DevCfg& c, RowMeta& r);

// Rows must form a CSR over hist_ids: 0 <= off[b] <= off[b+1] <= off[B].  A
// row outside that, or with a prompt longer than the row, is flagged bad.
__device__ __forceinline__ RowMeta row_meta(const DevCfg& c, const int32_t* hist, const int64_t* off,
                                            const int32_t* plen, int b, int B) {
  RowMeta r;
  long long o0 = off[b], o1 = off[b + 1], oend = off[B];
  int P = plen[b];
  r.h0 = o0;
  long long L = o1 - o0;
  r.bad = (o0 < 0) || (L < 0) || (o1 > oend) || (L > 0x7fffffffLL) || (P < 0) || (P > L) ||
          (hist == nullptr && L > 0);
  r.L = r.bad ? 0 : static_cast<int>(L);
  r.P = r.bad ? 0 : P;
  r.Lb = r.L;
  r.ext = nullptr;
  row_meta_rules(c, r);
  return r;
}

// The length rules of a row whose L and P are set.
__device__ __forceinline__ void row_meta_rules(const DevCfg& c, RowMeta& r) {
  int Li = r.L, new_tokens = r.L - r.P;
  if (c.min_new > 0) r.eos_off = new_tokens < c.min_new;
  else r.eos_off = c.min_length > 0 && Li < c.min_length;
  bool fb = c.bos >= 0 && Li == 1;
  r.forced_eos = c.n_feos > 0 && Li == r.P + c.max_new - 1;
  r.forced = fb || r.forced_eos;
  int bidx = (c.bos >= 0 && r.P == 1) ? r.P + 1 : r.P;
  r.bsup = c.n_bsup > 0 && Li == bidx;
}

// ---------------------------------------------------------------------------
// Per-row bitmaps in shared memory: N = banned (n-gram, bad words, eos under
// min length, suppress, begin-suppress); H = every token a processor changes:
// the banned ones and, when rho != 1, the history ids.  A token of H that is
// not in N is penalised.  nwords = ceil(V/32).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_bit(unsigned* bm, int t) { atomicOr(bm + (t >> 5), 1u << (t & 31)); }
__device__ __forceinline__ bool get_bit(const unsigned* bm, int t) { return (bm[t >> 5] >> (t & 31)) & 1u; }

//
// With `ctr` (a shared counter) and the history staged, the marked tokens are
// also listed, each once, in N's words (entry = t | banned << 31) and the
// count is returned; N then no longer holds the banned bitmap.  The return
// value is -1 when no list is made (not asked for, history not staged, or
// more marked tokens than fit), and N keeps the bitmap.
constexpr unsigned kBannedFlag = 0x80000000u;
constexpr unsigned kPlainFlag = 0x40000000u;   // listed from the processors' state only: no penalty
constexpr unsigned kIdMask = 0x3fffffffu;
//
// With `sids` (S ids of a row's processor state, -1 unused), the state ids
// are marked too and listed last: a state id that is no history id and not
// banned gets kPlainFlag (its score is x before the processors).
static __device__ __noinline__ int build_row_bitmaps(const DevCfg& c, const int32_t* hist, const RowMeta& r,
                                                     unsigned* H, unsigned* N, int nwords, int* stage = nullptr,
                                                     int stage_cap = 0, unsigned* ctr = nullptr,
                                                     const int32_t* sids = nullptr, int S = 0) {
  const int tid = threadIdx.x;
  for (int w = tid; w < nwords; w += kThreads) { H[w] = 0u; N[w] = 0u; }
  const int V = c.V;
  const int32_t* h = hist + r.h0;
  const int L = r.L;
  // With a shared-memory stage large enough, the history is copied there
  // first (coalesced, four reads in flight per thread) and every pass below
  // reads shared memory instead of waiting on global loads one at a time.
  // A row extended by ext (a verify position's candidates) is always staged.
  const bool staged = stage != nullptr && L <= stage_cap;
  if (staged) {
    const int Lb = r.Lb;
    for (int i0 = 0; i0 < L; i0 += 4 * kThreads) {
      int v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kThreads + tid;
        v[q] = i < L ? (i < Lb ? __ldg(h + i) : __ldg(r.ext + (i - Lb))) : 0;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kThreads + tid;
        if (i < L) stage[i] = v[q];
      }
    }
  }
  csync();
  const int32_t* hs = staged ? stage : h;
  bool bad_id = false;
  if (c.rho != 1.0f) {
    for (int i = tid; i < L; i += kThreads) {
      int t = hs[i];
      if (t >= 0 && t < V) set_bit(H, t); else bad_id = true;
    }
  } else {
    for (int i = tid; i < L; i += kThreads) {
      int t = hs[i];
      if (t < 0 || t >= V) bad_id = true;
    }
  }
  // no_repeat_ngram_size: start j bans h[j+n-1] when h[j..j+n-2] equals the
  // row's last n-1 tokens.
  const int n = c.ngram;
  if (n > 0 && L + 1 >= n) {
    const int last = L - n;  // last start of a complete n-gram
    const int s0 = L - n + 1;
    const int first_tok = n > 1 ? hs[s0] : 0;
    for (int j = tid; j <= last; j += kThreads) {
      bool eq = true;
      if (n > 1) {
        eq = hs[j] == first_tok;
        for (int q = 1; eq && q < n - 1; ++q) eq = hs[j + q] == hs[s0 + q];
      }
      if (eq) {
        int t = hs[j + n - 1];
        if (t >= 0 && t < V) set_bit(N, t);
      }
    }
  }
  // a4, bad words of several tokens: word s bans its last id when the row
  // ends with its other ids (one-token words are in the constant ban list)
  for (int s = tid; s < c.n_seq; s += kThreads) {
    const int o0 = __ldg(c.seq_off + s), o1 = __ldg(c.seq_off + s + 1), k = o1 - o0 - 1;
    bool hit = L >= k;
    for (int q = 0; hit && q < k; ++q) hit = hs[L - k + q] == __ldg(c.seq_ids + o0 + q);
    if (hit) set_bit(N, __ldg(c.seq_ids + o1 - 1));
  }
  for (int i = tid; i < c.n_ban; i += kThreads) set_bit(N, __ldg(c.ban_sorted + i));
  if (r.eos_off && tid < c.n_eos) set_bit(N, c.eos[tid]);
  if (r.bsup)
    for (int i = tid; i < c.n_bsup; i += kThreads) set_bit(N, __ldg(c.bsup_sorted + i));
  if (bad_id) atomicOr(c.status, kFlagBadId);
  for (int j = tid; j < S; j += kThreads) {
    const int t = __ldg(sids + j);
    if (t >= 0 && t < V) set_bit(H, t);
  }
  const bool listing = ctr != nullptr && staged;
  if (listing && tid == 0) *ctr = 0u;
  csync();
  // H becomes the marked set M = history | banned; N stays the banned set
  int cnt = 0;
  for (int w = tid; w < nwords; w += kThreads) {
    const unsigned m = H[w] | N[w];
    H[w] = m;
    cnt += __popc(m);
  }
  if (!listing) {
    csync();
    return -1;
  }
  // The list: every marked token is a history id or an id of a ban list.
  // The first thread to clear a token's bit in M lists it; M is restored
  // from the list afterwards.  A warp reserves room for its entries at once.
  for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) atomicAdd(ctr, static_cast<unsigned>(cnt));
  csync();
  const int total = static_cast<int>(*ctr);
  const int cap = min(stage_cap - L, nwords);
  csync();
  if (total > cap) return -1;
  if (tid == 0) *ctr = 0u;
  csync();
  int* tmp = stage + L;
  const int lane = tid & 31;
  auto claim = [&](int t, unsigned extra = 0u) {   // every lane of the warp calls, t < 0 for none
    bool own = false;
    unsigned e = 0u;
    if (t >= 0 && t < V) {
      const unsigned bit = 1u << (t & 31);
      own = (atomicAnd(&H[t >> 5], ~bit) & bit) != 0u;
      e = static_cast<unsigned>(t) | ((N[t >> 5] & bit) ? kBannedFlag : extra);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, own);
    if (bal) {
      int base = 0;
      if (lane == 0) base = static_cast<int>(atomicAdd(ctr, static_cast<unsigned>(__popc(bal))));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (own) tmp[base + __popc(bal & ((1u << lane) - 1u))] = static_cast<int>(e);
    }
  };
  for (int i0 = 0; i0 < L; i0 += kThreads) claim(i0 + tid < L ? hs[i0 + tid] : -1);
  for (int i0 = 0; i0 < c.n_ban; i0 += kThreads) claim(i0 + tid < c.n_ban ? __ldg(c.ban_sorted + i0 + tid) : -1);
  for (int i0 = 0; i0 < c.n_seq; i0 += kThreads)
    claim(i0 + tid < c.n_seq ? __ldg(c.seq_ids + __ldg(c.seq_off + i0 + tid + 1) - 1) : -1);
  if (r.eos_off) claim(tid < c.n_eos ? c.eos[tid] : -1);
  if (r.bsup)
    for (int i0 = 0; i0 < c.n_bsup; i0 += kThreads) claim(i0 + tid < c.n_bsup ? __ldg(c.bsup_sorted + i0 + tid) : -1);
  // last: what is still unclaimed of the state is neither history nor banned
  for (int i0 = 0; i0 < S; i0 += kThreads) claim(i0 + tid < S ? __ldg(sids + i0 + tid) : -1, kPlainFlag);
  csync();
  const int nl = static_cast<int>(*ctr);
  const bool whole = nl == total;   // always, unless a marked token had no source
  for (int i = tid; i < nl; i += kThreads) {
    const unsigned e = static_cast<unsigned>(tmp[i]);
    if (whole) N[i] = e;
    atomicOr(&H[(e & kIdMask) >> 5], 1u << (e & 31u));
  }
  csync();
  return whole ? nl : -1;
}

// The task's processors (Transmuter.Generation, section "Processors") on one
// token's score s, in list order: processor k finds t among the ids in use of
// its state columns (ascending, -1 padding after them) by binary search; an
// entry (t, v) makes s + v ("bias", one f32 add) or v ("set"), never below
// the filter value.  The state may be in global or shared memory.
// Column of t among one processor's n columns (ids in use ascending, -1
// padding after them), or -1.
__device__ __forceinline__ int state_find(const int* ids, int n, int t) {
  int lo = 0, hi = n;   // first column whose id is unused (-1) or >= t
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = ids[mid];
    if (v != -1 && v < t) lo = mid + 1; else hi = mid;
  }
  return (lo < n && ids[lo] == t) ? lo : -1;
}

__device__ __forceinline__ float apply_state_at(const DevCfg& c, const int* sids, const float* svals, float s,
                                                int t) {
  for (int k = 0; k < c.nproc; ++k) {
    const int c0 = c.pcol[k];
    const int j = state_find(sids + c0, c.pcol[k + 1] - c0, t);
    if (j >= 0) {
      const float v = svals[c0 + j];
      s = clampf(c.pkind[k] == 0 ? __fadd_rn(s, v) : v);
    }
  }
  return s;
}
__device__ __forceinline__ float apply_state(const DevCfg& c, float s, int t) {
  return apply_state_at(c, c.pst_ids, c.pst_vals, s, t);
}

// a2-a9 and the task's processors for one token of a row that has a state
// (or is forced): forced rows score 0 at the forced ids and F elsewhere;
// other rows take the row bitmaps; then the processors, for tokens whose
// bit is set in the row's state bitmap.
static __device__ __noinline__ float process_state_elem(const DevCfg& c, const unsigned* H, const unsigned* N,
                                                        float x, int i) {
  float s;
  if (c.forced_row) {
    s = kFilter;
    for (int q = 0; q < c.nfz; ++q) s = c.fz[q] == i ? 0.0f : s;
  } else if (get_bit(N, i)) {
    s = kFilter;
  } else if (get_bit(H, i)) {
    s = penalize(x, c.rho);
  } else {
    s = x;
  }
  if (c.pst_ids != nullptr && get_bit(c.pbits, i)) s = apply_state(c, s, i);
  return s;
}

// Processed score of one token from its raw value and the row bitmaps
// (a2-a9 for a row that is not forced), then temperature when sampling.
__device__ __forceinline__ float process_elem(const DevCfg& c, const unsigned* H, const unsigned* N,
                                              float x, int i, bool sample) {
  float s = x;
  if (c.prow) s = process_state_elem(c, H, N, x, i);
  else if (get_bit(N, i)) s = kFilter;
  else if (get_bit(H, i)) s = penalize(x, c.rho);
  if (sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
  return s;
}

// Processed score of a marked token (its row-bitmap bit is set) from its raw
// value: the filter value when banned, else penalised; then temperature when
// sampling.  The same result as process_elem for such a token.
__device__ __forceinline__ float process_marked(const DevCfg& c, float x, bool banned, bool sample) {
  float s = banned ? kFilter : penalize(x, c.rho);
  if (sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
  return s;
}

// A 1,024-bit filter of a row's state ids (bit t mod 1024): a token whose bit
// is clear is no state id.
constexpr int kStateFilterWords = 32;
__device__ __forceinline__ bool state_filter_hit(const unsigned* f, int t) {
  return (f[(t >> 5) & (kStateFilterWords - 1)] >> (t & 31)) & 1u;
}

// Processed score of a listed marked token from its raw value and its list
// entry e (banned, plain or a penalised history id), then the row's processor
// state when sids is given (sfilt: the state ids' filter), then temperature
// when sampling.
__device__ __forceinline__ float process_listed(const DevCfg& c, float x, unsigned e, const int* sids,
                                                const float* svals, const unsigned* sfilt, bool sample) {
  float s = (e & kBannedFlag) ? kFilter : ((e & kPlainFlag) ? x : penalize(x, c.rho));
  const int t = static_cast<int>(e & kIdMask);
  if (sids != nullptr && state_filter_hit(sfilt, t)) s = apply_state_at(c, sids, svals, s, t);
  if (sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
  return s;
}

// ---------------------------------------------------------------------------
// Forced rows (a6/a7 active): every token is the filter value except the
// forced ids, which score 0, unless suppress_tokens or begin_suppress_tokens
// remove them again (a8, a9 run after the forcing).  The zero-scored ids are
// returned sorted and unique in zs[0..nz).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int forced_zeros(const DevCfg& c, const RowMeta& r, int* zs) {
  int cand[8];
  int nc = 0;
  if (r.forced_eos) {
    for (int i = 0; i < c.n_feos; ++i) cand[nc++] = c.feos[i];
  } else {
    cand[nc++] = c.bos;
  }
  int nz = 0;
  for (int i = 0; i < nc; ++i) {
    int t = cand[i];
    bool gone = in_sorted(c.sup_sorted, c.n_sup, t) || (r.bsup && in_sorted(c.bsup_sorted, c.n_bsup, t));
    if (!gone) zs[nz++] = t;
  }
  return nz;
}

// n-th member (1-based) of a group of equal-weight items whose running mass
// starting at `above` first reaches the target: >= target (cut) or > target
// (draw).  Always in [1, cnt].
__device__ __forceinline__ unsigned long long group_pick(unsigned long long above, unsigned long long w,
                                                         unsigned long long cnt, unsigned long long target,
                                                         bool strict) {
  unsigned long long n;
  if (w == 0ull) return cnt;
  if (target < above) return 1ull;
  unsigned long long need = target - above;
  n = strict ? need / w + 1ull : (need + w - 1ull) / w;
  if (n < 1ull) n = 1ull;
  if (n > cnt) n = cnt;
  return n;
}

// p * Z for a float p in [0, 1] and a 64-bit Z, exactly: p = mant * 2^-k
// with a 24-bit mant, so p * Z = (mant * Z) / 2^k with a 128-bit numerator.
// Returns floor(p * Z) and whether p * Z is not an integer.
__device__ __forceinline__ unsigned long long mul_frac(float p, unsigned long long Z, bool* inexact) {
  const unsigned b = __float_as_uint(p);
  const int e = static_cast<int>((b >> 23) & 0xffu);
  *inexact = false;
  if (e == 0 || (b >> 31) || Z == 0ull) { *inexact = false; return 0ull; }
  const unsigned long long mant = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u);
  const int k = 150 - e;                       // p = mant * 2^-k
  const unsigned long long lo = mant * Z, hi = __umul64hi(mant, Z);
  if (k <= 0) return lo << (-k);               // p >= 2^23: not reached for p <= 1
  if (k >= 128) { *inexact = (lo | hi) != 0ull; return 0ull; }
  unsigned long long q, rem_nonzero;
  if (k >= 64) {
    q = k == 64 ? hi : hi >> (k - 64);
    rem_nonzero = lo | (k == 64 ? 0ull : (hi & ((1ull << (k - 64)) - 1ull)));
  } else {
    q = (lo >> k) | (hi << (64 - k));
    rem_nonzero = lo & ((1ull << k) - 1ull);
  }
  *inexact = rem_nonzero != 0ull;
  return q;
}

// Mass target of the top-p cut: the smallest integer >= p * Z.
__device__ __forceinline__ unsigned long long topp_target(float p, unsigned long long Z) {
  bool inexact;
  const unsigned long long f = mul_frac(p, Z, &inexact);
  const unsigned long long T = f + (inexact ? 1ull : 0ull);
  return T > Z ? Z : T;
}
// Mass target of the draw: the largest integer <= u * S, u in [0, 1).
__device__ __forceinline__ unsigned long long draw_target(float u, unsigned long long S) {
  if (!(u >= 0.0f)) u = 0.0f;               // NaN or negative -> 0
  if (u >= 1.0f) u = 0x1.fffffep-1f;        // largest float below 1
  bool inexact;
  const unsigned long long T = mul_frac(u, S, &inexact);
  return (T >= S && S > 0) ? S - 1 : T;
}

// ---------------------------------------------------------------------------
// Warp-parallel search over N buckets (run by one full warp): the first
// bucket, in scan order (descending bucket index when `desc`), at which the
// running sum of v reaches `reached(cum)`.  `cnt` marks non-empty buckets;
// when the sum never reaches the target the last non-empty bucket is
// returned with found = 0.
// ---------------------------------------------------------------------------
template <class T>
struct FindOut {
  int b;          // bucket
  T before;       // sum of v over buckets before b in scan order
  int found;
};

template <int N, class T, class Reached>
__device__ __forceinline__ FindOut<T> warp_find(const T* v, const unsigned* cnt, bool desc, Reached reached) {
  constexpr int PER = N / 32;
  const int lane = threadIdx.x & 31;
  T local = 0;
  int last_ne = -1;
#pragma unroll 8
  for (int j = 0; j < PER; ++j) {
    const int p = lane * PER + j;
    const int b = desc ? N - 1 - p : p;
    local += v[b];
    if (cnt[b]) last_ne = p;
  }
  T incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const T excl = incl - local;
  FindOut<T> r;
  r.b = 0;
  r.before = 0;
  r.found = 0;
  const unsigned hit = __ballot_sync(0xffffffffu, reached(incl));
  if (hit) {
    const int L = __ffs(hit) - 1;
    int b = 0;
    T cum = 0;
    if (lane == L) {
      cum = excl;
      for (int j = 0; j < PER; ++j) {
        const int p = lane * PER + j;
        b = desc ? N - 1 - p : p;
        const T nx = cum + v[b];
        if (reached(nx)) break;
        cum = nx;
      }
    }
    r.b = __shfl_sync(0xffffffffu, b, L);
    r.before = __shfl_sync(0xffffffffu, cum, L);
    r.found = 1;
  } else {
    const unsigned ne = __ballot_sync(0xffffffffu, last_ne >= 0);
    if (ne) {
      const int L = 31 - __clz(ne);
      const int p = __shfl_sync(0xffffffffu, last_ne, L);
      const int b = desc ? N - 1 - p : p;
      // sum of v strictly before position p in scan order
      T part = 0;
      for (int j = 0; j < PER; ++j) {
        const int q = lane * PER + j;
        if (q < p) part += v[desc ? N - 1 - q : q];
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      r.b = b;
      r.before = part;
    }
  }
  return r;
}

// ---------------------------------------------------------------------------
// Radix selection engine.  A Source visits every item (score s, index i) of
// one row, once per pass, on all threads of the CTA:
//     src.pass([&](float s, unsigned i) { ... });
// Items are ordered by (s desc, i asc).  Weights come from a functor (WExact
// or WFast) so that every pass of one selection uses the same weights.
// ---------------------------------------------------------------------------
struct Hist {
  unsigned long long mass[256];
  unsigned cnt[256];
  unsigned mw[4][256];   // the weights in four 11-bit limbs: exact sums with 32-bit atomics
  // broadcast slots
  unsigned sel_bucket;
  unsigned long long sel_above;
  unsigned long long sel_mass;
  unsigned sel_cnt;
  unsigned sel_found;
};

// Kept-set filter: key >= klo, and, when `cut` is set, (key > kcut) or
// (key == kcut and i <= icut).
struct KeepFilter {
  unsigned klo;
  bool cut;
  unsigned kcut, icut;
  __device__ __forceinline__ bool operator()(unsigned key, unsigned i) const {
    if (key < klo) return false;
    if (!cut) return true;
    return key > kcut || (key == kcut && i <= icut);
  }
};

struct MassSel {
  unsigned key;               // key of the selected item
  unsigned idx;               // its index
  unsigned long long mass;    // running mass up to and including it
  bool found;
};

// Clear the histogram (all threads) -- followed by a barrier.
__device__ __forceinline__ void hist_clear(Hist* h) {
  for (int i = threadIdx.x; i < 256; i += kThreads) {
    h->mass[i] = 0ull;
    h->cnt[i] = 0u;
    h->mw[0][i] = 0u; h->mw[1][i] = 0u; h->mw[2][i] = 0u; h->mw[3][i] = 0u;
  }
  csync();
}

// The rank-th smallest index (1-based) among items with key == key and
// passing flt.  Counting radix select over the index bits, high digit first.
template <class Src, class Flt>
__device__ unsigned nth_index(const Src& src, Flt flt, unsigned key, unsigned rank, Hist* h) {
  unsigned prefix = 0u;
  for (int shift = 16; shift >= 0; shift -= 8) {
    hist_clear(h);
    const unsigned hi_mask = shift == 16 ? 0u : (0xffffffffu << (shift + 8));
    src.pass([&](float s, unsigned i) {
      unsigned k = fkey(s);
      if (k == key && flt(k, i) && (i & hi_mask) == prefix) atomicAdd(&h->cnt[(i >> shift) & 255u], 1u);
    });
    csync();
    if (threadIdx.x < 32) {
      const unsigned need = rank;
      FindOut<unsigned> f = warp_find<256>(h->cnt, h->cnt, false, [need](unsigned c) { return c >= need; });
      if (threadIdx.x == 0) { h->sel_bucket = static_cast<unsigned>(f.b); h->sel_cnt = f.before; }
    }
    csync();
    rank -= h->sel_cnt;
    prefix |= h->sel_bucket << shift;
    csync();
  }
  return prefix;
}

// The k-th largest key (with multiplicity) among items passing flt.
template <class Src, class Flt>
__device__ unsigned kth_key(const Src& src, Flt flt, unsigned k, Hist* h) {
  unsigned prefix = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    hist_clear(h);
    const unsigned hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    src.pass([&](float s, unsigned i) {
      unsigned key = fkey(s);
      if (flt(key, i) && (key & hi_mask) == prefix) atomicAdd(&h->cnt[(key >> shift) & 255u], 1u);
    });
    csync();
    if (threadIdx.x < 32) {
      const unsigned need = k;
      FindOut<unsigned> f = warp_find<256>(h->cnt, h->cnt, true, [need](unsigned c) { return c >= need; });
      if (threadIdx.x == 0) { h->sel_bucket = static_cast<unsigned>(f.b); h->sel_cnt = f.before; }
    }
    csync();
    k -= h->sel_cnt;
    prefix |= h->sel_bucket << shift;
    csync();
  }
  return prefix;
}

// First item, in (s desc, i asc) order among items passing flt, at which
// the running mass reaches the target: >= target (strict == false) or
// > target (strict == true).  found == false when the filtered mass never
// reaches it (the last item is returned then).
template <class Src, class Flt, class Wt>
__device__ MassSel mass_select(const Src& src, Flt flt, Wt wf, unsigned long long target, bool strict,
                               Hist* h) {
  unsigned prefix = 0u;
  unsigned long long above = 0ull;
  unsigned long long gmass = 0ull;
  unsigned gcnt = 0u;
  bool found = true;
  for (int shift = 24; shift >= 0; shift -= 8) {
    hist_clear(h);
    const unsigned hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    src.pass([&](float s, unsigned i) {
      unsigned key = fkey(s);
      if (flt(key, i) && (key & hi_mask) == prefix) {
        unsigned b = (key >> shift) & 255u;
        const unsigned long long w = wf(s);   // <= 2^44
        atomicAdd(&h->mw[0][b], static_cast<unsigned>(w & 0x7ffull));
        atomicAdd(&h->mw[1][b], static_cast<unsigned>((w >> 11) & 0x7ffull));
        atomicAdd(&h->mw[2][b], static_cast<unsigned>((w >> 22) & 0x7ffull));
        atomicAdd(&h->mw[3][b], static_cast<unsigned>(w >> 33));
        atomicAdd(&h->cnt[b], 1u);
      }
    });
    csync();
    for (int i = threadIdx.x; i < 256; i += kThreads)
      h->mass[i] = static_cast<unsigned long long>(h->mw[0][i]) + (static_cast<unsigned long long>(h->mw[1][i]) << 11) +
                   (static_cast<unsigned long long>(h->mw[2][i]) << 22) + (static_cast<unsigned long long>(h->mw[3][i]) << 33);
    csync();
    if (threadIdx.x < 32) {
      const unsigned long long base = above;
      const unsigned long long tgt = target;
      FindOut<unsigned long long> f = warp_find<256>(
          h->mass, h->cnt, true,
          [base, tgt, strict](unsigned long long c) { return strict ? base + c > tgt : base + c >= tgt; });
      if (threadIdx.x == 0) {
        h->sel_bucket = static_cast<unsigned>(f.b);
        h->sel_above = above + f.before;
        h->sel_mass = h->mass[f.b];
        h->sel_cnt = h->cnt[f.b];
        h->sel_found = static_cast<unsigned>(f.found);
      }
    }
    csync();
    prefix |= h->sel_bucket << shift;
    above = h->sel_above;
    gmass = h->sel_mass;
    gcnt = h->sel_cnt;
    found = found && h->sel_found;
    csync();
  }
  MassSel r;
  r.key = prefix;
  r.found = found && gcnt > 0u;
  if (gcnt == 0u) { r.idx = 0u; r.mass = above; return r; }
  unsigned long long w = gmass / gcnt;  // every item of the group has the same weight
  unsigned long long n = r.found ? group_pick(above, w, gcnt, target, strict) : gcnt;
  r.idx = nth_index(src, flt, prefix, static_cast<unsigned>(n), h);
  r.mass = above + n * w;
  return r;
}

// Sum of weights over items passing flt.
template <class Src, class Flt, class Wt>
__device__ unsigned long long mass_sum(const Src& src, Flt flt, Wt wf, RedScratch* red) {
  unsigned long long acc = 0ull;
  src.pass([&](float s, unsigned i) {
    unsigned key = fkey(s);
    if (flt(key, i)) acc += wf(s);
  });
  return block_sum_u64(acc, red);
}

template <class Src, class Flt>
__device__ unsigned count_items(const Src& src, Flt flt, RedScratch* red) {
  unsigned acc = 0u;
  src.pass([&](float s, unsigned i) {
    if (flt(fkey(s), i)) ++acc;
  });
  return static_cast<unsigned>(block_sum_u64(acc, red));
}

// Full sampling selection over a source holding EVERY token of the row:
// top_k, top_p, then the draw.  m = the row's maximum score.
// Returns the drawn token, and (optionally) the kept-set filter and its mass.
template <class Src>
__device__ unsigned sample_exact(const DevCfg& c, const Src& src, float m, float u, unsigned V,
                                 Hist* h, RedScratch* red, KeepFilter* kept_out,
                                 unsigned long long* S_out, unsigned* key_out = nullptr) {
  KeepFilter f{0u, false, 0u, 0u};
  if (c.top_k > 0 && static_cast<unsigned>(c.top_k) < V)
    f.klo = kth_key(src, f, static_cast<unsigned>(c.top_k), h);
  const WExact wx{m};
  unsigned long long Z = mass_sum(src, f, wx, red);
  unsigned long long S = Z;
  if (c.top_p < 1.0f) {
    unsigned long long T = topp_target(c.top_p, Z);
    MassSel cut = mass_select(src, f, wx, T, false, h);
    f.cut = true;
    f.kcut = cut.key;
    f.icut = cut.idx;
    S = cut.mass;
  }
  unsigned long long Td = draw_target(u, S);
  MassSel d = mass_select(src, f, wx, Td, true, h);
  if (kept_out) *kept_out = f;
  if (S_out) *S_out = S;
  if (key_out) *key_out = d.key;
  return d.idx;
}

}  // namespace tg
