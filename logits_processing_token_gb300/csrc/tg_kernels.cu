// Token-selection kernels for sm_103a.
//
//  select_kernel  -- tg_select and tg_verify.  One CTA of 16 warps per SM,
//                    persistent over the rows it owns.  Every row is streamed
//                    once from HBM with 32 KB bulk copies (TMA) into a ring of
//                    shared-memory stages.  Each warp copies its 2 KB slice of
//                    a stage into registers and counts itself done; the last
//                    of the 16 warps to do so refills the stage, so loads are
//                    in flight while every warp computes on registers.
//  process_kernel -- tg_process (diagnostic): processed scores, ban bits and
//                    the final distribution, written to global memory.
//
// Processors.  A per-row bitmap M marks every token that a processor changes
// (history ids under a repetition penalty, n-gram bans, bad words, eos under
// min length, suppress and begin-suppress ids); N marks the banned ones.
// The streaming loop never computes a processed score: greedy treats marked
// tokens as -inf, sampling counts their raw weight.  At the end of the row the
// marked tokens are read again (from L2), processed exactly, and merged in:
// greedy compares them with the best unmarked token, sampling replaces their
// raw weight with the processed one.
//
// Sampling in one pass.  While streaming, every lane adds the weight
// 2^((x - m0) log2e / T) of its raw logits x to its running mass (m0 = the
// first sub-chunk's maximum), and sets one bit per sub-chunk when its slice
// holds a logit at or above the row's raw threshold theta (chosen from the
// first sub-chunk's level counts).  At the end of the row the flagged slices
// are read again and every unmarked token whose processed score reaches
// theta_f becomes a candidate; theta_f is chosen so that no token below the
// raw threshold can reach it.  top_k, the top_p cut and the draw then run
// exactly on the candidates with fixed-point weights; every other token sits
// after all candidates in the (score desc, index asc) order, so the result is
// exact whenever the candidates hold the k largest scores (top_k), or more
// mass than the cut (top_p) or the draw target needs.  A row where that check
// fails is read once more with a lower threshold, and then, if needed,
// decided by the multi-pass exact selection over the whole row.
#include <mutex>

#include "../../include/tg.h"
#include "tg_device.cuh"

namespace tg {

#ifdef TG_DEBUG
// Debug builds only: per-row record {path, reason, m, theta, E, Zc, Z, ncand}.
__device__ double* g_dbg = nullptr;
#define TG_DBG(row, slot, val) do { if (g_dbg && threadIdx.x == 0) g_dbg[(row) * 32 + (slot)] = (double)(val); } while (0)
#else
#define TG_DBG(row, slot, val) do { } while (0)
#endif
#ifdef TG_DEBUG
#define TG_GIVEUP(bit) atomicOr(&sm.misc.gcause, (bit))
__device__ __forceinline__ unsigned long long tg_now() { return clock64(); }
// phase timestamps of a row (SM cycles), thread 0 only
#define TG_T(row, slot) do { if (g_dbg && threadIdx.x == 0) g_dbg[(row) * 32 + 8 + (slot)] = (double)tg_now(); } while (0)
#define TG_TF(slot) TG_T(sm.misc.dbg_row, slot)
#else
#define TG_TF(slot) do { } while (0)
#define TG_GIVEUP(bit) do { } while (0)
#define TG_T(row, slot) do { } while (0)
#endif

constexpr int kMaxRowsPerCta = kThreads;   // rows one CTA owns in one launch (the host splits larger batches)
constexpr int kEvCap = 4096;               // flagged units a row may list

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier + 1-D bulk copy global -> shared
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Shared-memory atomic add with acquire-release ordering at block scope.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 1-D bulk copy global -> shared, completing on `bar`.  No eviction hint:
// the row stays in L2 for the reads at the end of the row.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Bounded wait: false after ~1 s without completion.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > kWaitLimitCycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Shared-memory layout of select_kernel:
//   [SelSmem up to `fin`] [fin | row bitmaps M, N (aliased)] [stage ring]
// The bitmaps are needed until the marked tokens of a row are merged;
// FinSmem only after that; the rare paths that need the bitmaps afterwards
// rebuild them.
// ---------------------------------------------------------------------------
constexpr int kMaxStages = 8;

struct Misc {
  unsigned long long full[kMaxStages];   // stage loaded (one arrive + the copy's transaction bytes)
  unsigned cnt[kMaxStages];              // warps done with each stage (grows by 16 per use)
  int iss[kMaxStages];                   // copies issued into each stage
  int nrow;                              // streamed rows of this CTA
  int ncand;                             // candidates in the list
  unsigned lctr;                         // counter of the marked-token list while it is built
  int error;                             // a wait timed out; the kernel stops loading
  int err_snap;                          // thread 0's snapshot of `error`, read by all threads
  int gcause;                            // debug builds: why a row left the one-pass path
  int dbg_row;                           // debug builds: the row being finished
  float wf[kWarps];                      // per-warp scratch
  unsigned wu[kWarps];
  unsigned lvl[kWarps][4];               // first sub-chunk: packed counts per level of 2 below m0
  unsigned sfilt[kStateFilterWords];     // the row's state ids, as a 1,024-bit filter
  int nfst;                              // forced rows with a state of this CTA (after the streamed ones)
};

constexpr int kLevels = 1024;   // value levels between the lowest candidate and the row max
constexpr int kGroupCap = 256;  // largest level group sorted exactly in shared memory

struct FinSmem {
  unsigned long long lm[kLevels];  // weight of each level
  unsigned lc[kLevels];            // items in each level
  unsigned lw[3][kLevels];         // the weights in three 15-bit limbs (exact sums with 32-bit atomics)
  unsigned gk[kGroupCap];          // gathered group: key, index, weight
  unsigned gi[kGroupCap];
  unsigned long long gw[kGroupCap];
  unsigned sk[kGroupCap];          // the group sorted by (key desc, index asc)
  unsigned si[kGroupCap];
  unsigned long long sw[kGroupCap];
  unsigned long long wsum[kWarps]; // per-warp partial sums of a block scan
  unsigned wcnt[kWarps];
  unsigned short clv[kCandCap];    // level of each candidate
  int gn;
  int fb;                          // broadcast: bucket / position
  unsigned long long fbefore;      // broadcast: mass or count before it
  int ffound;
  int lastne;                      // last non-empty level (a search that finds nothing)
  unsigned long long fmass;        // broadcast: mass before the found level
};

struct SelSmem {
  float cand_s[kCandCap];
  unsigned cand_i[kCandCap];
  int rows[kMaxRowsPerCta];   // this CTA's streamed rows, in order
  unsigned ev[kEvCap];         // flagged units, then marked tokens, of the row being finished
  Hist hist;
  RedScratch red;
  Misc misc;
  FinSmem fin;   // last: the row bitmaps alias it and may run past its end
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int bitmap_bytes(int nwords) { return align_up(nwords * 4, 128); }
__host__ __device__ constexpr int fin_offset() { return static_cast<int>(offsetof(SelSmem, fin)); }
__host__ __device__ constexpr int union_bytes(int nwords) {
  return align_up(static_cast<int>(sizeof(FinSmem)) > 2 * bitmap_bytes(nwords) ? static_cast<int>(sizeof(FinSmem))
                                                                                : 2 * bitmap_bytes(nwords),
                  128);
}
__host__ __device__ constexpr int ring_offset(int nwords) { return align_up(fin_offset() + union_bytes(nwords), 128); }

// Sources for the radix engine -----------------------------------------------
struct CandSource {
  const float* s;
  const unsigned* idx;
  int n;
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    for (int i = threadIdx.x; i < n; i += kThreads) f(s[i], idx[i]);
  }
};

template <int DT>
__device__ __forceinline__ float load_logit(const void* row, int i) {
  if (DT == kF32) return __ldg(static_cast<const float*>(row) + i);
  return __uint_as_float(static_cast<unsigned>(__ldg(static_cast<const unsigned short*>(row) + i)) << 16);
}

template <int DT>
struct RowGlobalSource {
  const void* row;
  int V;
  const DevCfg* c;
  const unsigned* H;
  const unsigned* N;
  bool bitmaps;
  bool sample;
  // rows with the task's processors (state_kernel): P marks the state ids
  // and forced ids; a token in neither H nor P is plain (or F when forced)
  bool prow = false;
  bool forced = false;
  bool sparse = false;   // a forced row: only its tokens above F (final scores, listed once)
  const unsigned* P = nullptr;
  float temp = 1.0f;
  const float* sp_s = nullptr;
  const unsigned* sp_i = nullptr;
  int sp_n = 0;
  __device__ __forceinline__ void state_row(const DevCfg& cr) {
    prow = cr.prow;
    forced = cr.forced_row;
    sparse = cr.sparse_row;
    P = cr.pbits;
    temp = cr.temp;
    sp_s = cr.sp_s;
    sp_i = cr.sp_i;
    sp_n = cr.sp_n;
  }
  __device__ __forceinline__ float score(float x, int i) const {
    if (prow) {
      float s;
      if (get_bit(H, i) || get_bit(P, i)) s = process_state_elem(*c, H, N, x, i);
      else s = forced ? kFilter : x;
      if (sample && temp != 1.0f) s = clampf(__fdiv_rn(s, temp));
      return s;
    }
    if (bitmaps) return process_elem(*c, H, N, x, i, sample);
    if (sample && c->temp != 1.0f) return clampf(__fdiv_rn(x, c->temp));
    return x;
  }
  // Every token of the row once.  A 16-byte aligned row is read a vector
  // (16 bytes) per thread at a time, four vectors in flight; the tail and an
  // unaligned row element by element.
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    if (sparse) {
      // every other token scores F and weighs nothing: the listed ones only
      for (int j = threadIdx.x; j < sp_n; j += kThreads) f(sp_s[j], sp_i[j]);
      return;
    }
    constexpr int PER = DT == kF32 ? 4 : 8;
    constexpr int NV = 4;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) {
      const int nvec = V / PER;
      const uint4* rv = static_cast<const uint4*>(row);
      for (int v0 = 0; v0 < nvec; v0 += NV * kThreads) {
        uint4 q[NV];
        int vi[NV];
#pragma unroll
        for (int h = 0; h < NV; ++h) {
          vi[h] = v0 + h * kThreads + static_cast<int>(threadIdx.x);
          q[h] = vi[h] < nvec ? __ldg(rv + vi[h]) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll 1
        for (int h = 0; h < NV; ++h) {
          if (vi[h] < nvec) {
            uint4 v = q[0];
#pragma unroll
            for (int hh = 1; hh < NV; ++hh) v = hh == h ? q[hh] : v;
            const unsigned ps[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < PER; ++e) {
              const float x = DT == kF32 ? __uint_as_float(ps[e]) : ((e & 1) ? bf16hi(ps[e >> 1]) : bf16lo(ps[e >> 1]));
              const int i = vi[h] * PER + e;
              f(score(x, i), static_cast<unsigned>(i));
            }
          }
        }
      }
      done = nvec * PER;
    }
    for (int i = done + static_cast<int>(threadIdx.x); i < V; i += kThreads) f(score(load_logit<DT>(row, i), i), static_cast<unsigned>(i));
  }
};

// ---------------------------------------------------------------------------
// warp-level helpers (all 32 lanes, converged)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// Exact selection over the candidate list (all tokens with s >= theta).
//
// One pass sorts every candidate into one of kLevels value levels between
// the lowest candidate and the row maximum (level = floor((m - s) * inv),
// monotone in s) and sums each level's fixed-point weight.  A warp scan over
// the levels finds the level that holds the k-th token, the top-p cut or the
// draw; only that level's tokens are gathered and sorted exactly by (key
// desc, index asc).  A level larger than kGroupCap runs the generic radix
// selection over its members instead.
// ---------------------------------------------------------------------------
struct LevelMap {
  float m, inv;
  __device__ __forceinline__ int operator()(float s) const {
    float l = (m - s) * inv;
    return static_cast<int>(fminf(fmaxf(l, 0.0f), static_cast<float>(kLevels - 1)));
  }
};

// Candidates of one level (and key >= klo), as a radix-engine source.
struct CandLevelSource {
  const float* s;
  const unsigned* idx;
  int n;
  LevelMap lv;
  int level;
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      float v = s[i];
      if (lv(v) == level) f(v, idx[i]);
    }
  }
};

// Gather the candidates of `level` with key >= klo into fin.g*, then sort
// them into fin.s*.  Returns the group size, or -1 when it exceeds kGroupCap.
__device__ int gather_sort_level(SelSmem& sm, int n, const LevelMap& lv, int level, unsigned klo, float cc) {
  FinSmem& f = sm.fin;
  if (threadIdx.x == 0) f.gn = 0;
  csync();
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    bool has = false;
    float s = 0.0f;
    unsigned key = 0u;
    if (i < n) {
      s = sm.cand_s[i];
      key = fkey(s);
      has = lv(s) == level && key >= klo;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, has);
    if (bal) {
      const int lane = threadIdx.x & 31;
      const int leader = __ffs(bal) - 1;
      int pos = 0;
      if (lane == leader) pos = atomicAdd(&f.gn, __popc(bal));
      pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(bal & ((1u << lane) - 1u));
      if (has && pos < kGroupCap) { f.gk[pos] = key; f.gi[pos] = sm.cand_i[i]; f.gw[pos] = wfix_fast(s, cc); }
    }
  }
  csync();
  const int gn = f.gn;
  if (gn > kGroupCap) return -1;
  for (int t = threadIdx.x; t < gn; t += kThreads) {
    const unsigned kt = f.gk[t], it = f.gi[t];
    int r = 0;
    for (int j = 0; j < gn; ++j) {
      const unsigned kj = f.gk[j];
      r += (kj > kt) || (kj == kt && f.gi[j] < it);
    }
    f.sk[r] = kt;
    f.si[r] = it;
    f.sw[r] = f.gw[t];
  }
  csync();
  return gn;
}

// One warp: the first sorted position j < cnt where base + sum(sw[0..j])
// reaches the target (>= or >).  Writes fin.fb = j (or cnt-1 when never),
// fin.fbefore = base + sum(sw[0..j-1]), fin.ffound.  The warp scans 32
// positions at a time (lane = position within the chunk).
__device__ __forceinline__ void walk_sorted(SelSmem& sm, int cnt, unsigned long long base,
                                            unsigned long long target, bool strict) {
  FinSmem& f = sm.fin;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long run = base;
    bool done = false;
    for (int c0 = 0; c0 < cnt && !done; c0 += 32) {
      const int q = c0 + lane;
      const unsigned long long w = q < cnt ? f.sw[q] : 0ull;
      unsigned long long incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned long long tot = run + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, q < cnt && (strict ? tot > target : tot >= target));
      if (hit) {
        const int L = __ffs(hit) - 1;
        if (lane == L) {
          f.fb = q;
          f.fbefore = tot - w;
          f.ffound = 1;
        }
        done = true;
      } else {
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (!done && lane == 0) {
      unsigned long long all = base;
      for (int j = 0; j + 1 < cnt; ++j) all += f.sw[j];
      f.fb = cnt - 1;
      f.fbefore = all;
      f.ffound = 0;
    }
  }
  csync();
}

// End of a row, listed marked tokens: entry j of list[0..n) (t and the
// banned / plain flags) is read back from global memory and passed to
// fn(x, t, entry, j).
// Thread t takes entries t, t + kThreads, ... four at a time with the four
// reads in flight.
template <int DT, class Fn>
__device__ __forceinline__ void for_listed(const unsigned* list, int n, const unsigned char* rowp, Fn fn) {
  constexpr int kMB = 4;
  for (int j0 = 0; j0 < n; j0 += kMB * kThreads) {
    unsigned e[kMB];
    float xs[kMB];
#pragma unroll
    for (int q = 0; q < kMB; ++q) {
      const int j = j0 + q * kThreads + static_cast<int>(threadIdx.x);
      e[q] = j < n ? list[j] : 0xffffffffu;
    }
#pragma unroll
    for (int q = 0; q < kMB; ++q) xs[q] = e[q] != 0xffffffffu ? load_logit<DT>(rowp, static_cast<int>(e[q] & kIdMask)) : 0.0f;
#pragma unroll
    for (int q = 0; q < kMB; ++q)
      if (e[q] != 0xffffffffu)
        fn(xs[q], static_cast<int>(e[q] & kIdMask), e[q], j0 + q * kThreads + static_cast<int>(threadIdx.x));
  }
}

// Block-wide search over the levels: the first level l where the running
// sum of fin.lm reaches the target (Reached); fin.fb = l, fin.fbefore = the
// sum of the levels before l, fin.ffound = 1.  When no level reaches it:
// fin.fb = the last non-empty level, fin.fbefore = the sum before it,
// fin.ffound = 0.  Every thread calls; thread t owns levels 2t and 2t+1.
template <class T, class Reached>
__device__ __forceinline__ void level_find(SelSmem& sm, const T* vals, Reached r) {
  static_assert(kLevels == 2 * kThreads, "two levels per thread");
  FinSmem& f = sm.fin;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned long long v0 = vals[2 * tid], v1 = vals[2 * tid + 1];
  const bool ne0 = f.lc[2 * tid] != 0u, ne1 = f.lc[2 * tid + 1] != 0u;
  const unsigned long long local = v0 + v1;
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) f.wsum[wid] = incl;
  if (tid == 0) { f.ffound = 0; f.lastne = -1; }
  csync();
  unsigned long long before = 0ull;
  for (int q = 0; q < wid; ++q) before += f.wsum[q];
  const unsigned long long excl = before + incl - local;
  if (r(excl + local) && (tid == 0 || !r(excl))) {
    if (r(excl + v0)) { f.fb = 2 * tid; f.fbefore = excl; }
    else { f.fb = 2 * tid + 1; f.fbefore = excl + v0; }
    f.ffound = 1;
  }
  csync();
  if (!f.ffound) {
    // nothing reached the target: the last non-empty level
    int last = ne1 ? 2 * tid + 1 : (ne0 ? 2 * tid : -1);
    for (int o = 16; o; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0 && last >= 0) atomicMax(&f.lastne, last);
    csync();
    const int L = f.lastne;
    if (L >= 0 && (L >> 1) == tid) {
      f.fb = L;
      f.fbefore = (L & 1) ? excl + v0 : excl;
    }
    csync();
  }
}
template <class Reached>
__device__ __forceinline__ void level_find_mass(SelSmem& sm, Reached r) { level_find(sm, sm.fin.lm, r); }

// Keep only levels < L in full and the first `mass`/`cnt` of level L.
__device__ __forceinline__ void level_limit(SelSmem& sm, int L, unsigned long long mass, unsigned cnt) {
  for (int l = threadIdx.x; l < kLevels; l += kThreads) {
    if (l > L) { sm.fin.lm[l] = 0ull; sm.fin.lc[l] = 0u; }
    else if (l == L) { sm.fin.lm[l] = mass; sm.fin.lc[l] = cnt; }
  }
  csync();
}

struct FinResult {
  bool ok;                 // false: the candidates cannot decide this row
  int reason;
  unsigned token;
  float score;             // the token's processed score
  unsigned long long S;    // mass of the kept set (weights relative to the row maximum)
};

// top_k, top_p and the draw over the candidates.  Z_all = fixed-point mass
// of every token of the row (candidates included), relative to m.
__device__ __noinline__ FinResult finalize_candidates(const DevCfg& c, SelSmem& sm, float m, float lo,
                                                      unsigned long long Z_all, float u, bool topk, bool topp) {
  const float cc = m * kLog2e;
  const WFast wf{cc};
  FinResult res{false, 0, 0u};
  FinSmem& f = sm.fin;
  const int n = min(sm.misc.ncand, kCandCap);
  if (n <= 0) { res.reason = 9; return res; }
  // level map from the threshold (every candidate is at or above it) to the maximum
  TG_TF(8);
  const float range = m - lo;
  LevelMap lv{m, range > 0.0f ? static_cast<float>(kLevels - 1) / range : 0.0f};
  for (int l = threadIdx.x; l < kLevels; l += kThreads) { f.lc[l] = 0u; f.lw[0][l] = 0u; f.lw[1][l] = 0u; f.lw[2][l] = 0u; }
  csync();
  unsigned long long zc = 0ull;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const float s = sm.cand_s[i];
    const int l = lv(s);
    const unsigned long long w = wfix_fast(s, cc);   // <= 2^44
    zc += w;
    atomicAdd(&f.lc[l], 1u);
    atomicAdd(&f.lw[0][l], static_cast<unsigned>(w & 0x7fffull));
    atomicAdd(&f.lw[1][l], static_cast<unsigned>((w >> 15) & 0x7fffull));
    atomicAdd(&f.lw[2][l], static_cast<unsigned>(w >> 30));
  }
  csync();
  for (int l = threadIdx.x; l < kLevels; l += kThreads)
    f.lm[l] = static_cast<unsigned long long>(f.lw[0][l]) + (static_cast<unsigned long long>(f.lw[1][l]) << 15) +
              (static_cast<unsigned long long>(f.lw[2][l]) << 30);
  const unsigned long long Zc = block_sum_u64(zc, &sm.red);
  TG_TF(9);
  unsigned klo = 0u;
  unsigned long long Z;
  if (topk) {
    if (n < c.top_k) { res.reason = 4; return res; }
    // level holding the k-th largest token
    const unsigned long long need = static_cast<unsigned long long>(c.top_k);
    level_find(sm, f.lc, [need](unsigned long long x) { return x >= need; });
    const int Lk = f.fb;
    const unsigned rank = static_cast<unsigned>(c.top_k) - static_cast<unsigned>(f.fbefore);
    const int gn = gather_sort_level(sm, n, lv, Lk, 0u, cc);
    unsigned long long kept_mass = 0ull;
    unsigned kept_cnt = 0u;
    if (gn >= 0) {
      klo = f.sk[rank - 1];
      for (int j = 0; j < gn; ++j)
        if (f.sk[j] >= klo) { kept_mass += f.sw[j]; ++kept_cnt; }
    } else {
      CandLevelSource ls{sm.cand_s, sm.cand_i, n, lv, Lk};
      KeepFilter none{0u, false, 0u, 0u};
      klo = kth_key(ls, none, rank, &sm.hist);
      KeepFilter kf{klo, false, 0u, 0u};
      kept_mass = mass_sum(ls, kf, wf, &sm.red);
      kept_cnt = count_items(ls, kf, &sm.red);
    }
    csync();
    level_limit(sm, Lk, kept_mass, kept_cnt);
    Z = 0ull;
    for (int l = threadIdx.x; l < kLevels; l += kThreads) Z += f.lm[l];
    Z = block_sum_u64(Z, &sm.red);
  } else {
    Z = Z_all > Zc ? Z_all : Zc;
  }
  unsigned long long S = Z;
  int Lc = kLevels;          // level of the cut (kLevels: no cut)
  int nc = 0;                // kept members of the cut level, in sorted order
  bool cut_sorted = false;
  KeepFilter keep{klo, false, 0u, 0u};
  if (topp) {
    const unsigned long long T = topp_target(c.top_p, Z);
    if (!topk && Zc < T) { res.reason = 5; return res; }
    level_find_mass(sm, [T](unsigned long long x) { return x >= T; });
    TG_TF(10);
    if (!f.ffound) { res.reason = 6; return res; }
    Lc = f.fb;
    const unsigned long long before = f.fbefore;
    csync();
    const int gn = gather_sort_level(sm, n, lv, Lc, klo, cc);
    TG_TF(11);
    unsigned long long inlevel;
    if (gn >= 0) {
      walk_sorted(sm, gn, before, T, false);
      nc = f.fb + 1;
      S = f.fbefore + f.sw[f.fb];
      inlevel = S - before;
      keep.cut = true; keep.kcut = f.sk[f.fb]; keep.icut = f.si[f.fb];
      cut_sorted = true;
    } else {
      CandLevelSource ls{sm.cand_s, sm.cand_i, n, lv, Lc};
      MassSel cs = mass_select(ls, keep, wf, T - before, false, &sm.hist);
      if (!cs.found) { res.reason = 6; return res; }
      keep.cut = true; keep.kcut = cs.key; keep.icut = cs.idx;
      S = before + cs.mass;
      inlevel = cs.mass;
      nc = static_cast<int>(count_items(ls, keep, &sm.red));
    }
    csync();
    level_limit(sm, Lc, inlevel, static_cast<unsigned>(nc));
    TG_TF(12);
  }
  const unsigned long long Td = draw_target(u, S);
  if (!topk && !topp && !(Zc > Td)) { res.reason = 7; return res; }
  level_find_mass(sm, [Td](unsigned long long x) { return x > Td; });
  TG_TF(13);
  if (!f.ffound) { res.reason = 8; return res; }
  const int Ld = f.fb;
  const unsigned long long before = f.fbefore;
  csync();
  if (Ld == Lc && cut_sorted) {
    walk_sorted(sm, nc, before, Td, true);
    res.token = f.si[f.fb];
    res.score = key2f(f.sk[f.fb]);
  } else {
    const int gn = gather_sort_level(sm, n, lv, Ld, klo, cc);
    if (gn >= 0) {
      const int lim = (Ld == Lc) ? nc : gn;
      walk_sorted(sm, lim, before, Td, true);
      res.token = f.si[f.fb];
      res.score = key2f(f.sk[f.fb]);
    } else {
      CandLevelSource ls{sm.cand_s, sm.cand_i, n, lv, Ld};
      MassSel d = mass_select(ls, keep, wf, Td - before, true, &sm.hist);
      if (!d.found) { res.reason = 8; return res; }
      res.token = d.idx;
      res.score = key2f(d.key);
    }
  }
  res.S = S;
  csync();
  TG_TF(14);
  res.ok = true;
  return res;
}

// ---------------------------------------------------------------------------
// Per-warp slice work.  Warp w owns elements [w*SW, (w+1)*SW) of every
// sub-chunk (SW = SE / kWarps: 1024 bf16 or 512 f32, i.e. 2 KB).  Lane l
// holds the slice's 16-byte vectors l, l+32, l+64 and l+96 in registers;
// element e = i*PER + j of the lane is token tok0 + (lane + 32 i)*PER + j.
// ---------------------------------------------------------------------------
struct Slice {
  uint4 q[4];
  int nv;    // vectors of the slice inside the row
};

template <int DT>
__device__ __forceinline__ void load_slice(const unsigned char* stage, int soff, int scnt, Slice& sl) {
  constexpr int PER = DT == kF32 ? 4 : 8;
  const int lane = threadIdx.x & 31;
  const uint4* v4 = reinterpret_cast<const uint4*>(stage + soff * (DT == kF32 ? 4 : 2));
  sl.nv = scnt / PER;
  const unsigned fill = DT == kF32 ? 0xff800000u : 0xff80ff80u;   // -inf
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = lane + 32 * i;
    sl.q[i] = v < sl.nv ? v4[v] : make_uint4(fill, fill, fill, fill);
  }
}

// The slice's raw logits as f32 (padding is -inf).
template <int DT>
__device__ __forceinline__ void slice_values(const Slice& sl, float (&x)[DT == kF32 ? 16 : 32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned ps[4] = {sl.q[i].x, sl.q[i].y, sl.q[i].z, sl.q[i].w};
    if (DT == kF32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) x[i * 4 + j] = __uint_as_float(ps[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[i * 8 + j] = (j & 1) ? bf16hi(ps[j >> 1]) : bf16lo(ps[j >> 1]);
    }
  }
}

// Bits of the lane's elements that the bitmap marks (bit e for element e).
template <int DT>
__device__ __forceinline__ unsigned slice_marks(const Slice& sl, int tok0, const unsigned* M) {
  constexpr int PER = DT == kF32 ? 4 : 8;
  const int lane = threadIdx.x & 31;
  unsigned mk = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = lane + 32 * i;
    if (v < sl.nv) {
      const int t = tok0 + v * PER;   // PER divides 32, so the vector's bits share one word
      mk |= ((M[t >> 5] >> (t & 31)) & ((1u << PER) - 1u)) << (i * PER);
    }
  }
  return mk;
}

template <int NE>
__device__ __forceinline__ float tree_max(const float (&x)[NE]) {
  float t[NE / 2];
#pragma unroll
  for (int j = 0; j < NE / 2; ++j) t[j] = fmaxf(x[j], x[j + NE / 2]);
#pragma unroll
  for (int w = NE / 4; w >= 1; w >>= 1) {
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
  }
  return t[0];
}

// Greedy: the lane's best (score, lowest index) over its unmarked tokens.
// The lane's tokens increase with e, so only a strictly larger maximum
// replaces the best, and the lowest e holding it wins.
template <int DT>
__device__ __forceinline__ void slice_greedy(const Slice& sl, int tok0, const unsigned* M, bool bitmaps, float& bv,
                                             unsigned& bi) {
  constexpr int PER = DT == kF32 ? 4 : 8;
  constexpr int NE = 4 * PER;
  const int lane = threadIdx.x & 31;
  float x[NE];
  slice_values<DT>(sl, x);
  if (bitmaps) {
    const unsigned mk = slice_marks<DT>(sl, tok0, M);
#pragma unroll
    for (int e = 0; e < NE; ++e) x[e] = ((mk >> e) & 1u) ? -INFINITY : x[e];
  }
  const float vm = tree_max<NE>(x);
  if (vm > bv) {
    int ee = NE - 1;
#pragma unroll
    for (int e = NE - 2; e >= 0; --e) ee = x[e] == vm ? e : ee;
    bv = vm;
    bi = static_cast<unsigned>(tok0 + (lane + 32 * (ee / PER)) * PER + (ee % PER));
  }
}

// Error-free sum hi + x = s + e (Knuth's TwoSum); the lane's running mass.
__device__ __forceinline__ void acc_add(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  hi = s;
  lo = __fadd_rn(lo, e);
}

// Units of eight elements: a lane's slice holds four (bf16: one vector each)
// or two (f32: vectors i and i+1 of the lane).  Unit u covers elements
// 8u .. 8u+7 of the lane's slice.
template <int DT>
struct Units {
  static constexpr int kPerSlice = DT == kF32 ? 2 : 4;
};

// Sampling: the lane's raw weights 2^(x*ascale - ccl) over its unmarked tokens join (ah, al); bit
// k*UPS + u of emask is set when unit u of the lane's slice in sub-chunk k
// holds a logit at or above theta_raw.  ccl is the lane's own reference
// (first the block's m0 * ascale): when a slice's maximum lies more than 64
// binary orders above it, the lane rebases its mass to that maximum, so
// heavy-tailed rows whose maximum comes late cannot overflow.
template <int DT>
__device__ __forceinline__ void slice_sample(const Slice& sl, int tok0, const unsigned* M, bool bitmaps, float ascale,
                                             float& ccl, float theta_raw, int k, float& ah, float& al, float& mxt,
                                             unsigned long long& emask) {
  constexpr int NE = DT == kF32 ? 16 : 32;
  constexpr int UPS = Units<DT>::kPerSlice;
  float x[NE];
  slice_values<DT>(sl, x);
  if (bitmaps) {
    // marked tokens are merged exactly at the end of the row: they count nothing here
    const unsigned mk = slice_marks<DT>(sl, tok0, M);
#pragma unroll
    for (int e = 0; e < NE; ++e) x[e] = ((mk >> e) & 1u) ? -INFINITY : x[e];
  }
  float um[UPS];
#pragma unroll
  for (int u = 0; u < UPS; ++u) {
    float t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = fmaxf(x[8 * u + j], x[8 * u + j + 4]);
    um[u] = fmaxf(fmaxf(t[0], t[2]), fmaxf(t[1], t[3]));
  }
  float vm = um[0];
  unsigned bits = um[0] >= theta_raw ? 1u : 0u;
#pragma unroll
  for (int u = 1; u < UPS; ++u) {
    vm = fmaxf(vm, um[u]);
    bits |= (um[u] >= theta_raw ? 1u : 0u) << u;
  }
  mxt = fmaxf(mxt, vm);
  const float top = vm * ascale;
  if (top - ccl > 64.0f) {
    const float f = ex2_approx(ccl - top);
    ah *= f;
    al *= f;
    ccl = top;
  }
  const float2 A = make_float2(ascale, ascale);
  const float2 C = make_float2(-ccl, -ccl);
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int e = 0; e < NE; e += 2) {
    float2 w = __ffma2_rn(make_float2(x[e], x[e + 1]), A, C);
    w.x = ex2_approx(w.x);
    w.y = ex2_approx(w.y);
    acc[(e >> 1) & 3] = __fadd2_rn(acc[(e >> 1) & 3], w);
  }
  const float2 t = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  acc_add(ah, al, t.x + t.y);
  emask |= static_cast<unsigned long long>(bits) << (k * UPS);
}

// First sub-chunk: per level l = floor((m0 - x) * inv_w), counts of levels
// 0..7 summed over the warp, as four words of two 16-bit counts
// (cw[0] = levels 0 and 2, cw[1] = 1 and 3, cw[2] = 4 and 6, cw[3] = 5 and 7).
template <int DT>
__device__ __forceinline__ void slice_level_counts(const Slice& sl, float m0, float inv_w, unsigned (&cw)[4]) {
  constexpr int NE = DT == kF32 ? 16 : 32;
  float x[NE];
  slice_values<DT>(sl, x);
  // one 8-bit field per level 0..7 in a 64-bit word (at most 32 per lane); level 8 = below
  unsigned long long f = 0ull;
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int l = static_cast<int>(fminf((m0 - x[e]) * inv_w, 8.0f));
    f += l < 8 ? (1ull << (8 * l)) : 0ull;
  }
  const unsigned lo4 = static_cast<unsigned>(f), hi4 = static_cast<unsigned>(f >> 32);
  unsigned v[4] = {lo4 & 0x00ff00ffu, (lo4 >> 8) & 0x00ff00ffu, hi4 & 0x00ff00ffu, (hi4 >> 8) & 0x00ff00ffu};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    for (int o = 16; o; o >>= 1) v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
    cw[q] = v[q];
  }
}

// Element e (0 .. N-1) of a register array, without dynamic indexing.
template <int N>
__device__ __forceinline__ float pick_n(const float (&s)[N], int e) {
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = s[i];
#pragma unroll
  for (int w = N / 2, b = 0; w >= 1; w >>= 1, ++b) {
    const bool hi = (e >> b) & 1;
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = hi ? t[2 * i + 1] : t[2 * i];
  }
  return t[0];
}

// Append (s, t) to the block's candidate list for every lane with `ok`.
__device__ __forceinline__ void push_candidate(SelSmem& sm, bool ok, float s, unsigned t) {
  const int lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  if (!bal) return;
  const int leader = __ffs(bal) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(&sm.misc.ncand, __popc(bal));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (ok) {
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = t; }
  }
}

// Append (s, t) for every set bit e of cm (s = sv[e], t = tok[e]) to the
// block's candidate list: one reservation per warp, then each lane writes
// its own.  Every lane of the warp calls.
__device__ __forceinline__ void push_units(SelSmem& sm, unsigned cm, const float (&sv)[8], const unsigned (&tok)[8]) {
  const int lane = threadIdx.x & 31;
  const int cnt = __popc(cm);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total == 0) return;
  int base = 0;
  if (lane == 31) base = atomicAdd(&sm.misc.ncand, total);
  base = __shfl_sync(0xffffffffu, base, 31);
  int pos = base + incl - cnt;
  while (cm) {
    const int e = __ffs(cm) - 1;
    cm &= cm - 1u;
    if (pos < kCandCap) {
      float v = sv[0];
      unsigned ti = tok[0];
#pragma unroll
      for (int q = 1; q < 8; ++q) {
        v = e == q ? sv[q] : v;
        ti = e == q ? tok[q] : ti;
      }
      sm.cand_s[pos] = v;
      sm.cand_i[pos] = ti;
    }
    ++pos;
  }
}

// End of a sampled row: the units that lanes flagged while streaming, as one
// list for the block (entry = k << 11 | warp << 7 | lane << 2 | unit).
// Returns the number of flagged units (the list holds at most kEvCap).
template <int DT>
__device__ __forceinline__ int list_flagged(SelSmem& sm, unsigned long long emask) {
  constexpr int UPS = Units<DT>::kPerSlice;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int cnt = __popcll(emask);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.misc.wu[wid] = static_cast<unsigned>(incl);
  csync();
  int base = 0, total = 0;
  for (int q = 0; q < kWarps; ++q) {
    const int cq = static_cast<int>(sm.misc.wu[q]);
    base += q < wid ? cq : 0;
    total += cq;
  }
  int pos = base + incl - cnt;
  const unsigned tag = static_cast<unsigned>((wid << 7) | (lane << 2));
  // the two halves in turn: 32-bit bit scans are half the work of 64-bit ones
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    unsigned bits = static_cast<unsigned>(half ? (emask >> 32) : emask);
    while (bits) {
      const unsigned b = static_cast<unsigned>(__ffs(bits) - 1) + 32u * half;
      bits &= bits - 1u;
      if (pos < kEvCap) sm.ev[pos] = ((b / UPS) << 11) | tag | (b % UPS);
      ++pos;
    }
  }
  csync();
  return total;
}

// Read units back (from L2), eight logits each, and append every unmarked
// token whose processed score reaches theta_f (its raw logit is at or above
// theta_raw).  The units are the listed ones (nev of them), or with `every`
// all units of the row.  Thread t takes entries t, t + kThreads, ...; a batch
// issues all of its reads first, then reserves room for all of its
// candidates with one warp-wide reservation.  Every thread calls.
template <int DT>
__device__ void expand_units(const DevCfg& c, SelSmem& sm, const unsigned char* rowp, int V, int nev, bool every,
                             const unsigned* M, bool bitmaps, float theta_raw, float theta_f, bool temp_on) {
  constexpr int esz = DT == kF32 ? 4 : 2;
  constexpr int PER = DT == kF32 ? 4 : 8;
  constexpr int SE = kStageBytes / esz;
  constexpr int SW = SE / kWarps;
  constexpr int UPS = Units<DT>::kPerSlice;
  constexpr int NQ = DT == kF32 ? 2 : 1;    // 16-byte vectors per unit
  constexpr int B = DT == kF32 ? 4 : 8;     // entries per thread per batch (B * 8 candidate bits <= 64)
  const int lane = threadIdx.x & 31;
  const int nsub = (V + SE - 1) / SE;
  const int n = every ? (nsub << 11) : min(nev, kEvCap);
  const unsigned fill = DT == kF32 ? 0xff800000u : 0xff80ff80u;
  for (int j0 = 0; j0 < n; j0 += B * kThreads) {
    const int nb = min(B, (n - j0 + kThreads - 1) / kThreads);   // uniform
    uint4 q[B][NQ];
    int t0[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      t0[b] = -1;
#pragma unroll
      for (int h = 0; h < NQ; ++h) q[b][h] = make_uint4(fill, fill, fill, fill);
      const int j = j0 + b * kThreads + static_cast<int>(threadIdx.x);
      if (b < nb && j < n) {
        const unsigned en = every ? static_cast<unsigned>(j) : sm.ev[j];
        const int kk = static_cast<int>(en >> 11), w = static_cast<int>((en >> 7) & 15u);
        const int ln = static_cast<int>((en >> 2) & 31u), uu = static_cast<int>(en & 3u);
        const int nv = max(0, min(SW, min(SE, V - kk * SE) - w * SW)) / PER;   // vectors inside the row
        const int base = kk * SE + w * SW;
        const int v0 = ln + 32 * (NQ * uu);
        if (uu < UPS && v0 < nv) {
          t0[b] = base + v0 * PER;
#pragma unroll
          for (int h = 0; h < NQ; ++h)
            if (v0 + 32 * h < nv)
              q[b][h] = __ldg(reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(base + (v0 + 32 * h) * PER) * esz));
        }
      }
    }
    unsigned long long cmall = 0ull;
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (b < nb && t0[b] >= 0) {
        float x[8];
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          const unsigned ps[4] = {q[b][h].x, q[b][h].y, q[b][h].z, q[b][h].w};
#pragma unroll
          for (int e = 0; e < 8 / NQ; ++e)
            x[h * (8 / NQ) + e] = DT == kF32 ? __uint_as_float(ps[e]) : ((e & 1) ? bf16hi(ps[e >> 1]) : bf16lo(ps[e >> 1]));
        }
        unsigned cm = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) cm |= (x[e] >= theta_raw ? 1u : 0u) << e;
        if (bitmaps && cm) {
          unsigned mk;
          if (DT == kF32) {
            const int a0 = t0[b], a1 = t0[b] + 32 * PER;
            mk = (M[a0 >> 5] >> (a0 & 31)) & 15u;
            if (cm >> 4) mk |= ((M[a1 >> 5] >> (a1 & 31)) & 15u) << 4;
          } else {
            mk = (M[t0[b] >> 5] >> (t0[b] & 31)) & 255u;
          }
          cm &= ~mk;
        }
        if (temp_on && cm) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if ((cm >> e) & 1u) x[e] = clampf(__fdiv_rn(x[e], c.temp));
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cm &= ~((x[e] >= theta_f ? 0u : 1u) << e);
        cmall |= static_cast<unsigned long long>(cm) << (8 * b);
      }
    }
    // one reservation per warp for all of this batch's candidates
    const int cnt = __popcll(cmall);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) continue;
    int base = 0;
    if (lane == 31) base = atomicAdd(&sm.misc.ncand, total);
    base = __shfl_sync(0xffffffffu, base, 31);
    int pos = base + incl - cnt;
    while (cmall) {
      const int bit = __ffsll(static_cast<long long>(cmall)) - 1;
      cmall &= cmall - 1ull;
      const int b = bit >> 3, e = bit & 7;
      const int h = e / (8 / NQ), ee = e % (8 / NQ);
      uint4 v = q[0][0];
      int tb = t0[0];
#pragma unroll
      for (int bb = 0; bb < B; ++bb)
#pragma unroll
        for (int hh = 0; hh < NQ; ++hh)
          if (bb == b && hh == h) { v = q[bb][hh]; tb = t0[bb]; }
      const unsigned wsel = (ee >> (DT == kF32 ? 0 : 1)) == 0 ? v.x : (ee >> (DT == kF32 ? 0 : 1)) == 1 ? v.y
                          : (ee >> (DT == kF32 ? 0 : 1)) == 2 ? v.z : v.w;
      float xv = DT == kF32 ? __uint_as_float(wsel) : ((ee & 1) ? bf16hi(wsel) : bf16lo(wsel));
      if (temp_on) xv = clampf(__fdiv_rn(xv, c.temp));
      if (pos < kCandCap) {
        sm.cand_s[pos] = xv;
        sm.cand_i[pos] = static_cast<unsigned>(tb + h * 32 * PER + ee);
      }
      ++pos;
    }
  }
}

// End of a row: every marked token (a set bit of M), read back from global
// memory and passed to fn(x, t).  The marked tokens are first listed in
// sm.ev (block prefix over the threads' bitmap words), then thread t takes
// list entries t, t + kThreads, ... four at a time with the four reads in
// flight.  When more tokens are marked than the list holds, each thread walks
// its own bitmap words instead, in batches of eight that every lane of a warp
// runs together.  Every thread calls; sm.ev must be free.
template <int DT, class Fn>
__device__ __forceinline__ void for_marked(SelSmem& sm, const unsigned char* rowp, const unsigned* M, int nwords,
                                           Fn fn) {
  constexpr int kMB = 4;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int cnt = 0;
  for (int w = threadIdx.x; w < nwords; w += kThreads) cnt += __popc(M[w]);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.misc.wu[wid] = static_cast<unsigned>(incl);
  csync();
  int base = 0, total = 0;
  for (int q = 0; q < kWarps; ++q) {
    const int cq = static_cast<int>(sm.misc.wu[q]);
    base += q < wid ? cq : 0;
    total += cq;
  }
  if (total > kEvCap) {
    csync();
    constexpr int kWB = 8;
    int mx = cnt;
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int wcur = threadIdx.x;
    unsigned bits = wcur < nwords ? M[wcur] : 0u;
    for (int b0 = 0; b0 < mx; b0 += kWB) {
      int tb[kWB];
#pragma unroll
      for (int q = 0; q < kWB; ++q) {
        while (bits == 0u && wcur < nwords) {
          wcur += kThreads;
          bits = wcur < nwords ? M[wcur] : 0u;
        }
        if (bits) {
          tb[q] = (wcur << 5) + __ffs(bits) - 1;
          bits &= bits - 1u;
        } else {
          tb[q] = -1;
        }
      }
      float xs[kWB];
#pragma unroll
      for (int q = 0; q < kWB; ++q) xs[q] = tb[q] >= 0 ? load_logit<DT>(rowp, tb[q]) : 0.0f;
#pragma unroll
      for (int q = 0; q < kWB; ++q)
        if (tb[q] >= 0) fn(xs[q], tb[q]);
    }
    return;
  }
  int pos = base + incl - cnt;
  for (int w = threadIdx.x; w < nwords; w += kThreads) {
    unsigned bits = M[w];
    while (bits) {
      sm.ev[pos++] = static_cast<unsigned>((w << 5) + __ffs(bits) - 1);
      bits &= bits - 1u;
    }
  }
  csync();
  for (int j0 = 0; j0 < total; j0 += kMB * kThreads) {
    int tb[kMB];
    float xs[kMB];
#pragma unroll
    for (int q = 0; q < kMB; ++q) {
      const int j = j0 + q * kThreads + static_cast<int>(threadIdx.x);
      tb[q] = j < total ? static_cast<int>(sm.ev[j]) : -1;
    }
#pragma unroll
    for (int q = 0; q < kMB; ++q) xs[q] = tb[q] >= 0 ? load_logit<DT>(rowp, tb[q]) : 0.0f;
#pragma unroll
    for (int q = 0; q < kMB; ++q)
      if (tb[q] >= 0) fn(xs[q], tb[q]);
  }
}

// Gather the candidates whose stored level is `level` into fin.g*, then sort
// them into fin.s* by (key desc, index asc).  Returns the group size, or -1
// when it exceeds kGroupCap.  Every thread calls.
__device__ __noinline__ int gather_sort_stored(SelSmem& sm, int n, int level, float cc) {
  FinSmem& f = sm.fin;
  if (threadIdx.x == 0) f.gn = 0;
  csync();
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    const bool has = i < n && f.clv[i] == level;
    const unsigned bal = __ballot_sync(0xffffffffu, has);
    if (bal) {
      const int leader = __ffs(bal) - 1;
      int pos = 0;
      if (lane == leader) pos = atomicAdd(&f.gn, __popc(bal));
      pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(bal & ((1u << lane) - 1u));
      if (has && pos < kGroupCap) {
        const float s = sm.cand_s[i];
        f.gk[pos] = fkey(s);
        f.gi[pos] = sm.cand_i[i];
        f.gw[pos] = wfix_fast(s, cc);
      }
    }
  }
  csync();
  const int gn = f.gn;
  if (gn > kGroupCap) return -1;
  for (int t = threadIdx.x; t < gn; t += kThreads) {
    const unsigned kt = f.gk[t], it = f.gi[t];
    int r = 0;
    for (int j = 0; j < gn; ++j) {
      const unsigned kj = f.gk[j];
      r += (kj > kt) || (kj == kt && f.gi[j] < it);
    }
    f.sk[r] = kt;
    f.si[r] = it;
    f.sw[r] = f.gw[t];
  }
  csync();
  return gn;
}

// top_k, top_p and the draw over the candidate list (every candidate s is in
// [lo, m]).  Z_all = fixed-point mass of every token of the row, relative to
// m.  One pass sorts the candidates into kLevels value levels (count and exact
// mass per level); one block scan gives every thread the mass and count
// before its two levels, so each later search (the k-th token, the top-p cut,
// the draw) is one step in which the thread owning the crossing publishes it.
// Only the crossing level's members are sorted.  Falls back to
// finalize_candidates when such a level holds more than kGroupCap tokens.
__device__ __noinline__ FinResult finalize2(const DevCfg& c, SelSmem& sm, float m, float lo,
                                           unsigned long long Z_all, float u, bool topk, bool topp) {
  static_assert(kLevels == 2 * kThreads, "two levels per thread");
  FinSmem& f = sm.fin;
  FinResult res{false, 0, 0u};
  const int n = min(sm.misc.ncand, kCandCap);
  if (n <= 0) { res.reason = 9; return res; }
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float cc = m * kLog2e;
  const float range = m - lo;
  const LevelMap lv{m, range > 0.0f ? static_cast<float>(kLevels - 1) / range : 0.0f};
  for (int l = tid; l < kLevels; l += kThreads) { f.lc[l] = 0u; f.lw[0][l] = 0u; f.lw[1][l] = 0u; f.lw[2][l] = 0u; }
  csync();
  for (int i = tid; i < n; i += kThreads) {
    const float s = sm.cand_s[i];
    const int l = lv(s);
    f.clv[i] = static_cast<unsigned short>(l);
    const unsigned long long w = wfix_fast(s, cc);   // <= 2^44
    atomicAdd(&f.lc[l], 1u);
    atomicAdd(&f.lw[0][l], static_cast<unsigned>(w & 0x7fffull));
    atomicAdd(&f.lw[1][l], static_cast<unsigned>((w >> 15) & 0x7fffull));
    atomicAdd(&f.lw[2][l], static_cast<unsigned>(w >> 30));
  }
  csync();
  // exact mass and count of this thread's two levels, and of everything before them
  const int l0 = 2 * tid, l1 = l0 + 1;
  auto lmass = [&](int l) {
    return static_cast<unsigned long long>(f.lw[0][l]) + (static_cast<unsigned long long>(f.lw[1][l]) << 15) +
           (static_cast<unsigned long long>(f.lw[2][l]) << 30);
  };
  const unsigned long long m0 = lmass(l0), m1 = lmass(l1);
  const unsigned c0 = f.lc[l0], c1 = f.lc[l1];
  unsigned long long im = m0 + m1;
  unsigned ic = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tm = __shfl_up_sync(0xffffffffu, im, o);
    const unsigned tc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) { im += tm; ic += tc; }
  }
  if (lane == 31) { f.wsum[wid] = im; f.wcnt[wid] = ic; }
  csync();
  unsigned long long bm = 0ull, Zc = 0ull;
  unsigned bc = 0u;
  for (int q = 0; q < kWarps; ++q) {
    const unsigned long long sq = f.wsum[q];
    Zc += sq;
    if (q < wid) { bm += sq; bc += f.wcnt[q]; }
  }
  bm += im - (m0 + m1);   // mass before level l0
  bc += ic - (c0 + c1);   // count before level l0

  unsigned long long Z;
  int Lk = kLevels;                  // level of the k-th token (kLevels: no top_k)
  int rk = 0;                        // kept members of level Lk (in sorted order)
  unsigned long long kept_lk = 0ull; // their mass
  int sorted_level = -1;             // level currently held sorted in fin.s*
  int sorted_n = 0;
  if (topk) {
    const unsigned k = static_cast<unsigned>(c.top_k);
    if (n < c.top_k) { res.reason = 4; return res; }
    if (bc < k && bc + c0 + c1 >= k) {
      if (bc + c0 >= k) { f.fb = l0; f.fbefore = bc; f.fmass = bm; }
      else { f.fb = l1; f.fbefore = bc + c0; f.fmass = bm + m0; }
    }
    csync();
    Lk = f.fb;
    rk = static_cast<int>(k - static_cast<unsigned>(f.fbefore));
    const unsigned long long before_k = f.fmass;
    const int gn = gather_sort_stored(sm, n, Lk, cc);
    if (gn < 0) return finalize_candidates(c, sm, m, lo, Z_all, u, topk, topp);
    sorted_level = Lk;
    sorted_n = gn;
    if (tid == 0) {
      // top_k keeps every token tied with the k-th score: extend over equal keys
      const unsigned klo = f.sk[rk - 1];
      int r = rk;
      while (r < gn && f.sk[r] == klo) ++r;
      unsigned long long s = 0ull;
      for (int j = 0; j < r; ++j) s += f.sw[j];
      f.fmass = s;
      f.fb = r;
    }
    csync();
    kept_lk = f.fmass;
    rk = f.fb;
    Z = before_k + kept_lk;
    csync();
  } else {
    Z = Z_all > Zc ? Z_all : Zc;
  }
  // mass of level l over the kept set so far (levels past Lk dropped, Lk cut at rk)
  auto kept_mass = [&](int l, unsigned long long ml) { return l > Lk ? 0ull : (l == Lk ? kept_lk : ml); };

  unsigned long long S = Z;
  int Lc = kLevels;                  // level of the top-p cut (kLevels: no cut)
  int nc = 0;                        // kept members of level Lc (sorted order)
  unsigned long long before_c = 0ull;
  if (topp) {
    const unsigned long long T = topp_target(c.top_p, Z);
    if (!topk && Zc < T) { res.reason = 5; return res; }
    if (tid == 0) f.ffound = 0;
    csync();
    {
      const unsigned long long e0 = kept_mass(l0, m0), e1 = kept_mass(l1, m1);
      if (bm < T && bm + e0 + e1 >= T) {
        if (bm + e0 >= T) { f.fb = l0; f.fmass = bm; } else { f.fb = l1; f.fmass = bm + e0; }
        f.ffound = 1;
      }
    }
    csync();
    if (!f.ffound) { res.reason = 6; return res; }
    Lc = f.fb;
    before_c = f.fmass;
    int lim;
    if (Lc == sorted_level) {
      lim = Lc == Lk ? rk : sorted_n;
    } else {
      const int gn = gather_sort_stored(sm, n, Lc, cc);
      if (gn < 0) return finalize_candidates(c, sm, m, lo, Z_all, u, topk, topp);
      sorted_level = Lc;
      sorted_n = gn;
      lim = gn;
    }
    walk_sorted(sm, lim, before_c, T, false);
    if (!f.ffound) { res.reason = 6; return res; }
    nc = f.fb + 1;
    S = f.fbefore + f.sw[f.fb];
    csync();
  }
  const unsigned long long Td = draw_target(u, S);
  if (!topk && !topp && !(Zc > Td)) { res.reason = 7; return res; }
  // level of the draw among the kept levels (levels past Lc dropped, Lc cut at nc)
  if (tid == 0) f.ffound = 0;
  csync();
  {
    auto dmass = [&](int l, unsigned long long ml) {
      if (l > Lc) return 0ull;
      if (l == Lc) return S - before_c;
      return kept_mass(l, ml);
    };
    const unsigned long long e0 = dmass(l0, m0), e1 = dmass(l1, m1);
    if (bm <= Td && bm + e0 + e1 > Td) {
      if (bm + e0 > Td) { f.fb = l0; f.fmass = bm; } else { f.fb = l1; f.fmass = bm + e0; }
      f.ffound = 1;
    }
  }
  csync();
  if (!f.ffound) { res.reason = 8; return res; }
  const int Ld = f.fb;
  const unsigned long long before_d = f.fmass;
  int lim;
  if (Ld == sorted_level) {
    lim = Ld == Lc ? nc : (Ld == Lk ? rk : sorted_n);
  } else {
    const int gn = gather_sort_stored(sm, n, Ld, cc);
    if (gn < 0) return finalize_candidates(c, sm, m, lo, Z_all, u, topk, topp);
    lim = gn;
  }
  walk_sorted(sm, lim, before_d, Td, true);
  if (!f.ffound) { res.reason = 8; return res; }
  res.token = f.si[f.fb];
  res.score = key2f(f.sk[f.fb]);
  res.S = S;
  csync();
  res.ok = true;
  return res;
}

// The candidates could not hold the cut or the draw: read the whole row
// again (from L2) and take every token at or above a lower threshold.  The
// row's total mass Z does not change.  Every thread calls.
template <int DT>
__device__ __noinline__ FinResult second_chance(const DevCfg& c, const SelArgs& a, SelSmem& sm, const RowMeta& rm,
                                                const unsigned char* rowp, unsigned* M, unsigned* N, bool bitmaps,
                                                float theta_raw, bool tempered, float m, unsigned long long Z,
                                                float u, bool topk, bool topp) {
  const int V = a.V;
  const float theta_f = tempered ? nextafterf(__fdiv_rn(theta_raw, c.temp), INFINITY) : theta_raw;
  FinResult res{false, 20, 0u};
  csync();
  if (threadIdx.x == 0) sm.misc.ncand = 0;
  if (bitmaps) build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, reinterpret_cast<int*>(sm.cand_s), 2 * kCandCap);
  else csync();
  expand_units<DT>(c, sm, rowp, V, 0, true, M, bitmaps, theta_raw, theta_f, tempered);
  if (bitmaps) {
    for_marked<DT>(sm, rowp, M, a.nwords, [&](float x, int t) {
      const float s = process_elem(c, M, N, x, t, true);
      if (s >= theta_f) {
        const int pos = atomicAdd(&sm.misc.ncand, 1);
        if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = static_cast<unsigned>(t); }
      }
    });
  }
  csync();
  if (sm.misc.ncand > kCandCap) { res.reason = 24; return res; }
  return finalize2(c, sm, m, theta_f, Z, u, topk, topp);
}

struct LevelPick {
  bool ok;
  unsigned idx;                 // the selected token
  unsigned key;                 // its order-preserving score key
  unsigned long long cum;       // mass of every token up to and including it
};

// The first candidate, in (score desc, index asc) order over the list
// cand_s/cand_i[0..n) (every score in [lo, hi]), at which the running mass
// (weights relative to cc / log2e) reaches `target` (>= target, or > target
// when strict).  `base` is added to the returned running mass.  A level
// histogram over [lo, hi] finds the level; only its members are sorted.
// Every thread calls.  Uses FinSmem (which aliases the row bitmaps).
__device__ __forceinline__ LevelPick list_pick(SelSmem& sm, int n, float hi, float lo, float cc,
                                            unsigned long long target, bool strict, unsigned long long base) {
  FinSmem& f = sm.fin;
  LevelPick res{false, 0u, 0u, 0ull};
  if (n <= 0) return res;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float range = hi - lo;
  const LevelMap lv{hi, range > 0.0f ? static_cast<float>(kLevels - 1) / range : 0.0f};
  for (int l = tid; l < kLevels; l += kThreads) { f.lc[l] = 0u; f.lw[0][l] = 0u; f.lw[1][l] = 0u; f.lw[2][l] = 0u; }
  csync();
  for (int i = tid; i < n; i += kThreads) {
    const float s = sm.cand_s[i];
    const int l = lv(s);
    f.clv[i] = static_cast<unsigned short>(l);
    const unsigned long long w = wfix_fast(s, cc);
    atomicAdd(&f.lc[l], 1u);
    atomicAdd(&f.lw[0][l], static_cast<unsigned>(w & 0x7fffull));
    atomicAdd(&f.lw[1][l], static_cast<unsigned>((w >> 15) & 0x7fffull));
    atomicAdd(&f.lw[2][l], static_cast<unsigned>(w >> 30));
  }
  csync();
  const int l0 = 2 * tid, l1 = l0 + 1;
  auto lmass = [&](int l) {
    return static_cast<unsigned long long>(f.lw[0][l]) + (static_cast<unsigned long long>(f.lw[1][l]) << 15) +
           (static_cast<unsigned long long>(f.lw[2][l]) << 30);
  };
  const unsigned long long m0 = lmass(l0), m1 = lmass(l1);
  unsigned long long im = m0 + m1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tm = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) im += tm;
  }
  if (lane == 31) f.wsum[wid] = im;
  if (tid == 0) f.ffound = 0;
  csync();
  unsigned long long bm = 0ull;
  for (int q = 0; q < wid; ++q) bm += f.wsum[q];
  bm += im - (m0 + m1);
  auto reached = [&](unsigned long long x) { return strict ? x > target : x >= target; };
  if (!reached(bm) && reached(bm + m0 + m1)) {
    if (reached(bm + m0)) { f.fb = l0; f.fmass = bm; } else { f.fb = l1; f.fmass = bm + m0; }
    f.ffound = 1;
  }
  csync();
  if (!f.ffound) return res;
  const int L = f.fb;
  const unsigned long long before = f.fmass;
  const int gn = gather_sort_stored(sm, n, L, cc);
  if (gn < 0) return res;
  walk_sorted(sm, gn, before, target, strict);
  if (!f.ffound) return res;
  res.ok = true;
  res.idx = f.si[f.fb];
  res.key = f.sk[f.fb];
  res.cum = base + f.fbefore + f.sw[f.fb];
  csync();
  return res;
}

// Items whose key (order-preserving score key) lies in [klo, khi).
struct InWindow {
  unsigned klo, khi;
  __device__ __forceinline__ bool operator()(unsigned key, unsigned) const { return key >= klo && key < khi; }
};
struct AtLeast {
  unsigned k;
  __device__ __forceinline__ bool operator()(unsigned key, unsigned) const { return key >= k; }
};


// The first token, in (score desc, index asc) order over the whole row, at
// which the running mass (exact weights relative to m) reaches `target`
// (>= target, or > target when strict).  m >= every score; only tokens with
// score > m - 32 can carry mass at the 2^-44 quantum.  One pass counts the
// tokens in 2,048 levels of 1/64 below m; the level where the estimated
// running mass (count x the level's middle weight, rescaled to the exact
// total Z) crosses the target gives a narrow score window; one pass sums the
// exact mass above the window and inside it; when the target lies inside,
// the radix selection runs over the window's few tokens.  ok = false when
// four windows miss.  Every thread calls; the candidate list is free.
template <int DT>
__device__ __forceinline__ LevelPick level_pick(const RowGlobalSource<DT>& src, SelSmem& sm, float m,
                                             unsigned long long Z, unsigned long long target, bool strict) {
  constexpr int kL = 2048;
  constexpr float kPer = 64.0f;   // levels per score unit
  static_assert(kEvCap >= 2048, "level counts live in the unit list");
  unsigned* cnt = sm.ev;
  LevelPick res{false, 0u, 0u, 0ull};
  for (int l = threadIdx.x; l < kL; l += kThreads) cnt[l] = 0u;
  csync();
  src.pass([&](float s, unsigned) {
    const float d = (m - s) * kPer;
    if (d < static_cast<float>(kL)) atomicAdd(&cnt[d > 0.0f ? static_cast<int>(d) : 0], 1u);
  });
  csync();
  // estimated mass of each level (relative to m); thread t owns levels 4t .. 4t+3
  {
    constexpr int PT = kL / kThreads;
    static_assert(kL % kThreads == 0, "levels per thread");
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float e[PT];
    float loc = 0.0f;
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int l = PT * static_cast<int>(threadIdx.x) + j;
      e[j] = static_cast<float>(cnt[l]) * expf(-(static_cast<float>(l) + 0.5f) / kPer);
      loc += e[j];
    }
    float incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sm.misc.wf[wid] = incl;
    if (threadIdx.x == 0) sm.misc.wu[0] = static_cast<unsigned>(kL - 1);
    csync();
    float before = 0.0f, tot = 0.0f;
    for (int q = 0; q < kWarps; ++q) {
      const float v = sm.misc.wf[q];
      tot += v;
      before += q < wid ? v : 0.0f;
    }
    before += incl - loc;
    // the exact total rescales the estimate; the target in the same units
    const float unit = 1.0f / 17592186044416.0f;
    const float scale = tot > 0.0f ? (static_cast<float>(Z) * unit) / tot : 1.0f;
    const float want = static_cast<float>(target) * unit / scale;
    if (before < want && before + loc >= want) {
      float run = before;
      int le_t = PT * static_cast<int>(threadIdx.x) + PT - 1;
#pragma unroll
      for (int j = 0; j < PT; ++j) {
        run += e[j];
        if (run >= want) { le_t = PT * static_cast<int>(threadIdx.x) + j; break; }
      }
      sm.misc.wu[0] = static_cast<unsigned>(le_t);
    }
    csync();
  }
  int le = static_cast<int>(sm.misc.wu[0]);
  const WFast wx{m * kLog2e};
  for (int attempt = 0, half = 3; attempt < 4; ++attempt, half *= 4) {
    // window (m - l1/64, m - l0/64], narrowed until its tokens fit the list
    int l0 = 0, l1 = 0;
    unsigned wn = 0u;
    for (int h = half;; h >>= 1) {
      l0 = max(0, le - h);
      l1 = min(kL, le + h + 1);
      unsigned t = 0u;
      for (int l = l0 + static_cast<int>(threadIdx.x); l < l1; l += kThreads) t += cnt[l];
      wn = static_cast<unsigned>(block_sum_u64(t, &sm.red));
      if (wn <= static_cast<unsigned>(kCandCap) || h == 0) break;
    }
    if (wn > static_cast<unsigned>(kCandCap)) break;
    // keys: higher score = larger key
    const unsigned khi = l0 == 0 ? 0xffffffffu : fkey(m - static_cast<float>(l0) / kPer);
    const unsigned klo = l1 >= kL ? 0u : fkey(m - static_cast<float>(l1) / kPer);
    // exact mass above the window, and the window's tokens gathered into the
    // candidate list, in one pass
    if (threadIdx.x == 0) sm.misc.ncand = 0;
    csync();
    unsigned long long a_t = 0ull, w_t = 0ull;
    src.pass([&](float s, unsigned i) {
      const unsigned key = fkey(s);
      bool in = false;
      if (key >= klo) {
        const unsigned long long w = wx(s);
        if (key >= khi) a_t += w; else { w_t += w; in = true; }
      }
      if (in) {
        const int pos = atomicAdd(&sm.misc.ncand, 1);
        if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = i; }
      }
    });
    const unsigned long long A = block_sum_u64(a_t, &sm.red);
    const unsigned long long W = block_sum_u64(w_t, &sm.red);
    const bool below = strict ? target < A : target <= A;            // the crossing is above the window
    const bool past = strict ? target >= A + W : target > A + W;     // ... or below it
    if (!below && !past) {
      const int nw = min(sm.misc.ncand, kCandCap);
      const float top = l0 == 0 ? m : m - static_cast<float>(l0) / kPer;
      const float bot = m - static_cast<float>(l1) / kPer;
      return list_pick(sm, nw, top, bot, m * kLog2e, target - A, strict, A);
    }
    if (below && l0 == 0) break;
    if (past && l1 >= kL) break;
    le = below ? max(0, l0 - 1) : min(kL - 1, l1);
  }
  return res;
}

// Multi-pass exact selection over the whole row, read from global memory
// (it is normally in L2).  top_k rows run the generic radix selection;
// the others locate the top-p cut and the draw with level_pick.
struct SlowPick {
  unsigned token;
  float score;            // its processed score
  float ref;              // the masses' reference: m * log2e (fast weights) or m (accurate weights)
  bool fast;              // weights 2^(s * log2e - ref) (ex2.approx), else exp(s - ref)
  unsigned long long S;   // mass of the kept set
};
template <int DT>
__device__ __noinline__ SlowPick slow_select(const DevCfg& c, const SelArgs& a, SelSmem& sm, const RowMeta& rm,
                                             const unsigned char* rowp, unsigned* H, unsigned* N, bool bitmaps,
                                             float u, bool count = true) {
  csync();
  if (count && threadIdx.x == 0) { atomicOr(c.status, kFlagSlow); atomicAdd(c.slow_rows, 1ull); }
  TG_TF(15);
  if (bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords, reinterpret_cast<int*>(sm.cand_s), 2 * kCandCap);
  TG_TF(16);
  RowGlobalSource<DT> src{rowp, a.V, &c, H, N, bitmaps, true};
  if (c.prow) src.state_row(c);
  float mm = -INFINITY;
  src.pass([&](float s, unsigned) { mm = fmaxf(mm, s); });
  mm = block_max(mm, &sm.red);
  TG_TF(17);
  const bool topk = c.top_k > 0 && static_cast<unsigned>(c.top_k) < static_cast<unsigned>(a.V);
  if (!topk && mm > kFilter) {
    unsigned long long z_t = 0ull;
    const WFast wz{mm * kLog2e};
    src.pass([&](float s, unsigned) { z_t += wz(s); });
    const unsigned long long Z = block_sum_u64(z_t, &sm.red);
    TG_TF(18);
    unsigned long long S = Z;
    bool ok = Z > 0ull;
    // an exact pick over a window uses the finishing area, which holds the
    // row bitmaps: they are rebuilt before the next pass that reads them
    auto restore = [&]() {
      if (bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords, reinterpret_cast<int*>(sm.cand_s), 2 * kCandCap);
    };
    if (ok && c.top_p < 1.0f) {
      const LevelPick cut = level_pick<DT>(src, sm, mm, Z, topp_target(c.top_p, Z), false);
      TG_TF(19);
      restore();
      TG_TF(20);
      ok = cut.ok;
      S = cut.cum;
    }
    if (ok) {
      const LevelPick d = level_pick<DT>(src, sm, mm, Z, draw_target(u, S), true);
      TG_TF(21);
      if (d.ok) return SlowPick{d.idx, key2f(d.key), mm * kLog2e, true, S};
    }
    restore();
  }
  unsigned long long S = 0ull;
  unsigned key = 0u;
  const unsigned t = sample_exact(c, src, mm, u, static_cast<unsigned>(a.V), &sm.hist, &sm.red, nullptr, &S, &key);
  return SlowPick{t, key2f(key), mm, false, S};
}

// ---------------------------------------------------------------------------
// select_kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Verify position `row` (row b, position j) with the processors: the row's
// history followed by its first j candidates.  An empty history is a padding
// row.  The extended history is staged in shared memory, so it must fit the
// stage (2 * kCandCap ids); a longer one makes the position a bad row.
__device__ __forceinline__ RowMeta verify_meta(const DevCfg& c, const SelArgs& a, int row) {
  const int K1 = a.K + 1;
  const int b = row / K1, j = row % K1;
  RowMeta r = row_meta(c, a.hist, a.off, a.plen, b, a.nrows_total / K1);
  if (r.bad || r.L == 0) return r;
  r.ext = a.cand + static_cast<size_t>(b) * a.K;
  r.Lb = r.L;
  r.L += j;
  if (r.L > 2 * kCandCap) {
    r.bad = true;
    r.L = 0;
    return r;
  }
  row_meta_rules(c, r);
  return r;
}

// Verify, steps 4-5: the last of a row's K+1 positions to finish counts the
// left-to-right matches and writes -1 after the first divergent token.  One
// thread, after writing its position's token.
__device__ __forceinline__ void verify_ticket(const DevCfg& c, const SelArgs& a, int row) {
  const int vb = row / (a.K + 1);
  __threadfence();
  const unsigned prev = atomicAdd(&c.tickets[vb], 1u);
  if (prev == static_cast<unsigned>(a.K)) {
    __threadfence();
    const int K = a.K;
    volatile int32_t* nxt = a.out + static_cast<size_t>(vb) * (K + 1);
    int nm = 0;
    while (nm < K && nxt[nm] == a.cand[static_cast<size_t>(vb) * K + nm]) ++nm;
    for (int j = nm + 1; j <= K; ++j) nxt[j] = -1;
    a.out_match[vb] = nm;
    c.tickets[vb] = 0u;
  }
}

// Forced rows do not depend on the logits: the forced ids score 0, all
// others the filter value; greedy takes the lowest, sampling draws among them.
// *kept = how many equal-scored tokens the step selects from.
// Among cnt equal-scored tokens in index order: greedy takes the first;
// sampling keeps the top-p prefix and draws in it.  Returns the position;
// *kept = the tokens the step selects from.
__device__ __forceinline__ int equal_pick(const DevCfg& c, unsigned long long cnt, float u, bool sample,
                                          unsigned long long* kept) {
  *kept = cnt;
  if (!sample) return 0;
  const unsigned long long W = 1ull << kFixShift;
  unsigned long long ncut = cnt;
  if (c.top_p < 1.0f) ncut = group_pick(0ull, W, cnt, topp_target(c.top_p, cnt * W), false);
  *kept = ncut;
  const unsigned long long nd = group_pick(0ull, W, ncut, draw_target(u, ncut * W), true);
  return static_cast<int>(nd - 1);
}

__device__ __forceinline__ int forced_token(const DevCfg& c, const RowMeta& rm, int V, float u, bool sample,
                                            unsigned long long* kept) {
  int zs[8];
  const int nz = forced_zeros(c, rm, zs);
  const unsigned long long cnt = nz ? static_cast<unsigned long long>(nz) : static_cast<unsigned long long>(V);
  const int pos = equal_pick(c, cnt, u, sample, kept);
  return nz ? zs[pos] : pos;
}

// Log-probability of a selected token (the log-softmax of the scores the
// step selects from, at the token): the log of its weight, in the same
// arithmetic as the weights summed into the kept set's mass S (2^-44 units),
// less log S.  Fast weights are 2^(fma(s, log2e, -ref)); accurate ones
// exp(s - ref).  log2 S = its binary exponent plus log2f of its mantissa in
// [1, 2) (f32 S, 6e-8 relative): no fp64 transcendental, which is slow here.
__device__ __forceinline__ float token_logprob(float score, float ref, bool fast, unsigned long long S) {
  constexpr double kLn2 = 0.6931471805599453;
  const double lnw = fast ? static_cast<double>(fmaf(score, kLog2e, -ref)) * kLn2
                          : static_cast<double>(score) - static_cast<double>(ref);
  const unsigned b = __float_as_uint(__ull2float_rn(S));   // S >= 1: a normal float
  const int e = static_cast<int>(b >> 23) - 127;
  const float mant = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
  const double log2S = static_cast<double>(e - kFixShift) + static_cast<double>(log2f(mant));
  return static_cast<float>(lnw - log2S * kLn2);
}

// Block-uniform choice of the sampling threshold from the first sub-chunk's
// level counts (level l holds tempered scores in (m0 - 2(l+1), m0 - 2l]).
// Returns l: the threshold is m0 - 2(l+1).  top_k: the first level where the
// row is expected to hold 4k tokens; otherwise the first level where the mass
// expected below it is at most a quarter of the (1 - q) the cut or draw
// allows; never beyond the level where the row's candidates would fill three
// quarters of the list.  -1: even level 0 would overfill it.
__device__ __forceinline__ int pilot_level(const unsigned (&cnt)[8], unsigned n_seen, float scale, bool topk,
                                           int top_k, float qfrac) {
  const float cap = 0.75f * static_cast<float>(kCandCap);
  float cum = 0.0f, Z = 0.0f;
  float wl[8];
#pragma unroll
  for (int l = 0; l < 8; ++l) {
    wl[l] = static_cast<float>(cnt[l]) * __expf(-2.0f * l - 1.0f);
    Z += wl[l];
  }
  unsigned seen = 0u;
#pragma unroll
  for (int l = 0; l < 8; ++l) seen += cnt[l];
  const float rest = static_cast<float>(n_seen - min(seen, n_seen)) * __expf(-17.0f);
  Z += rest;
  int jcap = -1, jsel = -1;
  float below = Z;
#pragma unroll
  for (int l = 0; l < 8; ++l) {
    cum += static_cast<float>(cnt[l]);
    below -= wl[l];
    if (cum * scale <= cap) jcap = l;
    if (jsel < 0) {
      if (topk ? (cum * scale >= 4.0f * static_cast<float>(top_k)) : (below <= 0.25f * (1.0f - qfrac) * Z)) jsel = l;
    }
  }
  if (jsel < 0) jsel = 7;
  return jcap < 0 ? -1 : min(jsel, jcap);
}

// One barrier for all of a sampled row's sums: the exact fixed-point mass
// (two's complement, so signed parts add up exactly), the raw streaming mass,
// the raw mass of the marked tokens, and whether any processed score exceeded
// the reference maximum.  Every thread calls; all get the totals.
struct RowSums {
  unsigned long long z;
  float hot, wr;
  bool over;
};
__device__ __forceinline__ RowSums block_row_sums(SelSmem& sm, unsigned long long z, float hot, float wr, bool over) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o; o >>= 1) {
    z += __shfl_xor_sync(0xffffffffu, z, o);
    hot += __shfl_xor_sync(0xffffffffu, hot, o);
    wr += __shfl_xor_sync(0xffffffffu, wr, o);
  }
  const bool ov = __any_sync(0xffffffffu, over);
  csync();
  if (lane == 0) {
    sm.red.q[wid] = z;
    sm.red.f[wid] = hot;
    sm.red.u[wid] = __float_as_uint(wr);
    sm.misc.wu[wid] = ov ? 1u : 0u;
  }
  csync();
  RowSums r{0ull, 0.0f, 0.0f, false};
  for (int q = 0; q < kWarps; ++q) {
    r.z += sm.red.q[q];
    r.hot += sm.red.f[q];
    r.wr += __uint_as_float(sm.red.u[q]);
    r.over |= sm.misc.wu[q] != 0u;
  }
  return r;
}

// A row's processor state breaks its layout (this thread's columns): an id
// outside [-1, V), or within a processor's columns an unused (-1) column
// before a used one, or used ids not strictly ascending.
__device__ __forceinline__ bool state_layout_bad(const DevCfg& c, const int32_t* ids) {
  const int S = c.pcol[c.nproc];
  bool bad = false;
  for (int j = threadIdx.x; j < S; j += kThreads) {
    int end = S;
    for (int k = 0; k < c.nproc; ++k)
      if (j < c.pcol[k + 1]) { end = c.pcol[k + 1]; break; }
    const int t = __ldg(ids + j);
    if (t < -1 || t >= c.V) {
      bad = true;
    } else if (j + 1 < end) {
      const int t2 = __ldg(ids + j + 1);
      if (t == -1 ? t2 != -1 : (t2 != -1 && t2 <= t)) bad = true;
    }
  }
  return bad;
}

// A forced row with a processor state, block-wide: its tokens score F except
// the forced ids (0) and the state ids (a processor's value), so the tokens
// above F are listed once (a state id in its first processor's columns, a
// forced id that is no state id) with their final scores, and the one-pass
// finish selects from them (they hold all of the row's mass).  Every token at
// F: all V tie.  Left at kDeferred for state_kernel when the list overflows
// or the finish cannot decide.
template <bool SAMPLE>
__device__ __noinline__ void forced_state_row(const DevCfg& c, const SelArgs& a, SelSmem& sm, int row, int S) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int V = a.V;
  const RowMeta rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows_total);
  int zs[8];
  const int nz = forced_zeros(c, rm, zs);
  const int32_t* ids = a.st_ids + static_cast<size_t>(row) * S;
  const float* vals = a.st_vals + static_cast<size_t>(row) * S;
  csync();
  const bool bad = __syncthreads_or(state_layout_bad(c, ids) ? 1 : 0) != 0;
  if (tid == 0) {
    if (bad) atomicOr(c.status, kFlagBadState);
    sm.misc.ncand = 0;
  }
  csync();
  for (int j = tid; j < S + nz; j += kThreads) {
    int t;
    bool dup = false;
    if (j < S) {
      t = bad ? -1 : __ldg(ids + j);
      if (t < 0) continue;
      for (int k = 0; k < c.nproc && c.pcol[k + 1] <= j; ++k)
        dup = dup || state_find(ids + c.pcol[k], c.pcol[k + 1] - c.pcol[k], t) >= 0;
    } else {
      t = zs[j - S];
      for (int k = 0; !bad && k < c.nproc; ++k)
        dup = dup || state_find(ids + c.pcol[k], c.pcol[k + 1] - c.pcol[k], t) >= 0;
    }
    if (dup) continue;
    float s = kFilter;
    for (int q = 0; q < nz; ++q) s = zs[q] == t ? 0.0f : s;
    if (!bad) s = apply_state_at(c, ids, vals, s, t);
    if (SAMPLE && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
    if (s > kFilter) {
      const int pos = atomicAdd(&sm.misc.ncand, 1);
      if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = static_cast<unsigned>(t); }
    }
  }
  csync();
  const int n = sm.misc.ncand;
  if (n > kCandCap) return;
  const float u = (SAMPLE && a.uniforms) ? a.uniforms[row] : 0.0f;
  if (n == 0) {
    if (tid == 0) {
      unsigned long long kept = 1ull;
      a.out[row] = equal_pick(c, static_cast<unsigned long long>(V), u, SAMPLE, &kept);
      if (SAMPLE && a.logprobs) a.logprobs[row] = -logf(static_cast<float>(kept));
    }
    csync();
    return;
  }
  if (!SAMPLE) {
    float bv = -INFINITY;
    unsigned bi = 0xffffffffu;
    for (int j = tid; j < n; j += kThreads) {
      const float v = sm.cand_s[j];
      const unsigned i = sm.cand_i[j];
      if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
    }
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const unsigned i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
    }
    if (lane == 0) { sm.misc.wf[wid] = bv; sm.misc.wu[wid] = bi; }
    csync();
    if (tid == 0) {
      float v = sm.misc.wf[0];
      unsigned b = sm.misc.wu[0];
      for (int q = 1; q < kWarps; ++q) {
        const float v2 = sm.misc.wf[q];
        const unsigned i2 = sm.misc.wu[q];
        if (v2 > v || (v2 == v && i2 < b)) { v = v2; b = i2; }
      }
      a.out[row] = static_cast<int>(b);
    }
    csync();
    return;
  }
  float mx = -INFINITY, mn = INFINITY;
  for (int j = tid; j < n; j += kThreads) {
    mx = fmaxf(mx, sm.cand_s[j]);
    mn = fminf(mn, sm.cand_s[j]);
  }
  const float m = block_max(mx, &sm.red);
  const float lo = -block_max(-mn, &sm.red);
  const float cc = m * kLog2e;
  unsigned long long z = 0ull;
  for (int j = tid; j < n; j += kThreads) z += wfix_fast(sm.cand_s[j], cc);
  const unsigned long long Z = block_sum_u64(z, &sm.red);
  // top_k at or above the tokens above F keeps all of them (the rest weigh nothing)
  const bool topk = c.top_k > 0 && c.top_k < n;
  const FinResult fr = finalize2(c, sm, m, lo, Z, u, topk, c.top_p < 1.0f);
  if (tid == 0) {
    if (fr.ok) {
      a.out[row] = static_cast<int>(fr.token);
      if (a.logprobs) a.logprobs[row] = token_logprob(fr.score, cc, true, fr.S);
    } else {
      atomicOr(c.status, kFlagSlow);
      atomicAdd(c.slow_rows, 1ull);
    }
  }
  csync();
}

// VMODE: 0 select, 1 verify, 2 verify with the processors at every position
// (a compile-time choice, so plain verify carries none of the bitmap code).
template <int DT, int VMODE, bool SAMPLE>
__global__ void __launch_bounds__(kThreads, 1) select_kernel(const DevCfg c, const SelArgs a) {
  constexpr bool VERIFY = VMODE != 0;
  constexpr bool VHIST = VMODE == 2;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  unsigned* M = reinterpret_cast<unsigned*>(smem_raw + fin_offset());   // marked (history | banned)
  unsigned* N = M + bitmap_bytes(a.nwords) / 4;                         // banned
  unsigned char* ring = smem_raw + ring_offset(a.nwords);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int esz = DT == kF32 ? 4 : 2;
  constexpr int PER = DT == kF32 ? 4 : 8;
  constexpr int SE = kStageBytes / esz;   // elements per sub-chunk
  constexpr int SW = SE / kWarps;         // elements per warp slice
  static_assert(SW == 4 * 32 * PER, "a warp slice is four 16-byte vectors per lane");
  const int V = a.V;
  const int nsub = (V + SE - 1) / SE;
  const int nst = a.nstage;
  const bool tempered = SAMPLE && c.temp != 1.0f;
  // rows take the TMA ring when every row starts on a 16-byte boundary
  const bool tma_ok = ((reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0u) && ((static_cast<size_t>(V) * esz) % 16u == 0u);
  // rows with the task's processors: their state ids are marked and listed;
  // a row that cannot finish on the one-pass path is left to state_kernel
  const bool state = !VERIFY && a.st_ids != nullptr;
  const int S = state ? c.pcol[c.nproc] : 0;
  const bool bitmaps = (!VERIFY || VHIST) && (state || c.rho != 1.0f || c.ngram > 0 || c.n_ban > 0 || c.n_bsup > 0 ||
                                               c.n_seq > 0 || (c.n_eos > 0 && (c.min_length > 0 || c.min_new > 0)));

  // Inputs may come from the kernel before this one in the stream.
  grid_dependency_wait();

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&sm.misc.full[s], 1u);
      sm.misc.cnt[s] = 0u;
      sm.misc.iss[s] = 0;
    }
    sm.misc.error = 0;
    sm.misc.gcause = 0;
    fence_mbar_init();
  }

  // ---- this CTA's rows: row_begin + blockIdx.x + i * gridDim.x, one per thread ----
  const int rel = a.nrows - a.row_begin - static_cast<int>(blockIdx.x);
  const int nmine = rel > 0 ? min(kMaxRowsPerCta, (rel - 1) / static_cast<int>(gridDim.x) + 1) : 0;
  bool streamed = false;
  bool fstate = false;   // a forced row with a processor state: finished after the streamed rows
  int myrow = 0;
  if (tid < nmine) {
    myrow = a.row_begin + static_cast<int>(blockIdx.x) + tid * static_cast<int>(gridDim.x);
    if (VERIFY && !VHIST) {
      streamed = true;
    } else {
      const RowMeta rm = VERIFY ? verify_meta(c, a, myrow) : row_meta(c, a.hist, a.off, a.plen, myrow, a.nrows_total);
      if (rm.bad || rm.L == 0) {
        a.out[myrow] = -1;
        if (!VERIFY && SAMPLE && a.logprobs) a.logprobs[myrow] = __int_as_float(0x7fc00000);   // no token: NaN
        if (rm.bad) atomicOr(c.status, kFlagBadRow);
        if (VERIFY) verify_ticket(c, a, myrow);
      } else if (rm.forced && state) {
        a.out[myrow] = kDeferred;   // until this CTA finishes it (or state_kernel does)
        fstate = true;
      } else if (rm.forced) {
        const float u = (SAMPLE && a.uniforms) ? a.uniforms[myrow] : 0.0f;
        unsigned long long kept = 1ull;
        a.out[myrow] = forced_token(c, rm, V, u, SAMPLE, &kept);
        // the kept tokens score equally: each has probability 1 / kept
        if (!VERIFY && SAMPLE && a.logprobs) a.logprobs[myrow] = -logf(static_cast<float>(kept));
        if (VERIFY) verify_ticket(c, a, myrow);
      } else {
        streamed = true;
      }
    }
  }
  {
    // compact the streamed rows, keeping their order
    const unsigned bal = __ballot_sync(0xffffffffu, streamed);
    if (lane == 0) sm.misc.wu[wid] = static_cast<unsigned>(__popc(bal));
    __syncthreads();
    int before = 0, total = 0;
    for (int q = 0; q < kWarps; ++q) {
      const int cq = static_cast<int>(sm.misc.wu[q]);
      before += q < wid ? cq : 0;
      total += cq;
    }
    if (streamed) sm.rows[before + __popc(bal & ((1u << lane) - 1u))] = myrow;
    if (tid == 0) sm.misc.nrow = total;
    __syncthreads();
    if (state) {
      // then the forced rows with a state, after them
      const unsigned bal2 = __ballot_sync(0xffffffffu, fstate);
      if (lane == 0) sm.misc.wu[wid] = static_cast<unsigned>(__popc(bal2));
      __syncthreads();
      int before2 = 0, total2 = 0;
      for (int q = 0; q < kWarps; ++q) {
        const int cq = static_cast<int>(sm.misc.wu[q]);
        before2 += q < wid ? cq : 0;
        total2 += cq;
      }
      if (fstate) sm.rows[total + before2 + __popc(bal2 & ((1u << lane) - 1u))] = myrow;
      if (tid == 0) sm.misc.nfst = total2;
      __syncthreads();
    }
  }
  const int nrow = sm.misc.nrow;
  const int total_seq = nrow * nsub;   // <= kMaxRowsPerCta * (TG_MAX_VOCAB * 4 / kStageBytes)

  // Load sub-chunk kk of the schedule's row ri into stage st.
  auto issue = [&](int st, int ri, int kk) {
    const int row = sm.rows[ri];
    const int lo = kk * SE, n = min(SE, V - lo);
    const unsigned char* src = static_cast<const unsigned char*>(a.logits) + (static_cast<size_t>(row) * V + lo) * esz;
    mbar_expect_tx(&sm.misc.full[st], static_cast<unsigned>(n * esz));
    bulk_g2s(ring + st * kStageBytes, src, static_cast<unsigned>(n * esz), &sm.misc.full[st]);
    sm.misc.iss[st] += 1;
  };
  if (tma_ok && tid == 0) {
    for (int q = 0; q < nst && q < total_seq; ++q) issue(q, q / nsub, q % nsub);
  }
  grid_dependents_launch();

  int cur_st = 0;          // stage and phase of the next sub-chunk of the schedule
  unsigned cur_ph = 0u;
  for (int ri = 0; ri < nrow; ++ri) {
    const int row = sm.rows[ri];
    const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * esz;
    RowMeta rm;
    if (VERIFY && VHIST) {
      rm = verify_meta(c, a, row);
    } else if (VERIFY) {
      rm.bad = false; rm.L = 1; rm.P = 0; rm.h0 = 0; rm.Lb = 1; rm.ext = nullptr;
      rm.eos_off = rm.forced = rm.forced_eos = rm.bsup = false;
    } else {
      rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows_total);
    }
    const float u = (SAMPLE && a.uniforms) ? a.uniforms[row] : 0.0f;
    const bool topk = SAMPLE && c.top_k > 0 && c.top_k < V;
    const bool topp = SAMPLE && c.top_p < 1.0f;
    const float qfrac = topp ? c.top_p : fminf(fmaxf(u, 0.0f), 1.0f);
#ifdef TG_DEBUG
    if (tid == 0) sm.misc.dbg_row = row;
#endif
    TG_T(row, 0);
    // the row's processor state: its layout is checked first (a row whose
    // state breaks it is deferred, and state_kernel flags and drops it)
    const int32_t* sids = nullptr;
    const float* svals = nullptr;
    bool defer = false;
    if (state) {
      sids = a.st_ids + static_cast<size_t>(row) * S;
      svals = a.st_vals + static_cast<size_t>(row) * S;
      if (tid < kStateFilterWords) sm.misc.sfilt[tid] = 0u;
      csync();
      for (int j = tid; j < S; j += kThreads) {
        const int t = __ldg(sids + j);
        if (t >= 0) atomicOr(&sm.misc.sfilt[(t >> 5) & (kStateFilterWords - 1)], 1u << (t & 31));
      }
      defer = __syncthreads_or(state_layout_bad(c, sids) ? 1 : 0) != 0;
    }
    // the candidate list is free at the start of a row: it stages the history
    // the marked tokens are listed too (in N's words) when they fit
    const int nlist = bitmaps ? build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, reinterpret_cast<int*>(sm.cand_s),
                                                  2 * kCandCap, &sm.misc.lctr, sids, S)
                              : -1;
    if (state && nlist < 0) defer = true;
    TG_T(row, 1);

    float bv = -INFINITY;            // greedy: this lane's best unmarked score and index
    unsigned bi = 0xffffffffu;
    float ah = 0.0f, al = 0.0f;      // sampling: this lane's raw mass relative to ccl (hi + lo)
    float mxt = -INFINITY;           // sampling: largest raw logit this lane saw
    unsigned long long emask = 0ull; // sampling: units (sub-chunk, unit) of this lane that reached theta_raw
    float theta_raw = INFINITY;      // sampling: raw threshold (block-uniform)
    float ascale = kLog2e, cc0 = 0.0f;
    float ccl = 0.0f;                // sampling: this lane's reference for its running mass
    bool decided = false;            // sampling: m0 and theta_raw are set

    if (tma_ok) {
      for (int k = 0; k < nsub; ++k) {
        const int st = cur_st;
        const unsigned parity = cur_ph;
        if (++cur_st == nst) { cur_st = 0; cur_ph ^= 1u; }
        if (!*reinterpret_cast<volatile int*>(&sm.misc.error)) {
          if (!mbar_wait(&sm.misc.full[st], parity)) atomicExch(&sm.misc.error, 1);
        }
        const int lo = k * SE;
        const int n = min(SE, V - lo);
        const int scnt = max(0, min(SW, n - wid * SW));
        const int tok0 = lo + wid * SW;
        Slice sl;
        load_slice<DT>(ring + st * kStageBytes, wid * SW, scnt, sl);
        // the slice is in registers; the sixteenth warp to get here refills the stage
        __syncwarp();
        if (lane == 0) {
          // release: this warp's reads of the stage happen before the count;
          // acquire (for the sixteenth): every warp's reads happen before the refill
          const unsigned done = atom_add_acq_rel(&sm.misc.cnt[st], 1u);
          if ((done & (kWarps - 1)) == kWarps - 1) {
            fence_proxy_async();
            // the stage's next use: sub-chunk k + nst of this row, or of a later one
            int nk = k + nst, nri = ri;
            while (nk >= nsub) { nk -= nsub; ++nri; }
            if (nri < nrow && !*reinterpret_cast<volatile int*>(&sm.misc.error)) issue(st, nri, nk);
          }
        }
        if (!SAMPLE) {
          slice_greedy<DT>(sl, tok0, M, bitmaps, bv, bi);
          continue;
        }
        if (k == 0) {
          // First sub-chunk: the reference maximum m0 and the raw threshold.
          float mx = -INFINITY;
          {
            float x[4 * PER];
            slice_values<DT>(sl, x);
            if (bitmaps) {
              const unsigned mk = slice_marks<DT>(sl, tok0, M);
#pragma unroll
              for (int e = 0; e < 4 * PER; ++e) x[e] = ((mk >> e) & 1u) ? -INFINITY : x[e];
            }
            mx = tree_max<4 * PER>(x);
          }
          const float m0 = block_max(mx, &sm.red);
          if (m0 > kFilter && m0 < INFINITY) {
            const float T = tempered ? c.temp : 1.0f;
            unsigned cw[4];
            slice_level_counts<DT>(sl, m0, 0.5f / T, cw);
            if (lane == 0) {
#pragma unroll
              for (int q = 0; q < 4; ++q) sm.misc.lvl[wid][q] = cw[q];
            }
            csync();
            unsigned tot[4] = {0u, 0u, 0u, 0u};
            for (int w = 0; w < kWarps; ++w) {
#pragma unroll
              for (int q = 0; q < 4; ++q) tot[q] += sm.misc.lvl[w][q];
            }
            const unsigned cnt[8] = {tot[0] & 0xffffu, tot[1] & 0xffffu, tot[0] >> 16, tot[1] >> 16,
                                     tot[2] & 0xffffu, tot[3] & 0xffffu, tot[2] >> 16, tot[3] >> 16};
            const int n0 = min(V, SE);
            const int jl = pilot_level(cnt, static_cast<unsigned>(n0), static_cast<float>(V) / static_cast<float>(n0),
                                       topk, c.top_k, qfrac);
            theta_raw = jl >= 0 ? m0 - 2.0f * T * static_cast<float>(jl + 1) : m0;
            ascale = tempered ? kLog2e / c.temp : kLog2e;
            cc0 = m0 * ascale;
            ccl = cc0;
            decided = true;
          }
        }
        if (decided) slice_sample<DT>(sl, tok0, M, bitmaps, ascale, ccl, theta_raw, k, ah, al, mxt, emask);
      }
    } else {
      // rows not on a 16-byte boundary: read the logits directly
      if (!SAMPLE) {
        for (int i = tid; i < V; i += kThreads) {
          if (bitmaps && get_bit(M, i)) continue;
          const float x = load_logit<DT>(rowp, i);
          if (x > bv) { bv = x; bi = static_cast<unsigned>(i); }
        }
      }
    }

    // ---------------- finish the row (all threads) ----------------
    TG_T(row, 2);
    int token = -1;
    float tok_score = 0.0f, tok_ref = 0.0f;   // sampling: for the log-probability
    bool tok_fast = true;
    unsigned long long tok_S = 1ull;
    if (!SAMPLE) {
      // marked tokens, processed exactly, against the best unmarked one
      auto merge = [&](float s, int t) {
        if (s > bv || (s == bv && static_cast<unsigned>(t) < bi)) { bv = s; bi = static_cast<unsigned>(t); }
      };
      if (bitmaps && nlist >= 0) {
        for_listed<DT>(N, nlist, rowp, [&](float x, int t, unsigned e, int) {
          merge(process_listed(c, x, e, sids, svals, sm.misc.sfilt, false), t);
        });
      } else if (bitmaps) {
        for_marked<DT>(sm, rowp, M, a.nwords, [&](float x, int t) { merge(process_elem(c, M, N, x, t, false), t); });
      }
      for (int o = 16; o; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const unsigned i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
      }
      if (lane == 0) { sm.misc.wf[wid] = bv; sm.misc.wu[wid] = bi; }
      if (tid == 0) sm.misc.err_snap = *reinterpret_cast<volatile int*>(&sm.misc.error);
      csync();
      if (sm.misc.err_snap) break;   // uniform: every thread reads the same snapshot
      if (tid == 0) {
        float v = sm.misc.wf[0];
        unsigned b = sm.misc.wu[0];
        for (int q = 1; q < kWarps; ++q) {
          const float v2 = sm.misc.wf[q];
          const unsigned i2 = sm.misc.wu[q];
          if (v2 > v || (v2 == v && i2 < b)) { v = v2; b = i2; }
        }
        token = static_cast<int>(b);
      }
    } else {
      const float wmx = warp_max(mxt);
      if (lane == 0) sm.misc.wf[wid] = wmx;
      if (tid == 0) {
        sm.misc.err_snap = *reinterpret_cast<volatile int*>(&sm.misc.error);
        sm.misc.ncand = 0;
      }
      csync();
      TG_T(row, 15);
      if (sm.misc.err_snap) break;
      float m_raw = -INFINITY;
      for (int q = 0; q < kWarps; ++q) m_raw = fmaxf(m_raw, sm.misc.wf[q]);
      bool slow = !decided || !tma_ok || !(m_raw > kFilter);
      int reason = slow ? 3 : 0;
      unsigned tok = 0u;
      const float T = tempered ? c.temp : 1.0f;
      // every unmarked token with a processed score >= theta_f has x >= theta_raw
      const float theta_f = tempered ? nextafterf(__fdiv_rn(theta_raw, T), INFINITY) : theta_raw;
      float m = tempered ? clampf(__fdiv_rn(m_raw, T)) : m_raw;   // >= every unmarked score
      float cc_m = m * kLog2e;
      if (!slow) {
        const int nev = list_flagged<DT>(sm, emask);
        TG_T(row, 16);
        expand_units<DT>(c, sm, rowp, V, nev, false, M, bitmaps, theta_raw, theta_f, tempered);
        TG_T(row, 17);
        TG_T(row, 3);
        // marked tokens, processed exactly: their weight (against a thread-local
        // reference, raised when a processed score exceeds it) and their maximum
        float wp = 0.0f, pref = cc_m, mk_max = -INFINITY;
        auto push = [&](float s, int t) {
          if (s >= theta_f) {
            const int pos = atomicAdd(&sm.misc.ncand, 1);
            if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = static_cast<unsigned>(t); }
          }
        };
        if (bitmaps && nlist >= 0) {
          // listed: each processed score replaces its entry; the weights follow once m is known
          for_listed<DT>(N, nlist, rowp, [&](float x, int t, unsigned e, int j) {
            const float s = process_listed(c, x, e, sids, svals, sm.misc.sfilt, true);
            mk_max = fmaxf(mk_max, s);
            push(s, t);
            N[j] = __float_as_uint(s);
          });
        } else if (bitmaps) {
          // their weight against a thread-local reference, raised when a processed score exceeds it
          for_marked<DT>(sm, rowp, M, a.nwords, [&](float x, int t) {
            const float s = process_elem(c, M, N, x, t, true);
            const float sc = s * kLog2e;
            if (sc > pref) { wp *= ex2_approx(pref - sc); pref = sc; }
            wp += ex2_approx(sc - pref);
            mk_max = fmaxf(mk_max, s);
            push(s, t);
          });
        }
        // the reference maximum of the row: the larger of the unmarked maximum and the marked scores
        m = fmaxf(m, block_max(mk_max, &sm.red));
        cc_m = m * kLog2e;
        const float hot = decided ? (ah + al) * ex2_approx(ccl - cc_m) : 0.0f;
        unsigned long long zt;
        if (bitmaps && nlist >= 0) {
          // exact per-token weights: the same integers the candidates carry
          zt = fix44(hot);
          for (int j = tid; j < nlist; j += kThreads) zt += wfix_fast(__uint_as_float(N[j]), cc_m);
        } else {
          zt = fix44(hot + wp * ex2_approx(pref - cc_m));
        }
        const RowSums rs = block_row_sums(sm, zt, hot, 0.0f, false);
        TG_T(row, 18);
        const long long Zsigned = static_cast<long long>(rs.z);
        if (!(rs.hot < 3.0e38f) || Zsigned <= 0) { slow = true; reason = 2; }
        if (nev > kEvCap) { slow = true; reason = 25; }
        const int ncand = sm.misc.ncand;
        if (!slow && ncand > kCandCap) { slow = true; reason = 4; }
        TG_DBG(row, 2, m); TG_DBG(row, 3, theta_f); TG_DBG(row, 4, static_cast<double>(Zsigned) / kFixScale);
        TG_DBG(row, 7, ncand);
        TG_T(row, 4);
        if (!slow) {
          const FinResult fr = finalize2(c, sm, m, theta_f, static_cast<unsigned long long>(Zsigned), u, topk, topp);
          slow = !fr.ok;
          if (slow) reason = fr.reason;
          tok = fr.token;
          tok_score = fr.score;
          tok_ref = m * kLog2e;   // the finish weighs 2^(s log2e - m log2e)
          tok_S = fr.S;
          // Too little candidate mass for the cut or draw: one more pass, read
          // directly (the row is likely still in L2), with a lower threshold.
          // (a draw without top_p that misses its target lies in the bulk of the
          // row; only the exact path helps there)
          if (slow && reason == 5 && !state) {
            TG_T(row, 5);
            const FinResult fr2 = second_chance<DT>(c, a, sm, rm, rowp, M, N, bitmaps, theta_raw - 2.0f * T, tempered, m,
                                                    static_cast<unsigned long long>(Zsigned), u, topk, topp);
            slow = !fr2.ok;
            if (slow) reason = 10 + fr2.reason;
            tok = fr2.token;
            tok_score = fr2.score;
            tok_S = fr2.S;
          }
        }
      }
      TG_DBG(row, 0, slow ? 1 : 0); TG_DBG(row, 1, reason);
      TG_T(row, 6);
      if (slow && state) {
        defer = true;
      } else if (slow) {
        const SlowPick sp = slow_select<DT>(c, a, sm, rm, rowp, M, N, bitmaps, u);
        tok = sp.token;
        tok_score = sp.score;
        tok_ref = sp.ref;
        tok_fast = sp.fast;
        tok_S = sp.S;
      }
      token = static_cast<int>(tok);
    }

    // ---------------- outputs ----------------
    TG_T(row, 7);
    if (tid == 0) {
      // a row deferred here takes state_kernel's exact path: counted as slow
      if (defer) { atomicOr(c.status, kFlagSlow); atomicAdd(c.slow_rows, 1ull); }
      a.out[row] = defer ? kDeferred : token;
      if (SAMPLE && !VERIFY && a.logprobs && !defer) a.logprobs[row] = token_logprob(tok_score, tok_ref, tok_fast, tok_S);
      if (VERIFY) verify_ticket(c, a, row);
    }
    csync();
  }

  // error: wait (bounded) for the copies still in flight, then leave
  __syncthreads();
  if (sm.misc.error && tid == 0) {
    atomicOr(c.status, kFlagTimeout);
    for (int s = 0; s < nst; ++s) {
      const int n = sm.misc.iss[s];
      if (n > 0) mbar_wait(&sm.misc.full[s], static_cast<unsigned>((n - 1) & 1));
    }
  }
  // forced rows with a state, block-wide (the row bitmaps' area is free now);
  // after an error they stay deferred to state_kernel
  if (state && !sm.misc.error) {
    const int nf = sm.misc.nfst;
    for (int q = 0; q < nf; ++q) forced_state_row<SAMPLE>(c, a, sm, sm.rows[nrow + q], S);
  }
}

// ---------------------------------------------------------------------------
// process_kernel (diagnostic): one CTA per row, global-memory passes
// ---------------------------------------------------------------------------
struct ScoreSource {
  const float* s;
  int V;
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    for (int i = threadIdx.x; i < V; i += kThreads) f(s[i], static_cast<unsigned>(i));
  }
};

struct ProcSmem {
  Hist hist;
  RedScratch red;
};

// The task's processors, once per row, every thread: check the row's state
// (ids in [-1, V); within a processor's columns the ids in use ascend
// strictly and the unused -1 come after them), set the bitmap P of its ids
// and of a forced row's forced ids (a token outside P and the row bitmaps
// needs no processing), and fill the per-row fields of cr.  A state that breaks its layout is
// dropped for the row and raises kFlagBadState.  P has nwords words.
__device__ __forceinline__ void state_row_setup(DevCfg& cr, const RowMeta& rm, const int32_t* st_ids,
                                                const float* st_vals, int row, unsigned* P, int nwords,
                                                int* stage_ids, float* stage_vals) {
  const int S = cr.pcol[cr.nproc];
  const int32_t* ids = st_ids + static_cast<size_t>(row) * S;
  const float* vals = st_vals + static_cast<size_t>(row) * S;
  for (int w = threadIdx.x; w < nwords; w += kThreads) P[w] = 0u;
  __syncthreads();
  // the state is staged in shared memory: the processors search it per token
  for (int j = threadIdx.x; j < S; j += kThreads) {
    const int t = __ldg(ids + j);
    stage_ids[j] = t;
    stage_vals[j] = __ldg(vals + j);
    if (t >= 0 && t < cr.V) set_bit(P, t);
  }
  const bool bad = __syncthreads_or(state_layout_bad(cr, ids) ? 1 : 0) != 0;
  if (bad && threadIdx.x == 0) atomicOr(cr.status, kFlagBadState);
  cr.prow = true;
  cr.forced_row = rm.forced;
  cr.nfz = rm.forced ? forced_zeros(cr, rm, cr.fz) : 0;
  if (threadIdx.x < cr.nfz) set_bit(P, cr.fz[threadIdx.x]);
  __syncthreads();
  cr.pst_ids = bad ? nullptr : stage_ids;
  cr.pst_vals = bad ? nullptr : stage_vals;
  cr.pbits = P;
}

// Shared memory after the row bitmaps' area in state_kernel (where select_kernel
// keeps its TMA ring): the state bitmap P, the staged state (S ids, S values),
// and a forced row's list of tokens above F (S + 8 scores and ids).
__host__ __device__ constexpr int state_stage_bytes(int S) { return align_up(8 * S, 128); }
__host__ __device__ constexpr int sparse_list_bytes(int S) { return align_up(8 * (S + 8), 128); }

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    process_kernel(const DevCfg c, const SelArgs a, float* out_scores, unsigned* out_banbits, float* out_probs,
                   const int32_t* st_ids, const float* st_vals) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ProcSmem& sm = *reinterpret_cast<ProcSmem*>(smem_raw);
  const int fixed = align_up(static_cast<int>(sizeof(ProcSmem)), 128);
  unsigned* H = reinterpret_cast<unsigned*>(smem_raw + fixed);
  unsigned* N = reinterpret_cast<unsigned*>(smem_raw + fixed + bitmap_bytes(a.nwords));
  const int V = a.V;
  const int row = blockIdx.x;
  const bool sample = c.mode == kSample;
  RowMeta rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows);
  if (rm.bad || rm.L == 0) {
    if (rm.bad && threadIdx.x == 0) atomicOr(c.status, kFlagBadRow);
    return;
  }
  DevCfg cr = c;
  if (st_ids != nullptr) {
    unsigned char* area = smem_raw + fixed + 2 * bitmap_bytes(a.nwords);
    unsigned* P = reinterpret_cast<unsigned*>(area);
    int* sid = reinterpret_cast<int*>(area + bitmap_bytes(a.nwords));
    const int S = c.pcol[c.nproc];
    state_row_setup(cr, rm, st_ids, st_vals, row, P, a.nwords, sid, reinterpret_cast<float*>(sid + S));
  }
  const void* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * (DT == kF32 ? 4 : 2);
  float* sc = out_scores + static_cast<size_t>(row) * V;
  build_row_bitmaps(cr, a.hist, rm, H, N, a.nwords);
  int zs[8];
  int nz = rm.forced ? forced_zeros(c, rm, zs) : 0;
  for (int i = threadIdx.x; i < V; i += kThreads) {
    float s;
    if (rm.forced && !cr.prow) {
      s = kFilter;
      for (int q = 0; q < nz; ++q) if (zs[q] == i) s = 0.0f;
    } else {
      float x = DT == kF32 ? __ldg(static_cast<const float*>(rowp) + i)
                           : __uint_as_float(static_cast<unsigned>(__ldg(static_cast<const unsigned short*>(rowp) + i)) << 16);
      s = process_elem(cr, H, N, x, i, false);
    }
    if (!c.renorm && sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
    sc[i] = s;
  }
  if (c.renorm) {
    // renormalize_logits: (s - m) - ln S with S = sum exp(s - m), ln S as
    // hi + lo from S's exponent and log2f of its mantissa, then temperature.
    // The maximum comes off first: a row of equal scores at the filter value
    // gives -ln V (m + ln S would round back to m there).
    csync();
    float tm = -INFINITY;
    for (int i = threadIdx.x; i < V; i += kThreads) tm = fmaxf(tm, sc[i]);
    const float m = block_max(tm, &sm.red);
    float ts = 0.0f;
    for (int i = threadIdx.x; i < V; i += kThreads) ts += expf(sc[i] - m);
    const float S = block_sum_f(ts, &sm.red);
    constexpr double kLn2 = 0.6931471805599453;
    const unsigned b = __float_as_uint(S);
    const int e = static_cast<int>(b >> 23) - 127;
    const float mant = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
    const double lnS = (static_cast<double>(e) + static_cast<double>(log2f(mant))) * kLn2;
    const float hi = static_cast<float>(lnS), lo = static_cast<float>(lnS - static_cast<double>(hi));
    for (int i = threadIdx.x; i < V; i += kThreads) {
      float s = clampf(__fsub_rn(__fsub_rn(__fsub_rn(sc[i], m), hi), lo));
      if (sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
      sc[i] = s;
    }
  }
  if (out_banbits) {
    unsigned* bb = out_banbits + static_cast<size_t>(row) * a.nwords;
    for (int w = threadIdx.x; w < a.nwords; w += kThreads) {
      unsigned v;
      if (rm.forced) {
        v = 0xffffffffu;
        for (int q = 0; q < nz; ++q) if ((zs[q] >> 5) == w) v &= ~(1u << (zs[q] & 31));
      } else {
        v = N[w];
      }
      const int rem = V - w * 32;
      if (rem < 32) v &= (1u << rem) - 1u;
      bb[w] = v;
    }
  }
  csync();
  if (!out_probs) return;
  ScoreSource src{sc, V};
  float m = -INFINITY;
  src.pass([&](float s, unsigned) { m = fmaxf(m, s); });
  m = block_max(m, &sm.red);
  KeepFilter kept{0u, false, 0u, 0u};
  unsigned long long S;
  if (sample) {
    const float u = a.uniforms ? a.uniforms[row] : 0.0f;
    sample_exact(c, src, m, u, static_cast<unsigned>(V), &sm.hist, &sm.red, &kept, &S);
  } else {
    S = mass_sum(src, kept, WExact{m}, &sm.red);
  }
  float* pr = out_probs + static_cast<size_t>(row) * V;
  const double invS = 1.0 / static_cast<double>(S);
  for (int i = threadIdx.x; i < V; i += kThreads) {
    float s = sc[i];
    pr[i] = kept(fkey(s), static_cast<unsigned>(i)) ? static_cast<float>(static_cast<double>(wfix(s, m)) * invS) : 0.0f;
  }
}


// ---------------------------------------------------------------------------
// state_kernel: the rows of tg_select_state that select_kernel deferred
// (out == kDeferred): forced rows, rows whose marked tokens do not fit the
// list, rows that need the exact path, rows whose state breaks its layout
// (Transmuter.Generation, section "Processors").  One CTA per row at a time
// (grid-stride over the rows).  Per row: the state is checked and its ids
// (and a forced row's forced ids) set in a bitmap P, in the space the TMA
// ring takes in select_kernel; the row bitmaps are built; every token is
// processed by process_elem, which takes the processor path.  Greedy: one
// pass and a block argmax (lowest index on ties).  Sampling: the exact
// multi-pass selection of select_kernel's slow path, uncounted.  A forced row
// scores F except at its P tokens, which are all the passes visit (F tokens
// weigh nothing); when none scores above F every token ties.
// ---------------------------------------------------------------------------
template <int DT, bool SAMPLE>
__global__ void __launch_bounds__(kThreads, 1)
    state_kernel(const DevCfg c, const SelArgs a, const int32_t* st_ids, const float* st_vals) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  unsigned* H = reinterpret_cast<unsigned*>(smem_raw + fin_offset());
  unsigned* N = H + bitmap_bytes(a.nwords) / 4;
  unsigned char* area = smem_raw + ring_offset(a.nwords);
  unsigned* P = reinterpret_cast<unsigned*>(area);
  const int S = c.pcol[c.nproc];
  int* stage_ids = reinterpret_cast<int*>(area + bitmap_bytes(a.nwords));
  float* stage_vals = reinterpret_cast<float*>(stage_ids + S);
  float* sp_s = reinterpret_cast<float*>(area + bitmap_bytes(a.nwords) + state_stage_bytes(S));
  unsigned* sp_i = reinterpret_cast<unsigned*>(sp_s + S + 8);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int V = a.V;
  constexpr int esz = DT == kF32 ? 4 : 2;
  for (int row = blockIdx.x; row < a.nrows; row += gridDim.x) {
    if (a.fixup && __ldcg(a.out + row) != kDeferred) continue;
#ifdef TG_DEBUG
    if (tid == 0) sm.misc.dbg_row = row;
#endif
    TG_T(row, 0);
    const RowMeta rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows_total);
    if (rm.bad || rm.L == 0) {
      if (tid == 0) {
        a.out[row] = -1;
        if (SAMPLE && a.logprobs) a.logprobs[row] = __int_as_float(0x7fc00000);
        if (rm.bad) atomicOr(c.status, kFlagBadRow);
      }
      continue;
    }
    DevCfg cr = c;
    state_row_setup(cr, rm, st_ids, st_vals, row, P, a.nwords, stage_ids, stage_vals);
    TG_T(row, 1);
    // a forced row scores F, 0 or a processor's value: it needs no row bitmaps
    if (!rm.forced) build_row_bitmaps(cr, a.hist, rm, H, N, a.nwords, reinterpret_cast<int*>(sm.cand_s), 2 * kCandCap);
    TG_T(row, 2);
    const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * esz;
    const float u = (SAMPLE && a.uniforms) ? a.uniforms[row] : 0.0f;
    unsigned long long live = 1ull;
    if (rm.forced) {
      // list the tokens above F once (forced ids and state ids; final scores)
      if (tid == 0) sm.misc.ncand = 0;
      __syncthreads();
      for (int w = tid; w < a.nwords; w += kThreads) {
        unsigned bits = P[w];
        while (bits) {
          const int i = w * 32 + __ffs(bits) - 1;
          bits &= bits - 1u;
          float sc = process_state_elem(cr, H, N, 0.0f, i);
          if (SAMPLE && cr.temp != 1.0f) sc = clampf(__fdiv_rn(sc, cr.temp));
          if (sc > kFilter) {
            const int pos = atomicAdd(&sm.misc.ncand, 1);
            sp_s[pos] = sc;
            sp_i[pos] = static_cast<unsigned>(i);
          }
        }
      }
      __syncthreads();
      cr.sparse_row = true;
      cr.sp_s = sp_s;
      cr.sp_i = sp_i;
      cr.sp_n = sm.misc.ncand;
      live = static_cast<unsigned long long>(cr.sp_n);
      // top_k at or above the tokens above F keeps all of them (the rest weigh nothing)
      if (live > 0ull && static_cast<unsigned long long>(cr.top_k) >= live) cr.top_k = 0;
    }
    TG_T(row, 3);
    if (live == 0ull) {
      // every token scores F: all V tie
      if (tid == 0) {
        unsigned long long kept = 1ull;
        a.out[row] = equal_pick(cr, static_cast<unsigned long long>(V), u, SAMPLE, &kept);
        if (SAMPLE && a.logprobs) a.logprobs[row] = -logf(static_cast<float>(kept));
      }
    } else if (!SAMPLE) {
      RowGlobalSource<DT> src{rowp, V, &cr, H, N, !rm.forced, false};
      src.state_row(cr);
      float bv = -INFINITY;
      unsigned bi = 0xffffffffu;
      src.pass([&](float s, unsigned i) {
        if (s > bv || (s == bv && i < bi)) { bv = s; bi = i; }
      });
      for (int o = 16; o; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const unsigned i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
      }
      csync();
      if (lane == 0) { sm.misc.wf[wid] = bv; sm.misc.wu[wid] = bi; }
      csync();
      if (tid == 0) {
        float v = sm.misc.wf[0];
        unsigned b = sm.misc.wu[0];
        for (int q = 1; q < kWarps; ++q) {
          const float v2 = sm.misc.wf[q];
          const unsigned i2 = sm.misc.wu[q];
          if (v2 > v || (v2 == v && i2 < b)) { v = v2; b = i2; }
        }
        a.out[row] = static_cast<int>(b);
      }
    } else {
      bool done = false;
      if (rm.forced && cr.sp_n <= kCandCap) {
        // the one-pass path's candidate finish: the listed tokens hold all of
        // the row's mass (the rest score F and weigh nothing)
        const int n = cr.sp_n;
        float mx = -INFINITY, mn = INFINITY;
        for (int j = tid; j < n; j += kThreads) {
          sm.cand_s[j] = sp_s[j];
          sm.cand_i[j] = sp_i[j];
          mx = fmaxf(mx, sp_s[j]);
          mn = fminf(mn, sp_s[j]);
        }
        const float m = block_max(mx, &sm.red);
        const float lo = -block_max(-mn, &sm.red);
        const float cc = m * kLog2e;
        unsigned long long z = 0ull;
        for (int j = tid; j < n; j += kThreads) z += wfix_fast(sp_s[j], cc);
        const unsigned long long Z = block_sum_u64(z, &sm.red);
        if (tid == 0) sm.misc.ncand = n;
        csync();
        const bool topk = cr.top_k > 0 && cr.top_k < V;
        const bool topp = cr.top_p < 1.0f;
        const FinResult fr = finalize2(cr, sm, m, lo, Z, u, topk, topp);
        if (fr.ok) {
          if (tid == 0) {
            a.out[row] = static_cast<int>(fr.token);
            if (a.logprobs) a.logprobs[row] = token_logprob(fr.score, cc, true, fr.S);
          }
          done = true;
        }
      }
      if (!done) {
        const SlowPick sp = slow_select<DT>(cr, a, sm, rm, rowp, H, N, !rm.forced, u, false);
        if (tid == 0) {
          a.out[row] = static_cast<int>(sp.token);
          if (a.logprobs) a.logprobs[row] = token_logprob(sp.score, sp.ref, sp.fast, sp.S);
        }
      }
    }
    TG_T(row, 4);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// host-side launch helpers (C++ linkage, used by tg_api.cu)
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// tg_verify_noalloc: the verify step for callers that may not allocate.
//
// tg_verify keeps its per-row tickets in memory that tg_config_create
// allocates.  Some callers cannot allocate device memory at all: a serving
// engine that hands every byte of HBM to its KV-cache pool at start-up and
// forbids later allocations, or a decode loop where a cudaMalloc would
// synchronise the device in the middle of a pipelined step.  This variant
// takes the settings by value and keeps its tickets in a fixed array in the
// library's own device memory, so a call allocates nothing.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxBatch = TG_NOALLOC_MAX_BATCH;
// tickets [kNoAllocMaxBatch], then the status word, a pad and the slow-row counter
constexpr int kNoAllocWords = kNoAllocMaxBatch + 4;

// Shared by every tg_verify_noalloc call on a device; holds what the last
// call left (the tickets are cleared at the start of each call).  Every GPU
// that loads the library keeps this array until the process exits.
static __device__ __align__(256) unsigned g_noalloc_scratch[kNoAllocWords];

struct NoAllocDevice {
  bool ready;
  unsigned* scratch;   // device address of g_noalloc_scratch on this device
  int nsm;
  int nstage[2], smem[2], bps[2];   // launch plan per dtype
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: resolve the scratch array's
// device address, zero it, and plan the verify launch.
cudaError_t noalloc_setup(int dev, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, sizeof(g_noalloc_scratch));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev);
    int optin = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    for (int dt = 0; dt < 2 && e == cudaSuccess; ++dt) {
      const int ns = min(kRingStages, (optin - select_smem_bytes(0, 0)) / kStageBytes);
      d.nstage[dt] = ns;
      d.smem[dt] = select_smem_bytes(ns, 0);
      e = select_occupancy(dt, true, d.smem[dt], &d.bps[dt]);
      if (e == cudaSuccess && (ns < 2 || d.bps[dt] < 1)) e = cudaErrorInvalidConfiguration;
      d.bps[dt] = 1;
    }
    if (e != cudaSuccess) return e;
    d.scratch = static_cast<unsigned*>(p);
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_verify_noalloc(const void* target_logits, int32_t B, int32_t V, const int32_t* cand_ids,
                                       int32_t K, const tg_params* params, const float* uniforms,
                                       int32_t* out_match, int32_t* out_next, tg_stream stream) {
  using namespace tg;
  if (!params || V != params->vocab || V < 1 || B < 0 || K < 1) return TG_ERR_INVALID_ARGUMENT;
  if (V > TG_MAX_VOCAB) return TG_ERR_UNSUPPORTED;
  if (params->logits_dtype != TG_DTYPE_F32 && params->logits_dtype != TG_DTYPE_BF16) return TG_ERR_INVALID_ARGUMENT;
  if (params->mode != TG_GREEDY && params->mode != TG_SAMPLE) return TG_ERR_INVALID_ARGUMENT;
  if (!(params->temperature > 0.0f) || !(params->temperature < INFINITY)) return TG_ERR_INVALID_ARGUMENT;
  if (params->top_k < 0 || !(params->top_p > 0.0f && params->top_p <= 1.0f)) return TG_ERR_INVALID_ARGUMENT;
  if (B == 0) return TG_OK;
  if (B > kNoAllocMaxBatch) return TG_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * (K + 1) > 0x7fffffffLL) return TG_ERR_INVALID_ARGUMENT;
  if (!target_logits || !cand_ids || !out_match || !out_next) return TG_ERR_INVALID_ARGUMENT;
  if (params->mode == TG_SAMPLE && !uniforms) return TG_ERR_INVALID_ARGUMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return TG_ERR_CUDA;
  NoAllocDevice* d = nullptr;
  if (noalloc_setup(dev, &d) != cudaSuccess) return TG_ERR_CUDA;

  DevCfg c;
  memset(&c, 0, sizeof(c));
  c.V = V;
  c.dtype = params->logits_dtype;
  c.mode = params->mode;
  c.rho = 1.0f;
  c.bos = -1;
  c.temp = params->temperature;
  c.top_k = params->top_k;
  c.top_p = params->top_p;
  c.tickets = d->scratch;
  c.status = d->scratch + kNoAllocMaxBatch;
  c.slow_rows = reinterpret_cast<unsigned long long*>(d->scratch + kNoAllocMaxBatch + 2);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the tickets of this call start at zero
  if (cudaMemsetAsync(c.tickets, 0, static_cast<size_t>(B) * sizeof(unsigned), s) != cudaSuccess) return TG_ERR_CUDA;

  SelArgs a;
  memset(&a, 0, sizeof(a));
  a.logits = target_logits;
  a.nrows = B * (K + 1);
  a.nrows_total = a.nrows;
  a.V = V;
  a.uniforms = uniforms;
  a.out = out_next;
  a.cand = cand_ids;
  a.K = K;
  a.out_match = out_match;
  const int dt = c.dtype == kBF16 ? 1 : 0;
  a.nstage = d->nstage[dt];
  a.nwords = 0;
  const int grid = static_cast<int>(min(static_cast<long long>(a.nrows), static_cast<long long>(d->bps[dt]) * d->nsm));
  return launch_select(c, a, true, grid, d->smem[dt], s) == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

namespace tg {

int select_smem_bytes(int nstage, int nwords) { return ring_offset(nwords) + nstage * kStageBytes; }
int process_smem_bytes(int nwords, int S) {
  // the row bitmaps, the state bitmap and the staged state
  return align_up(static_cast<int>(sizeof(ProcSmem)), 128) + 3 * bitmap_bytes(nwords) + state_stage_bytes(S);
}
int state_smem_bytes(int nwords, int S) {
  return ring_offset(nwords) + bitmap_bytes(nwords) + state_stage_bytes(S) + sparse_list_bytes(S);
}

// One launch per kMaxRowsPerCta * grid rows; each is a programmatic dependent
// of the kernel before it in the stream (its launch overlaps that kernel's
// tail; it waits for it before touching global memory).
template <int DT, int VMODE, bool SAMPLE>
static cudaError_t launch_sel(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  auto k = select_kernel<DT, VMODE, SAMPLE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long per_launch = static_cast<long long>(grid) * kMaxRowsPerCta;
  for (long long r0 = 0; r0 < a.nrows_total; r0 += per_launch) {
    SelArgs b = a;
    b.row_begin = static_cast<int>(r0);
    b.nrows = static_cast<int>(r0 + per_launch < a.nrows_total ? r0 + per_launch : a.nrows_total);
    e = cudaLaunchKernelEx(&cfg, k, c, b);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

template <int DT, int VMODE>
static cudaError_t launch_sel_m(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  return c.mode == kSample ? launch_sel<DT, VMODE, true>(c, a, grid, smem, s) : launch_sel<DT, VMODE, false>(c, a, grid, smem, s);
}

template <int DT>
static cudaError_t launch_sel_v(const DevCfg& c, const SelArgs& a, bool verify, int grid, int smem, cudaStream_t s) {
  if (!verify) return launch_sel_m<DT, 0>(c, a, grid, smem, s);
  return a.vhist ? launch_sel_m<DT, 2>(c, a, grid, smem, s) : launch_sel_m<DT, 1>(c, a, grid, smem, s);
}

cudaError_t launch_select(const DevCfg& c, const SelArgs& a, bool verify, int grid, int smem, cudaStream_t s) {
  if (a.nstage < 2 || a.nstage > kMaxStages || grid < 1) return cudaErrorInvalidValue;
  return c.dtype == kF32 ? launch_sel_v<kF32>(c, a, verify, grid, smem, s) : launch_sel_v<kBF16>(c, a, verify, grid, smem, s);
}

cudaError_t launch_process(const DevCfg& c, const SelArgs& a, float* scores, unsigned* banbits, float* probs,
                           int smem, cudaStream_t s, const int32_t* st_ids, const float* st_vals) {
  cudaError_t e;
  if (c.dtype == kF32) {
    e = cudaFuncSetAttribute(process_kernel<kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    process_kernel<kF32><<<a.nrows, kThreads, smem, s>>>(c, a, scores, banbits, probs, st_ids, st_vals);
  } else {
    e = cudaFuncSetAttribute(process_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    process_kernel<kBF16><<<a.nrows, kThreads, smem, s>>>(c, a, scores, banbits, probs, st_ids, st_vals);
  }
  return cudaGetLastError();
}

template <int DT, bool SAMPLE>
static cudaError_t launch_state_t(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s,
                                  const int32_t* st_ids, const float* st_vals) {
  auto k = state_kernel<DT, SAMPLE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, s>>>(c, a, st_ids, st_vals);
  return cudaGetLastError();
}

cudaError_t launch_state(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s,
                         const int32_t* st_ids, const float* st_vals) {
  if (grid < 1) return cudaErrorInvalidValue;
  const bool sample = c.mode == kSample;
  if (c.dtype == kF32)
    return sample ? launch_state_t<kF32, true>(c, a, grid, smem, s, st_ids, st_vals)
                  : launch_state_t<kF32, false>(c, a, grid, smem, s, st_ids, st_vals);
  return sample ? launch_state_t<kBF16, true>(c, a, grid, smem, s, st_ids, st_vals)
                : launch_state_t<kBF16, false>(c, a, grid, smem, s, st_ids, st_vals);
}

cudaError_t select_occupancy(int dtype, bool verify, int smem, int* blocks_per_sm) {
  // the most demanding instantiation decides
  int worst = 1 << 20;
  for (int t = 0; t < 2; ++t) {
    void (*k)(DevCfg, SelArgs);
    if (dtype == kF32) k = verify ? (t ? select_kernel<kF32, 1, true> : select_kernel<kF32, 1, false>)
                                  : (t ? select_kernel<kF32, 0, true> : select_kernel<kF32, 0, false>);
    else k = verify ? (t ? select_kernel<kBF16, 1, true> : select_kernel<kBF16, 1, false>)
                    : (t ? select_kernel<kBF16, 0, true> : select_kernel<kBF16, 0, false>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, smem);
    if (e != cudaSuccess) return e;
    worst = occ < worst ? occ : worst;
  }
  *blocks_per_sm = worst;
  return cudaSuccess;
}

#ifdef TG_DEBUG
extern "C" int tg_debug_set(double* p) { return (int)cudaMemcpyToSymbol(g_dbg, &p, sizeof(p)); }
#endif

}  // namespace tg
