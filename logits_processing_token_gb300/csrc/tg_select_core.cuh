// Shared device machinery of the select kernels (sm_103a): PTX wrappers for
// mbarriers and 1-D bulk copies, the shared-memory layout, the exact finish
// over a candidate list, the multi-pass exact path over a row in global
// memory, forced rows, verify tickets and log-probabilities.  Included by
// tg_kernels.cu (select_kernel, process_kernel, state_kernel) and by
// tg_pipe.cu (the three-kernel path); internal to the library.
#pragma once

#include "../../include/tg.h"
#include "tg_device.cuh"

namespace tg {
// Internal linkage: every translation unit that includes this header gets its
// own copy of these functions.
namespace {


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
// Limit of the streaming waits in SM cycles (kWaitLimitCycles, ~1 s; a
// test may shorten it to make the waits run out).
__device__ unsigned long long g_wait_limit = kWaitLimitCycles;

// Bounded wait: false when the phase did not complete within `limit`
// cycles.  (try_wait may itself suspend the thread until the phase completes,
// so a completion seen later than the limit counts as a timeout too.)
__device__ __forceinline__ bool mbar_wait_for(unsigned long long* bar, unsigned parity, unsigned long long limit) {
  const long long t0 = clock64();
  for (;;) {
    const bool done = mbar_try_wait(bar, parity);
    const unsigned long long dt = static_cast<unsigned long long>(clock64() - t0);
    if (done) return dt <= limit;
    if (dt > limit) return false;
  }
}
// A streaming wait (g_wait_limit).
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity) {
  return mbar_wait_for(bar, parity, *static_cast<volatile unsigned long long*>(&g_wait_limit));
}
// The wait for copies still in flight after an error: always the full ~1 s.
__device__ __forceinline__ bool mbar_drain(unsigned long long* bar, unsigned parity) {
  return mbar_wait_for(bar, parity, kWaitLimitCycles);
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
  int nrow_done;                         // after a timeout: the first streamed row left unfinished
  int tbin;                              // tail_pick: the bin of the draw
  unsigned long long tbefore;            // tail_pick: the tail's mass before that bin
};

constexpr int kLevels = 2 * kThreads;   // value levels between the lowest candidate and the row max
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
  // pass() with eight vectors in flight per thread and the per-vector work
  // unrolled, for a row read again at the end of its finish (from L2 or
  // HBM, latency-bound at four vectors).  A small f only: it is inlined
  // eight times.
  template <class Fn>
  __device__ __forceinline__ void pass_deep(Fn f) const {
    constexpr int PER = DT == kF32 ? 4 : 8;
    constexpr int NV = 8;
    if (sparse || (reinterpret_cast<uintptr_t>(row) & 15u) != 0u) {
      pass(f);
      return;
    }
    const int nvec = V / PER;
    const uint4* rv = static_cast<const uint4*>(row);
    for (int v0 = 0; v0 < nvec; v0 += NV * kThreads) {
      uint4 q[NV];
#pragma unroll
      for (int h = 0; h < NV; ++h) {
        const int vi = v0 + h * kThreads + static_cast<int>(threadIdx.x);
        q[h] = vi < nvec ? __ldg(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < NV; ++h) {
        const int vi = v0 + h * kThreads + static_cast<int>(threadIdx.x);
        if (vi < nvec) {
          const unsigned ps[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
#pragma unroll
          for (int e = 0; e < PER; ++e) {
            const float x = DT == kF32 ? __uint_as_float(ps[e]) : ((e & 1) ? bf16hi(ps[e >> 1]) : bf16lo(ps[e >> 1]));
            const int i = vi * PER + e;
            f(score(x, i), static_cast<unsigned>(i));
          }
        }
      }
    }
    for (int i = nvec * PER + static_cast<int>(threadIdx.x); i < V; i += kThreads)
      f(score(load_logit<DT>(row, i), i), static_cast<unsigned>(i));
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
// A draw without top_k and top_p whose target lies past every candidate (the
// candidates hold the tokens scoring theta_f or more).  The row's tail
// (scores below theta_f) is read again from L2 into an exact histogram of
// the tail's fixed-point mass over kLevels bins of [m - 32, theta_f) (a score
// further below weighs less than 2^-44 of the maximum's weight and falls into
// the last bin); one block scan finds the bin in which the running mass,
// taken in (score desc, index asc) order after the candidates', passes the
// draw target; a third read lists that bin's tokens, and list_pick walks
// them in that order.  Every thread calls; the candidate list, sm.ev and the
// row bitmaps' area are free (the bitmaps are rebuilt).  Not ok when the bin
// holds more tokens than the candidate list.
template <int DT>
__device__ __noinline__ FinResult tail_pick(const DevCfg& c, const SelArgs& a, SelSmem& sm, const RowMeta& rm,
                                           const unsigned char* rowp, unsigned* M, unsigned* N, bool bitmaps,
                                           float theta_f, float m, unsigned long long Z, float u) {
  FinResult res{false, 40, 0u};
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float cc = m * kLog2e;
  // the candidates' exact mass, in the weights of the finish
  const int n = min(sm.misc.ncand, kCandCap);
  unsigned long long zc = 0ull;
  for (int i = tid; i < n; i += kThreads) zc += wfix_fast(sm.cand_s[i], cc);
  const unsigned long long Zc = block_sum_u64(zc, &sm.red);
  const unsigned long long Td = draw_target(u, Z);
  if (Td < Zc) { res.reason = 41; return res; }
  const unsigned long long R = Td - Zc;   // the draw's target within the tail
  TG_TF(19);
  // each bin's mass in two 32-bit words: the low words of the weights, and
  // their high words plus one for every add that carried out of the low word
  // (the thread whose add wrapped sees it in the value the atomic returns).
  // A tail weight is below 2^44 and V <= 2^18, so the high word stays below 2^32.
  static_assert(kEvCap >= 2 * kLevels, "tail histogram");
  unsigned* hlo = sm.ev;
  unsigned* hhi = sm.ev + kLevels;
  for (int l = tid; l < kLevels; l += kThreads) { hlo[l] = 0u; hhi[l] = 0u; }
  if (bitmaps) build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, reinterpret_cast<int*>(sm.cand_s), 2 * kCandCap);
  else csync();
  const float hi = theta_f, lo = m - 32.0f;
  const float scale = hi > lo ? static_cast<float>(kLevels) / (hi - lo) : 0.0f;
  auto bin = [&](float s) { return min(max(static_cast<int>((hi - s) * scale), 0), kLevels - 1); };
  RowGlobalSource<DT> src{rowp, a.V, &c, M, N, bitmaps, true};
  src.pass_deep([&](float s, unsigned) {
    if (s < hi) {
      const unsigned long long w = wfix_fast(s, cc);
      const int b = bin(s);
      const unsigned wl = static_cast<unsigned>(w);
      const unsigned old = atomicAdd(&hlo[b], wl);
      const unsigned wh = static_cast<unsigned>(w >> 32) + (old + wl < old ? 1u : 0u);
      if (wh) atomicAdd(&hhi[b], wh);
    }
  });
  csync();
  TG_TF(20);
  // bins 2t and 2t+1 per thread: the tail's mass before them, then the bin
  // whose running mass first passes R
  const int l0 = 2 * tid, l1 = l0 + 1;
  const unsigned long long m0 = (static_cast<unsigned long long>(hhi[l0]) << 32) + hlo[l0];
  const unsigned long long m1 = (static_cast<unsigned long long>(hhi[l1]) << 32) + hlo[l1];
  unsigned long long im = m0 + m1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) im += t;
  }
  if (lane == 31) sm.red.q[wid] = im;
  if (tid == 0) sm.misc.tbin = -1;
  csync();
  unsigned long long bm = im - (m0 + m1);
  for (int q = 0; q < wid; ++q) bm += sm.red.q[q];
  if (bm <= R && bm + m0 + m1 > R) {
    if (bm + m0 > R) { sm.misc.tbin = l0; sm.misc.tbefore = bm; }
    else { sm.misc.tbin = l1; sm.misc.tbefore = bm + m0; }
  }
  csync();
  const int bs = sm.misc.tbin;
  const unsigned long long before = sm.misc.tbefore;
  if (bs < 0) { res.reason = 42; return res; }
  // that bin's tokens become the candidates
  if (tid == 0) sm.misc.ncand = 0;
  csync();
  float smax = -INFINITY, smin = INFINITY;
  src.pass_deep([&](float s, unsigned t) {
    if (s < hi && bin(s) == bs) {
      const int pos = atomicAdd(&sm.misc.ncand, 1);
      if (pos < kCandCap) { sm.cand_s[pos] = s; sm.cand_i[pos] = t; }
      smax = fmaxf(smax, s);
      smin = fminf(smin, s);
    }
  });
  const float bhi = block_max(smax, &sm.red);
  const float blo = -block_max(-smin, &sm.red);
  if (sm.misc.ncand > kCandCap) { res.reason = 43; return res; }   // (read after block_max's barriers)
  const int nb = sm.misc.ncand;
  TG_TF(21);
  TG_DBG(sm.misc.dbg_row, 6, nb);
  const LevelPick d = list_pick(sm, nb, bhi, blo, cc, R - before, true, Zc + before);
  TG_TF(22);
  if (!d.ok) { res.reason = 44; return res; }
  res.ok = true;
  res.token = d.idx;
  res.score = key2f(d.key);
  res.S = Z;
  return res;
}

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


}  // namespace
}  // namespace tg
