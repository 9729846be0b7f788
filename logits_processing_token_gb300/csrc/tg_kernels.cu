// Token-selection kernels for sm_103a.
//
//  select_kernel  -- tg_select and tg_verify.  One CTA per row at a time
//                    (persistent over rows).  A producer warp streams every
//                    row once from HBM with 32 KB TMA bulk copies into a ring
//                    of shared-memory stages; 16 consumer warps each own a
//                    fixed slice of every stage and process it on their own
//                    (no CTA barrier while a row streams), releasing the
//                    stage through an mbarrier.
//  process_kernel -- tg_process (diagnostic): processed scores, ban bits and
//                    the final distribution, written to global memory.
//
// Processors.  Tokens that a history/ban bitmap marks are patched in the
// stage before a warp reads its slice (f32: the processed score in place;
// bf16: -inf in place and the exact f32 score in a per-warp side list).
//
// Sampling in one pass.  While streaming, every token's weight exp(s - m)
// (m = the warp's reference maximum) either joins the warp's excluded mass E
// (s below the warp's threshold theta) or the token joins the warp's
// candidate segment (s >= theta).  At the end of the row every warp drops
// candidates below the largest theta, so the candidates are exactly the
// tokens with s >= theta_final and all others are in E.  top_k, the top_p cut
// and the draw then run exactly on the candidates with fixed-point weights;
// the excluded tokens all sit after every candidate in the (score desc,
// index asc) order, so the result is exact whenever the candidates hold the
// k largest scores (top_k) or more mass than the cut (top_p) or the draw
// target needs.  A row where that check fails is streamed once more with a
// lower threshold, and then, if needed, decided by the multi-pass exact
// selection over the whole row.
#include <mutex>

#include "../../include/tg.h"
#include "tg_device.cuh"

namespace tg {

#ifdef TG_DEBUG
// Debug builds only: per-row record {path, reason, m, theta, E, Zc, Z, ncand}.
__device__ double* g_dbg = nullptr;
#define TG_DBG(row, slot, val) do { if (g_dbg && threadIdx.x == 0) g_dbg[(row) * 16 + (slot)] = (double)(val); } while (0)
#else
#define TG_DBG(row, slot, val) do { } while (0)
#endif
#ifdef TG_DEBUG
#define TG_GIVEUP(bit) atomicOr(&sm.misc.gcause, (bit))
#else
#define TG_GIVEUP(bit) do { } while (0)
#endif

constexpr int kProducerThreads = 32;                 // one producer warp
constexpr int kSelThreads = kThreads + kProducerThreads;

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
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         unsigned long long* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ unsigned long long evict_first_policy() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
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
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<unsigned long long>(clock64() - t0) > kWaitLimitCycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Shared-memory layout of select_kernel:
//   [SelSmem up to `fin`] [fin | row bitmaps H, N (aliased)] [stage ring]
// The bitmaps are needed while a row streams; FinSmem only while it is
// finished; the rare paths that need the bitmaps afterwards rebuild them.
// ---------------------------------------------------------------------------
constexpr int kMaxStages = 8;
constexpr int kSpecPerWarp = 128;                    // bf16 side list per warp and sub-chunk

struct Misc {
  unsigned long long full[kMaxStages];   // stage loaded (producer arrive + transaction bytes)
  unsigned long long empty[kMaxStages];  // stage released (one arrive per consumer warp)
  int wcnt[kWarps];                      // candidates in each warp's segment
  float wtheta[kWarps];                  // each warp's threshold at the end of a row
  float wmref[kWarps];                   // each warp's reference maximum
  int wflags[kWarps];                    // bit 0: decided, bit 1: gave up
  int ncand;                             // packed (contiguous) candidates, for the finish
  int error;                             // a wait timed out; the kernel stops
  int err_snap;                          // thread 0's snapshot of `error`, read by all consumers
  int gcause;                            // debug builds: why a warp gave up (bit mask)
  int issued;                            // sub-chunks the producer has issued (for the error path)
  float pr_mass[kWarps][32];             // per-warp prune histograms: levels of 0.5 below the max
  unsigned pr_cnt[kWarps][32];
};

// Each warp appends candidates to its own segment of the list (no atomics).
constexpr int kSeg = kCandCap / kWarps;

constexpr int kLevels = 1024;   // value levels between the lowest candidate and the row max
constexpr int kGroupCap = 256;  // largest level group sorted exactly in shared memory

struct FinSmem {
  unsigned long long lm[kLevels];  // weight of each level
  unsigned lc[kLevels];            // items in each level
  unsigned gk[kGroupCap];          // gathered group: key, index, weight
  unsigned gi[kGroupCap];
  unsigned long long gw[kGroupCap];
  unsigned sk[kGroupCap];          // the group sorted by (key desc, index asc)
  unsigned si[kGroupCap];
  unsigned long long sw[kGroupCap];
  int gn;
  int fb;                          // broadcast: bucket / position
  unsigned long long fbefore;      // broadcast: mass or count before it
  int ffound;
};

struct SelSmem {
  float cand_s[kCandCap];
  unsigned cand_i[kCandCap];
  float spec_s[kWarps * kSpecPerWarp];
  unsigned spec_i[kWarps * kSpecPerWarp];
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
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    for (int i = threadIdx.x; i < V; i += kThreads) {
      const float x = load_logit<DT>(row, i);
      float s = x;
      if (bitmaps) s = process_elem(*c, H, N, x, i, sample);
      else if (sample && c->temp != 1.0f) s = clampf(__fdiv_rn(x, c->temp));
      f(s, static_cast<unsigned>(i));
    }
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

// Append one (value, index) per lane that has one to this warp's segment.
// wc is the warp's count, kept uniform across the warp.
__device__ __forceinline__ void warp_push(bool has, float v, unsigned i, SelSmem& sm, int& wc) {
  const unsigned bal = __ballot_sync(0xffffffffu, has);
  if (bal == 0u) return;
  const int lane = threadIdx.x & 31;
  if (has) {
    const int pos = wc + __popc(bal & ((1u << lane) - 1u));
    if (pos < kSeg) {
      const int q = (threadIdx.x >> 5) * kSeg + pos;
      sm.cand_s[q] = v;
      sm.cand_i[q] = i;
    }
  }
  wc += __popc(bal);
}

// Fast mass (relative to c = m * log2e) of this warp's candidates.
__device__ __forceinline__ float warp_cand_mass(const SelSmem& sm, int wc, float c) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(wc, kSeg);
  float acc = 0.0f;
  for (int j = lane; j < n; j += 32) acc += wfast(sm.cand_s[w * kSeg + j], c);
  return warp_sum(acc);
}

// Drop this warp's candidates below theta (in place); returns the new count
// and, in `dropped` (all lanes), their fast mass relative to c.
__device__ __forceinline__ int warp_compact(SelSmem& sm, int wc, float theta, float c, float& dropped) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(wc, kSeg);
  float* S = sm.cand_s + w * kSeg;
  unsigned* I = sm.cand_i + w * kSeg;
  int out = 0;
  float dr = 0.0f;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const bool in = j < n;
    const float s = in ? S[j] : -INFINITY;
    const unsigned id = in ? I[j] : 0u;
    const bool keep = in && s >= theta;
    if (in && !keep) dr += wfast(s, c);
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) {
      const int pos = out + __popc(bal & ((1u << lane) - 1u));
      S[pos] = s;
      I[pos] = id;
    }
    out += __popc(bal);
    __syncwarp();
  }
  dropped = warp_sum(dr);
  return out;
}

// A higher threshold for this warp's candidates.  top_k: keep at least k of
// them; otherwise drop at most `allowed` fast mass.  Returns theta' >= theta.
__device__ float warp_choose_theta(SelSmem& sm, int wc, float theta, float m, float c, bool topk, int k,
                                   float allowed) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sm.misc.pr_mass[w][lane] = 0.0f;
  sm.misc.pr_cnt[w][lane] = 0u;
  __syncwarp();
  const int n = min(wc, kSeg);
  for (int j = lane; j < n; j += 32) {
    const float s = sm.cand_s[w * kSeg + j];
    const int lv = static_cast<int>(fminf(fmaxf((m - s) * 2.0f, 0.0f), 31.0f));
    atomicAdd(&sm.misc.pr_mass[w][lv], wfast(s, c));
    atomicAdd(&sm.misc.pr_cnt[w][lv], 1u);
  }
  __syncwarp();
  int jstar = 32;
  if (topk) {
    unsigned cum = 0u;
    for (int j = 0; j < 32; ++j) {
      cum += sm.misc.pr_cnt[w][j];
      if (cum >= static_cast<unsigned>(k)) { jstar = j + 1; break; }
    }
  } else {
    float tail = 0.0f;
    for (int j = 31; j >= 0; --j) {
      const float t2 = tail + sm.misc.pr_mass[w][j];
      if (t2 > allowed) break;
      tail = t2;
      jstar = j;
    }
  }
  __syncwarp();
  const float cand = (jstar >= 32) ? theta : m - 0.5f * static_cast<float>(jstar);
  return fmaxf(theta, cand);
}

// Largest t in [lo, hi] with at least `keep` of this warp's candidates at
// or above t (bisection on the score; all lanes get the same result).
__device__ __forceinline__ float warp_keep_score(const SelSmem& sm, int wc, int keep, float lo, float hi) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(wc, kSeg);
  for (int it = 0; it < 20; ++it) {
    const float mid = 0.5f * (lo + hi);
    int cnt = 0;
    for (int j = lane; j < n; j += 32) cnt += sm.cand_s[w * kSeg + j] >= mid ? 1 : 0;
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (cnt >= keep) lo = mid; else hi = mid;
  }
  return lo;
}

// Fast mass of this warp's candidates below t (all lanes).
__device__ __forceinline__ float warp_mass_below(const SelSmem& sm, int wc, float t, float c) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(wc, kSeg);
  float acc = 0.0f;
  for (int j = lane; j < n; j += 32) {
    const float s = sm.cand_s[w * kSeg + j];
    if (s < t) acc += wfast(s, c);
  }
  return warp_sum(acc);
}

// Make room in this warp's segment: raise theta so that about half of it
// stays, but never past the point where the excluded mass E (+ what is
// dropped) exceeds `allowed_frac` of everything this warp has seen; top_k
// keeps at least k.  Returns the new theta (>= theta).
__device__ __forceinline__ float warp_make_room(SelSmem& sm, int wc, float theta, float mx, float c, float et_sum,
                                                bool topk, int k, float allowed_frac) {
  const int keep = topk ? max(kSeg / 2, k) : kSeg / 2;
  const float tcap = warp_keep_score(sm, wc, keep, theta, fmaxf(mx, theta));
  const float zc = warp_cand_mass(sm, wc, c);
  const float dropped = warp_mass_below(sm, wc, tcap, c);
  if (topk || et_sum + dropped <= allowed_frac * (et_sum + zc)) return fmaxf(theta, tcap);
  // the budget stops short of the capacity target: go as far as it allows
  return warp_choose_theta(sm, wc, theta, mx, c, false, 0, allowed_frac * (et_sum + zc) - et_sum);
}

// Block-wide choice of a higher threshold over all warps' candidates: top_k
// keeps at least 2k; otherwise the excluded mass may grow by `allowed`.
// Every consumer thread calls; all get the same theta' >= theta.
__device__ float block_choose_theta(SelSmem& sm, int wc, float theta, float m, float c, bool topk, int k,
                                    float allowed) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sm.misc.pr_mass[w][lane] = 0.0f;
  sm.misc.pr_cnt[w][lane] = 0u;
  __syncwarp();
  const int n = min(wc, kSeg);
  for (int j = lane; j < n; j += 32) {
    const float s = sm.cand_s[w * kSeg + j];
    const int lv = static_cast<int>(fminf(fmaxf((m - s) * 2.0f, 0.0f), 31.0f));
    atomicAdd(&sm.misc.pr_mass[w][lv], wfast(s, c));
    atomicAdd(&sm.misc.pr_cnt[w][lv], 1u);
  }
  csync();
  if (threadIdx.x < 32) {
    float tm = 0.0f;
    unsigned tc = 0u;
    for (int q = 0; q < kWarps; ++q) { tm += sm.misc.pr_mass[q][threadIdx.x]; tc += sm.misc.pr_cnt[q][threadIdx.x]; }
    sm.misc.pr_mass[0][threadIdx.x] = tm;
    sm.misc.pr_cnt[0][threadIdx.x] = tc;
  }
  csync();
  int jstar = 32;
  if (topk) {
    unsigned cum = 0u;
    for (int j = 0; j < 32; ++j) {
      cum += sm.misc.pr_cnt[0][j];
      if (cum >= static_cast<unsigned>(2 * k)) { jstar = j + 1; break; }
    }
  } else {
    float tail = 0.0f;
    for (int j = 31; j >= 0; --j) {
      const float t2 = tail + sm.misc.pr_mass[0][j];
      if (t2 > allowed) break;
      tail = t2;
      jstar = j;
    }
  }
  csync();
  const float cand = (jstar >= 32) ? theta : m - 0.5f * static_cast<float>(jstar);
  return fmaxf(theta, cand);
}

// Block-wide: the lowest threshold theta' >= theta (on levels of 0.5 below
// m) at which the candidates at or above it, times `scale` (the row's
// sub-chunks per sub-chunk seen), fill at most three quarters of the list.
__device__ float block_capacity_theta(SelSmem& sm, int wc, float theta, float m, float scale) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sm.misc.pr_cnt[w][lane] = 0u;
  __syncwarp();
  const int n = min(wc, kSeg);
  for (int j = lane; j < n; j += 32) {
    const float s = sm.cand_s[w * kSeg + j];
    const int lv = static_cast<int>(fminf(fmaxf((m - s) * 2.0f, 0.0f), 31.0f));
    atomicAdd(&sm.misc.pr_cnt[w][lv], 1u);
  }
  csync();
  if (threadIdx.x < 32) {
    unsigned tc = 0u;
    for (int q = 0; q < kWarps; ++q) tc += sm.misc.pr_cnt[q][threadIdx.x];
    sm.misc.pr_cnt[0][threadIdx.x] = tc;
  }
  csync();
  // level j holds scores in (m - 0.5(j+1), m - 0.5j]; keeping levels < j
  // means theta' = m - 0.5 j
  const float cap = 0.75f * static_cast<float>(kCandCap);
  int jbest = 0;
  float cum = 0.0f;
  for (int j = 1; j <= 32; ++j) {
    cum += static_cast<float>(sm.misc.pr_cnt[0][j - 1]);
    if (cum * scale <= cap) jbest = j; else break;
  }
  csync();
  const float cand = m - 0.5f * static_cast<float>(jbest);
  return fmaxf(theta, cand);
}

// Move the warp segments into one contiguous list [0, ncand).
__device__ void pack_candidates(SelSmem& sm) {
  constexpr int kPer = kSeg / 32;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int off = 0;
  for (int q = 0; q < w; ++q) off += min(sm.misc.wcnt[q], kSeg);
  const int n = min(sm.misc.wcnt[w], kSeg);
  float vs[kPer];
  unsigned is[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int q = lane + 32 * j;
    vs[j] = q < n ? sm.cand_s[w * kSeg + q] : 0.0f;
    is[j] = q < n ? sm.cand_i[w * kSeg + q] : 0u;
  }
  csync();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int q = lane + 32 * j;
    if (q < n) { sm.cand_s[off + q] = vs[j]; sm.cand_i[off + q] = is[j]; }
  }
  if (threadIdx.x == 0) {
    int t = 0;
    for (int q = 0; q < kWarps; ++q) t += min(sm.misc.wcnt[q], kSeg);
    sm.misc.ncand = t;
  }
  csync();
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
// fin.fbefore = base + sum(sw[0..j-1]), fin.ffound.
__device__ __forceinline__ void walk_sorted(SelSmem& sm, int cnt, unsigned long long base,
                                            unsigned long long target, bool strict) {
  FinSmem& f = sm.fin;
  if (threadIdx.x < 32) {
    constexpr int PER = kGroupCap / 32;
    const int lane = threadIdx.x;
    unsigned long long local = 0ull;
    for (int j = 0; j < PER; ++j) {
      const int q = lane * PER + j;
      if (q < cnt) local += f.sw[q];
    }
    unsigned long long incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned long long excl = incl - local;
    const unsigned long long tot = base + incl;
    const unsigned hit = __ballot_sync(0xffffffffu, strict ? tot > target : tot >= target);
    if (hit) {
      const int L = __ffs(hit) - 1;
      if (lane == L) {
        unsigned long long cum = base + excl;
        int j = lane * PER;
        for (; j < lane * PER + PER && j < cnt; ++j) {
          const unsigned long long nx = cum + f.sw[j];
          if (strict ? nx > target : nx >= target) break;
          cum = nx;
        }
        f.fb = j;
        f.fbefore = cum;
        f.ffound = 1;
      }
    } else if (lane == 0) {
      unsigned long long all = 0ull;
      for (int j = 0; j + 1 < cnt; ++j) all += f.sw[j];
      f.fb = cnt - 1;
      f.fbefore = base + all;
      f.ffound = 0;
    }
  }
  csync();
}

// Level search by warp 0 over fin.lm / fin.lc; results in fin.fb/fbefore/ffound.
template <class Reached>
__device__ __forceinline__ void level_find_mass(SelSmem& sm, Reached r) {
  if (threadIdx.x < 32) {
    FindOut<unsigned long long> o = warp_find<kLevels>(sm.fin.lm, sm.fin.lc, false, r);
    if (threadIdx.x == 0) { sm.fin.fb = o.b; sm.fin.fbefore = o.before; sm.fin.ffound = o.found; }
  }
  csync();
}

// Keep only levels < L in full and the first `mass`/`cnt` of level L.
__device__ __forceinline__ void level_limit(SelSmem& sm, int L, unsigned long long mass, unsigned cnt) {
  for (int l = threadIdx.x; l < kLevels; l += kThreads) {
    if (l > L) { sm.fin.lm[l] = 0ull; sm.fin.lc[l] = 0u; }
    else if (l == L) { sm.fin.lm[l] = mass; sm.fin.lc[l] = cnt; }
  }
  csync();
}

struct FinResult {
  bool ok;        // false: the candidates cannot decide this row
  int reason;
  unsigned token;
};

// top_k, top_p and the draw over the candidates.  E_fix = fixed-point mass
// of every token below theta.
__device__ FinResult finalize_candidates(const DevCfg& c, SelSmem& sm, float m, unsigned long long E_fix,
                                         float u, bool topk, bool topp) {
  const float cc = m * kLog2e;
  const WFast wf{cc};
  FinResult res{false, 0, 0u};
  FinSmem& f = sm.fin;
  const int n = min(sm.misc.ncand, kCandCap);
  if (n <= 0) { res.reason = 9; return res; }
  // level map from the lowest candidate to the maximum
  float smin = INFINITY;
  for (int i = threadIdx.x; i < n; i += kThreads) smin = fminf(smin, sm.cand_s[i]);
  smin = -block_max(-smin, &sm.red);
  const float range = m - smin;
  LevelMap lv{m, range > 0.0f ? static_cast<float>(kLevels - 1) / range : 0.0f};
  for (int l = threadIdx.x; l < kLevels; l += kThreads) { f.lm[l] = 0ull; f.lc[l] = 0u; }
  csync();
  unsigned long long zc = 0ull;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const float s = sm.cand_s[i];
    const int l = lv(s);
    const unsigned long long w = wfix_fast(s, cc);
    zc += w;
    atomicAdd(&f.lm[l], w);
    atomicAdd(&f.lc[l], 1u);
  }
  const unsigned long long Zc = block_sum_u64(zc, &sm.red);
  unsigned klo = 0u;
  unsigned long long Z;
  if (topk) {
    if (n < c.top_k) { res.reason = 4; return res; }
    // level holding the k-th largest token
    if (threadIdx.x < 32) {
      const unsigned need = static_cast<unsigned>(c.top_k);
      FindOut<unsigned> o = warp_find<kLevels>(f.lc, f.lc, false, [need](unsigned x) { return x >= need; });
      if (threadIdx.x == 0) { f.fb = o.b; f.fbefore = o.before; }
    }
    csync();
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
    Z = Zc + E_fix;
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
    if (!f.ffound) { res.reason = 6; return res; }
    Lc = f.fb;
    const unsigned long long before = f.fbefore;
    csync();
    const int gn = gather_sort_level(sm, n, lv, Lc, klo, cc);
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
  }
  const unsigned long long Td = draw_target(u, S);
  if (!topk && !topp && !(Zc > Td)) { res.reason = 7; return res; }
  level_find_mass(sm, [Td](unsigned long long x) { return x > Td; });
  if (!f.ffound) { res.reason = 8; return res; }
  const int Ld = f.fb;
  const unsigned long long before = f.fbefore;
  csync();
  if (Ld == Lc && cut_sorted) {
    walk_sorted(sm, nc, before, Td, true);
    res.token = f.si[f.fb];
  } else {
    const int gn = gather_sort_level(sm, n, lv, Ld, klo, cc);
    if (gn >= 0) {
      const int lim = (Ld == Lc) ? nc : gn;
      walk_sorted(sm, lim, before, Td, true);
      res.token = f.si[f.fb];
    } else {
      CandLevelSource ls{sm.cand_s, sm.cand_i, n, lv, Ld};
      MassSel d = mass_select(ls, keep, wf, Td - before, true, &sm.hist);
      if (!d.found) { res.reason = 8; return res; }
      res.token = d.idx;
    }
  }
  csync();
  res.ok = true;
  return res;
}

// Select element j (0..N-1) of a register array without dynamic indexing.
template <int N>
__device__ __forceinline__ float pick(const float (&s)[N], int j) {
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = s[i];
#pragma unroll
  for (int w = N / 2, b = 0; w >= 1; w >>= 1, ++b) {
    const bool hi = (j >> b) & 1;
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = hi ? t[2 * i + 1] : t[2 * i];
  }
  return t[0];
}

// ---------------------------------------------------------------------------
// Per-warp slice work.  Warp w owns elements [w*SW, (w+1)*SW) of every
// sub-chunk (SW = SE / kWarps: 1024 bf16 or 512 f32, i.e. 2 KB); `soff` is
// that offset within the stage, `tok0` the slice's first token.
// ---------------------------------------------------------------------------

// Patch the tokens the row bitmaps mark in this warp's slice (a2-a9).  f32:
// the processed score replaces the logit.  bf16: the slot becomes -inf and
// the exact f32 score goes to the warp's side list; returns its length.
template <int DT>
__device__ __forceinline__ int warp_patch(unsigned char* stage, int soff, int scnt, int tok0, const unsigned* H,
                                          const unsigned* N, float rho, float* ss, unsigned* si, bool& ovf) {
  const int lane = threadIdx.x & 31;
  const int nw = (scnt + 31) >> 5;
  unsigned bits = 0u, nb = 0u;
  if (lane < nw) {
    const int wd = (tok0 >> 5) + lane;
    bits = H[wd] | N[wd];
    nb = N[wd];
    const int rem = scnt - lane * 32;
    if (rem < 32) bits &= (1u << rem) - 1u;
  }
  int pos = 0, total = 0;
  if (DT == kBF16) {
    const int cnt = __popc(bits);
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    pos = incl - cnt;
    if (total > kSpecPerWarp) ovf = true;
  }
  while (bits) {
    const int b = __ffs(bits) - 1;
    bits &= bits - 1u;
    const int local = soff + lane * 32 + b;
    if (DT == kF32) {
      float* sf = reinterpret_cast<float*>(stage);
      sf[local] = ((nb >> b) & 1u) ? kFilter : penalize(sf[local], rho);
    } else {
      unsigned short* sh = reinterpret_cast<unsigned short*>(stage);
      const float x = __uint_as_float(static_cast<unsigned>(sh[local]) << 16);
      const float s = ((nb >> b) & 1u) ? kFilter : penalize(x, rho);
      if (pos < kSpecPerWarp) { ss[pos] = s; si[pos] = static_cast<unsigned>(tok0 + lane * 32 + b); }
      ++pos;
      sh[local] = 0xff80u;  // -inf: counted through the side list
    }
  }
  __syncwarp();
  return DT == kBF16 ? min(total, kSpecPerWarp) : 0;
}

// Raw (pre-temperature) maximum of this warp's slice, all lanes.
template <int DT>
__device__ __forceinline__ float warp_slice_max(const unsigned char* stage, int soff, int scnt, int nspec,
                                                const float* ss) {
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY;
  if (DT == kF32) {
    const float4* v4 = reinterpret_cast<const float4*>(stage + soff * 4);
    const int nv = scnt >> 2;
    for (int v = lane; v < nv; v += 32) {
      const float4 q = v4[v];
      mx = fmaxf(mx, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
    }
    const float* sf = reinterpret_cast<const float*>(stage) + soff;
    for (int i = (nv << 2) + lane; i < scnt; i += 32) mx = fmaxf(mx, sf[i]);
  } else {
    const uint4* v4 = reinterpret_cast<const uint4*>(stage + soff * 2);
    const int nv = scnt >> 3;
    __nv_bfloat162 m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    for (int v = lane; v < nv; v += 32) {
      uint4 q = v4[v];
      m2 = __hmax2(m2, __hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.x), *reinterpret_cast<__nv_bfloat162*>(&q.y)),
                               __hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.z), *reinterpret_cast<__nv_bfloat162*>(&q.w))));
    }
    mx = fmaxf(__low2float(m2), __high2float(m2));
    const unsigned short* sh = reinterpret_cast<const unsigned short*>(stage) + soff;
    for (int i = (nv << 3) + lane; i < scnt; i += 32) mx = fmaxf(mx, __uint_as_float(static_cast<unsigned>(sh[i]) << 16));
    for (int i = lane; i < nspec; i += 32) mx = fmaxf(mx, ss[i]);
  }
  return warp_max(mx);
}

// Greedy over this warp's slice: each lane keeps its best (score, lowest index).
template <int DT>
__device__ __forceinline__ void warp_greedy(const unsigned char* stage, int soff, int scnt, int tok0, int nspec,
                                            const float* ss, const unsigned* si, float& bv, unsigned& bi) {
  const int lane = threadIdx.x & 31;
  if (DT == kF32) {
    const float4* v4 = reinterpret_cast<const float4*>(stage + soff * 4);
    const int nv = scnt >> 2;
    for (int v = lane; v < nv; v += 32) {
      const float4 q = v4[v];
      const float vm = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
      if (vm > bv) {
        const int j = q.x == vm ? 0 : q.y == vm ? 1 : q.z == vm ? 2 : 3;
        bv = vm;
        bi = static_cast<unsigned>(tok0 + 4 * v + j);
      }
    }
    const float* sf = reinterpret_cast<const float*>(stage) + soff;
    for (int i = (nv << 2) + lane; i < scnt; i += 32)
      if (sf[i] > bv) { bv = sf[i]; bi = static_cast<unsigned>(tok0 + i); }
  } else {
    const uint4* v4 = reinterpret_cast<const uint4*>(stage + soff * 2);
    const int nv = scnt >> 3;
    for (int v = lane; v < nv; v += 32) {
      uint4 q = v4[v];
      __nv_bfloat162 m2 = __hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.x), *reinterpret_cast<__nv_bfloat162*>(&q.y)),
                                  __hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.z), *reinterpret_cast<__nv_bfloat162*>(&q.w)));
      const float vm = fmaxf(__low2float(m2), __high2float(m2));
      if (vm > bv) {
        const unsigned ps[4] = {q.x, q.y, q.z, q.w};
        int jj = 7;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          const float x = (j & 1) ? bf16hi(ps[j >> 1]) : bf16lo(ps[j >> 1]);
          if (x == vm) jj = j;
        }
        bv = vm;
        bi = static_cast<unsigned>(tok0 + 8 * v + jj);
      }
    }
    const unsigned short* sh = reinterpret_cast<const unsigned short*>(stage) + soff;
    for (int i = (nv << 3) + lane; i < scnt; i += 32) {
      const float x = __uint_as_float(static_cast<unsigned>(sh[i]) << 16);
      if (x > bv) { bv = x; bi = static_cast<unsigned>(tok0 + i); }
    }
    for (int i = lane; i < nspec; i += 32) {
      const float s = ss[i];
      const unsigned id = si[i];
      if (s > bv || (s == bv && id < bi)) { bv = s; bi = id; }
    }
  }
}

// Number of this warp's slice tokens (tempered) at or above t, all lanes.
template <int DT, bool TEMP>
__device__ __forceinline__ int warp_slice_count(const unsigned char* stage, int soff, int scnt, int nspec,
                                                const float* ss, float temp, float t) {
  const int lane = threadIdx.x & 31;
  int cnt = 0;
  for (int i = lane; i < scnt; i += 32) {
    float s = DT == kF32 ? reinterpret_cast<const float*>(stage)[soff + i]
                         : __uint_as_float(static_cast<unsigned>(reinterpret_cast<const unsigned short*>(stage)[soff + i]) << 16);
    if (TEMP) s = temper(s, temp);
    cnt += s >= t ? 1 : 0;
  }
  for (int i = lane; i < nspec; i += 32) cnt += (TEMP ? clampf(__fdiv_rn(ss[i], temp)) : ss[i]) >= t ? 1 : 0;
  for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt;
}

// A slice overflowed the warp's segment: the lowest t (bisection) at which
// the listed candidates plus the slice's tokens at or above t fill at most
// three quarters of the segment.
template <int DT, bool TEMP>
__device__ float warp_overflow_theta(const SelSmem& sm, int wc, const unsigned char* stage, int soff, int scnt,
                                     int nspec, const float* ss, float temp, float lo, float hi) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(wc, kSeg);
  const int target = (3 * kSeg) / 4;
  for (int it = 0; it < 20; ++it) {
    const float mid = 0.5f * (lo + hi);
    int cnt = 0;
    for (int j = lane; j < n; j += 32) cnt += sm.cand_s[w * kSeg + j] >= mid ? 1 : 0;
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    cnt += warp_slice_count<DT, TEMP>(stage, soff, scnt, nspec, ss, temp, mid);
    if (cnt <= target) hi = mid; else lo = mid;
  }
  return hi;
}

// Sampling over this warp's slice: tokens below theta add their weight
// 2^(s*log2e - cc) to et, the others go to the warp's candidate segment; mxt
// tracks the largest (tempered) score.
template <int DT, bool TEMP>
__device__ __forceinline__ void warp_pass(const unsigned char* stage, int soff, int scnt, int tok0, int nspec,
                                          const float* ss, const unsigned* si, SelSmem& sm, float temp, float theta,
                                          float cc, float& et, float& mxt, int& wc) {
  constexpr int PER = DT == kF32 ? 4 : 8;      // elements per 16-byte vector
  constexpr int NE = 2 * PER;                  // elements per lane and round
  const int lane = threadIdx.x & 31;
  const int nv = scnt / PER;
  const unsigned char* base_ptr = stage + soff * (DT == kF32 ? 4 : 2);
  float* S = sm.cand_s + (threadIdx.x >> 5) * kSeg;
  unsigned* I = sm.cand_i + (threadIdx.x >> 5) * kSeg;
  int v0 = 0;
  // rounds of two vectors per lane: every weight first, then one warp scan
  for (; v0 + 64 <= nv; v0 += 64) {
    float s[NE];
    float vm;
    const int va = v0 + lane, vb = v0 + 32 + lane;
    if (DT == kF32) {
      const float4* v4 = reinterpret_cast<const float4*>(base_ptr);
      const float4 a = v4[va], b = v4[vb];
      s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
      s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
      vm = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
    } else {
      const uint4* v4 = reinterpret_cast<const uint4*>(base_ptr);
      uint4 a = v4[va], b = v4[vb];
      const unsigned ps[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] = (j & 1) ? bf16hi(ps[j >> 1]) : bf16lo(ps[j >> 1]);
      __nv_bfloat162 m2 = __hmax2(__hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&a.x), *reinterpret_cast<__nv_bfloat162*>(&a.y)),
                                          __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a.z), *reinterpret_cast<__nv_bfloat162*>(&a.w))),
                                  __hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&b.x), *reinterpret_cast<__nv_bfloat162*>(&b.y)),
                                          __hmax2(*reinterpret_cast<__nv_bfloat162*>(&b.z), *reinterpret_cast<__nv_bfloat162*>(&b.w))));
      vm = fmaxf(__low2float(m2), __high2float(m2));
    }
    if (TEMP) {
      vm = temper(vm, temp);
#pragma unroll
      for (int j = 0; j < NE; ++j) s[j] = temper(s[j], temp);
    }
    mxt = fmaxf(mxt, vm);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    unsigned cm = 0u;
#pragma unroll
    for (int j = 0; j < NE; ++j) {
      const float w = wfast(s[j], cc);
      const bool cnd = s[j] >= theta;
      cm |= cnd ? (1u << j) : 0u;
      acc[j & 3] += cnd ? 0.0f : w;
    }
    et += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    if (__any_sync(0xffffffffu, cm != 0u)) {
      const int cnt = __popc(cm);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      int pos = wc + incl - cnt;
      wc += total;
      while (cm) {
        const int j = __ffs(cm) - 1;
        cm &= cm - 1u;
        const unsigned id = static_cast<unsigned>(tok0 + (j < PER ? PER * va + j : PER * vb + (j - PER)));
        if (pos < kSeg) { S[pos] = pick<NE>(s, j); I[pos] = id; }
        ++pos;
      }
    }
  }
  // remaining whole vectors, then single elements
  for (; v0 < nv; v0 += 32) {
    const int v = v0 + lane;
    const bool in = v < nv;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      float s = -INFINITY;
      if (in) {
        if (DT == kF32) s = reinterpret_cast<const float*>(base_ptr)[v * PER + j];
        else s = __uint_as_float(static_cast<unsigned>(reinterpret_cast<const unsigned short*>(base_ptr)[v * PER + j]) << 16);
        if (TEMP) s = temper(s, temp);
      }
      mxt = fmaxf(mxt, s);
      const bool cnd = s >= theta;
      if (!cnd) et += wfast(s, cc);
      warp_push(cnd, s, static_cast<unsigned>(tok0 + v * PER + j), sm, wc);
    }
  }
  for (int base = nv * PER; base < scnt; base += 32) {
    const int i = base + lane;
    float s = -INFINITY;
    if (i < scnt) {
      if (DT == kF32) s = reinterpret_cast<const float*>(base_ptr)[i];
      else s = __uint_as_float(static_cast<unsigned>(reinterpret_cast<const unsigned short*>(base_ptr)[i]) << 16);
      if (TEMP) s = temper(s, temp);
    }
    mxt = fmaxf(mxt, s);
    const bool cnd = s >= theta;
    if (!cnd) et += wfast(s, cc);
    warp_push(cnd, s, static_cast<unsigned>(tok0 + i), sm, wc);
  }
  for (int base = 0; base < nspec; base += 32) {
    const int i = base + lane;
    float s = -INFINITY;
    unsigned id = 0u;
    if (i < nspec) {
      s = TEMP ? clampf(__fdiv_rn(ss[i], temp)) : ss[i];
      id = si[i];
    }
    mxt = fmaxf(mxt, s);
    const bool cnd = s >= theta;
    if (!cnd) et += wfast(s, cc);
    warp_push(cnd, s, id, sm, wc);
  }
}

// Row-wide direct pass from global memory (unaligned rows, the second
// chance): every token's processed score from the logits and the bitmaps.
// Greedy: each thread's best.  Sampling with a known theta and cc: tokens
// below theta add to et, the others join the warp segments (wc).
template <int DT>
__device__ void direct_pass(const DevCfg& c, const void* rowp, int V, const unsigned* H, const unsigned* N,
                            bool bitmaps, bool sample, float theta, float cc, SelSmem& sm, float& bv, unsigned& bi,
                            float& et, float& mxt, int& wc) {
  for (int base = 0; base < V; base += kThreads) {
    const int i = base + threadIdx.x;
    float s = -INFINITY;
    if (i < V) {
      const float x = load_logit<DT>(rowp, i);
      s = bitmaps ? process_elem(c, H, N, x, i, sample)
                  : ((sample && c.temp != 1.0f) ? clampf(__fdiv_rn(x, c.temp)) : x);
    }
    if (!sample) {
      if (s > bv) { bv = s; bi = static_cast<unsigned>(i); }
    } else {
      mxt = fmaxf(mxt, s);
      const bool cnd = s >= theta;
      if (!cnd) et += wfast(s, cc);
      warp_push(cnd, s, static_cast<unsigned>(i), sm, wc);
    }
  }
}

// ---------------------------------------------------------------------------
// select_kernel
// ---------------------------------------------------------------------------
template <int DT, bool VERIFY, bool TEMP>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const DevCfg c, const SelArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  unsigned* H = reinterpret_cast<unsigned*>(smem_raw + fin_offset());
  unsigned* N = H + bitmap_bytes(a.nwords) / 4;
  unsigned char* ring = smem_raw + ring_offset(a.nwords);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int esz = DT == kF32 ? 4 : 2;
  constexpr int SE = kStageBytes / esz;   // elements per sub-chunk
  constexpr int SW = SE / kWarps;         // elements per warp slice
  static_assert(SW % 32 == 0 && SW / 32 <= 32, "a warp slice is at most one bitmap word per lane");
  const int V = a.V;
  const int nsub = (V + SE - 1) / SE;
  const int nst = a.nstage;
  const bool sample = c.mode == kSample;
  // rows take the TMA ring when every row starts on a 16-byte boundary
  const bool tma_ok = ((reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0u) && ((static_cast<size_t>(V) * esz) % 16u == 0u);

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&sm.misc.full[s], 1u);
      mbar_init(&sm.misc.empty[s], static_cast<unsigned>(kWarps));
    }
    sm.misc.error = 0;
    sm.misc.issued = 0;
    sm.misc.gcause = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------- producer warp: every sub-chunk of every streamed row ----------------
  if (wid == kWarps) {
    if (lane == 0) {
      const unsigned long long policy = evict_first_policy();
      long long seq = 0;
      for (int row = blockIdx.x; row < a.nrows && tma_ok; row += gridDim.x) {
        if (!VERIFY) {
          const RowMeta rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows);
          if (rm.bad || rm.L == 0 || rm.forced) continue;
        }
        const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * esz;
        for (int k = 0; k < nsub; ++k, ++seq) {
          const int st = static_cast<int>(seq % nst);
          const long long use = seq / nst;
          if (use > 0 && !mbar_wait(&sm.misc.empty[st], static_cast<unsigned>((use - 1) & 1))) {
            atomicExch(&sm.misc.error, 1);
            return;
          }
          if (*reinterpret_cast<volatile int*>(&sm.misc.error)) return;
          const int lo = k * SE, n = min(SE, V - lo);
          mbar_expect_tx(&sm.misc.full[st], static_cast<unsigned>(n * esz));
          bulk_g2s(ring + st * kStageBytes, rowp + static_cast<size_t>(lo) * esz, static_cast<unsigned>(n * esz),
                   &sm.misc.full[st], policy);
          *reinterpret_cast<volatile int*>(&sm.misc.issued) = static_cast<int>(seq + 1);
        }
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  long long seq = 0;
  for (int row = blockIdx.x; row < a.nrows; row += gridDim.x) {
    const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * esz;
    RowMeta rm;
    int vb = 0;
    if (VERIFY) {
      vb = row / (a.K + 1);
      rm.bad = false; rm.L = 1; rm.P = 0; rm.h0 = 0;
      rm.eos_off = rm.forced = rm.forced_eos = rm.bsup = false;
    } else {
      rm = row_meta(c, a.hist, a.off, a.plen, row, a.nrows);
    }
    const float u = (sample && a.uniforms) ? a.uniforms[row] : 0.0f;
    int token = -1;

    if (!VERIFY && (rm.bad || rm.L == 0)) {
      if (rm.bad && tid == 0) atomicOr(c.status, kFlagBadRow);
    } else if (!VERIFY && rm.forced) {
      // Forced rows do not depend on the logits: nothing is read.
      int zs[8];
      const int nz = forced_zeros(c, rm, zs);
      if (!sample) {
        token = nz ? zs[0] : 0;
      } else {
        const unsigned long long W = 1ull << kFixShift;
        const unsigned long long cnt = nz ? static_cast<unsigned long long>(nz) : static_cast<unsigned long long>(V);
        unsigned long long ncut = cnt;
        if (c.top_p < 1.0f) ncut = group_pick(0ull, W, cnt, topp_target(c.top_p, cnt * W), false);
        const unsigned long long nd = group_pick(0ull, W, ncut, draw_target(u, ncut * W), true);
        token = nz ? zs[nd - 1] : static_cast<int>(nd - 1);
      }
    } else {
      const bool bitmaps = !VERIFY;
      const bool topk = sample && c.top_k > 0 && c.top_k < V;
      const bool topp = sample && c.top_p < 1.0f;
      const float qfrac = topp ? c.top_p : fminf(fmaxf(u, 0.0f), 1.0f);
      const float budget = 0.5f * (1.0f - qfrac);
      if (bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords);

      float bv = -INFINITY;          // greedy: this lane's best score and index
      unsigned bi = 0xffffffffu;
      float et = 0.0f;               // sampling: this lane's excluded mass, relative to mref
      float mxt = -INFINITY;         // sampling: largest score this lane saw
      int wc = 0;                    // this warp's candidates (uniform in the warp)
      float mref = -INFINITY;        // this warp's reference maximum
      float cc = 0.0f;               // mref * log2e
      float theta = -INFINITY;       // this warp's threshold
      bool decided = false;          // mref and theta are set
      bool give_up = false;          // the one-pass path cannot decide this row
      float* ss = sm.spec_s + wid * kSpecPerWarp;
      unsigned* si = sm.spec_i + wid * kSpecPerWarp;

      if (tma_ok) {
        for (int k = 0; k < nsub; ++k, ++seq) {
          const int st = static_cast<int>(seq % nst);
          const unsigned parity = static_cast<unsigned>((seq / nst) & 1);
          if (!*reinterpret_cast<volatile int*>(&sm.misc.error)) {
            if (!mbar_wait(&sm.misc.full[st], parity)) atomicExch(&sm.misc.error, 1);
          }
          unsigned char* stage = ring + st * kStageBytes;
          const int lo = k * SE;
          const int n = min(SE, V - lo);
          const int soff = wid * SW;
          const int scnt = max(0, min(SW, n - soff));
          const int tok0 = lo + soff;
          int nspec = 0;
          if (scnt > 0) {
            bool sovf = false;
            if (bitmaps) nspec = warp_patch<DT>(stage, soff, scnt, tok0, H, N, c.rho, ss, si, sovf);
            if (sovf) { give_up = true; TG_GIVEUP(1); }
            if (!sample) {
              warp_greedy<DT>(stage, soff, scnt, tok0, nspec, ss, si, bv, bi);
            } else if (!give_up) {
              bool first = false;
              if (!decided) {
                float mx = warp_slice_max<DT>(stage, soff, scnt, nspec, ss);
                if (TEMP) mx = temper(mx, c.temp);
                if (mx > kFilter) {
                  mref = mx;
                  cc = mref * kLog2e;
                  theta = mref - 8.0f;
                  decided = true;
                  first = true;
                }
              }
              if (decided) {
                bool raised = false;
                for (int attempt = 0;; ++attempt) {
                  const float et0 = et, mxt0 = mxt;
                  const int wc0 = wc;
                  warp_pass<DT, TEMP>(stage, soff, scnt, tok0, nspec, ss, si, sm, c.temp, theta, cc, et, mxt, wc);
                  const bool ovf = wc > kSeg;
                  // (k == 0 is settled block-wide below; later first slices check themselves)
                  const bool pilot = first && k > 0 && !topk && !raised && attempt < 4;
                  if (!ovf && !pilot) break;
                  if (!ovf) {
                    // first slice: lower theta while too much of its mass lies below it
                    const float E = warp_sum(et);
                    const float zc = warp_cand_mass(sm, wc, cc);
                    if (E <= budget * (E + zc) || theta < mref - 40.0f) break;
                    et = 0.0f; mxt = mxt0; wc = 0;
                    theta -= 4.0f;
                    continue;
                  }
                  // overflow: undo the slice, make room, redo
                  et = et0; mxt = mxt0; wc = wc0;
                  if (attempt >= 12) { give_up = true; TG_GIVEUP(2); break; }
                  float hi = fmaxf(mref, warp_max(mxt));
                  if (TEMP) hi = fmaxf(hi, temper(warp_slice_max<DT>(stage, soff, scnt, nspec, ss), c.temp));
                  else hi = fmaxf(hi, warp_slice_max<DT>(stage, soff, scnt, nspec, ss));
                  float th2 = warp_overflow_theta<DT, TEMP>(sm, wc, stage, soff, scnt, nspec, ss, c.temp, theta, hi);
                  if (topk) th2 = fminf(th2, warp_keep_score(sm, wc, min(wc, c.top_k), theta, hi));
                  if (!(th2 > theta)) { give_up = true; TG_GIVEUP(4); break; }
                  if (th2 >= hi) { give_up = true; TG_GIVEUP(8); break; }
                  theta = th2;
                  raised = true;
                  float dropped;
                  wc = warp_compact(sm, wc, theta, cc, dropped);
                  if (lane == 0) et += dropped;
                }
                // keep a quarter of the segment free
                if (!give_up && wc > (3 * kSeg) / 4) {
                  const float th2 = warp_make_room(sm, wc, theta, warp_max(mxt), cc, warp_sum(et), topk, c.top_k,
                                                   0.9f * (1.0f - qfrac));
                  if (th2 > theta) {
                    theta = th2;
                    float dropped;
                    wc = warp_compact(sm, wc, theta, cc, dropped);
                    if (lane == 0) et += dropped;
                  }
                }
              }
            }
          }
          // First sub-chunk: one block-wide decision of theta from all sixteen
          // slices (its stage is kept until then, so it can be redone).
          if (sample && k == 0) {
            for (int round = 0;; ++round) {
              csync();
              if (lane == 0) {
                sm.misc.wmref[wid] = mref;
                sm.misc.wflags[wid] = (decided ? 1 : 0) | (give_up ? 2 : 0);
              }
              csync();
              float m0 = -INFINITY;
              bool any_gu = false;
              for (int q = 0; q < kWarps; ++q) {
                const int fl = sm.misc.wflags[q];
                if (fl & 1) m0 = fmaxf(m0, sm.misc.wmref[q]);
                any_gu |= (fl & 2) != 0;
              }
              if (any_gu || !(m0 > kFilter)) break;   // each warp goes on by itself
              // one reference maximum and one threshold for every warp
              const float cc0 = m0 * kLog2e;
              et = decided ? et * expf(mref - m0) : 0.0f;
              if (!decided) { wc = 0; mxt = -INFINITY; }
              mref = m0;
              cc = cc0;
              decided = true;
              const float th0 = round == 0 ? m0 - 8.0f : theta;
              float dropped;
              wc = warp_compact(sm, wc, th0, cc, dropped);
              if (lane == 0) et += dropped;
              theta = th0;
              // project the first sub-chunk over the whole row
              const float scale = static_cast<float>(V) / static_cast<float>(min(V, SE));
              const float E = block_sum_f(et, &sm.red);
              const float zcw = warp_cand_mass(sm, wc, cc);
              const float zc = block_sum_f(lane == 0 ? zcw : 0.0f, &sm.red);
              const float nct = block_sum_f(lane == 0 ? static_cast<float>(min(wc, kSeg)) : 0.0f, &sm.red);
              if (!topk && E * scale > 0.5f * (1.0f - qfrac) * (E + zc) && nct * scale < 0.5f * kCandCap &&
                  round < 3 && theta > m0 - 40.0f) {
                // too much mass below theta and room to spare: lower it, redo the sub-chunk
                theta -= 2.0f;
                et = 0.0f; mxt = -INFINITY; wc = 0;
                if (scnt > 0) {
                  warp_pass<DT, TEMP>(stage, soff, scnt, tok0, nspec, ss, si, sm, c.temp, theta, cc, et, mxt, wc);
                  if (wc > kSeg) give_up = true;
                }
                continue;
              }
              // as low a threshold as the list's capacity allows
              const float th1 = block_capacity_theta(sm, wc, theta, m0, scale);
              if (th1 > theta) {
                theta = th1;
                wc = warp_compact(sm, wc, theta, cc, dropped);
                if (lane == 0) et += dropped;
              }
              break;
            }
          }
          // release the stage to the producer
          if (bitmaps) fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.misc.empty[st]);
        }
      } else {
        // rows not on a 16-byte boundary: read the logits directly
        if (!sample) {
          float et_unused = 0.0f, mxt_unused = -INFINITY;
          int wc_unused = 0;
          direct_pass<DT>(c, rowp, V, H, N, bitmaps, false, 0.0f, 0.0f, sm, bv, bi, et_unused, mxt_unused, wc_unused);
        } else {
          float mx = -INFINITY;
          for (int i = tid; i < V; i += kThreads) {
            const float x = load_logit<DT>(rowp, i);
            mx = fmaxf(mx, bitmaps ? process_elem(c, H, N, x, i, true)
                                   : ((c.temp != 1.0f) ? clampf(__fdiv_rn(x, c.temp)) : x));
          }
          mx = block_max(mx, &sm.red);
          if (mx > kFilter) {
            mref = mx;
            cc = mref * kLog2e;
            theta = mref - 8.0f;
            decided = true;
            direct_pass<DT>(c, rowp, V, H, N, bitmaps, true, theta, cc, sm, bv, bi, et, mxt, wc);
            if (wc > kSeg) give_up = true;
          }
        }
      }

      // ---------------- finish the row (all consumer warps) ----------------
      csync();
      if (tid == 0) sm.misc.err_snap = *reinterpret_cast<volatile int*>(&sm.misc.error);
      csync();
      if (sm.misc.err_snap) break;   // uniform: every consumer reads the same snapshot
      if (!sample) {
        const float m = block_max(bv, &sm.red);
        token = static_cast<int>(block_min_u(bv == m ? bi : 0xffffffffu, &sm.red));
      } else {
        if (lane == 0) {
          sm.misc.wtheta[wid] = theta;
          sm.misc.wmref[wid] = mref;
          sm.misc.wflags[wid] = (decided ? 1 : 0) | ((give_up || wc > kSeg) ? 2 : 0);
          if (wc > kSeg) TG_GIVEUP(16);
        }
        csync();
        bool any_give_up = false, any_decided = false;
        float theta_f = -INFINITY, mref_max = -INFINITY;
        for (int q = 0; q < kWarps; ++q) {
          const int fl = sm.misc.wflags[q];
          any_give_up |= (fl & 2) != 0;
          if (fl & 1) {
            any_decided = true;
            theta_f = fmaxf(theta_f, sm.misc.wtheta[q]);
            mref_max = fmaxf(mref_max, sm.misc.wmref[q]);
          }
        }
        const float m = fmaxf(mref_max, block_max(mxt, &sm.red));
        bool slow = any_give_up || !any_decided || !(m > kFilter);
        int reason = any_give_up ? 1 : slow ? 3 : 0;
        unsigned tok = 0u;
        const float cc_m = m * kLog2e;
        if (!slow) {
          // every warp drops its candidates below the largest theta
          et = decided ? et * expf(mref - m) : 0.0f;
          float dropped;
          wc = warp_compact(sm, wc, theta_f, cc_m, dropped);
          if (lane == 0) { et += dropped; sm.misc.wcnt[wid] = wc; }
          const float E = block_sum_f(et, &sm.red);
          pack_candidates(sm);
          TG_DBG(row, 2, m); TG_DBG(row, 3, theta_f); TG_DBG(row, 4, E); TG_DBG(row, 7, sm.misc.ncand);
          const FinResult fr = finalize_candidates(
              c, sm, m, static_cast<unsigned long long>(llrint(static_cast<double>(E) * kFixScale)), u, topk, topp);
          slow = !fr.ok;
          if (slow) reason = fr.reason;
          tok = fr.token;
          // Too little candidate mass for the cut or draw: one more pass, read
          // directly (the row is likely still in L2), with a lower threshold.
          if (slow && (reason == 5 || reason == 7)) {
            csync();
            if (bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords);
            float et2 = 0.0f, mxt2 = -INFINITY;
            int wc2 = 0;
            float bv2 = -INFINITY;
            unsigned bi2 = 0u;
            direct_pass<DT>(c, rowp, V, H, N, bitmaps, true, theta_f - 1.5f, cc_m, sm, bv2, bi2, et2, mxt2, wc2);
            if (lane == 0) sm.misc.wflags[wid] = wc2 > kSeg ? 2 : 0;
            csync();
            bool ovf2 = false;
            for (int q = 0; q < kWarps; ++q) ovf2 |= (sm.misc.wflags[q] & 2) != 0;
            if (!ovf2) {
              if (lane == 0) sm.misc.wcnt[wid] = wc2;
              const float E2 = block_sum_f(et2, &sm.red);
              pack_candidates(sm);
              const FinResult fr2 = finalize_candidates(
                  c, sm, m, static_cast<unsigned long long>(llrint(static_cast<double>(E2) * kFixScale)), u, topk, topp);
              slow = !fr2.ok;
              if (slow) reason = 10 + fr2.reason;
              tok = fr2.token;
            }
          }
        }
        TG_DBG(row, 0, slow ? 1 : 0); TG_DBG(row, 1, reason);
#ifdef TG_DEBUG
        TG_DBG(row, 5, sm.misc.gcause);
        csync();
        if (tid == 0) sm.misc.gcause = 0;
#endif
        if (slow) {
          // Multi-pass exact selection over the whole row.
          csync();
          if (tid == 0) { atomicOr(c.status, kFlagSlow); atomicAdd(c.slow_rows, 1ull); }
          if (bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords);
          RowGlobalSource<DT> src{rowp, V, &c, H, N, bitmaps, true};
          float mm = -INFINITY;
          src.pass([&](float s, unsigned) { mm = fmaxf(mm, s); });
          mm = block_max(mm, &sm.red);
          tok = sample_exact(c, src, mm, u, static_cast<unsigned>(V), &sm.hist, &sm.red, nullptr, nullptr);
        }
        token = static_cast<int>(tok);
      }
    }

    // ---------------- outputs ----------------
    if (tid == 0) {
      a.out[row] = token;
      if (VERIFY) {
        // Last of the K+1 positions of row vb counts the matches (steps 4-5).
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
    }
    csync();
  }

  // error: wait (bounded) for every copy the producer issued, then leave
  if (*reinterpret_cast<volatile int*>(&sm.misc.error)) {
    if (tid == 0) {
      atomicOr(c.status, kFlagTimeout);
      for (int tries = 0; tries < 4 * kMaxStages && seq < *reinterpret_cast<volatile int*>(&sm.misc.issued); ++tries, ++seq) {
        const int st = static_cast<int>(seq % nst);
        mbar_wait(&sm.misc.full[st], static_cast<unsigned>((seq / nst) & 1));
      }
    }
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

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    process_kernel(const DevCfg c, const SelArgs a, float* out_scores, unsigned* out_banbits, float* out_probs) {
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
  const void* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * (DT == kF32 ? 4 : 2);
  float* sc = out_scores + static_cast<size_t>(row) * V;
  build_row_bitmaps(c, a.hist, rm, H, N, a.nwords);
  int zs[8];
  int nz = rm.forced ? forced_zeros(c, rm, zs) : 0;
  for (int i = threadIdx.x; i < V; i += kThreads) {
    float s;
    if (rm.forced) {
      s = kFilter;
      for (int q = 0; q < nz; ++q) if (zs[q] == i) s = 0.0f;
    } else {
      float x = DT == kF32 ? __ldg(static_cast<const float*>(rowp) + i)
                           : __uint_as_float(static_cast<unsigned>(__ldg(static_cast<const unsigned short*>(rowp) + i)) << 16);
      s = process_elem(c, H, N, x, i, false);
    }
    if (sample && c.temp != 1.0f) s = clampf(__fdiv_rn(s, c.temp));
    sc[i] = s;
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
      const int ns = min(8, (optin - select_smem_bytes(0, 0)) / kStageBytes);
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
int process_smem_bytes(int nwords) {
  return align_up(static_cast<int>(sizeof(ProcSmem)), 128) + 2 * bitmap_bytes(nwords);
}

template <int DT, bool VERIFY, bool TEMP>
static cudaError_t launch_sel(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  auto k = select_kernel<DT, VERIFY, TEMP>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kSelThreads, smem, s>>>(c, a);
  return cudaGetLastError();
}

template <int DT, bool VERIFY>
static cudaError_t launch_sel_t(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  const bool temp = c.mode == kSample && c.temp != 1.0f;
  return temp ? launch_sel<DT, VERIFY, true>(c, a, grid, smem, s) : launch_sel<DT, VERIFY, false>(c, a, grid, smem, s);
}

cudaError_t launch_select(const DevCfg& c, const SelArgs& a, bool verify, int grid, int smem, cudaStream_t s) {
  if (a.nstage < 2 || a.nstage > kMaxStages) return cudaErrorInvalidValue;
  if (c.dtype == kF32) return verify ? launch_sel_t<kF32, true>(c, a, grid, smem, s) : launch_sel_t<kF32, false>(c, a, grid, smem, s);
  return verify ? launch_sel_t<kBF16, true>(c, a, grid, smem, s) : launch_sel_t<kBF16, false>(c, a, grid, smem, s);
}

cudaError_t launch_process(const DevCfg& c, const SelArgs& a, float* scores, unsigned* banbits, float* probs,
                           int smem, cudaStream_t s) {
  cudaError_t e;
  if (c.dtype == kF32) {
    e = cudaFuncSetAttribute(process_kernel<kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    process_kernel<kF32><<<a.nrows, kThreads, smem, s>>>(c, a, scores, banbits, probs);
  } else {
    e = cudaFuncSetAttribute(process_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    process_kernel<kBF16><<<a.nrows, kThreads, smem, s>>>(c, a, scores, banbits, probs);
  }
  return cudaGetLastError();
}

cudaError_t select_occupancy(int dtype, bool verify, int smem, int* blocks_per_sm) {
  // the most demanding instantiation decides
  int worst = 1 << 20;
  for (int t = 0; t < 2; ++t) {
    void (*k)(DevCfg, SelArgs);
    if (dtype == kF32) k = verify ? (t ? select_kernel<kF32, true, true> : select_kernel<kF32, true, false>)
                                  : (t ? select_kernel<kF32, false, true> : select_kernel<kF32, false, false>);
    else k = verify ? (t ? select_kernel<kBF16, true, true> : select_kernel<kBF16, true, false>)
                    : (t ? select_kernel<kBF16, false, true> : select_kernel<kBF16, false, false>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kSelThreads, smem);
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
