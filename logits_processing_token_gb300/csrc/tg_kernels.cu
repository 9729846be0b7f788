// Token-selection kernels for sm_103a.
//
//  select_kernel  -- tg_select and tg_verify: one CTA per row at a time
//                    (persistent over rows), the row streamed once from HBM
//                    through a ring of 16 KB TMA bulk copies into shared
//                    memory, processors applied by patching the few tokens
//                    the history/ban bitmaps mark, then greedy argmax or the
//                    one-pass sampling path below.
//  process_kernel -- tg_process (diagnostic): processed scores, ban bits and
//                    the final distribution, written to global memory.
//
// Sampling in one pass.  While streaming, every token's weight exp(s - m)
// (m = running maximum) either joins the excluded mass E (s below a value
// threshold theta) or the token joins a small candidate list (s >= theta).
// theta only rises, so at the end the candidates are exactly the tokens with
// s >= theta.  top_k, the top_p cut and the draw then run exactly on the
// candidates with 44-bit fixed-point weights; the excluded tokens all sit
// after every candidate in the (score desc, index asc) order, so the result
// is exact whenever the candidates hold the k largest scores (top_k) or more
// mass than the cut (top_p) or the draw target needs.  A row where that check
// fails runs the multi-pass exact selection over the whole row instead.
#include <mutex>

#include "../../include/tg.h"
#include "tg_device.cuh"

namespace tg {

#ifdef TG_DEBUG
// Debug builds only: per-row record {path, reason, m, theta, E, Zc, Z, ncand,
// then clock64 totals of: setup, wait, patch, passA, passB, prune, finalize, restream}.
__device__ double* g_dbg = nullptr;
#define TG_DBG(row, slot, val) do { if (g_dbg && threadIdx.x == 0) g_dbg[(row) * 16 + (slot)] = (double)(val); } while (0)
#define TG_T0(name) long long name = clock64()
#define TG_TACC(row, slot, t0) do { if (g_dbg && threadIdx.x == 0) g_dbg[(row) * 16 + (slot)] += (double)(clock64() - (t0)); } while (0)
#else
#define TG_DBG(row, slot, val) do { } while (0)
#define TG_T0(name) do { } while (0)
#define TG_TACC(row, slot, t0) do { } while (0)
#endif

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
// Shared-memory layout of select_kernel
// ---------------------------------------------------------------------------
struct Misc {
  unsigned long long mbar[8];
  int wcnt[kWarps];    // candidates in each warp's segment of the list
  int ncand;           // packed (contiguous) candidates, for the finish
  int nspec[2];        // side-list length, double-buffered by sub-chunk parity
  int overflow;        // a warp's segment ran out of room
  int prune;           // a warp's segment is three-quarters full
  int spec_overflow;
  int timeout;
  float pr_mass[kWarps][32];   // prune histogram per warp: levels of 0.5 below the running max
  unsigned pr_cnt[kWarps][32];
  float pr_tmass[32];
  unsigned pr_tcnt[32];
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
  float spec_s[kSpecCap];
  unsigned spec_i[kSpecCap];
  Hist hist;
  FinSmem fin;
  RedScratch red;
  Misc misc;
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int sel_fixed_bytes() { return align_up(static_cast<int>(sizeof(SelSmem)), 128); }
__host__ __device__ constexpr int bitmap_bytes(int nwords) { return align_up(nwords * 4, 128); }

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
      float x;
      if (DT == kF32) x = __ldg(static_cast<const float*>(row) + i);
      else x = __uint_as_float(static_cast<unsigned>(__ldg(static_cast<const unsigned short*>(row) + i)) << 16);
      float s = x;
      if (bitmaps) s = process_elem(*c, H, N, x, i, sample);
      else if (sample && c->temp != 1.0f) s = clampf(__fdiv_rn(x, c->temp));
      f(s, static_cast<unsigned>(i));
    }
  }
};

// Append one (value, index) per lane that has one to this warp's segment.
// All 32 lanes call (converged); wc is the warp's count, kept uniform.
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
    } else {
      sm.misc.overflow = 1;
    }
  }
  wc += __popc(bal);
}

__device__ __forceinline__ int cand_total(const SelSmem& sm) {
  int t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += min(sm.misc.wcnt[w], kSeg);
  return t;
}

// Fast mass (relative to c = m * log2e) of every listed candidate.
__device__ __forceinline__ float cand_fast_mass(SelSmem& sm, float c) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(sm.misc.wcnt[w], kSeg);
  float acc = 0.0f;
  for (int j = lane; j < n; j += 32) acc += wfast(sm.cand_s[w * kSeg + j], c);
  return block_sum_f(acc, &sm.red);
}

// Drop candidates below theta, each warp compacting its own segment in
// place; returns the dropped fast mass.  All threads call.
__device__ float compact_candidates(SelSmem& sm, float theta, float c) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = min(sm.misc.wcnt[w], kSeg);
  float* S = sm.cand_s + w * kSeg;
  unsigned* I = sm.cand_i + w * kSeg;
  int out = 0;
  float dropped = 0.0f;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const bool in = j < n;
    const float s = in ? S[j] : -INFINITY;
    const unsigned id = in ? I[j] : 0u;
    const bool keep = in && s >= theta;
    if (in && !keep) dropped += wfast(s, c);
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
  if (lane == 0) sm.misc.wcnt[w] = out;
  __syncthreads();
  return block_sum_f(dropped, &sm.red);
}

// Choose a higher threshold for the candidate list.  top_k: keep at least
// 2k candidates; otherwise drop at most `allowed` fast mass.  Returns the new
// theta (>= old).  All threads call.
__device__ float choose_theta(SelSmem& sm, float theta, float m, float c, bool topk, int k, float allowed) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sm.misc.pr_mass[w][lane] = 0.0f;
  sm.misc.pr_cnt[w][lane] = 0u;
  __syncwarp();
  const int n = min(sm.misc.wcnt[w], kSeg);
  for (int j = lane; j < n; j += 32) {
    const float s = sm.cand_s[w * kSeg + j];
    const int lv = static_cast<int>(fminf(fmaxf((m - s) * 2.0f, 0.0f), 31.0f));
    atomicAdd(&sm.misc.pr_mass[w][lv], wfast(s, c));
    atomicAdd(&sm.misc.pr_cnt[w][lv], 1u);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float tm = 0.0f;
    unsigned tc = 0u;
    for (int q = 0; q < kWarps; ++q) { tm += sm.misc.pr_mass[q][threadIdx.x]; tc += sm.misc.pr_cnt[q][threadIdx.x]; }
    sm.misc.pr_tmass[threadIdx.x] = tm;
    sm.misc.pr_tcnt[threadIdx.x] = tc;
  }
  __syncthreads();
  // every thread scans the 32 levels identically
  int jstar = 32;
  if (topk) {
    unsigned cum = 0u;
    for (int j = 0; j < 32; ++j) {
      cum += sm.misc.pr_tcnt[j];
      if (cum >= static_cast<unsigned>(2 * k)) { jstar = j + 1; break; }
    }
  } else {
    float tail = 0.0f;
    for (int j = 31; j >= 0; --j) {
      float t2 = tail + sm.misc.pr_tmass[j];
      if (t2 > allowed) break;
      tail = t2;
      jstar = j;
    }
  }
  __syncthreads();
  float cand = (jstar >= 32) ? theta : m - 0.5f * static_cast<float>(jstar);
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
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int q = lane + 32 * j;
    if (q < n) { sm.cand_s[off + q] = vs[j]; sm.cand_i[off + q] = is[j]; }
  }
  if (threadIdx.x == 0) sm.misc.ncand = cand_total(sm);
  __syncthreads();
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
__device__ int gather_sort_level(SelSmem& sm, int n, const LevelMap& lv, int level, unsigned klo, float m) {
  FinSmem& f = sm.fin;
  if (threadIdx.x == 0) f.gn = 0;
  __syncthreads();
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
      if (has && pos < kGroupCap) { f.gk[pos] = key; f.gi[pos] = sm.cand_i[i]; f.gw[pos] = wfix(s, m); }
    }
  }
  __syncthreads();
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
  __syncthreads();
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
  __syncthreads();
}

// Level search by warp 0 over fin.lm / fin.lc; results in fin.fb/fbefore/ffound.
template <class Reached>
__device__ __forceinline__ void level_find_mass(SelSmem& sm, Reached r) {
  if (threadIdx.x < 32) {
    FindOut<unsigned long long> o = warp_find<kLevels>(sm.fin.lm, sm.fin.lc, false, r);
    if (threadIdx.x == 0) { sm.fin.fb = o.b; sm.fin.fbefore = o.before; sm.fin.ffound = o.found; }
  }
  __syncthreads();
}

// Keep only levels < L in full and the first `mass`/`cnt` of level L.
__device__ __forceinline__ void level_limit(SelSmem& sm, int L, unsigned long long mass, unsigned cnt) {
  for (int l = threadIdx.x; l < kLevels; l += kThreads) {
    if (l > L) { sm.fin.lm[l] = 0ull; sm.fin.lc[l] = 0u; }
    else if (l == L) { sm.fin.lm[l] = mass; sm.fin.lc[l] = cnt; }
  }
  __syncthreads();
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
  __syncthreads();
  unsigned long long zc = 0ull;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const float s = sm.cand_s[i];
    const int l = lv(s);
    const unsigned long long w = wfix(s, m);
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
    __syncthreads();
    const int Lk = f.fb;
    const unsigned rank = static_cast<unsigned>(c.top_k) - static_cast<unsigned>(f.fbefore);
    const int gn = gather_sort_level(sm, n, lv, Lk, 0u, m);
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
      kept_mass = mass_sum(ls, kf, m, &sm.red);
      kept_cnt = count_items(ls, kf, &sm.red);
    }
    __syncthreads();
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
    __syncthreads();
    const int gn = gather_sort_level(sm, n, lv, Lc, klo, m);
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
      MassSel cs = mass_select(ls, keep, m, T - before, false, &sm.hist);
      if (!cs.found) { res.reason = 6; return res; }
      keep.cut = true; keep.kcut = cs.key; keep.icut = cs.idx;
      S = before + cs.mass;
      inlevel = cs.mass;
      nc = static_cast<int>(count_items(ls, keep, &sm.red));
    }
    __syncthreads();
    level_limit(sm, Lc, inlevel, static_cast<unsigned>(nc));
  }
  const unsigned long long Td = draw_target(u, S);
  if (!topk && !topp && !(Zc > Td)) { res.reason = 7; return res; }
  level_find_mass(sm, [Td](unsigned long long x) { return x > Td; });
  if (!f.ffound) { res.reason = 8; return res; }
  const int Ld = f.fb;
  const unsigned long long before = f.fbefore;
  __syncthreads();
  if (Ld == Lc && cut_sorted) {
    walk_sorted(sm, nc, before, Td, true);
    res.token = f.si[f.fb];
  } else {
    const int gn = gather_sort_level(sm, n, lv, Ld, klo, m);
    if (gn >= 0) {
      const int lim = (Ld == Lc) ? nc : gn;
      walk_sorted(sm, lim, before, Td, true);
      res.token = f.si[f.fb];
    } else {
      CandLevelSource ls{sm.cand_s, sm.cand_i, n, lv, Ld};
      MassSel d = mass_select(ls, keep, m, Td - before, true, &sm.hist);
      if (!d.found) { res.reason = 8; return res; }
      res.token = d.idx;
    }
  }
  __syncthreads();
  res.ok = true;
  return res;
}

// ---------------------------------------------------------------------------
// select_kernel
// ---------------------------------------------------------------------------

// Maximum over one sub-chunk (raw values, before temperature), this thread's part.
template <int DT>
__device__ __forceinline__ float stage_max(const unsigned char* stage, int n, int nspec, const SelSmem& sm) {
  float mx = -INFINITY;
  if (DT == kF32) {
    const float4* v4 = reinterpret_cast<const float4*>(stage);
    const int nv = n >> 2;
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      const float4 q = v4[v];
      mx = fmaxf(mx, fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w)));
    }
    for (int i = (nv << 2) + threadIdx.x; i < n; i += kThreads) mx = fmaxf(mx, reinterpret_cast<const float*>(stage)[i]);
  } else {
    const uint4* v4 = reinterpret_cast<const uint4*>(stage);
    const int nv = n >> 3;
    __nv_bfloat162 m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      uint4 q = v4[v];
      m2 = __hmax2(m2, __hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.x), *reinterpret_cast<__nv_bfloat162*>(&q.y)),
                               __hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.z), *reinterpret_cast<__nv_bfloat162*>(&q.w))));
    }
    mx = fmaxf(__low2float(m2), __high2float(m2));
    const unsigned short* sh = reinterpret_cast<const unsigned short*>(stage);
    for (int i = (nv << 3) + threadIdx.x; i < n; i += kThreads) mx = fmaxf(mx, __uint_as_float(static_cast<unsigned>(sh[i]) << 16));
    for (int i = threadIdx.x; i < nspec; i += kThreads) mx = fmaxf(mx, sm.spec_s[i]);
  }
  return mx;
}

// Greedy: this thread's best (value, lowest index) over one sub-chunk.
template <int DT>
__device__ __forceinline__ void greedy_scan(const unsigned char* stage, int n, int lo, int nspec, const SelSmem& sm,
                                            float& bv, unsigned& bi) {
  if (DT == kF32) {
    const float4* v4 = reinterpret_cast<const float4*>(stage);
    const int nv = n >> 2;
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      const float4 q = v4[v];
      const float vm = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
      if (vm > bv) {
        const int j = q.x == vm ? 0 : q.y == vm ? 1 : q.z == vm ? 2 : 3;
        bv = vm;
        bi = static_cast<unsigned>(lo + 4 * v + j);
      }
    }
    const float* sf = reinterpret_cast<const float*>(stage);
    for (int i = (nv << 2) + threadIdx.x; i < n; i += kThreads)
      if (sf[i] > bv) { bv = sf[i]; bi = static_cast<unsigned>(lo + i); }
  } else {
    const uint4* v4 = reinterpret_cast<const uint4*>(stage);
    const int nv = n >> 3;
    for (int v = threadIdx.x; v < nv; v += kThreads) {
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
        bi = static_cast<unsigned>(lo + 8 * v + jj);
      }
    }
    const unsigned short* sh = reinterpret_cast<const unsigned short*>(stage);
    for (int i = (nv << 3) + threadIdx.x; i < n; i += kThreads) {
      const float x = __uint_as_float(static_cast<unsigned>(sh[i]) << 16);
      if (x > bv) { bv = x; bi = static_cast<unsigned>(lo + i); }
    }
    for (int i = threadIdx.x; i < nspec; i += kThreads) {
      const float s = sm.spec_s[i];
      const unsigned id = sm.spec_i[i];
      if (s > bv || (s == bv && id < bi)) { bv = s; bi = id; }
    }
  }
}

// Sampling pass over one sub-chunk: every token below theta adds its weight
// 2^(s*log2e - cc) to et; the others are appended to the warp's segment.
// mxt tracks the largest (tempered) score seen.
template <int DT, bool TEMP>
__device__ __forceinline__ void stage_pass(const unsigned char* stage, int n, int lo, int nspec, SelSmem& sm,
                                           float temp, float theta, float cc, float& et, float& mxt, int& wc) {
  const int tid = threadIdx.x;
  if (DT == kF32) {
    const float4* v4 = reinterpret_cast<const float4*>(stage);
    const int nv = n >> 2;
    for (int base = 0; base < nv; base += kThreads) {
      const int v = base + tid;
      const float4 q = v < nv ? v4[v] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      float s[4] = {q.x, q.y, q.z, q.w};
      float vm = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
      if (TEMP) {
        vm = temper(vm, temp);
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j] = temper(s[j], temp);
      }
      mxt = fmaxf(mxt, vm);
      const unsigned t0 = static_cast<unsigned>(lo + 4 * v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool cnd = s[j] >= theta;
        const float w = wfast(s[j], cc);
        if (!cnd) et += w;
        warp_push(cnd, s[j], t0 + static_cast<unsigned>(j), sm, wc);
      }
    }
    const float* sf = reinterpret_cast<const float*>(stage);
    for (int base = nv << 2; base < n; base += kThreads) {
      const int i = base + tid;
      float s = -INFINITY;
      if (i < n) s = TEMP ? temper(sf[i], temp) : sf[i];
      mxt = fmaxf(mxt, s);
      const bool cnd = s >= theta;
      if (!cnd) et += wfast(s, cc);
      warp_push(cnd, s, static_cast<unsigned>(lo + i), sm, wc);
    }
  } else {
    const uint4* v4 = reinterpret_cast<const uint4*>(stage);
    const int nv = n >> 3;
    for (int base = 0; base < nv; base += kThreads) {
      const int v = base + tid;
      uint4 q = v < nv ? v4[v] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      __nv_bfloat162 m2 = __hmax2(__hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.x), *reinterpret_cast<__nv_bfloat162*>(&q.y)),
                                  __hmax2(*reinterpret_cast<__nv_bfloat162*>(&q.z), *reinterpret_cast<__nv_bfloat162*>(&q.w)));
      float vm = fmaxf(__low2float(m2), __high2float(m2));
      if (TEMP) vm = temper(vm, temp);
      mxt = fmaxf(mxt, vm);
      const unsigned ps[4] = {q.x, q.y, q.z, q.w};
      const unsigned t0 = static_cast<unsigned>(lo + 8 * v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float s = (j & 1) ? bf16hi(ps[j >> 1]) : bf16lo(ps[j >> 1]);
        if (TEMP) s = temper(s, temp);
        const bool cnd = s >= theta;
        const float w = wfast(s, cc);
        if (!cnd) et += w;
        warp_push(cnd, s, t0 + static_cast<unsigned>(j), sm, wc);
      }
    }
    const unsigned short* sh = reinterpret_cast<const unsigned short*>(stage);
    for (int base = nv << 3; base < n; base += kThreads) {
      const int i = base + tid;
      float s = -INFINITY;
      if (i < n) {
        s = __uint_as_float(static_cast<unsigned>(sh[i]) << 16);
        if (TEMP) s = temper(s, temp);
      }
      mxt = fmaxf(mxt, s);
      const bool cnd = s >= theta;
      if (!cnd) et += wfast(s, cc);
      warp_push(cnd, s, static_cast<unsigned>(lo + i), sm, wc);
    }
    for (int base = 0; base < nspec; base += kThreads) {
      const int i = base + tid;
      float s = -INFINITY;
      unsigned id = 0u;
      if (i < nspec) {
        s = TEMP ? clampf(__fdiv_rn(sm.spec_s[i], temp)) : sm.spec_s[i];
        id = sm.spec_i[i];
      }
      mxt = fmaxf(mxt, s);
      const bool cnd = s >= theta;
      if (!cnd) et += wfast(s, cc);
      warp_push(cnd, s, id, sm, wc);
    }
  }
}

template <int DT, bool VERIFY, bool TEMP>
__global__ void __launch_bounds__(kThreads, 1) select_kernel(const DevCfg c, const SelArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  unsigned* H = reinterpret_cast<unsigned*>(smem_raw + sel_fixed_bytes());
  unsigned* N = reinterpret_cast<unsigned*>(smem_raw + sel_fixed_bytes() + bitmap_bytes(a.nwords));
  unsigned char* ring = smem_raw + sel_fixed_bytes() + 2 * bitmap_bytes(a.nwords);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int esz = DT == kF32 ? 4 : 2;
  constexpr int SE = kStageBytes / esz;   // elements per sub-chunk
  static_assert(SE / 32 <= kThreads, "one bitmap word per thread per sub-chunk");
  const int V = a.V;
  const int nsub = (V + SE - 1) / SE;
  const bool sample = c.mode == kSample;

  if (tid == 0) {
    for (int s = 0; s < a.nstage; ++s) mbar_init(&sm.misc.mbar[s], 1u);
    fence_mbar_init();
  }
  __syncthreads();
  unsigned phase = 0u;  // bit s: parity of the next wait on stage s
  const unsigned long long policy = evict_first_policy();

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
      int nz = forced_zeros(c, rm, zs);
      if (!sample) {
        token = nz ? zs[0] : 0;
      } else {
        const unsigned long long W = 1ull << kFixShift;
        unsigned long long cnt = nz ? static_cast<unsigned long long>(nz) : static_cast<unsigned long long>(V);
        unsigned long long ncut = cnt;
        if (c.top_p < 1.0f) ncut = group_pick(0ull, W, cnt, topp_target(c.top_p, cnt * W), false);
        unsigned long long nd = group_pick(0ull, W, ncut, draw_target(u, ncut * W), true);
        token = nz ? zs[nd - 1] : static_cast<int>(nd - 1);
      }
    } else {
      const bool tma_ok = ((reinterpret_cast<uintptr_t>(rowp) & 15u) == 0u) && ((static_cast<size_t>(V) * esz) % 16u == 0u);
      const bool bitmaps = !VERIFY;
      const bool topk = sample && c.top_k > 0 && c.top_k < V;
      const bool topp = sample && c.top_p < 1.0f;
      const float qfrac = topp ? c.top_p : fminf(fmaxf(u, 0.0f), 1.0f);
      const float budget = 0.5f * (1.0f - qfrac);
      // Chance 0 adapts theta while streaming; a sampling row whose
      // candidates cannot decide it streams once more (chance 1) with a
      // fixed, lower theta before the multi-pass exact path is used.
      float theta_fixed = 0.0f;
      for (int chance = 0;; ++chance) {
        if (tma_ok && tid == 0) {
          for (int k = 0; k < a.nstage && k < nsub; ++k) {
            const int lo = k * SE, n = min(SE, V - lo);
            mbar_expect_tx(&sm.misc.mbar[k], static_cast<unsigned>(n * esz));
            bulk_g2s(ring + k * kStageBytes, rowp + static_cast<size_t>(lo) * esz, static_cast<unsigned>(n * esz),
                     &sm.misc.mbar[k], policy);
          }
        }
        TG_T0(t_setup);
        if (chance == 0 && bitmaps) build_row_bitmaps(c, a.hist, rm, H, N, a.nwords);
        TG_TACC(row, 8, t_setup);
        if (lane == 0) sm.misc.wcnt[wid] = 0;
        if (tid == 0) {
          sm.misc.ncand = 0; sm.misc.overflow = 0; sm.misc.prune = 0; sm.misc.spec_overflow = 0;
          sm.misc.timeout = 0; sm.misc.nspec[0] = 0; sm.misc.nspec[1] = 0;
        }
        __syncthreads();

        float bv = -INFINITY;          // greedy: this thread's best score and index
        unsigned bi = 0xffffffffu;
        float mxt = -INFINITY;         // sampling: largest score this thread saw
        float et = 0.0f;               // sampling: this thread's excluded mass, relative to mref
        int wc = 0;                    // this warp's candidate count (uniform in the warp)
        float mref = -INFINITY;        // reference maximum of the weights
        float cc = 0.0f;               // mref * log2e
        float theta = chance ? theta_fixed : -INFINITY;
        bool decided = false;          // mref and theta are set
        bool give_up = false;          // the one-pass path cannot decide this row

        for (int k = 0; k < nsub; ++k) {
          const int st = k % a.nstage;
          const int lo = k * SE;
          const int n = min(SE, V - lo);
          unsigned char* stage = ring + st * kStageBytes;
          TG_T0(t_wait);
          if (tma_ok) {
            if (!mbar_wait(&sm.misc.mbar[st], (phase >> st) & 1u)) sm.misc.timeout = 1;
            phase ^= 1u << st;
          } else {
            // unaligned rows: cooperative copy through registers
            for (int i = tid; i < n * esz / 2; i += kThreads)
              reinterpret_cast<unsigned short*>(stage)[i] =
                  __ldg(reinterpret_cast<const unsigned short*>(rowp + static_cast<size_t>(lo) * esz) + i);
            __syncthreads();
          }
          TG_TACC(row, 9, t_wait);
          TG_T0(t_patch);
          // ---- patch the tokens the bitmaps mark (a2-a9) ----
          if (bitmaps) {
            const int w0 = lo >> 5;
            const int nw = (n + 31) >> 5;
            unsigned bits = 0u, nb = 0u;
            if (tid < nw) {
              bits = H[w0 + tid] | N[w0 + tid];
              nb = N[w0 + tid];
              const int rem = n - tid * 32;
              if (rem < 32) bits &= (1u << rem) - 1u;
            }
            int base = 0;
            if (DT == kBF16) {
              const int cntb = __popc(bits);
              int incl = cntb;
              for (int o = 1; o < 32; o <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
              }
              const int total = __shfl_sync(0xffffffffu, incl, 31);
              if (lane == 31 && total) base = atomicAdd(&sm.misc.nspec[k & 1], total);
              base = __shfl_sync(0xffffffffu, base, 31) + incl - cntb;
            }
            while (bits) {
              const int bpos = __ffs(bits) - 1;
              bits &= bits - 1u;
              const int local = tid * 32 + bpos;
              if (DT == kF32) {
                float* sf = reinterpret_cast<float*>(stage);
                sf[local] = ((nb >> bpos) & 1u) ? kFilter : penalize(sf[local], c.rho);
              } else {
                unsigned short* sh = reinterpret_cast<unsigned short*>(stage);
                const float x = __uint_as_float(static_cast<unsigned>(sh[local]) << 16);
                const float s = ((nb >> bpos) & 1u) ? kFilter : penalize(x, c.rho);
                if (base < kSpecCap) { sm.spec_s[base] = s; sm.spec_i[base] = static_cast<unsigned>(lo + local); }
                else sm.misc.spec_overflow = 1;
                ++base;
                sh[local] = 0xff80u;  // -inf: counted through the side list
              }
            }
          }
          if (tid == 0) sm.misc.nspec[(k + 1) & 1] = 0;
          __syncthreads();                                    // S1: data patched
          TG_TACC(row, 10, t_patch);
          if (sm.misc.timeout) {
            if (tid == 0) atomicOr(c.status, kFlagTimeout);
            for (int k2 = k + 1; k2 < nsub && k2 < k + a.nstage; ++k2) {   // drain copies in flight
              const int st2 = k2 % a.nstage;
              if (tma_ok) mbar_wait(&sm.misc.mbar[st2], (phase >> st2) & 1u);
            }
            return;
          }
          const int nspec = DT == kBF16 ? min(sm.misc.nspec[k & 1], kSpecCap) : 0;
          if (DT == kBF16 && sm.misc.spec_overflow) give_up = true;

          TG_T0(t_passB);
          if (!sample) {
            greedy_scan<DT>(stage, n, lo, nspec, sm, bv, bi);
          } else if (!give_up) {
            bool first = false;        // this sub-chunk sets mref and theta
            if (!decided) {
              // first sub-chunk with a score above the filter value: set the
              // reference maximum and theta from it
              float mx = block_max(stage_max<DT>(stage, n, nspec, sm), &sm.red);
              if (TEMP) mx = temper(mx, c.temp);
              if (mx > kFilter) {
                mref = mx;
                cc = mref * kLog2e;
                if (chance == 0) theta = mref - 8.0f;
                decided = true;
                first = true;
              }
            }
            if (decided) {
              bool raised = false;
              for (int attempt = 0;; ++attempt) {
                const float et0 = et, mxt0 = mxt;
                const int wc0 = wc;
                stage_pass<DT, TEMP>(stage, n, lo, nspec, sm, c.temp, theta, cc, et, mxt, wc);
                if (lane == 0) sm.misc.wcnt[wid] = wc;
                __syncthreads();
                const bool ovf = sm.misc.overflow != 0;
                const bool pilot = first && chance == 0 && !topk && !raised && attempt < 4;
                if (!ovf && !pilot) break;
                if (!ovf) {
                  // first sub-chunk: lower theta while too much of its mass lies below it
                  const float E = block_sum_f(et, &sm.red);
                  const float zc = cand_fast_mass(sm, cc);
                  if (E <= budget * (E + zc) || theta < mref - 40.0f) break;
                  et = 0.0f; mxt = mxt0; wc = 0;
                  if (lane == 0) sm.misc.wcnt[wid] = 0;
                  theta -= 4.0f;
                  __syncthreads();
                  continue;
                }
                // overflow: undo this sub-chunk, raise theta, compact, redo
                et = et0; mxt = mxt0; wc = wc0;
                if (lane == 0) sm.misc.wcnt[wid] = wc0;
                __syncthreads();
                if (tid == 0) sm.misc.overflow = 0;
                if (chance != 0 || attempt >= 12) { give_up = true; break; }
                const float E = block_sum_f(et, &sm.red);
                float th2 = theta;
                const bool have = cand_total(sm) > 0;
                if (have) {
                  const float zc = cand_fast_mass(sm, cc);
                  th2 = choose_theta(sm, theta, mref, cc, topk, c.top_k, 0.8f * (1.0f - qfrac) * (E + zc) - E);
                }
                if (!(th2 > theta)) th2 = theta + fmaxf(1.0f, fabsf(theta) * 1e-6f);
                if (th2 >= fmaxf(mref, block_max(mxt, &sm.red))) { give_up = true; break; }
                theta = th2;
                raised = true;
                if (have) {
                  const float dropped = compact_candidates(sm, theta, cc);
                  if (tid == 0) et += dropped;
                  wc = sm.misc.wcnt[wid];
                }
              }
              if (lane == 0 && wc > (3 * kSeg) / 4) sm.misc.prune = 1;
            }
          }
          TG_TACC(row, 12, t_passB);

          // ---- end of sub-chunk: release the stage (and prune if a list is filling up) ----
          fence_proxy_async();
          __syncthreads();                                    // S2
          if (sample && decided && !give_up && chance == 0 && sm.misc.prune) {
            TG_T0(t_prune);
            __syncthreads();
            if (tid == 0) sm.misc.prune = 0;
            // move the reference maximum up to the current one first
            const float mnow = fmaxf(mref, block_max(mxt, &sm.red));
            if (mnow > mref) { et *= expf(mref - mnow); mref = mnow; cc = mref * kLog2e; }
            const float E = block_sum_f(et, &sm.red);
            const float zc = cand_fast_mass(sm, cc);
            const float th2 = choose_theta(sm, theta, mref, cc, topk, c.top_k, budget * (E + zc) - E);
            if (th2 > theta) {
              theta = th2;
              const float dropped = compact_candidates(sm, theta, cc);
              if (tid == 0) et += dropped;
              wc = sm.misc.wcnt[wid];
            }
            __syncthreads();
            TG_TACC(row, 13, t_prune);
          }
          if (tma_ok && tid == 0 && k + a.nstage < nsub) {
            const int k2 = k + a.nstage;
            const int lo2 = k2 * SE, n2 = min(SE, V - lo2);
            mbar_expect_tx(&sm.misc.mbar[st], static_cast<unsigned>(n2 * esz));
            bulk_g2s(stage, rowp + static_cast<size_t>(lo2) * esz, static_cast<unsigned>(n2 * esz), &sm.misc.mbar[st],
                     policy);
          }
        }

        // ---------------- finish the row ----------------
        if (!sample) {
          const float m = block_max(bv, &sm.red);
          token = static_cast<int>(block_min_u(bv == m ? bi : 0xffffffffu, &sm.red));
          break;
        }
        const float m = fmaxf(mref, block_max(mxt, &sm.red));
        const float E = block_sum_f(et, &sm.red) * (decided ? expf(mref - m) : 0.0f);
        bool slow = give_up || !decided || m <= kFilter;
        int reason = give_up ? 1 : slow ? 3 : 0;
        unsigned tok = 0u;
        pack_candidates(sm);
        TG_DBG(row, 2, m); TG_DBG(row, 3, theta); TG_DBG(row, 4, E); TG_DBG(row, 7, sm.misc.ncand);
        TG_T0(t_fin);
        if (!slow) {
          FinResult fr = finalize_candidates(c, sm, m, static_cast<unsigned long long>(llrint(static_cast<double>(E) * kFixScale)),
                                             u, topk, topp);
          slow = !fr.ok;
          if (slow) reason = fr.reason;
          tok = fr.token;
        }
        TG_TACC(row, 14, t_fin);
        TG_DBG(row, 0, slow ? 1 + chance : 0); TG_DBG(row, 1, reason);
        if (!slow) {
          token = static_cast<int>(tok);
          break;
        }
        // Too little candidate mass for the cut or draw: one more pass with a
        // lower threshold, unless the list itself was the problem.
        if (chance == 0 && (reason == 5 || reason == 7) && theta > kFilter) {
          theta_fixed = theta - 1.5f;
          __syncthreads();
          continue;
        }
        // Multi-pass exact selection over the whole row.
        if (tid == 0) { atomicOr(c.status, kFlagSlow); atomicAdd(c.slow_rows, 1ull); }
        RowGlobalSource<DT> src{rowp, V, &c, H, N, bitmaps, true};
        float mm = -INFINITY;
        src.pass([&](float s, unsigned) { mm = fmaxf(mm, s); });
        mm = block_max(mm, &sm.red);
        tok = sample_exact(c, src, mm, u, static_cast<unsigned>(V), &sm.hist, &sm.red, nullptr, nullptr);
        token = static_cast<int>(tok);
        break;
      }  // chance
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
    __syncthreads();
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
  __syncthreads();
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
    S = mass_sum(src, kept, m, &sm.red);
  }
  float* pr = out_probs + static_cast<size_t>(row) * V;
  const double invS = 1.0 / static_cast<double>(S);
  for (int i = threadIdx.x; i < V; i += kThreads) {
    float s = sc[i];
    pr[i] = kept(fkey(s), static_cast<unsigned>(i)) ? static_cast<float>(static_cast<double>(wfix(s, m)) * invS) : 0.0f;
  }
}

#ifdef TG_DEBUG
extern "C" int tg_debug_set(double* p) { return (int)cudaMemcpyToSymbol(g_dbg, &p, sizeof(p)); }
#endif

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

int select_smem_bytes(int nstage, int nwords) {
  return sel_fixed_bytes() + 2 * bitmap_bytes(nwords) + nstage * kStageBytes;
}
int process_smem_bytes(int nwords) {
  return align_up(static_cast<int>(sizeof(ProcSmem)), 128) + 2 * bitmap_bytes(nwords);
}

template <int DT, bool VERIFY, bool TEMP>
static cudaError_t launch_sel(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  auto k = select_kernel<DT, VERIFY, TEMP>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, s>>>(c, a);
  return cudaGetLastError();
}

template <int DT, bool VERIFY>
static cudaError_t launch_sel_t(const DevCfg& c, const SelArgs& a, int grid, int smem, cudaStream_t s) {
  const bool temp = c.mode == kSample && c.temp != 1.0f;
  return temp ? launch_sel<DT, VERIFY, true>(c, a, grid, smem, s) : launch_sel<DT, VERIFY, false>(c, a, grid, smem, s);
}

cudaError_t launch_select(const DevCfg& c, const SelArgs& a, bool verify, int grid, int smem, cudaStream_t s) {
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, smem);
    if (e != cudaSuccess) return e;
    worst = occ < worst ? occ : worst;
  }
  *blocks_per_sm = worst;
  return cudaSuccess;
}

}  // namespace tg
