// Beam search, the device part of one step (Transmuter.Generation, module
// intro, the paragraphs on num_beams): for each beam row the log-softmax of
// its logits, the processors on it and the beam's score; for each prompt the
// best max(2, 1 + eos tokens) * num_beams of its num_beams * V candidates, in
// the order (score desc, flat index asc) with flat index = beam * V + token.
// The host's part of the step (finished hypotheses, length penalty,
// stopping) is not here.
//
// One thread-block cluster per prompt, one CTA (8 warps) per beam row.  A
// CTA reads its row once for the log-sum-exp, then selects its own best keep
// candidates with the radix k-th-key engine over the processed scores (the
// row is in L2 by then); after a cluster barrier, CTA 0 of the cluster reads
// every beam's candidates from the other CTAs' shared memory (distributed
// shared memory), ranks them and writes the prompt's result.  A second
// cluster barrier keeps each CTA's shared memory alive until CTA 0 is done.
#include <cstdint>

#include <cuda_runtime.h>

// 8 warps per beam row: two CTAs share an SM, so a step's clusters run in
// one wave and one CTA's barriers overlap the other's passes
#define TG_THREADS 256
#include "../../include/tg.h"
#include "tg_device.cuh"

namespace tg {
namespace {

constexpr int kBeamRowCap = 128;                          // candidates one beam row hands over
constexpr int kMergeCap = kBeamRowCap * kMaxClusterBeams;  // candidates of one prompt
constexpr int kBeamStage = 8192;                           // history ids staged for the marked-token list
constexpr int kLevelsBeam = 8;                             // level l: within 2^l / 4 of the top unmarked logit

__host__ __device__ constexpr int beam_bitmap_words(int nwords) { return (nwords * 4 + 127) / 128 * 32; }

struct BeamSmem {
  Hist hist;
  RedScratch red;
  float cs[kBeamRowCap];     // this row's candidates: score, token
  unsigned ci[kBeamRowCap];
  float ms[kMergeCap];       // CTA 0: the prompt's candidates: score, flat index
  unsigned mi[kMergeCap];
  int n;                     // this row's candidate count (read by CTA 0 of the cluster)
  int ngt;                   // candidates strictly above the k-th key
  int moff[kMaxClusterBeams + 1];
  int wcnt[kWarps];
  unsigned lctr;
  int lvl[kWarps][kLevelsBeam];
  float lse_hi, lse_lo;
  int stage[kBeamStage];     // the row's history while its bitmaps and marked-token list are built
};

constexpr int kBeamFixed = (static_cast<int>(sizeof(BeamSmem)) + 127) / 128 * 128;

#ifdef TG_DEBUG
__device__ long long* g_beam_dbg = nullptr;
#define TB_T(slot) do { if (g_beam_dbg && threadIdx.x == 0) g_beam_dbg[blockIdx.x * 16 + (slot)] = clock64(); } while (0)
#else
#define TB_T(slot) do { } while (0)
#endif

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; release / acquire order the
// shared-memory writes before it against the reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ unsigned peer_addr(const void* p, unsigned rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned ld_peer_u32(unsigned addr) {
  unsigned v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <int DT>
__device__ __forceinline__ float beam_logit(const unsigned char* row, int i) {
  if (DT == kF32) return __ldg(reinterpret_cast<const float*>(row) + i);
  return __uint_as_float(static_cast<unsigned>(__ldg(reinterpret_cast<const unsigned short*>(row) + i)) << 16);
}

// Level of an unmarked logit x against the row's largest unmarked logit mu
// (d = mu - x >= 0): the smallest l with d <= 2^l / 4, or kLevelsBeam.
__device__ __forceinline__ int beam_level(float d) {
  const float d4 = d * 4.0f;
  if (!(d4 > 1.0f)) return 0;
  const unsigned b = __float_as_uint(d4);
  const int e = static_cast<int>(b >> 23) - 127 + ((b & 0x007fffffu) != 0u ? 1 : 0);
  return min(e, kLevelsBeam);
}

// One (not forced) beam row's candidate scores: the log-softmax x - lse
// (lse carried as hi + lo), the processors (bitmaps M = marked, N = banned),
// plus the beam's score, never below the filter value.  Register-only
// members: the per-token work reads no local memory.
template <int DT>
struct BeamRow {
  const unsigned char* row;
  int V;
  float rho;
  const unsigned* M;
  const unsigned* N;
  bool bitmaps;
  float lse_hi, lse_lo, bs;
  // renormalize_logits: the processed log-probabilities less their own
  // log-sum-exp (r_hi + r_lo); when every token is removed, all score -ln V
  bool renorm, allf;
  float r_hi, r_lo, lnv;

  // processed log-probability -> candidate score
  __device__ __forceinline__ float fin(float ls) const {
    if (renorm) ls = allf ? -lnv : clampf(__fsub_rn(__fsub_rn(ls, r_hi), r_lo));
    return clampf(__fadd_rn(ls, bs));
  }
  __device__ __forceinline__ float processed(float x, int i) const {
    float ls = __fsub_rn(__fsub_rn(x, lse_hi), lse_lo);
    if (bitmaps) {
      if (get_bit(N, i)) ls = kFilter;
      else if (get_bit(M, i)) ls = penalize(ls, rho);
    }
    return ls;
  }
  __device__ __forceinline__ float score(float x, int i) const { return fin(processed(x, i)); }
  // An unmarked token's score (no processor changes it).  The bitmaps are not
  // read: N may hold the marked-token list instead of the banned bitmap.
  __device__ __forceinline__ float score_unmarked(float x) const {
    return fin(__fsub_rn(__fsub_rn(x, lse_hi), lse_lo));
  }
  // Every token once: 16-byte vectors, four per thread in flight, when the
  // row is 16-byte aligned; the rest element by element.
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    constexpr int PER = DT == kF32 ? 4 : 8;
    constexpr int NV = 4;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) {
      const int nvec = V / PER;
      const uint4* rv = reinterpret_cast<const uint4*>(row);
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
              const float x = DT == kF32 ? __uint_as_float(ps[e])
                                         : __uint_as_float((e & 1) ? (ps[e >> 1] & 0xffff0000u) : (ps[e >> 1] << 16));
              const int i = vi * PER + e;
              f(x, i);
            }
          }
        }
      }
      done = nvec * PER;
    }
    for (int i = done + static_cast<int>(threadIdx.x); i < V; i += kThreads) f(beam_logit<DT>(row, i), i);
  }
  // Every token once, a 16-byte vector at a time: fv(x[PER], first index,
  // marked bits of the PER tokens) -- one bitmap read per vector -- and
  // fs(x, i, marked) for the tail (and every token of an unaligned row).
  template <class FV, class FS>
  __device__ __forceinline__ void pass_vec(FV fv, FS fs) const {
    constexpr int PER = DT == kF32 ? 4 : 8;
    constexpr int NV = 8;   // 64 KB of a row in flight per CTA
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) {
      const int nvec = V / PER;
      const uint4* rv = reinterpret_cast<const uint4*>(row);
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
            float x[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e)
              x[e] = DT == kF32 ? __uint_as_float(ps[e])
                                : __uint_as_float((e & 1) ? (ps[e >> 1] & 0xffff0000u) : (ps[e >> 1] << 16));
            const int i0 = vi * PER;
            const unsigned mk = bitmaps ? (M[i0 >> 5] >> (i0 & 31)) & ((1u << PER) - 1u) : 0u;
            fv(x, i0, mk);
          }
        }
      }
      done = nvec * PER;
    }
    for (int i = done + static_cast<int>(threadIdx.x); i < V; i += kThreads)
      fs(beam_logit<DT>(row, i), i, bitmaps && get_bit(M, i));
  }
};

// Scores (not raw logits) for kth_key.
template <int DT>
struct BeamScores {
  BeamRow<DT> br;   // a copy: taking the row's address would move it to local memory
  template <class Fn>
  __device__ __forceinline__ void pass(Fn f) const {
    br.pass([&](float x, int i) { f(br.score(x, i), static_cast<unsigned>(i)); });
  }
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) beam_kernel(const DevCfg c, const BeamArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BeamSmem& sm = *reinterpret_cast<BeamSmem*>(smem_raw);
  unsigned* M = reinterpret_cast<unsigned*>(smem_raw + kBeamFixed);
  unsigned* N = M + beam_bitmap_words(a.nwords);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int r = blockIdx.x;              // beam row
  const int prompt = r / a.nb;
  const unsigned beam = cluster_rank();  // == r % nb
  const int V = a.V;
  const int kk = min(a.keep, V);         // candidates this row can hand over

  grid_dep_wait();
  TB_T(0);
  if (tid == 0) { sm.n = 0; sm.ngt = 0; }

  const RowMeta rm = row_meta(c, a.hist, a.off, a.plen, r, a.nrows);
  if (rm.bad && tid == 0) atomicOr(c.status, kFlagBadRow);
  if (!rm.bad && rm.L > 0) {
    const unsigned char* row = static_cast<const unsigned char*>(a.logits) +
                               static_cast<size_t>(r) * V * (DT == kF32 ? 4 : 2);
    BeamRow<DT> br;
    br.row = row;
    br.V = V;
    br.rho = c.rho;
    br.M = M;
    br.N = N;
    br.bitmaps = !rm.forced && (c.rho != 1.0f || c.ngram > 0 || c.n_ban > 0 || c.n_bsup > 0 || c.n_seq > 0 ||
                                (c.n_eos > 0 && (c.min_length > 0 || c.min_new > 0)));
    br.bs = a.beam_scores[r];
    br.lse_hi = 0.0f;
    br.lse_lo = 0.0f;
    br.renorm = c.renorm != 0;
    br.allf = false;
    br.r_hi = 0.0f;
    br.r_lo = 0.0f;
    br.lnv = logf(static_cast<float>(V));
    if (rm.forced) {
      // every token scores the filter value except the forced ids (0), before
      // the beam's score: the forced ids in index order, then the lowest other ids
      if (tid == 0) {
        int zs[8];
        const int nzall = forced_zeros(c, rm, zs);
        // renormalized: the forced ids share the mass (-ln nz each), or every
        // token is removed and all score -ln V
        br.allf = nzall == 0;
        br.r_hi = nzall > 0 ? logf(static_cast<float>(nzall)) : 0.0f;
        const float s0 = br.fin(0.0f), sf = br.fin(kFilter);
        const int nz = s0 > sf ? nzall : 0;   // equal scores: index order alone
        int n = 0;
        for (int q = 0; q < nz && n < kk; ++q) {
          sm.cs[n] = s0;
          sm.ci[n++] = static_cast<unsigned>(zs[q]);
        }
        for (int t = 0; t < V && n < kk; ++t) {
          bool z = false;
          for (int q = 0; q < nz; ++q) z |= zs[q] == t;
          if (!z) {
            bool zero = false;
            for (int q = 0; q < nzall; ++q) zero |= zs[q] == t;
            sm.cs[n] = zero ? s0 : sf;
            sm.ci[n++] = static_cast<unsigned>(t);
          }
        }
        sm.n = n;
      }
    } else {
      // bitmaps, and the marked tokens listed (in N's words) when they fit
      const int nlist = br.bitmaps ? build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, sm.stage, kBeamStage, &sm.lctr)
                                   : 0;
      TB_T(1);
      // pass 1: log-sum-exp (each thread keeps (max, sum of exp(x - max)),
      // rescaled when its maximum grows) and the largest unmarked logit
      constexpr int PER = DT == kF32 ? 4 : 8;
      // (with renormalize_logits also the unmarked tokens' share, tsu)
      float tm = -INFINITY, ts = 0.0f, tu = -INFINITY, tsu = 0.0f;
      br.pass_vec(
          [&](const float (&x)[PER], int, unsigned mk) {
            float vm = x[0], vu = (mk & 1u) ? -INFINITY : x[0];
#pragma unroll
            for (int e = 1; e < PER; ++e) {
              vm = fmaxf(vm, x[e]);
              vu = ((mk >> e) & 1u) ? vu : fmaxf(vu, x[e]);
            }
            if (vm > tm) {
              const float f = tm > -INFINITY ? expf(tm - vm) : 0.0f;
              ts *= f;
              tsu *= f;
              tm = vm;
            }
            float add = 0.0f, addu = 0.0f;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
              const float ex = expf(x[e] - tm);
              add += ex;
              addu += ((mk >> e) & 1u) ? 0.0f : ex;
            }
            ts += add;
            tsu += addu;
            tu = fmaxf(tu, vu);
          },
          [&](float x, int, bool mkd) {
            if (x > tm) {
              const float f = tm > -INFINITY ? expf(tm - x) : 0.0f;
              ts *= f;
              tsu *= f;
              tm = x;
            }
            const float ex = expf(x - tm);
            ts += ex;
            tsu += mkd ? 0.0f : ex;
            if (!mkd) tu = fmaxf(tu, x);
          });
      const float m = block_max(tm, &sm.red);
      const float mu = block_max(tu, &sm.red);
      const float part = tm > -INFINITY ? ts * expf(tm - m) : 0.0f;
      const float S = block_sum_f(part, &sm.red);
      if (tid == 0) {
        // lse = m + ln S, S >= 1: ln S from S's binary exponent and log2f of
        // its mantissa (no fp64 transcendental), then split into hi + lo
        constexpr double kLn2 = 0.6931471805599453;
        const unsigned b = __float_as_uint(S);
        const int e = static_cast<int>(b >> 23) - 127;
        const float mant = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
        const double lse = static_cast<double>(m) + (static_cast<double>(e) + static_cast<double>(log2f(mant))) * kLn2;
        const float hi = static_cast<float>(lse);
        sm.lse_hi = hi;
        sm.lse_lo = static_cast<float>(lse - static_cast<double>(hi));
      }
      __syncthreads();
      br.lse_hi = sm.lse_hi;
      br.lse_lo = sm.lse_lo;
      if (br.renorm) {
        // log-sum-exp of the processed log-probabilities: the unmarked tokens'
        // share of the row's mass (U / S) plus each marked token's exp(ls)
        const float U = block_sum_f(tm > -INFINITY ? tsu * expf(tm - m) : 0.0f, &sm.red);
        float mk = 0.0f;
        if (nlist >= 0) {
          for (int j = tid; j < nlist; j += kThreads) {
            const unsigned ent = N[j];
            const int t = static_cast<int>(ent & ~kBannedFlag);
            const float ls = __fsub_rn(__fsub_rn(beam_logit<DT>(row, t), br.lse_hi), br.lse_lo);
            mk += expf((ent & kBannedFlag) ? kFilter : penalize(ls, br.rho));
          }
        } else {
          br.pass([&](float x, int i) {
            if (get_bit(M, i)) mk += expf(br.processed(x, i));
          });
        }
        mk = block_sum_f(mk, &sm.red);
        if (tid == 0) {
          constexpr double kLn2 = 0.6931471805599453;
          const double tot = static_cast<double>(U) / static_cast<double>(S) + static_cast<double>(mk);
          if (!(tot > 0.0)) {
            sm.lse_hi = 0.0f;
            sm.lse_lo = -1.0f;   // every token removed
          } else {
            const float tf = static_cast<float>(tot);
            const unsigned b = __float_as_uint(tf);
            const int e = static_cast<int>(b >> 23) - 127;
            const float mant = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
            const double lse2 = (static_cast<double>(e) + static_cast<double>(log2f(mant))) * kLn2;
            sm.lse_hi = static_cast<float>(lse2);
            sm.lse_lo = static_cast<float>(lse2 - static_cast<double>(sm.lse_hi));
          }
        }
        __syncthreads();
        br.allf = sm.lse_lo == -1.0f && sm.lse_hi == 0.0f;
        br.r_hi = br.allf ? 0.0f : sm.lse_hi;
        br.r_lo = br.allf ? 0.0f : sm.lse_lo;
      }
      TB_T(2);

      // Fast path.  An unmarked token's score rises with its logit, so the kk
      // best unmarked tokens lie within 2^l / 4 of mu for the first level l
      // that holds kk of them (pass 2 counts them per level); pass 3 gathers
      // those (C), every marked token scoring at least as much as the lowest
      // of them joins C (one scoring exactly as much waits for the tie walk),
      // and a rank sort picks C's kk best.  Every token outside C scores at
      // most s_out (the best unmarked one left out) or at most that lowest
      // score, so the kk-th score of C is the row's: the result is exact when
      // it beats both.  Otherwise (rounding made
      // tokens outside C tie it) the tokens above it come from C and the ties
      // from an index-order walk of the row; when the counts do not fit, the
      // radix path decides.
      bool done = false, have_klo = false;
      unsigned klo_known = 0u;
      int nc_known = 0;
      if (nlist >= 0 && mu > -INFINITY) {
        // gather every unmarked token with 4 (mu - x) <= lim4 into C, keeping
        // the best unmarked logit left out; returns how many
        float smin = INFINITY, xout = -INFINITY;
        auto gather_within = [&](float lim4) {
          if (tid == 0) sm.ngt = 0;
          __syncthreads();
          smin = INFINITY;
          xout = -INFINITY;
          auto gather = [&](float x, int i) {
            if ((mu - x) * 4.0f <= lim4) {
              const float s = br.score_unmarked(x);
              smin = fminf(smin, s);
              const int pos = atomicAdd(&sm.ngt, 1);
              if (pos < kMergeCap) { sm.ms[pos] = s; sm.mi[pos] = static_cast<unsigned>(i); }
            } else {
              xout = fmaxf(xout, x);
            }
          };
          br.pass_vec(
              [&](const float (&x)[PER], int i0, unsigned mk) {
#pragma unroll
                for (int e = 0; e < PER; ++e)
                  if (!((mk >> e) & 1u)) gather(x[e], i0 + e);
              },
              [&](float x, int i, bool mkd) {
                if (!mkd) gather(x, i);
              });
          __syncthreads();
          return sm.ngt;
        };
        // usually a few tokens lie within 2 of mu, at least kk of them: one
        // pass gathers them (level 3)
        int ng = gather_within(8.0f);
        bool ok = ng >= kk && ng <= kMergeCap;
        TB_T(3);
        if (!ok) {
          // count levels 0-7 and gather at the first that holds kk
          unsigned long long acc0 = 0ull, acc1 = 0ull;   // 16-bit counts of levels 0-3, 4-7
          auto count = [&](float x) {
            const float d4 = (mu - x) * 4.0f;
            if (d4 <= 8.0f) acc0 += 1ull << (16 * beam_level(mu - x));
            else if (d4 <= 128.0f) acc1 += 1ull << (16 * (beam_level(mu - x) - 4));
          };
          br.pass_vec(
              [&](const float (&x)[PER], int, unsigned mk) {
#pragma unroll
                for (int e = 0; e < PER; ++e)
                  if (!((mk >> e) & 1u)) count(x[e]);
              },
              [&](float x, int, bool mkd) {
                if (!mkd) count(x);
              });
          int cnt[kLevelsBeam];
#pragma unroll
          for (int l = 0; l < kLevelsBeam; ++l) {
            int v = static_cast<int>(((l < 4 ? acc0 : acc1) >> (16 * (l & 3))) & 0xffffull);
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            cnt[l] = v;
          }
          if (lane == 0) {
#pragma unroll
            for (int l = 0; l < kLevelsBeam; ++l) sm.lvl[wid][l] = cnt[l];
          }
          __syncthreads();
          int lsel = -1, cum = 0;
          for (int l = 0; l < kLevelsBeam && lsel < 0; ++l) {
            for (int q = 0; q < kWarps; ++q) cum += sm.lvl[q][l];
            if (cum >= kk) lsel = l;
          }
          if (lsel >= 0 && cum <= kMergeCap) {
            ng = gather_within(static_cast<float>(1 << lsel));
            ok = ng >= kk && ng <= kMergeCap;
          }
        }
        if (ok) {
          const float sbnd = -block_max(-smin, &sm.red);
          const float xo = block_max(xout, &sm.red);
          const float s_out = xo > -INFINITY ? br.score_unmarked(xo) : -INFINITY;
          TB_T(4);
          // marked tokens: their processed score (filter value when banned, else
          // penalised), plus the beam's score
          int mk_eq = 0;
          for (int j = tid; j < nlist; j += kThreads) {
            const unsigned ent = N[j];
            const int t = static_cast<int>(ent & ~kBannedFlag);
            const float x = beam_logit<DT>(row, t);
            float ls = __fsub_rn(__fsub_rn(x, br.lse_hi), br.lse_lo);
            ls = (ent & kBannedFlag) ? kFilter : penalize(ls, br.rho);
            const float s = br.fin(ls);
            if (s > sbnd) {
              const int pos = atomicAdd(&sm.ngt, 1);
              if (pos < kMergeCap) { sm.ms[pos] = s; sm.mi[pos] = static_cast<unsigned>(t); }
            }
            mk_eq += s == sbnd ? 1 : 0;
          }
          mk_eq = static_cast<int>(block_sum_u64(static_cast<unsigned long long>(mk_eq), &sm.red));
          const int nc = sm.ngt;
          TB_T(5);
          if (nc <= kMergeCap) {
            // the kk best by (score desc, index asc)
            float skk = INFINITY;
            for (int q = tid; q < nc; q += kThreads) {
              const unsigned kq = fkey(sm.ms[q]), iq = sm.mi[q];
              int rank = 0;
              for (int o = 0; o < nc; ++o) {
                const unsigned ko = fkey(sm.ms[o]);
                rank += (ko > kq) || (ko == kq && sm.mi[o] < iq);
              }
              if (rank < kk) {
                sm.cs[rank] = sm.ms[q];
                sm.ci[rank] = iq;
                if (rank == kk - 1) skk = sm.ms[q];
              }
            }
            const float kth = -block_max(-skk, &sm.red);
            // marked tokens at exactly sbnd are not in C: they can only tie
            done = kth > s_out && (kth > sbnd || mk_eq == 0);
            if (done && tid == 0) sm.n = kk;
            if (!done) {
              have_klo = true;
              klo_known = fkey(kth);
              nc_known = nc;
            }
          }
        }
      }
      if (!done) {
        // radix path: the kk-th largest key, then every token above it and the
        // lowest-index tokens at it (with the banned bitmap back in N's words)
        if (br.bitmaps) build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, sm.stage, kBeamStage);
        if (tid == 0) sm.ngt = 0;
        __syncthreads();
        unsigned klo;
        int neq;
        if (have_klo) {
          // the tokens above the kk-th score are all in C
          klo = klo_known;
          for (int q = tid; q < nc_known; q += kThreads) {
            if (fkey(sm.ms[q]) > klo) {
              const int pos = atomicAdd(&sm.ngt, 1);
              if (pos < kBeamRowCap) { sm.cs[pos] = sm.ms[q]; sm.ci[pos] = sm.mi[q]; }
            }
          }
          int myeq = 0;
          br.pass([&](float x, int i) { myeq += fkey(br.score(x, i)) == klo ? 1 : 0; });
          neq = static_cast<int>(block_sum_u64(static_cast<unsigned long long>(myeq), &sm.red));
        } else {
          // counted in the status word with the exact-path rows of tg_select
          if (tid == 0) {
            atomicOr(c.status, kFlagSlow);
            atomicAdd(c.slow_rows, 1ull);
          }
          BeamScores<DT> src{br};
          klo = kth_key(src, KeepFilter{0u, false, 0u, 0u}, static_cast<unsigned>(kk), &sm.hist);
          int myeq = 0;
          br.pass([&](float x, int i) {
            const float s = br.score(x, i);
            const unsigned key = fkey(s);
            if (key > klo) {
              const int pos = atomicAdd(&sm.ngt, 1);
              if (pos < kBeamRowCap) { sm.cs[pos] = s; sm.ci[pos] = static_cast<unsigned>(i); }
            } else if (key == klo) {
              ++myeq;
            }
          });
          neq = static_cast<int>(block_sum_u64(static_cast<unsigned long long>(myeq), &sm.red));
        }
        const int ngt = min(sm.ngt, kBeamRowCap);
        const int need = min(kk - ngt, kBeamRowCap - ngt);   // ties to take, lowest index first
        if (need > 0 && neq <= need) {
          // every tie is taken
          br.pass([&](float x, int i) {
            const float s = br.score(x, i);
            if (fkey(s) == klo) {
              const int pos = atomicAdd(&sm.ngt, 1);
              if (pos < kBeamRowCap) { sm.cs[pos] = s; sm.ci[pos] = static_cast<unsigned>(i); }
            }
          });
        } else if (need > 0) {
          // in index order, 8 consecutive tokens per thread, block by block,
          // until enough
          constexpr int kRun = 8;
          int taken = 0;
          for (int base = 0; base < V && taken < need; base += kRun * kThreads) {
            const int i0 = base + kRun * tid;
            unsigned hit = 0u;
#pragma unroll
            for (int e = 0; e < kRun; ++e) {
              const int i = i0 + e;
              if (i < V && fkey(br.score(beam_logit<DT>(row, i), i)) == klo) hit |= 1u << e;
            }
            const int mine = __popc(hit);
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int t = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += t;
            }
            if (lane == 31) sm.wcnt[wid] = incl;
            __syncthreads();
            int before = 0, total = 0;
            for (int q = 0; q < kWarps; ++q) {
              before += q < wid ? sm.wcnt[q] : 0;
              total += sm.wcnt[q];
            }
            int pos = taken + before + incl - mine;
            while (hit) {
              const int e = __ffs(hit) - 1;
              hit &= hit - 1u;
              if (pos < need) {
                sm.cs[ngt + pos] = key2f(klo);
                sm.ci[ngt + pos] = static_cast<unsigned>(i0 + e);
              }
              ++pos;
            }
            taken += total;
            __syncthreads();
          }
        }
        __syncthreads();
        if (tid == 0) sm.n = min(kk, kBeamRowCap);
      }
    }
  }

  TB_T(6);
  // ---- the prompt's merge, in CTA 0 of the cluster ----
  cluster_sync();
  TB_T(7);
  if (beam == 0) {
    const int nb = a.nb;
    if (tid == 0) {
      int o = 0;
      for (int j = 0; j < nb; ++j) {
        sm.moff[j] = o;
        o += static_cast<int>(ld_peer_u32(peer_addr(&sm.n, static_cast<unsigned>(j))));
      }
      sm.moff[nb] = o;
    }
    __syncthreads();
    const int total = sm.moff[nb];
    for (int e = tid; e < total; e += kThreads) {
      int j = 0;
      while (e >= sm.moff[j + 1]) ++j;
      const int q = e - sm.moff[j];
      const unsigned s = ld_peer_u32(peer_addr(&sm.cs[q], static_cast<unsigned>(j)));
      const unsigned t = ld_peer_u32(peer_addr(&sm.ci[q], static_cast<unsigned>(j)));
      sm.ms[e] = __uint_as_float(s);
      sm.mi[e] = static_cast<unsigned>(j) * static_cast<unsigned>(V) + t;
    }
    __syncthreads();
    const int K = a.keep;
    for (int e = tid; e < total; e += kThreads) {
      const unsigned ke = fkey(sm.ms[e]), fe = sm.mi[e];
      int rank = 0;
      for (int o = 0; o < total; ++o) {
        const unsigned ko = fkey(sm.ms[o]);
        rank += (ko > ke) || (ko == ke && sm.mi[o] < fe);
      }
      if (rank < K) {
        const size_t w = static_cast<size_t>(prompt) * K + rank;
        a.out_scores[w] = sm.ms[e];
        a.out_tokens[w] = static_cast<int32_t>(fe % static_cast<unsigned>(V));
        a.out_beams[w] = static_cast<int32_t>(fe / static_cast<unsigned>(V));
      }
    }
    // a prompt with fewer candidates than it keeps (padding rows)
    for (int e = total + tid; e < K; e += kThreads) {
      const size_t w = static_cast<size_t>(prompt) * K + e;
      a.out_scores[w] = kFilter;
      a.out_tokens[w] = -1;
      a.out_beams[w] = -1;
    }
  }
  grid_dep_launch();
  TB_T(8);
  cluster_sync();
}

}  // namespace

int beam_smem_bytes(int nwords) { return kBeamFixed + 2 * beam_bitmap_words(nwords) * 4; }

#ifdef TG_DEBUG
extern "C" void tg_beam_debug_set(long long* p) { cudaMemcpyToSymbol(g_beam_dbg, &p, sizeof(p)); }
#endif

cudaError_t launch_beam(const DevCfg& c, const BeamArgs& a, cudaStream_t s) {
  if (a.nb < 1 || a.nb > kMaxClusterBeams || a.nrows % a.nb != 0 || a.keep < 1) return cudaErrorInvalidValue;
  const int smem = beam_smem_bytes(a.nwords);
  void (*k)(DevCfg, BeamArgs) = c.dtype == kF32 ? beam_kernel<kF32> : beam_kernel<kBF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.nrows));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.nb);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, c, a);
}

}  // namespace tg
