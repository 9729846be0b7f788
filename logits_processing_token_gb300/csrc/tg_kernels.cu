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

#include "tg_select_core.cuh"

namespace tg {

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

  if (tid == 0) sm.misc.nrow_done = nrow;
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
      if (sm.misc.err_snap) { if (tid == 0) sm.misc.nrow_done = ri; break; }   // uniform snapshot
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
      if (sm.misc.err_snap) { if (tid == 0) sm.misc.nrow_done = ri; break; }
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
          } else if (slow && reason == 7 && !topk && !topp && !state) {
            // a draw over the whole distribution that lands below the
            // candidates: the tail's histogram, then the one bin it falls in
            TG_T(row, 9);
            const FinResult fr3 = tail_pick<DT>(c, a, sm, rm, rowp, M, N, bitmaps, theta_f, m,
                                                static_cast<unsigned long long>(Zsigned), u);
            slow = !fr3.ok;
            if (slow) reason = 40 + fr3.reason;
            tok = fr3.token;
            tok_score = fr3.score;
            tok_S = fr3.S;
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

  // error: wait (bounded) for the copies still in flight, then leave.  No
  // copy is issued once the error flag is set, and an issued bulk copy
  // completes unless the memory system itself fails.  The rows this CTA did
  // not finish get -1 (verify: their batch row's out_match too; its count of
  // finished positions never completes, so no other CTA writes it).
  __syncthreads();
  if (sm.misc.error && tid == 0) {
    atomicOr(c.status, kFlagTimeout);
    for (int s = 0; s < nst; ++s) {
      const int n = sm.misc.iss[s];
      if (n > 0) mbar_drain(&sm.misc.full[s], static_cast<unsigned>((n - 1) & 1));
    }
  }
  if (sm.misc.error) {
    for (int q = sm.misc.nrow_done + tid; q < nrow; q += kThreads) {
      const int row = sm.rows[q];
      a.out[row] = -1;
      if (VERIFY) a.out_match[row / (a.K + 1)] = -1;
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

// ---------------------------------------------------------------------------
// Greedy ids for a batch too small to fill the GPU: each row is split over
// gridDim.x CTAs of slice_tok tokens (grid: slices x rows), so a few rows are
// read by many SMs instead of one each.  Every CTA builds the row's bitmaps
// (2 x V/8 bytes of shared memory), takes the best processed score of its
// tokens with select_kernel's rules (the larger score, on a tie the smaller
// id; a marked token competes with its processed score, an unmarked one with
// its logit, and an unmarked -inf is never taken), and folds it into the
// row's 64-bit key in global memory with atomicMax: order-preserving score
// bits above the complemented id.  The last of the row's CTAs to count
// itself in takes the key, leaves the key and the count at zero for the next
// call, and writes the id.  No CTA waits for another.
// ---------------------------------------------------------------------------
constexpr int kSplitStage = 4096;   // history ids staged in shared memory (a longer history is read in place)
struct SplitSmem {
  float wf[kWarps];
  unsigned wu[kWarps];
};
__host__ __device__ constexpr int split_stage_off() { return align_up(static_cast<int>(sizeof(SplitSmem)), 128); }
__host__ __device__ constexpr int split_bits_off() { return align_up(split_stage_off() + kSplitStage * 4, 128); }
__host__ __device__ constexpr int split_smem(int nwords) { return split_bits_off() + 2 * bitmap_bytes(nwords); }

// Unsigned key in the order of the floats (no NaN reaches it).
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    split_greedy_kernel(const DevCfg c, const SelArgs a, int slice_tok, unsigned long long* best, unsigned* tick,
                        int verify) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SplitSmem& ss = *reinterpret_cast<SplitSmem*>(smem_raw);
  int* stage = reinterpret_cast<int*>(smem_raw + split_stage_off());
  unsigned* M = reinterpret_cast<unsigned*>(smem_raw + split_bits_off());
  unsigned* N = reinterpret_cast<unsigned*>(smem_raw + split_bits_off() + bitmap_bytes(a.nwords));
  constexpr int esz = DT == kF32 ? 4 : 2;
  constexpr int PER = 16 / esz;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int row = a.row_begin + static_cast<int>(blockIdx.y);
  const int V = a.V;

  // The logits and histories may come from the kernel before this one.
  grid_dependency_wait();
  grid_dependents_launch();
  // verify (no processors): every position is read
  const RowMeta rm = verify ? RowMeta{} : row_meta(c, a.hist, a.off, a.plen, row, a.nrows_total);
  if (!verify && (rm.bad || rm.L == 0 || rm.forced)) {
    // not read: the first slice writes the row's id
    if (blockIdx.x == 0 && tid == 0) {
      if (rm.bad || rm.L == 0) {
        a.out[row] = -1;
        if (rm.bad) atomicOr(c.status, kFlagBadRow);
      } else {
        unsigned long long kept = 1ull;
        a.out[row] = forced_token(c, rm, V, 0.0f, false, &kept);
      }
    }
    return;
  }
  const bool bitmaps = !verify && (c.rho != 1.0f || c.ngram > 0 || c.n_ban > 0 || c.n_bsup > 0 || c.n_seq > 0 ||
                                    (c.n_eos > 0 && (c.min_length > 0 || c.min_new > 0)));
  if (bitmaps) build_row_bitmaps(c, a.hist, rm, M, N, a.nwords, stage, kSplitStage);   // M = history | banned

  const int t0 = static_cast<int>(blockIdx.x) * slice_tok;
  const int t1 = min(V, t0 + slice_tok);
  const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + static_cast<size_t>(row) * V * esz;
  float bv = -INFINITY;
  unsigned bi = 0xffffffffu;
  // a thread's tokens come in increasing id order
  auto take = [&](float x, int i) {
    if (bitmaps && get_bit(M, i)) {
      const float s = process_elem(c, M, N, x, i, false);
      if (s > bv || (s == bv && static_cast<unsigned>(i) < bi)) { bv = s; bi = static_cast<unsigned>(i); }
    } else if (x > bv) {
      bv = x;
      bi = static_cast<unsigned>(i);
    }
  };
  const bool vec = ((reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0u) && ((static_cast<size_t>(V) * esz) % 16u == 0u);
  if (vec) {
    // whole 16-byte vectors (slice_tok is a multiple of 8 tokens), four in flight per thread
    const uint4* rv = reinterpret_cast<const uint4*>(rowp);
    const int v0 = t0 / PER, v1 = t1 / PER;
    for (int vb = v0; vb < v1; vb += 4 * kThreads) {
      uint4 q[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int vi = vb + h * kThreads + tid;
        q[h] = vi < v1 ? __ldg(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int vi = vb + h * kThreads + tid;
        if (vi < v1) {
          const unsigned ps[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
#pragma unroll
          for (int e = 0; e < PER; ++e)
            take(DT == kF32 ? __uint_as_float(ps[e]) : ((e & 1) ? bf16hi(ps[e >> 1]) : bf16lo(ps[e >> 1])), vi * PER + e);
        }
      }
    }
  } else {
    for (int i = t0 + tid; i < t1; i += kThreads) take(load_logit<DT>(rowp, i), i);
  }
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
    const unsigned i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
  }
  if (lane == 0) { ss.wf[wid] = bv; ss.wu[wid] = bi; }
  csync();
  if (tid == 0) {
    float v = ss.wf[0];
    unsigned b = ss.wu[0];
    for (int q = 1; q < kWarps; ++q) {
      const float v2 = ss.wf[q];
      const unsigned i2 = ss.wu[q];
      if (v2 > v || (v2 == v && i2 < b)) { v = v2; b = i2; }
    }
    // no candidate: -inf over id 0xffffffff, below every real key, and the id -1 if no slice has one
    atomicMax(best + row, (static_cast<unsigned long long>(order_key(v)) << 32) | static_cast<unsigned long long>(~b));
    __threadfence();
    const unsigned done = atomicAdd(tick + row, 1u);
    if (done == gridDim.x - 1) {
      __threadfence();
      const unsigned long long k = atomicExch(best + row, 0ull);
      tick[row] = 0u;
      a.out[row] = static_cast<int>(~static_cast<unsigned>(k & 0xffffffffull));
      if (verify) verify_ticket(c, a, row);   // the last position of a sequence writes its match
    }
  }
}

template <int DT>
static cudaError_t launch_split_t(const DevCfg& c, const SelArgs& a, int nslice, int slice_tok,
                                  unsigned long long* best, unsigned* tick, bool verify, cudaStream_t s) {
  auto k = split_greedy_kernel<DT>;
  const int smem = split_smem(a.nwords);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nslice), static_cast<unsigned>(a.nrows - a.row_begin));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, c, a, slice_tok, best, tick, verify ? 1 : 0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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

int split_greedy_smem(int nwords) { return split_smem(nwords); }

cudaError_t launch_split_greedy(const DevCfg& c, const SelArgs& a, int nslice, int slice_tok, unsigned long long* best,
                                unsigned* tick, bool verify, cudaStream_t s) {
  if (nslice < 1 || slice_tok < 8 || slice_tok % 8 != 0 || a.nrows <= a.row_begin || a.nrows - a.row_begin > 65535)
    return cudaErrorInvalidValue;
  return c.dtype == kF32 ? launch_split_t<kF32>(c, a, nslice, slice_tok, best, tick, verify, s)
                         : launch_split_t<kBF16>(c, a, nslice, slice_tok, best, tick, verify, s);
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

// Testing: the select kernels' streaming waits give up after `cycles` SM
// cycles (0: the default, about one second).
extern "C" tg_status tg_set_wait_limit(uint64_t cycles) {
  const unsigned long long v = cycles ? static_cast<unsigned long long>(cycles) : kWaitLimitCycles;
  return cudaMemcpyToSymbol(g_wait_limit, &v, sizeof(v)) == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

#ifdef TG_DEBUG
extern "C" int tg_debug_set(double* p) { return (int)cudaMemcpyToSymbol(g_dbg, &p, sizeof(p)); }
#endif

}  // namespace tg
