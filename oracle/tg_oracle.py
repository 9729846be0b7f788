"""Plain CPU oracle for per-step token selection and assisted-generation verify.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this module.  The CUDA library never imports, links or calls it, and it
shares no code with the CUDA path (no helpers, tables or constants).

What it computes, step by step, in the order the pages give:

* Transmuter.Generation (transmuter v2.0.0), module intro, paragraph on token
  selection: the processors run in the order repetition_penalty,
  no_repeat_ngram_size, single-token bad_words_ids, min_length /
  min_new_tokens, forced_bos_token_id, forced_eos_token_id, suppress_tokens,
  begin_suppress_tokens, the task's processors, renormalize_logits,
  temperature, top_k, top_p.
* Same page, section "Processors": a processor is a per-row state made on the
  host before each step plus a function of the row's scores and that state;
  the task's come at the end of the list.  Here the functions are "bias"
  (s + v) and "set" (v) over a sparse state of (id, value) entries, or one
  function given by the caller (``Params.custom``: the row's scores and its
  dense state row in, new scores out; f32, never below the filter value).
* Same page, section "Lengths": a row's length L counts the prompt and the new
  tokens; max_length = prompt + max_new_tokens; the rules for
  no_repeat_ngram_size, min_length, min_new_tokens, forced_bos, forced_eos and
  begin_suppress_tokens.
* Same page, section "Log-probabilities", last paragraph: scores are f32, a
  removed token gets the smallest finite f32 and no score goes below it.
* Same page, section "Batches": an empty prompt is a padding row that gives
  no token (-1 in the on_token map of generate/5).
* Assisted Generation: a new direction toward low-latency text generation,
  section "Greedy decoding with assisted generation", steps 1-6: select with
  argmax (greedy) or multinomial (sampling) at every candidate position, count
  left-to-right matches, keep the matches plus the first divergent token, and
  adjust the candidate count (+2 if all match, -1 otherwise, 5 at first).

The pages name the processors but do not print their formulas.  The readings
taken here are:

* repetition_penalty: each distinct id of the history in [0, V) takes
  x * rho if its ORIGINAL logit x < 0, else x / rho.
* top_k keeps every token whose score is >= the k-th largest score (ties at
  the k-th value are all kept).
* top_p keeps the shortest prefix of the order (score desc, index asc) whose
  softmax mass is >= p (at least one token).
* the multinomial draw with a supplied uniform u in [0, 1) is the first kept
  token, in that same order, whose cumulative normalised mass exceeds u; if
  rounding leaves none, the last kept token.
* greedy skips temperature/top_k/top_p and takes the lowest index among the
  maximal scores.
* the task's processors leave their function open; here "bias" (s + v) and
  "set" (v) over a sparse per-row state of (id, value) entries, in list
  order, never below the filter value.

Each function is pinned by tests/test_oracle_pins.py to these readings
(closed forms, worked rules of the pages, brute force, exact rationals).
Their equivalence with the transformers processors that the names refer to
is parity unpinned: that library is not available to test against.

Elementwise arithmetic is IEEE fp32 one operation at a time (numpy float32
scalars/arrays, no fused multiply-add).  Softmax masses and cumulative sums
are fp64.  Everything here is a straight loop or a library primitive (sort,
cumsum, argmax) over one row at a time; nothing is blocked or fused.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Sequence

import numpy as np

F32 = np.float32
# Filter value: a removed token scores -FLT_MAX (not -inf), and every score is
# kept at or above it (Transmuter.Generation, section Log-probabilities).
FILTER = F32(-np.finfo(np.float32).max)

# Rows whose decisive mass lies this close to p or to u are reported, not
# compared (the tolerance the spec contract states for sampled ids).
BOUNDARY_EPS = 1e-6


@dataclass
class Params:
    """Generation settings, named as in transformers' generation_config."""

    vocab: int
    logits_dtype: str = "f32"          # "f32" or "bf16"
    mode: str = "greedy"               # "greedy" or "sample"
    repetition_penalty: float = 1.0
    no_repeat_ngram_size: int = 0
    bad_words_ids: Sequence[int] = ()  # single-token bad words
    bad_word_seqs: Sequence[Sequence[int]] = ()   # bad words of one or more tokens
    suppress_tokens: Sequence[int] = ()
    begin_suppress_tokens: Sequence[int] = ()
    eos_token_ids: Sequence[int] = ()
    min_length: int = 0
    min_new_tokens: int = 0
    forced_bos_token_id: int = -1
    forced_eos_token_ids: Sequence[int] = ()
    max_new_tokens: int = 0
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    renormalize_logits: bool = False   # log-softmax after the processors (diagnostic scores, beam step)
    # the task's processors: (kind, size) pairs, kind "bias" (s + v) or "set" (v); each owns
    # `size` columns of the per-row state (ids, values) passed next to the logits
    processors: Sequence[tuple] = ()
    # or one task processor given as a function (scores [V] f32, state row) -> new scores [V];
    # the state passed next to the logits is then a dense [B, S] array
    custom: object = None


@dataclass
class RowInfo:
    """Per-row side results reported next to the selected id."""

    skipped_ids: int = 0             # history ids outside [0, V)
    topp_boundary: bool = False      # top-p cut within BOUNDARY_EPS of p
    u_boundary: bool = False         # u within BOUNDARY_EPS of a CDF value
    n_kept: int = 0                  # tokens kept for the draw
    forced: bool = False
    logprob: float = float("nan")    # log-softmax of the selected-from scores at the token
    bad_state: bool = False          # the processors' state broke its layout and was dropped


# ---------------------------------------------------------------------------
# a0: load + upcast
# ---------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32; widening appends 16 zero bits."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def upcast_row(row, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(row)
    return np.array(row, dtype=np.float32, copy=True)


def _clamp(s: np.ndarray) -> np.ndarray:
    """Keep scores at or above the filter value (Transmuter.Generation, Log-probabilities)."""
    return np.maximum(s, FILTER)


# ---------------------------------------------------------------------------
# Row conditions from the "Lengths" section
# ---------------------------------------------------------------------------
def eos_removed(L: int, P: int, p: Params) -> bool:
    """min_length / min_new_tokens (Transmuter.Generation, Lengths).

    When both limits are set, the min_new_tokens rule is the one that
    applies, so with min_new_tokens > 0 only the new tokens are counted.
    """
    new = L - P
    if p.min_new_tokens > 0:
        return new < p.min_new_tokens
    if p.min_length > 0:
        return L < p.min_length
    return False


def forced_bos_active(L: int, p: Params) -> bool:
    """forced_bos_token_id is forced when the row holds exactly one token (Lengths)."""
    return p.forced_bos_token_id >= 0 and L == 1


def forced_eos_active(L: int, P: int, p: Params) -> bool:
    """forced_eos_token_id is forced when the row is one token short of
    max_length = prompt + max_new_tokens (Lengths)."""
    return len(p.forced_eos_token_ids) > 0 and L == P + p.max_new_tokens - 1


def begin_index(P: int, p: Params) -> int:
    """Row length at which begin_suppress_tokens apply (Lengths): the step
    that picks the first new token, moved one step later when a one-token
    prompt is followed by a forced bos token."""
    if p.forced_bos_token_id >= 0 and P == 1:
        return P + 1
    return P


# ---------------------------------------------------------------------------
# a3: no_repeat_ngram_size, by brute force over every start position
# ---------------------------------------------------------------------------
def ngram_banned_tokens(h: Sequence[int], n: int) -> list[int]:
    """Tokens that would repeat an n-gram of the row (Lengths: every n-gram
    over prompt plus new tokens may appear at most once).

    The next token t is banned when (last n-1 tokens, t) already occurs as an
    n-gram of the row.  Every start j of a complete n-gram h[j .. j+n-1] is
    compared with the current (n-1)-token suffix.  Nothing is banned while the
    row has fewer than n-1 tokens.
    """
    L = len(h)
    if n <= 0 or L + 1 < n:
        return []
    suffix = list(h[L - n + 1:]) if n > 1 else []
    banned = []
    for j in range(0, L - n + 1):
        if list(h[j:j + n - 1]) == suffix:
            banned.append(int(h[j + n - 1]))
    return banned


# ---------------------------------------------------------------------------
# a0-a9: the processors, in order
# ---------------------------------------------------------------------------
def processor_state_valid(ids_row, p: Params) -> bool:
    """A row's processors' state keeps its layout: every id is -1 or in
    [0, V); within a processor's columns the used ids ascend strictly and the
    unused (-1) come after them."""
    col = 0
    for _, size in p.processors:
        block = [int(t) for t in ids_row[col:col + size]]
        col += size
        used = [t for t in block if t != -1]
        if any(t < -1 or t >= p.vocab for t in block):
            return False
        if block[:len(used)] != used or any(b <= a for a, b in zip(used, used[1:])):
            return False
    return True


def apply_processors(s: np.ndarray, state, p: Params, info) -> None:
    """The task's processors (Transmuter.Generation, section "Processors"),
    in list order, on the scores after a9: processor k reads its columns of
    the row's state; an entry (t, v) makes s[t] = s[t] + v ("bias", an f32
    add) or v ("set"), never below the filter value.  A state that breaks
    its layout is dropped (info.bad_state)."""
    ids_row, vals_row = state
    if not processor_state_valid(ids_row, p):
        info.bad_state = True
        return
    col = 0
    for kind, size in p.processors:
        bias = kind in ("bias", 0)
        for j in range(col, col + size):
            t = int(ids_row[j])
            if t < 0:
                continue
            v = F32(vals_row[j])
            with np.errstate(over="ignore"):
                new = F32(s[t] + v) if bias else v
            s[t] = max(new, FILTER)
        col += size


def process_row(x: np.ndarray, h: Sequence[int], P: int, p: Params, state=None):
    """Scores after a0-a9 and the task's processors for one non-empty row
    (state: the row's (ids, values), needed when p has processors).

    Returns (s, banned, info): s are fp32 scores, banned marks tokens a
    ban/force processor of a3-a9 set to the filter value.
    """
    V = p.vocab
    L = len(h)
    s = np.array(x, dtype=np.float32, copy=True)
    banned = np.zeros(V, dtype=bool)
    info = RowInfo()
    in_range = [int(t) for t in h if 0 <= int(t) < V]
    info.skipped_ids = L - len(in_range)

    # a2 repetition_penalty: uses the original x, so duplicates change nothing.
    rho = F32(p.repetition_penalty)
    if rho != F32(1.0):
        with np.errstate(over="ignore"):
            for t in sorted(set(in_range)):
                v = x[t]
                s[t] = v * rho if v < F32(0.0) else v / rho
        s = _clamp(s)

    # a3 no_repeat_ngram_size
    for t in ngram_banned_tokens(h, p.no_repeat_ngram_size):
        if 0 <= t < V:
            banned[t] = True
    # a4 bad_words_ids: a one-token bad word is always banned; a longer one
    # bans its last token when the row ends with the rest of it
    for t in p.bad_words_ids:
        banned[t] = True
    hl = [int(t) for t in h]
    for seq in p.bad_word_seqs:
        seq = [int(t) for t in seq]
        n = len(seq)
        if n == 1 or (L >= n - 1 and hl[L - (n - 1):] == seq[:-1]):
            banned[seq[-1]] = True
    # a5 min_length / min_new_tokens
    if eos_removed(L, P, p):
        for t in p.eos_token_ids:
            banned[t] = True
    s[banned] = FILTER

    # a6 forced_bos: everything removed except bos, which scores 0.
    if forced_bos_active(L, p):
        s[:] = FILTER
        banned[:] = True
        s[p.forced_bos_token_id] = F32(0.0)
        banned[p.forced_bos_token_id] = False
        info.forced = True
    # a7 forced_eos: everything removed except the forced ids, which score 0.
    if forced_eos_active(L, P, p):
        s[:] = FILTER
        banned[:] = True
        for t in p.forced_eos_token_ids:
            s[t] = F32(0.0)
            banned[t] = False
        info.forced = True

    # a8 suppress_tokens (a constant mask)
    for t in p.suppress_tokens:
        s[t] = FILTER
        banned[t] = True
    # a9 begin_suppress_tokens at the begin index
    if L == begin_index(P, p):
        for t in p.begin_suppress_tokens:
            s[t] = FILTER
            banned[t] = True
    # the task's processors, at the end of the list
    if p.processors:
        apply_processors(s, state, p, info)
    if p.custom is not None:
        s = _clamp(np.asarray(p.custom(s.copy(), state), dtype=np.float32))
    return s, banned, info


def apply_temperature(s: np.ndarray, p: Params) -> np.ndarray:
    """a10: scores / temperature in fp32, clamped at the filter value."""
    T = F32(p.temperature)
    if T == F32(1.0):
        return s.copy()
    with np.errstate(over="ignore"):
        return _clamp((s / T).astype(np.float32))


# ---------------------------------------------------------------------------
# a11-a13 on one row of scores
# ---------------------------------------------------------------------------
def order_desc(s: np.ndarray) -> np.ndarray:
    """Indices in the total order (score desc, index asc); +0 and -0 tie."""
    idx = np.arange(s.size)
    return np.lexsort((idx, -s.astype(np.float64)))


def softmax64(s: np.ndarray) -> np.ndarray:
    """Softmax in fp64 of fp32 scores."""
    d = s.astype(np.float64)
    e = np.exp(d - d.max())
    return e / e.sum()


def top_k_threshold(s: np.ndarray, k: int):
    """a11: the k-th largest score (with multiplicity), or None when off."""
    if k <= 0 or k >= s.size:
        return None
    return np.sort(s)[::-1][k - 1]


def sample_distribution(s_t: np.ndarray, p: Params):
    """a11-a12 on temperature-scaled scores.

    Returns (order, kept, probs, info) where ``order`` is the (score desc,
    index asc) order, ``kept`` the number of leading tokens of that order kept
    for the draw, ``probs`` the fp64 softmax of the scores after top_k (used
    for top_p and the draw).
    """
    info = RowInfo()
    s = s_t.copy()
    tau = top_k_threshold(s, p.top_k)
    if tau is not None:
        s[s < tau] = FILTER
    probs = softmax64(s)
    order = order_desc(s)
    cum = np.cumsum(probs[order])
    n_kept = s.size
    if p.top_p < 1.0:
        hits = np.nonzero(cum >= p.top_p)[0]
        n_kept = int(hits[0]) + 1 if hits.size else s.size
        lo = cum[n_kept - 2] if n_kept >= 2 else 0.0
        info.topp_boundary = bool(abs(lo - p.top_p) < BOUNDARY_EPS
                                  or abs(cum[n_kept - 1] - p.top_p) < BOUNDARY_EPS)
    elif tau is not None:
        # top_k alone: the draw runs over the tokens that kept a finite score.
        n_kept = int(np.count_nonzero(s >= tau))
    info.n_kept = n_kept
    return order, n_kept, probs, s, info


def draw(order: np.ndarray, n_kept: int, probs: np.ndarray, u: float):
    """a13 multinomial: inverse CDF over the kept tokens in (score desc, index asc)."""
    w = probs[order[:n_kept]]
    cdf = np.cumsum(w) / w.sum()
    hits = np.nonzero(cdf > u)[0]
    pos = int(hits[0]) if hits.size else n_kept - 1
    u_boundary = bool(np.min(np.abs(cdf - u)) < BOUNDARY_EPS)
    return int(order[pos]), u_boundary


def final_distribution(s_t: np.ndarray, p: Params) -> np.ndarray:
    """fp64 probabilities the draw uses: kept tokens renormalised, others 0."""
    order, n_kept, probs, _, _ = sample_distribution(s_t, p)
    out = np.zeros(s_t.size, dtype=np.float64)
    kept = order[:n_kept]
    out[kept] = probs[kept] / probs[kept].sum()
    return out


def log_softmax_at(scores: np.ndarray, tok: int) -> float:
    """Transmuter.Generation, section "Log-probabilities": the log-softmax of
    the scores a step selects from, at the selected token, in fp64:
    s_tok - m - log(sum_i exp(s_i - m)) with m the largest score.  Removed
    tokens hold the filter value and add exp(F - m) = 0, unless every token
    is removed (then all are equal and the result is -log V)."""
    d = scores.astype(np.float64)
    m = d.max()
    return float(d[tok] - m - np.log(np.sum(np.exp(d - m))))


def selected_from_scores(s_t: np.ndarray, order: np.ndarray, n_kept: int, s_k: np.ndarray) -> np.ndarray:
    """The scores a sampling step selects from: after the processors and
    temperature, top_k (``s_k``, removed tokens at the filter value) and top_p
    (tokens past the kept prefix of the order at the filter value)."""
    out = np.full(s_t.size, FILTER, dtype=F32)
    kept = order[:n_kept]
    out[kept] = s_k[kept]
    return out


def select_row(x: np.ndarray, h: Sequence[int], P: int, p: Params, u: float, state=None):
    """One row of tg_select.  Returns (token id or -1, RowInfo); the info
    carries the token's log-probability (NaN for a padding row).

    renormalize_logits shifts a row's scores by one constant; argmax,
    temperature, top_k, top_p, the draw and the log-probability do not change
    under it (exactly, before rounding), so selection leaves it out."""
    if len(h) == 0:
        return -1, RowInfo()
    s, _, info = process_row(x, h, P, p, state)
    if p.mode == "greedy":
        tok = int(np.argmax(s))
        info.logprob = log_softmax_at(s, tok)
        return tok, info
    s_t = apply_temperature(s, p)
    order, n_kept, probs, s_k, dinfo = sample_distribution(s_t, p)
    tok, ub = draw(order, n_kept, probs, u)
    info.topp_boundary = dinfo.topp_boundary
    info.u_boundary = ub
    info.n_kept = n_kept
    info.logprob = log_softmax_at(selected_from_scores(s_t, order, n_kept, s_k), tok)
    return tok, info


def _row_state(proc_state, r):
    if proc_state is None:
        return None
    if isinstance(proc_state, np.ndarray):   # a dense state (Params.custom)
        return proc_state[r]
    return (proc_state[0][r], proc_state[1][r])


def select(logits, hist_ids, hist_offsets, prompt_lens, p: Params, uniforms=None,
           rows=None, proc_state=None):
    """tg_select over a batch (or the listed ``rows``) -> (ids, infos).
    proc_state: (ids [B, S], values [B, S]) of the task's processors."""
    B = len(prompt_lens)
    rows = range(B) if rows is None else rows
    ids, infos = [], []
    for b in rows:
        h = hist_ids[int(hist_offsets[b]):int(hist_offsets[b + 1])]
        x = upcast_row(logits[b], p.logits_dtype)
        u = float(uniforms[b]) if uniforms is not None else 0.0
        t, info = select_row(x, h, int(prompt_lens[b]), p, u, _row_state(proc_state, b))
        ids.append(t)
        infos.append(info)
    return np.array(ids, dtype=np.int32), infos


def processed_scores(x, h, P, p: Params, state=None):
    """What the diagnostic entry point writes: scores after a0-a9 (greedy) or
    a0-a10 (sampling), and the mask of banned tokens."""
    s, banned, _ = process_row(x, h, P, p, state)
    if p.renormalize_logits:
        s = _clamp(log_softmax_row(s))
    if p.mode == "sample":
        s = apply_temperature(s, p)
    return s, banned


# ---------------------------------------------------------------------------
# Beam search, the device part of one step (Transmuter.Generation, module
# intro, the paragraphs on num_beams; the host's hypotheses are not here)
# ---------------------------------------------------------------------------
def log_softmax_row(x: np.ndarray) -> np.ndarray:
    """The log-softmax of one row of f32 logits: each x_i - logsumexp(x),
    in fp64, rounded once to f32.  The maximum m comes off first,
    (x_i - m) - log(sum exp(x - m)), so that a row of equal scores at the
    filter value (~3.4e38, where m + ln V rounds back to m) still gives -ln V."""
    d = x.astype(np.float64) - x.astype(np.float64).max()
    return (d - np.log(np.sum(np.exp(d)))).astype(np.float32)


def beam_keep(num_beams: int, p: Params) -> int:
    """Candidates a prompt keeps per step: max(2, 1 + eos tokens) * num_beams."""
    return max(2, 1 + len(p.eos_token_ids)) * num_beams


def beam_step(logits, beam_scores, hist_ids, hist_offsets, prompt_lens, num_beams: int, p: Params,
              proc_state=None):
    """One beam-search step on the device side.

    Rows i*num_beams .. i*num_beams+num_beams-1 are prompt i's beams.  Each
    row: the log-softmax of its logits, the processors on it (in the order
    of select), plus the beam's score, in f32, never below the filter value.
    Of a prompt's num_beams * V candidates (beam b, token t; flat index
    b*V + t), the best beam_keep() in the order (score desc, flat index asc).
    Returns (scores [P, K] f32, tokens [P, K] int32, beams [P, K] int32)."""
    R = len(prompt_lens)
    assert R % num_beams == 0
    P = R // num_beams
    V = p.vocab
    K = beam_keep(num_beams, p)
    out_s = np.zeros((P, K), np.float32)
    out_t = np.zeros((P, K), np.int32)
    out_b = np.zeros((P, K), np.int32)
    for i in range(P):
        cand, live = beam_candidates(logits, beam_scores, hist_ids, hist_offsets, prompt_lens, num_beams, p, i,
                                     proc_state)
        flat = order_desc(cand)
        flat = flat[live[flat]][:K]
        n = flat.size
        out_s[i, :n] = cand[flat]
        out_t[i, :n] = flat % V
        out_b[i, :n] = flat // V
        # fewer candidates than kept (empty rows give none)
        out_s[i, n:] = FILTER
        out_t[i, n:] = -1
        out_b[i, n:] = -1
    return out_s, out_t, out_b


def beam_candidates(logits, beam_scores, hist_ids, hist_offsets, prompt_lens, num_beams: int, p: Params, i: int,
                    proc_state=None):
    """Prompt i's num_beams * V candidate scores (flat index b*V + t) and a
    mask of the live ones (rows with an empty history give none)."""
    V = p.vocab
    cand = np.full(num_beams * V, FILTER, np.float32)
    live = np.zeros(num_beams * V, bool)
    for b in range(num_beams):
        r = i * num_beams + b
        h = hist_ids[int(hist_offsets[r]):int(hist_offsets[r + 1])]
        if len(h) == 0:
            continue
        x = upcast_row(logits[r], p.logits_dtype)
        ls = log_softmax_row(x)
        s, _, _ = process_row(ls, h, int(prompt_lens[r]), p, _row_state(proc_state, r))
        if p.renormalize_logits:
            s = _clamp(log_softmax_row(s))
        with np.errstate(over="ignore"):
            cand[b * V:(b + 1) * V] = _clamp((s + F32(beam_scores[r])).astype(np.float32))
        live[b * V:(b + 1) * V] = True
    return cand, live


# ---------------------------------------------------------------------------
# Assisted generation verify (steps 2-5) and the candidate heuristic (step 6)
# ---------------------------------------------------------------------------
def verify(target_logits, cand_ids, K: int, p: Params, uniforms=None, proc_state=None):
    """tg_verify: select at each of the K+1 positions, count left-to-right
    matches, keep the matches plus the first divergent token.

    Position j selects from target_logits[b, j] with the warpers only (no
    history processors run per position); with Params.custom, the task's
    function first, with state row b (K+1) + j of proc_state.
    """
    B = target_logits.shape[0]
    out_match = np.zeros(B, dtype=np.int32)
    out_next = np.full((B, K + 1), -1, dtype=np.int32)
    infos = []
    for b in range(B):
        nxt = []
        row_infos = []
        for j in range(K + 1):
            x = upcast_row(target_logits[b, j], p.logits_dtype)
            if p.custom is not None:
                x = _clamp(np.asarray(p.custom(x.copy(), proc_state[b * (K + 1) + j]), dtype=np.float32))
            if p.mode == "greedy":
                nxt.append(int(np.argmax(x)))
                row_infos.append(RowInfo())
            else:
                s_t = apply_temperature(x, p)
                order, n_kept, probs, _, dinfo = sample_distribution(s_t, p)
                u = float(uniforms[b, j])
                t, ub = draw(order, n_kept, probs, u)
                dinfo.u_boundary = ub
                nxt.append(t)
                row_infos.append(dinfo)
        n = matched_prefix(nxt, cand_ids[b], K)
        out_match[b] = n
        out_next[b, :n + 1] = nxt[:n + 1]
        infos.append((nxt, row_infos))
    return out_match, out_next, infos


def verify_history(target_logits, cand_ids, K: int, hist_ids, hist_offsets, prompt_lens, p: Params,
                   uniforms=None):
    """tg_verify_history: as verify, but position j of row b runs the whole
    processor chain with the history the target model saw there -- the row's
    history followed by its first j candidates (Assisted Generation, "Greedy
    decoding with assisted generation", step 2: the candidates extend the
    sequence each position continues).  A row with an empty history is a
    padding row: no tokens, no matches."""
    B = target_logits.shape[0]
    out_match = np.zeros(B, dtype=np.int32)
    out_next = np.full((B, K + 1), -1, dtype=np.int32)
    infos = []
    for b in range(B):
        h = [int(t) for t in hist_ids[int(hist_offsets[b]):int(hist_offsets[b + 1])]]
        if not h:
            infos.append(([-1] * (K + 1), [RowInfo() for _ in range(K + 1)]))
            continue
        nxt, row_infos = [], []
        for j in range(K + 1):
            x = upcast_row(target_logits[b, j], p.logits_dtype)
            u = float(uniforms[b, j]) if uniforms is not None else 0.0
            t, info = select_row(x, h + [int(c) for c in cand_ids[b][:j]], int(prompt_lens[b]), p, u)
            nxt.append(t)
            row_infos.append(info)
        n = matched_prefix(nxt, cand_ids[b], K)
        out_match[b] = n
        out_next[b, :n + 1] = nxt[:n + 1]
        infos.append((nxt, row_infos))
    return out_match, out_next, infos


def matched_prefix(next_tokens: Sequence[int], candidates: Sequence[int], K: int) -> int:
    """Step 4: count matches from the left and stop at the first mismatch;
    later candidates do not count even when they agree."""
    n = 0
    while n < K and int(next_tokens[n]) == int(candidates[n]):
        n += 1
    return n


def next_num_candidates(K: int, n_match: int, K_max: int) -> int:
    """Step 6: +2 when ALL candidates matched, -1 otherwise; bounded to [1, K_max]."""
    K2 = K + 2 if n_match >= K else K - 1
    return max(1, min(K_max, K2))


INITIAL_NUM_CANDIDATES = 5  # step 1: the first call asks the assistant for 5


# ---------------------------------------------------------------------------
# Prompt chunking (Transmuter.Generation intro): power-of-two step lengths
# ---------------------------------------------------------------------------
def chunk_plan(n: int) -> list[int]:
    """The powers of two a prompt of n tokens runs as, largest first."""
    out = []
    bit = 1
    while bit <= n:
        bit <<= 1
    bit >>= 1
    while bit >= 1:
        if n & bit:
            out.append(bit)
        bit >>= 1
    return out
