"""Pins that tie the CPU oracle to something other than itself.

Each test checks the oracle against a value the pages print (fixtures under
tests/golden/), a closed form, a library routine the oracle does not use for
that step, or brute force on tiny inputs.  A plausible slip in the oracle (a
dropped term, a wrong sign, an off-by-one in a length rule, a transposed
operand) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import tg_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_rules.json")
with open(GOLDEN) as f:
    RULES = json.load(f)

F = O.FILTER


def P(**kw):
    kw.setdefault("vocab", 16)
    return O.Params(**kw)


# --------------------------------------------------------------------------
# values printed on the pages
# --------------------------------------------------------------------------
def test_chunk_plan_worked_example():
    for n, plan in RULES["chunk_plan"]["cases"]:
        assert O.chunk_plan(n) == plan


def test_chunk_plan_properties():
    # powers of two, strictly decreasing, summing to n; empty for 0
    assert O.chunk_plan(0) == []
    for n in range(1, 3000):
        plan = O.chunk_plan(n)
        assert sum(plan) == n
        assert all(c & (c - 1) == 0 for c in plan)
        assert all(a > b for a, b in zip(plan, plan[1:]))


def test_candidate_heuristic_rules():
    assert O.INITIAL_NUM_CANDIDATES == RULES["initial_num_candidates"]["K0"]
    for K, n, K2 in RULES["candidate_heuristic"]["cases"]:
        assert O.next_num_candidates(K, n, 64) == K2
    # bounds
    assert O.next_num_candidates(1, 0, 16) == 1
    assert O.next_num_candidates(16, 16, 16) == 16


def test_verify_prefix_rules():
    for c in RULES["verify_prefix"]["cases"]:
        K = len(c["cand"])
        assert O.matched_prefix(c["next"], c["cand"], K) == c["n"]
        # the same through verify(), with one-hot target logits forcing argmax
        V = 10
        tl = np.zeros((1, K + 1, V), np.float32)
        for j, t in enumerate(c["next"]):
            tl[0, j, t] = 5.0
        m, nxt, _ = O.verify(tl, np.array([c["cand"]]), K, P(vocab=V))
        assert m[0] == c["n"]
        assert list(nxt[0]) == c["kept"][:K + 1]


# --------------------------------------------------------------------------
# the "Lengths" rules, one case on each side of every boundary
# --------------------------------------------------------------------------
EOS = 2


def _row(L, P_, V=16):
    h = [(7 + 3 * i) % V for i in range(L)]
    return h, P_


def _eos_banned(L, Plen, **kw):
    p = P(eos_token_ids=[EOS], **kw)
    x = np.linspace(-1, 1, p.vocab).astype(np.float32)
    h, _ = _row(L, Plen)
    s, banned, _ = O.process_row(x, h, Plen, p)
    return bool(banned[EOS])


def test_min_length_strict():
    assert _eos_banned(L=9, Plen=5, min_length=10)
    assert not _eos_banned(L=10, Plen=5, min_length=10)


def test_min_new_tokens_replaces_min_length():
    # L < min_length but new >= min_new_tokens: NOT removed when both are set
    assert not _eos_banned(L=12, Plen=10, min_length=50, min_new_tokens=1)
    assert _eos_banned(L=10, Plen=10, min_length=5, min_new_tokens=1)
    assert _eos_banned(L=14, Plen=10, min_new_tokens=5)
    assert not _eos_banned(L=15, Plen=10, min_new_tokens=5)


def _scores(L, Plen, **kw):
    p = P(**kw)
    x = np.linspace(-1, 1, p.vocab).astype(np.float32)
    h, _ = _row(L, Plen)
    return O.process_row(x, h, Plen, p)[0]


def test_forced_eos_only_at_max_length_minus_one():
    kw = dict(forced_eos_token_ids=[EOS], max_new_tokens=5)
    for L in (6, 8):
        s = _scores(L, 3, **kw)
        assert np.count_nonzero(s == F) == 0
    s = _scores(7, 3, **kw)          # 3 + 5 - 1
    assert s[EOS] == 0.0 and np.count_nonzero(s == F) == s.size - 1


def test_forced_bos_only_for_one_token():
    kw = dict(forced_bos_token_id=5)
    s = _scores(1, 1, **kw)
    assert s[5] == 0.0 and np.count_nonzero(s == F) == s.size - 1
    # decoder-only prompt of more than one token: no forced token
    s = _scores(3, 3, **kw)
    assert np.count_nonzero(s == F) == 0
    s = _scores(2, 1, **kw)
    assert np.count_nonzero(s == F) == 0


def test_begin_suppress_index_shift():
    kw = dict(begin_suppress_tokens=[4])
    assert _scores(4, 4, **kw)[4] == F          # first new token
    assert _scores(5, 4, **kw)[4] != F
    # a one-token prompt with a forced bos: removed at the SECOND new token
    kw2 = dict(begin_suppress_tokens=[4], forced_bos_token_id=9)
    assert _scores(2, 1, **kw2)[4] == F
    assert _scores(3, 1, **kw2)[4] != F
    # without forced bos a one-token prompt suppresses at L == 1
    assert _scores(1, 1, begin_suppress_tokens=[4])[4] == F


def test_processor_order_suppress_after_forced_eos():
    # suppress_tokens comes after forced_eos: a suppressed eos stays removed,
    # leaving an all-removed row whose argmax is index 0
    p = P(forced_eos_token_ids=[EOS], max_new_tokens=2, suppress_tokens=[EOS])
    x = np.linspace(-1, 1, 16).astype(np.float32)
    s, _, _ = O.process_row(x, [1, 2], 1, p)
    assert np.all(s == F)
    assert O.select_row(x, [1, 2], 1, p, 0.0)[0] == 0


def test_forced_eos_overrides_min_length_removal():
    p = P(eos_token_ids=[EOS], min_length=100, forced_eos_token_ids=[EOS], max_new_tokens=2)
    x = np.linspace(-1, 1, 16).astype(np.float32)
    s, _, _ = O.process_row(x, [1, 2], 1, p)
    assert s[EOS] == 0.0


# --------------------------------------------------------------------------
# repetition penalty: closed form
# --------------------------------------------------------------------------
def test_repetition_penalty_closed_form():
    p = P(vocab=5, repetition_penalty=2.0)
    x = np.array([1.0, -1.0, 0.0, 4.0, -3.0], np.float32)
    s, _, _ = O.process_row(x, [0, 1, 1, 2, 0], 5, p)
    assert list(s) == [0.5, -2.0, 0.0, 4.0, -3.0]


def test_repetition_penalty_fp32_rounding():
    # x / 1.1 rounds once in binary32, not in binary64
    p = P(vocab=2, repetition_penalty=1.1)
    x = np.array([1.0, -1.0], np.float32)
    s, _, _ = O.process_row(x, [0, 1], 2, p)
    assert s[0] == np.float32(np.float32(1.0) / np.float32(1.1))
    assert s[1] == np.float32(np.float32(-1.0) * np.float32(1.1))


def test_out_of_range_history_ids_skipped():
    p = P(vocab=4, repetition_penalty=2.0)
    x = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    s, _, info = O.process_row(x, [-1, 4, 1, 99], 4, p)
    assert list(s) == [1.0, 1.0, 3.0, 4.0]
    assert info.skipped_ids == 3


def test_filter_clamp():
    p = P(vocab=2, repetition_penalty=4.0, mode="sample", temperature=0.5)
    x = np.array([-3e38, 1.0], np.float32)
    s, _, _ = O.process_row(x, [0], 1, p)
    assert s[0] == F
    assert O.apply_temperature(np.array([F, 1.0], np.float32), p)[0] == F


# --------------------------------------------------------------------------
# no_repeat_ngram_size: brute force vs an independent dictionary enumeration
# --------------------------------------------------------------------------
def _ngram_dict_bans(h, n):
    """Map every (n-1)-token prefix of a complete n-gram to its next tokens,
    then look up the row's current (n-1)-token suffix."""
    if len(h) + 1 < n:
        return set()
    table = {}
    for g in zip(*[h[i:] for i in range(n)]):
        table.setdefault(tuple(g[:-1]), set()).add(g[-1])
    key = tuple(h[len(h) - n + 1:]) if n > 1 else ()
    return table.get(key, set())


def test_ngram_hand_cases():
    assert sorted(O.ngram_banned_tokens([1, 2, 3, 1, 2], 3)) == [3]
    assert sorted(set(O.ngram_banned_tokens([5, 6, 5], 2))) == [6]
    assert sorted(set(O.ngram_banned_tokens([4, 4, 7], 1))) == [4, 7]
    assert O.ngram_banned_tokens([1, 2], 4) == []
    # L + 1 == n: only the (n-1)-suffix exists, no complete n-gram yet
    assert O.ngram_banned_tokens([1, 2, 3], 4) == []
    assert sorted(O.ngram_banned_tokens([1, 2, 3, 9, 1, 2, 3], 4)) == [9]


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_ngram_matches_dictionary_enumeration(n):
    rng = np.random.default_rng(7 + n)
    for trial in range(300):
        L = int(rng.integers(0, 40))
        h = [int(t) for t in rng.integers(0, 4, size=L)]
        assert set(O.ngram_banned_tokens(h, n)) == _ngram_dict_bans(h, n), (h, n)


# --------------------------------------------------------------------------
# a0 upcast: against torch's own bfloat16 conversion
# --------------------------------------------------------------------------
def test_bf16_upcast_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert O.bf16_bits_to_f32(np.array([0x3F80, 0xC000], np.uint16)).tolist() == [1.0, -2.0]


# --------------------------------------------------------------------------
# a11 top_k: numpy.partition
# --------------------------------------------------------------------------
def test_top_k_threshold_matches_partition():
    rng = np.random.default_rng(3)
    for trial in range(200):
        V = int(rng.integers(2, 300))
        s = rng.integers(-5, 5, size=V).astype(np.float32)  # many ties
        k = int(rng.integers(1, V))
        tau = O.top_k_threshold(s, k)
        assert tau == np.partition(s, V - k)[V - k]
        kept = s >= tau
        assert kept.sum() >= k
    assert O.top_k_threshold(np.ones(5, np.float32), 0) is None
    assert O.top_k_threshold(np.ones(5, np.float32), 5) is None


# --------------------------------------------------------------------------
# a12 top_p: exact rational arithmetic with the ascending-cumsum removal rule
# --------------------------------------------------------------------------
def _topp_kept_ascending_exact(s, p):
    """Kept set by the "remove while the ascending cumulative mass <= 1 - p"
    rule, evaluated exactly on the fp64 exp weights, ties ordered so that the
    higher index is removed first."""
    V = len(s)
    m = max(float(v) for v in s)
    w = [Fraction(math.exp(float(v) - m)) for v in s]
    Z = sum(w)
    asc = sorted(range(V), key=lambda i: (float(s[i]), -i))
    cum = Fraction(0)
    kept = set(range(V))
    thr = 1 - Fraction(p)
    for pos, i in enumerate(asc):
        cum += w[i] / Z
        if cum <= thr and pos < V - 1:
            kept.discard(i)
    # exact distance of the decisive sums from the threshold (for skipping
    # cases too close to call in fp64)
    return kept


def test_top_p_matches_exact_ascending_rule():
    rng = np.random.default_rng(11)
    checked = 0
    for trial in range(3000):
        V = int(rng.integers(1, 9))
        s = (rng.integers(-6, 6, size=V) * 0.5).astype(np.float32)
        p = float(rng.choice([0.3, 0.5, 0.7, 0.9, 0.95]))
        params = P(vocab=V, mode="sample", top_p=p)
        order, n_kept, probs, _, info = O.sample_distribution(s, params)
        if info.topp_boundary:
            continue
        assert set(order[:n_kept].tolist()) == _topp_kept_ascending_exact(s, p), (s, p)
        checked += 1
    assert checked > 2000


# --------------------------------------------------------------------------
# a13 greedy: D3 lowest index among maxima
# --------------------------------------------------------------------------
def test_greedy_lowest_index_tie_break():
    p = P(vocab=4)
    assert O.select_row(np.array([1, 3, 3, 2], np.float32), [0], 1, p, 0)[0] == 1
    assert O.select_row(np.array([-0.0, 0.0, -1, -2], np.float32), [3], 1, p, 0)[0] == 0
    assert O.select_row(np.array([0.0, -0.0, -1, -2], np.float32), [3], 1, p, 0)[0] == 0


def test_padding_row():
    p = P(vocab=4)
    assert O.select_row(np.ones(4, np.float32), [], 0, p, 0.3)[0] == -1


# --------------------------------------------------------------------------
# a13 sampling: inverse CDF on the sorted CDF, and a chi-square check
# --------------------------------------------------------------------------
def test_draw_is_searchsorted_on_sorted_cdf():
    rng = np.random.default_rng(5)
    for trial in range(500):
        V = int(rng.integers(1, 50))
        s = rng.normal(0, 2, V).astype(np.float32)
        u = float(rng.random())
        params = P(vocab=V, mode="sample")
        tok, info = O.select_row(s, [0], 1, params, u)
        # independent: sort by -s with a stable sort, cumulative fp64 softmax
        idx = np.argsort(-s.astype(np.float64), kind="stable")
        e = np.exp(s.astype(np.float64)[idx] - s.max())
        cdf = np.cumsum(e) / e.sum()
        pos = min(int(np.searchsorted(cdf, u, side="right")), V - 1)
        if not info.u_boundary:
            assert tok == idx[pos]


def test_sampling_frequencies_chi_square():
    s = np.array([0.0, 1.0, -1.0, 2.0, 0.5], np.float32)
    params = P(vocab=5, mode="sample")
    rng = np.random.default_rng(123)
    N = 100_000
    us = rng.random(N)
    counts = np.zeros(5)
    order, n_kept, probs, _, _ = O.sample_distribution(s, params)
    for u in us:
        counts[O.draw(order, n_kept, probs, u)[0]] += 1
    e = np.exp(s.astype(np.float64) - s.max())
    expect = N * e / e.sum()
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 18.47  # 99.9% quantile, 4 degrees of freedom


def test_all_removed_row_is_uniform():
    p = P(vocab=4, mode="sample")
    s = np.full(4, F, np.float32)
    order, n_kept, probs, _, _ = O.sample_distribution(s, p)
    assert np.allclose(probs, 0.25)
    tok, ub = O.draw(order, n_kept, probs, 0.6)
    assert tok == 2 and not ub
    tok, ub = O.draw(order, n_kept, probs, 0.5)
    assert tok == 2 and ub


def test_temperature_then_top_k_then_top_p_order():
    # top_k keeps the two largest; top_p=0.5 then keeps only the first of them
    p = P(vocab=4, mode="sample", temperature=0.5, top_k=2, top_p=0.5)
    s = np.array([1.0, 0.9, 0.0, -1.0], np.float32)
    st = O.apply_temperature(s, p)
    assert list(st) == [2.0, np.float32(0.9) / np.float32(0.5), 0.0, -2.0]
    order, n_kept, probs, _, _ = O.sample_distribution(st, p)
    assert probs[2] == 0 and probs[3] == 0
    assert list(order[:n_kept]) == [0]


# --------------------------------------------------------------------------
# identities
# --------------------------------------------------------------------------
def test_identity_settings_leave_scores_unchanged():
    rng = np.random.default_rng(9)
    x = rng.normal(0, 3, 64).astype(np.float32)
    h = [int(t) for t in rng.integers(0, 64, 20)]
    p = P(vocab=64, mode="sample", repetition_penalty=1.0, temperature=1.0, top_k=0, top_p=1.0)
    s, banned, _ = O.process_row(x, h, 10, p)
    assert np.array_equal(s, x) and not banned.any()
    st = O.apply_temperature(s, p)
    assert np.array_equal(st, x)
    for k in (0, 64, 100):
        p.top_k = k
        _, n_kept, probs, filt, _ = O.sample_distribution(st, p)
        assert n_kept == 64 and np.array_equal(filt, x)


# --------------------------------------------------------------------------
# token log-probabilities (Transmuter.Generation, section "Log-probabilities":
# the log-softmax of the scores the step selects from, at the token)
# --------------------------------------------------------------------------
def test_logprob_two_tokens_closed_form():
    a, b = 2.5, 0.75
    x = np.array([a, b], np.float32)
    g = O.select_row(x, [0], 1, P(vocab=2), 0.0)[1].logprob
    assert g == pytest.approx(-math.log1p(math.exp(float(x[1]) - float(x[0]))), abs=1e-13)
    # sampling: a high uniform draws the second token; temperature divides first
    T = 0.5
    tok, info = O.select_row(x, [0], 1, P(vocab=2, mode="sample", temperature=T), 0.999)
    sa, sb = float(np.float32(x[0] / np.float32(T))), float(np.float32(x[1] / np.float32(T)))
    assert tok == 1
    assert info.logprob == pytest.approx((sb - sa) - math.log1p(math.exp(sb - sa)), abs=1e-12)


def test_logprob_over_the_kept_set():
    """Each kept token, drawn in turn, has log-probability s_i - log(sum over
    the kept set of exp(s_j)); the kept set is rebuilt here by sorting and
    math.fsum, independently of the oracle; the probabilities sum to one."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        V = int(rng.integers(4, 14))
        x = rng.normal(0, 2, V).astype(np.float32)
        T = float(rng.choice([1.0, 0.7]))
        k = int(rng.integers(0, V + 1))
        pp = float(rng.choice([1.0, 0.8, 0.5]))
        params = P(vocab=V, mode="sample", temperature=T, top_k=k, top_p=pp)
        s = (x / np.float32(T)).astype(np.float32) if T != 1.0 else x.copy()
        order = sorted(range(V), key=lambda i: (-float(s[i]), i))
        if 0 < k < V:
            tau = float(s[order[k - 1]])
            order = [i for i in order if float(s[i]) >= tau]
        m = float(s[order[0]])
        w = [math.exp(float(s[i]) - m) for i in order]
        tot = math.fsum(w)
        kept = len(order)
        if pp < 1.0:
            cum = 0.0
            for j in range(len(order)):
                cum = math.fsum(w[: j + 1]) / tot
                if cum >= pp:
                    kept = j + 1
                    break
            if abs(cum - pp) < 1e-9 or (kept >= 2 and abs(math.fsum(w[: kept - 1]) / tot - pp) < 1e-9):
                continue
        ks = math.fsum(w[:kept])
        probs = []
        for j in range(kept):
            lo, hi = math.fsum(w[:j]) / ks, math.fsum(w[: j + 1]) / ks
            if hi - lo < 1e-6:
                continue
            tok, info = O.select_row(x, [0], 1, params, (lo + hi) / 2)
            assert tok == order[j]
            expect = (float(s[tok]) - m) - math.log(ks)
            assert info.logprob == pytest.approx(expect, abs=1e-12)
            probs.append(math.exp(info.logprob))
        if len(probs) == kept:
            assert math.fsum(probs) == pytest.approx(1.0, abs=1e-12)


def test_logprob_equal_scores():
    V = 7
    x = np.full(V, 1.25, np.float32)
    assert O.select_row(x, [0], 1, P(vocab=V), 0.0)[1].logprob == pytest.approx(-math.log(V), abs=1e-14)
    # top_k keeps every token tied at the k-th score
    info = O.select_row(x, [0], 1, P(vocab=V, mode="sample", top_k=3), 0.4)[1]
    assert info.logprob == pytest.approx(-math.log(V), abs=1e-14)
    # top_p over equal scores keeps the shortest prefix with mass >= p: ceil(p V) tokens
    info = O.select_row(x, [0], 1, P(vocab=V, mode="sample", top_p=0.5), 0.4)[1]
    assert info.logprob == pytest.approx(-math.log(4), abs=1e-14)
    # every token removed: the scores are all the filter value, each -log V
    info = O.select_row(x, [0], 1, P(vocab=V, suppress_tokens=list(range(V))), 0.0)[1]
    assert info.logprob == pytest.approx(-math.log(V), abs=1e-14)


def test_logprob_forced_and_padding_rows():
    V = 10
    x = np.linspace(-1, 1, V).astype(np.float32)
    # forced eos with two eos ids at L = P + max_new - 1: both score 0, the rest the filter value
    p = P(vocab=V, eos_token_ids=[3, 7], forced_eos_token_ids=[3, 7], max_new_tokens=4)
    tok, info = O.select_row(x, [1, 2, 5, 6], 1, p, 0.0)
    assert tok == 3 and info.logprob == pytest.approx(-math.log(2), abs=1e-14)
    assert math.isnan(O.select_row(x, [], 0, p, 0.0)[1].logprob)


# --------------------------------------------------------------------------
# beam search, device part of a step (Transmuter.Generation, the paragraphs on
# num_beams): log-softmax, processors, + beam score, keep max(2, 1 + eos) * beams
# --------------------------------------------------------------------------
def test_log_softmax_two_tokens_closed_form():
    a, b = 1.75, -0.5
    ls = O.log_softmax_row(np.array([a, b], np.float32))
    d = b - a
    assert float(ls[0]) == pytest.approx(-math.log1p(math.exp(d)), abs=2e-7)
    assert float(ls[1]) == pytest.approx(d - math.log1p(math.exp(d)), abs=2e-7)


def test_beam_keep_rule():
    assert O.beam_keep(4, P(eos_token_ids=[])) == 8
    assert O.beam_keep(4, P(eos_token_ids=[2])) == 8
    assert O.beam_keep(3, P(eos_token_ids=[2, 5, 9])) == 12


def test_beam_step_brute_force():
    """Independent: log-softmax with math.fsum / math.log, the candidates of a
    prompt listed as Python tuples and sorted, flat index split by divmod.
    The processors are the oracle's own (pinned above)."""
    rng = np.random.default_rng(21)
    for trial in range(30):
        V = int(rng.integers(3, 9))
        nb = int(rng.integers(1, 4))
        Pn = int(rng.integers(1, 3))
        R = Pn * nb
        eos = [int(rng.integers(0, V))] if rng.random() < 0.7 else []
        params = P(vocab=V, repetition_penalty=float(rng.choice([1.0, 1.3])), eos_token_ids=eos,
                   min_length=int(rng.integers(0, 5)), bad_words_ids=[int(rng.integers(0, V))])
        logits = rng.normal(0, 2, (R, V)).astype(np.float32)
        hists = [rng.integers(0, V, int(rng.integers(1, 5))).astype(np.int32) for _ in range(R)]
        off = np.concatenate([[0], np.cumsum([len(h) for h in hists])]).astype(np.int64)
        ids = np.concatenate(hists).astype(np.int32)
        plens = np.array([1] * R, np.int32)
        bs = np.where(rng.random(R) < 0.3, -1e9, rng.normal(-3, 1, R)).astype(np.float32)
        got_s, got_t, got_b = O.beam_step(logits, bs, ids, off, plens, nb, params)
        K = max(2, 1 + len(eos)) * nb
        for i in range(Pn):
            cands = []
            for b in range(nb):
                r = i * nb + b
                x = [float(v) for v in logits[r]]
                m = max(x)
                lse = m + math.log(math.fsum(math.exp(v - m) for v in x))
                ls = np.array([v - lse for v in x], np.float32)
                s, _, _ = O.process_row(ls, list(hists[r]), 1, params)
                for t in range(V):
                    v = max(float(np.float32(s[t] + bs[r])), float(F))
                    cands.append((-v, b * V + t))
            cands.sort()
            for j in range(K):
                beam, tok = divmod(cands[j][1], V)
                assert (int(got_b[i, j]), int(got_t[i, j])) == (beam, tok)
                assert float(got_s[i, j]) == -cands[j][0]


def test_beam_first_step_counts_only_the_first_beam():
    V, nb = 12, 3
    x = np.random.default_rng(3).normal(0, 1, V).astype(np.float32)
    logits = np.stack([x] * nb)
    bs = np.array([0.0, -1e9, -1e9], np.float32)
    ids = np.array([1, 1, 1], np.int32)
    off = np.arange(nb + 1, dtype=np.int64)
    s, t, b = O.beam_step(logits, bs, ids, off, np.ones(nb, np.int32), nb, P(vocab=V, eos_token_ids=[0]))
    assert (b == 0).all()
    assert list(t[0]) == list(np.argsort(-x.astype(np.float64), kind="stable")[:6])


def test_beam_repetition_penalty_acts_on_log_probabilities():
    V = 4
    x = np.array([2.0, 1.0, 0.5, 3.0], np.float32)
    ls = O.log_softmax_row(x)
    s, t, b = O.beam_step(x[None], np.array([-1.0], np.float32), np.array([3], np.int32),
                          np.array([0, 1], np.int64), np.array([1], np.int32), 1,
                          P(vocab=V, repetition_penalty=2.0))
    # log-probabilities are negative: the penalty multiplies the history token's
    pen = float(np.float32(ls[3] * np.float32(2.0)))
    assert pen < float(ls[3]) < 0.0
    assert list(t[0]) == [3, 0]
    assert float(s[0, 0]) == float(np.float32(np.float32(pen) + np.float32(-1.0)))
    assert float(s[0, 1]) == float(np.float32(ls[0] + np.float32(-1.0)))


def test_beam_empty_rows_give_no_candidates():
    V, nb = 5, 2
    x = np.array([[0.5, 1.5, -1.0, 0.0, 2.0]] * 4, np.float32)
    # prompt 0: beam 0 empty; prompt 1: both empty
    off = np.array([0, 0, 2, 2, 2], np.int64)
    ids = np.array([1, 3], np.int32)
    s, t, b = O.beam_step(x, np.zeros(4, np.float32), ids, off, np.array([0, 1, 0, 0], np.int32), nb,
                          P(vocab=V, eos_token_ids=[4]))
    K = 4
    order = sorted(range(V), key=lambda j: (-float(x[1, j]), j))
    assert list(b[0]) == [1] * K and list(t[0]) == order[:K]
    assert list(t[1]) == [-1] * K and list(b[1]) == [-1] * K and all(v == float(F) for v in s[1])


# --------------------------------------------------------------------------
# a4 with bad words of several tokens (Transmuter.Generation: the bad_words_ids
# of generation_config.json, one processor in the list of the intro)
# --------------------------------------------------------------------------
def test_multi_token_bad_words_hand_cases():
    V = 12
    x = np.linspace(1, 2, V).astype(np.float32)
    p = P(vocab=V, bad_word_seqs=[[3, 4, 5], [7], [9, 10], [2, 6, 11]])
    # the row ends with 3, 4: bans 5; [7] always; ends with 9? no; [2, 6]? no
    s, banned, _ = O.process_row(x, [1, 9, 3, 4], 1, p)
    assert set(np.nonzero(banned)[0].tolist()) == {5, 7}
    # ends with 9: bans 10
    s, banned, _ = O.process_row(x, [3, 4, 9], 1, p)
    assert set(np.nonzero(banned)[0].tolist()) == {7, 10}
    # prefix longer than the row: nothing but the one-token word
    s, banned, _ = O.process_row(x, [6], 1, p)
    assert set(np.nonzero(banned)[0].tolist()) == {7}
    # ends with 2, 6: bans 11; the banned score is the filter value
    s, banned, _ = O.process_row(x, [0, 2, 6], 1, p)
    assert set(np.nonzero(banned)[0].tolist()) == {7, 11} and s[11] == F


def test_multi_token_bad_words_against_brute_force():
    """Independent: the row and each word written as text, one token a
    bracketed field, compared with str.endswith; random short rows over a
    tiny vocabulary."""
    rng = np.random.default_rng(41)
    for trial in range(200):
        V = 6
        words = [list(rng.integers(0, V, int(rng.integers(1, 4)))) for _ in range(int(rng.integers(1, 4)))]
        h = list(rng.integers(0, V, int(rng.integers(1, 7))))
        expect = set()
        row = "".join("<%d>" % t for t in h)
        for wd in words:
            # the row's text ends with the word's text without its last token
            if row.endswith("".join("<%d>" % t for t in wd[:-1])):
                expect.add(int(wd[-1]))
        _, banned, _ = O.process_row(np.zeros(V, np.float32), h, 1, P(vocab=V, bad_word_seqs=words))
        assert set(np.nonzero(banned)[0].tolist()) == expect


# --------------------------------------------------------------------------
# verify with the processors at every position (Assisted Generation, step 2:
# each position continues the sequence extended by the earlier candidates)
# --------------------------------------------------------------------------
def test_verify_history_without_processors_is_verify():
    rng = np.random.default_rng(51)
    B, K, V = 3, 4, 20
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    cand = rng.integers(0, V, (B, K)).astype(np.int32)
    ids = np.array([1, 2, 3, 4, 5, 6], np.int32)
    off = np.array([0, 2, 4, 6], np.int64)
    pl = np.ones(B, np.int32)
    a = O.verify(t, cand, K, P(vocab=V))
    b = O.verify_history(t, cand, K, ids, off, pl, P(vocab=V))
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all()


def test_verify_history_candidates_join_the_history():
    V, K = 6, 2
    # every position prefers token 3 by a little; token 3 is the first candidate
    t = np.zeros((1, K + 1, V), np.float32)
    t[0, :, 3] = 1.0
    t[0, :, 4] = 0.5
    cand = np.array([[3, 3]], np.int32)
    p = P(vocab=V, repetition_penalty=4.0)
    m, nxt, _ = O.verify_history(t, cand, K, np.array([0], np.int32), np.array([0, 1], np.int64),
                                 np.array([1], np.int32), p)
    # position 0: history [0], 3 wins (match); position 1: history [0, 3] penalises 3 to 0.25 < 0.5
    assert m[0] == 1 and list(nxt[0]) == [3, 4, -1]
    # a 2-gram ban that only the first candidate makes
    p2 = P(vocab=V, no_repeat_ngram_size=2)
    m2, nxt2, _ = O.verify_history(t, cand, K, np.array([3], np.int32), np.array([0, 1], np.int64),
                                   np.array([1], np.int32), p2)
    # position 0: history [3], no earlier (3, x) pair: 3 wins; position 1: [3, 3] ends with 3 and
    # (3, 3) occurred: 3 is banned, 4 wins
    assert m2[0] == 1 and list(nxt2[0]) == [3, 4, -1]
    # an empty history is a padding row
    m3, nxt3, _ = O.verify_history(t, cand, K, np.array([], np.int32), np.array([0, 0], np.int64),
                                   np.array([0], np.int32), p)
    assert m3[0] == 0 and list(nxt3[0]) == [-1, -1, -1]


# --------------------------------------------------------------------------
# renormalize_logits (Transmuter.Generation intro: after the task's
# processors, before temperature): a log-softmax of the processed scores
# --------------------------------------------------------------------------
def test_renormalize_logits_is_a_normalised_shift():
    rng = np.random.default_rng(61)
    V = 40
    x = rng.normal(0, 3, V).astype(np.float32)
    p = P(vocab=V, repetition_penalty=1.3, suppress_tokens=[3, 4], renormalize_logits=True)
    s, banned = O.processed_scores(x, [1, 2, 5], 1, p)
    s0, _ = O.processed_scores(x, [1, 2, 5], 1, P(vocab=V, repetition_penalty=1.3, suppress_tokens=[3, 4]))
    keep = ~banned
    # probabilities sum to one (math.fsum), removed tokens stay removed
    assert math.fsum(math.exp(float(v)) for v in s[keep]) == pytest.approx(1.0, abs=1e-6)
    assert (s[banned] == F).all()
    # the same shift for every kept token: log-sum-exp of the unnormalised scores
    lse = math.log(math.fsum(math.exp(float(v)) for v in s0[keep]))
    assert np.allclose(s[keep].astype(np.float64), s0[keep].astype(np.float64) - lse, atol=2e-6)
    # selection is unchanged by it
    for mode in ("greedy", "sample"):
        for u in (0.1, 0.5, 0.9):
            a = O.select_row(x, [1, 2, 5], 1, P(vocab=V, mode=mode, renormalize_logits=True, top_p=0.8), u)
            b = O.select_row(x, [1, 2, 5], 1, P(vocab=V, mode=mode, top_p=0.8), u)
            assert a[0] == b[0]


def test_renormalize_logits_degenerate_rows():
    """Equal scores give the uniform distribution, log 1/V, at any level:
    the filter value included (every token removed); one kept token gets
    log 1 = 0 and the rest stay removed."""
    V = 3000
    for level in (0.0, -7.5, 1e30, F):
        assert (O.log_softmax_row(np.full(V, level, np.float32)) == np.float32(-math.log(V))).all(), level
    x = np.random.default_rng(62).normal(0, 2, V).astype(np.float32)
    s, banned = O.processed_scores(x, [1, 2], 1, P(vocab=V, suppress_tokens=list(range(V)), renormalize_logits=True))
    assert banned.all() and (s == np.float32(-math.log(V))).all()
    # length 1 = max_length - 1 (prompt 1, one new token): eos 9 forced
    s, banned = O.processed_scores(x, [1], 1, P(vocab=V, max_new_tokens=1, forced_eos_token_ids=[9],
                                                    renormalize_logits=True))
    assert s[9] == 0.0 and (s[np.arange(V) != 9] == F).all()


# --------------------------------------------------------------------------
# The task's processors (Transmuter.Generation, section "Processors"): at the
# end of the list, after begin_suppress_tokens, before renormalize_logits and
# temperature; here "bias" (s + v) and "set" (v) over a sparse per-row state
# --------------------------------------------------------------------------
def _state(*blocks):
    """One row's state from per-processor lists of (id, value), padded to the block sizes given."""
    ids, vals = [], []
    for entries, size in blocks:
        for t, v in entries:
            ids.append(t)
            vals.append(v)
        ids += [-1] * (size - len(entries))
        vals += [0.0] * (size - len(entries))
    return np.array(ids, np.int32), np.array(vals, np.float32)


def test_processor_bias_after_the_penalty_and_only_on_listed_ids():
    V = 6
    x = np.array([2.0, -1.0, 0.5, 0.25, 3.0, -2.0], np.float32)
    p = P(vocab=V, repetition_penalty=2.0, processors=(("bias", 3),))
    st = _state(([(0, 0.25), (2, 0.5), (5, -1.0)], 3))
    s, banned, info = O.process_row(x, [0, 1], 1, p, st)
    # history ids 0, 1 penalised first (2 / 2 = 1, -1 * 2 = -2), then the bias;
    # token 2 is listed but not in the history: no penalty
    assert s.tolist() == [1.25, -2.0, 1.0, 0.25, 3.0, -3.0]
    assert not banned.any() and not info.bad_state


def test_processors_apply_in_list_order():
    V = 4
    x = np.zeros(V, np.float32)
    a = _state(([(1, 1.0)], 1), ([(1, 5.0)], 1))
    s, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("bias", 1), ("set", 1))), a)
    assert s[1] == 5.0
    s, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("set", 1), ("bias", 1))), a)
    assert s[1] == 6.0


def test_processor_set_to_filter_equals_suppress_and_set_after_suppress_restores():
    rng = np.random.default_rng(63)
    V = 50
    x = rng.normal(0, 2, V).astype(np.float32)
    h = [3, 4, 4, 9]
    removed = [5, 11, 30]
    st = _state(([(t, float(F)) for t in removed], 4))
    s1, _, _ = O.process_row(x, h, 2, P(vocab=V, repetition_penalty=1.3, processors=(("set", 4),)), st)
    s2, _, _ = O.process_row(x, h, 2, P(vocab=V, repetition_penalty=1.3, suppress_tokens=removed))
    assert np.array_equal(s1, s2)
    # the task's processors run after suppress_tokens: a set brings a token back
    s3, banned, _ = O.process_row(x, h, 2, P(vocab=V, suppress_tokens=[7], processors=(("set", 1),)),
                                  _state(([(7, 1.5)], 1)))
    assert s3[7] == np.float32(1.5) and banned[7]


def test_forced_row_bias_gives_the_closed_form_distribution():
    """Forced eos ids 2 and 5 both score 0; a bias of ln 3 on 5 makes the draw
    pick 5 with probability 3/4 (it comes first, higher score) and 2 with 1/4."""
    V = 20
    x = np.random.default_rng(64).normal(0, 1, V).astype(np.float32)
    st = _state(([(5, float(np.float32(math.log(3.0))))], 2))
    kw = dict(vocab=V, max_new_tokens=2, forced_eos_token_ids=[2, 5], processors=(("bias", 2),))
    h = [1, 9]          # prompt 1 + one new token: L = P + max_new - 1
    tok, info = O.select_row(x, h, 1, P(mode="greedy", **kw), 0.0, st)
    assert tok == 5 and info.logprob == pytest.approx(math.log(0.75), abs=1e-6)
    for u, want in ((0.0, 5), (0.74, 5), (0.76, 2), (0.999, 2)):
        tok, info = O.select_row(x, h, 1, P(mode="sample", **kw), u, st)
        assert tok == want, (u, tok)
        assert info.logprob == pytest.approx(math.log(0.75 if want == 5 else 0.25), abs=1e-6)


def test_temperature_after_the_processors():
    V = 8
    x = np.zeros(V, np.float32)
    s, _ = O.processed_scores(x, [1], 1, P(vocab=V, mode="sample", temperature=0.5, processors=(("set", 1),)),
                              _state(([(3, 3.0)], 1)))
    assert s[3] == 6.0 and s[0] == 0.0


def test_beam_candidates_with_a_bias_and_renormalize():
    """Equal logits: every log-probability is -ln 4; a bias of ln 3 on token 1
    and renormalize give log 3/6 there and log 1/6 elsewhere, plus the beam score."""
    V = 4
    logits = np.zeros((1, V), np.float32)
    ids, off = np.array([0], np.int32), np.array([0, 1], np.int64)
    st = _state(([(1, float(np.float32(math.log(3.0))))], 1))
    p = P(vocab=V, renormalize_logits=True, processors=(("bias", 1),))
    cand, live = O.beam_candidates(logits, np.array([-2.0], np.float32), ids, off, np.array([1], np.int32), 1, p, 0,
                                   (st[0][None, :], st[1][None, :]))
    want = np.array([math.log(1 / 6), math.log(3 / 6), math.log(1 / 6), math.log(1 / 6)]) - 2.0
    assert live.all() and np.allclose(cand, want, atol=1e-6)


def test_invalid_processor_state_is_dropped():
    V = 10
    x = np.arange(V, dtype=np.float32)
    p = P(vocab=V, processors=(("bias", 3),))
    for ids in ([4, 2, -1], [1, -1, 3], [2, 2, -1], [0, 10, -1], [-2, -1, -1]):
        st = (np.array(ids, np.int32), np.ones(3, np.float32))
        assert not O.processor_state_valid(st[0], p)
        s, _, info = O.process_row(x, [1], 1, p, st)
        assert info.bad_state and np.array_equal(s, x)
    assert O.processor_state_valid(np.array([0, 9, -1], np.int32), p)


def _full_bias(V, c):
    """A state that lists every token once in one bias processor, each with value c."""
    return np.arange(V, dtype=np.int32), np.full(V, c, np.float32)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_uniform_bias_changes_no_selection(mode):
    """Softmax, argmax, top_k, top_p and the draw are invariant under a shift of
    every score by one constant: a bias of c on every token (dyadic values, so
    the f32 adds are exact) must leave ids and log-probabilities unchanged.  A
    bias placed after temperature, or applied to a subset, breaks this."""
    rng = np.random.default_rng(31)
    V = 24
    for trial in range(40):
        x = (rng.integers(-24, 24, V) * 0.25).astype(np.float32)
        h = [int(t) for t in rng.integers(0, V, 6)]
        kw = dict(vocab=V, mode=mode, temperature=0.5, top_k=int(rng.integers(0, 6)),
                  top_p=float(rng.choice([1.0, 0.7])), repetition_penalty=2.0)
        u = float(rng.random())
        t0, i0 = O.select_row(x, h, 2, P(**kw), u)
        t1, i1 = O.select_row(x, h, 2, P(processors=(("bias", V),), **kw), u, _full_bias(V, 3.0))
        assert t1 == t0, trial
        assert abs(i1.logprob - i0.logprob) < 1e-9, trial


def test_bias_zero_and_set_to_current_score_are_identities():
    V = 10
    x = np.array([1.5, -2.0, 0.25, 3.0, -0.5, 0.0, 2.5, -1.25, 0.75, 1.0], np.float32)
    h = [3, 3, 6]
    base, banned0, _ = O.process_row(x, h, 1, P(vocab=V, repetition_penalty=1.5, suppress_tokens=[1]))
    s1, banned1, _ = O.process_row(x, h, 1, P(vocab=V, repetition_penalty=1.5, suppress_tokens=[1],
                                             processors=(("bias", V),)), _full_bias(V, 0.0))
    ids = np.arange(V, dtype=np.int32)
    s2, _, _ = O.process_row(x, h, 1, P(vocab=V, repetition_penalty=1.5, suppress_tokens=[1],
                                       processors=(("set", V),)), (ids, base.copy()))
    assert np.array_equal(s1.view(np.uint32), base.view(np.uint32))
    assert np.array_equal(s2.view(np.uint32), base.view(np.uint32))
    assert np.array_equal(banned1, banned0)


def test_two_biases_compose_and_a_huge_negative_bias_removes_a_token():
    V = 8
    x = np.array([0.5, 2.0, -1.0, 1.75, 0.0, -0.25, 1.0, 3.0], np.float32)
    # two processors biasing the same token add up (dyadic values: exact)
    two = (np.array([7, 7], np.int32), np.array([-1.5, -0.75], np.float32))
    s2, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("bias", 1), ("bias", 1))), two)
    one = (np.array([7], np.int32), np.array([-2.25], np.float32))
    s1, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("bias", 1),)), one)
    assert np.array_equal(s1, s2) and s1[7] == np.float32(0.75)
    # a bias of -FLT_MAX takes a finite score to the filter value (the f32 add rounds there)
    to_f = (np.array([7], np.int32), np.array([F], np.float32))
    s, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("bias", 1),)), to_f)
    assert s[7] == F
    # a bias of -3e38 leaves the token finite but without mass: never selected, as if suppressed
    far = (np.array([7], np.int32), np.array([-3e38], np.float32))
    s, _, _ = O.process_row(x, [0], 1, P(vocab=V, processors=(("bias", 1),)), far)
    assert s[7] == np.float32(-3e38) and s[7] > F
    for u in np.linspace(0.0, 0.999, 41):
        t, _ = O.select_row(x, [0], 1, P(vocab=V, mode="sample", processors=(("bias", 1),)), float(u), far)
        t_sup, _ = O.select_row(x, [0], 1, P(vocab=V, mode="sample", suppress_tokens=[7]), float(u))
        assert t == t_sup and t != 7


def test_final_distribution_closed_forms():
    """The distribution the draw uses: the kept set renormalised, 0 elsewhere.
    Weights 4:2:1:1 under top_p 0.7 keep the first two (0.75 >= 0.7): 2/3, 1/3;
    top_k 2 over scores (1, 1, 1, 0) keeps all three tied tokens: 1/3 each."""
    V = 4
    s = np.array([np.log(4.0), np.log(2.0), 0.0, 0.0], np.float32)
    d = O.final_distribution(s, P(vocab=V, mode="sample", top_p=0.7))
    assert np.allclose(d, [2 / 3, 1 / 3, 0.0, 0.0], rtol=0, atol=1e-7)
    d = O.final_distribution(np.array([1.0, 1.0, 1.0, 0.0], np.float32), P(vocab=V, mode="sample", top_k=2))
    assert np.allclose(d, [1 / 3, 1 / 3, 1 / 3, 0.0], rtol=0, atol=1e-12)
    # no warper: the plain softmax, summing to one
    x = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    d = O.final_distribution(x, P(vocab=V, mode="sample"))
    e = np.exp(x.astype(np.float64))
    assert np.allclose(d, e / e.sum(), rtol=1e-12) and abs(d.sum() - 1.0) < 1e-12


def test_log_softmax_at_closed_forms():
    # weights 1 : 3 -> log(3/4) at the larger; filter-value tokens add nothing
    s = np.array([0.0, np.log(3.0), F, F], np.float32)
    assert abs(O.log_softmax_at(s, 1) - math.log(0.75)) < 1e-7
    assert abs(O.log_softmax_at(s, 0) - math.log(0.25)) < 1e-7
    # every token at the filter value: uniform over V
    assert abs(O.log_softmax_at(np.full(5, F, np.float32), 3) + math.log(5.0)) < 1e-12


# --------------------------------------------------------------------------
# A task processor given as a function (Params.custom) of the row's scores and
# its dense state row, at the same place in the list as the sparse kinds
# --------------------------------------------------------------------------
def test_custom_processor_identity_changes_nothing():
    rng = np.random.default_rng(71)
    B, V = 6, 300
    logits = rng.normal(0, 2, (B, V)).astype(np.float32)
    lens = rng.integers(1, 20, B)
    ids = rng.integers(0, V, int(lens.sum())).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    plen = np.maximum(1, lens // 2).astype(np.int32)
    u = rng.random(B).astype(np.float32)
    kw = dict(vocab=V, mode="sample", repetition_penalty=1.3, top_p=0.8)
    a = O.select(logits, ids, off, plen, P(**kw), u)[0]
    b = O.select(logits, ids, off, plen, P(**kw, custom=lambda s, row: s), u,
                 proc_state=np.zeros((B, 4), np.float32))[0]
    assert np.array_equal(a, b)


def test_custom_dense_bias_equals_the_sparse_bias_kind():
    # the same bias written both ways: a function adding row[i] to every token,
    # and the "bias" kind listing every token with that value
    rng = np.random.default_rng(72)
    V = 40
    x = rng.normal(0, 2, V).astype(np.float32)
    h = [3, 3, 8, 11]
    bias = rng.normal(0, 1, V).astype(np.float32)
    kw = dict(vocab=V, repetition_penalty=1.2, suppress_tokens=[5], eos_token_ids=[2], min_length=10)
    s1, _, _ = O.process_row(x, h, 2, P(**kw, custom=lambda s, row: s + row), bias)
    s2, _, _ = O.process_row(x, h, 2, P(**kw, processors=(("bias", V),)),
                             (np.arange(V, dtype=np.int32), bias))
    assert np.array_equal(s1, s2)


def test_custom_processor_runs_after_suppress_and_before_temperature():
    V = 8
    x = np.zeros(V, np.float32)
    # it brings a suppressed token back (it runs after suppress_tokens) ...
    keep7 = lambda s, row: np.where(np.arange(V) == 7, np.float32(row[0]), s)
    s, banned = O.processed_scores(x, [1], 1, P(vocab=V, suppress_tokens=[7], custom=keep7),
                                   np.array([1.5], np.float32))
    assert s[7] == np.float32(1.5) and banned[7]
    # ... and the temperature divides what it gives
    s, _ = O.processed_scores(x, [1], 1, P(vocab=V, mode="sample", temperature=0.5, custom=keep7),
                              np.array([3.0], np.float32))
    assert s[7] == 6.0 and s[0] == 0.0
