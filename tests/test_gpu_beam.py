"""tg_beam_step on the GPU against the CPU oracle.

Per prompt, the kernel's kept candidates must be the oracle's: each (beam,
token) the oracle scores within TOL of the kernel's score, all distinct, in
non-increasing order, none scored (by the oracle) below the oracle's k-th
kept score by more than TOL.  Away from near-ties that is the oracle's list
exactly, which is also checked whenever the oracle's k-th and (k+1)-th
scores are further apart than TOL.  TOL: the kernel forms x - lse in f32 with
the log-sum-exp as a two-float pair (the oracle rounds x - lse once from
fp64), so a score may differ by a few ulp: 4e-6 * max(1, |score|).
"""
import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

from .gpu_util import to_device

pytestmark = pytest.mark.gpu


def tol(s):
    return 4e-6 * max(1.0, abs(float(s)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def gpu_beam(w, nb, bs):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params)
    dev = to_device(w)
    keep = tg.tg_beam_keep(cfg, nb)
    P = w.B // nb
    s = torch.full((P, keep), 7.0, dtype=torch.float32, device="cuda")
    t = torch.full((P, keep), -7, dtype=torch.int32, device="cuda")
    b = torch.full((P, keep), -7, dtype=torch.int32, device="cuda")
    tg.tg_beam_step(dev["logits"], torch.from_numpy(np.asarray(bs, np.float32)).cuda(), dev["hist_ids"],
                    dev["hist_offsets"], dev["prompt_lens"], cfg, nb, s, t, b)
    torch.cuda.synchronize()
    return s.cpu().numpy(), t.cpu().numpy(), b.cpu().numpy(), keep


def compare_beam(w, nb, bs):
    p = O.Params(**w.params)
    gs, gt, gb, keep = gpu_beam(w, nb, bs)
    assert keep == O.beam_keep(nb, p)
    os_, ot, ob = O.beam_step(w.logits, bs, w.hist_ids, w.hist_offsets, w.prompt_lens, nb, p)
    V = w.V
    for i in range(w.B // nb):
        cand, live = O.beam_candidates(w.logits, bs, w.hist_ids, w.hist_offsets, w.prompt_lens, nb, p, i)
        n_live = int(live.sum())
        n = min(keep, n_live)
        # unfilled slots
        assert all(int(x) == -1 for x in gt[i, n:]) and all(int(x) == -1 for x in gb[i, n:]), i
        flats = []
        for j in range(n):
            f = int(gb[i, j]) * V + int(gt[i, j])
            assert 0 <= int(gb[i, j]) < nb and 0 <= int(gt[i, j]) < V and live[f], (i, j)
            assert abs(float(gs[i, j]) - float(cand[f])) <= tol(cand[f]), (i, j, float(gs[i, j]), float(cand[f]))
            flats.append(f)
            if j:
                assert float(gs[i, j]) <= float(gs[i, j - 1]) + tol(gs[i, j]), (i, j)
        assert len(set(flats)) == n
        kth = float(os_[i, n - 1]) if n else 0.0
        for f in flats:
            assert float(cand[f]) >= kth - tol(kth), (i, f)
        # away from near-ties the lists are equal
        order = O.order_desc(np.where(live, cand, -np.inf).astype(np.float64))
        if n_live > n:
            gap = float(cand[order[n - 1]]) - float(cand[order[n]])
        else:
            gap = np.inf
        scores = [float(cand[order[j]]) for j in range(n)]
        distinct = all(scores[j] - scores[j + 1] > 2 * tol(scores[j]) for j in range(n - 1))
        if gap > 2 * tol(kth) and distinct:
            assert flats == [int(f) for f in order[:n]], i
    return gs, gt, gb


@pytest.mark.parametrize("nb", [1, 2, 4, 8])
def test_random_prompts(nb):
    for seed in range(2):
        w = W.random_case(900 + 10 * nb + seed, B=3 * nb, V=1000, dtype="f32", mode="greedy", L_max=40,
                          repetition_penalty=1.3, no_repeat_ngram_size=2, eos_token_ids=[3], min_length=20)
        bs = np.random.default_rng(seed).normal(-4, 2, w.B).astype(np.float32)
        compare_beam(w, nb, bs)


def test_first_step_only_beam_zero():
    V = 4099
    rng = np.random.default_rng(31)
    ids, off = W._pack([rng.integers(0, V, 3).astype(np.int32) for _ in range(8)])
    logits = rng.normal(0, 2, (8, V)).astype(np.float32)
    w = W.Workload("first", dict(vocab=V, logits_dtype="f32", eos_token_ids=[7, 9], repetition_penalty=1.1),
                   logits, ids, off, np.ones(8, np.int32), rng.random(8, dtype=np.float32))
    bs = np.tile(np.array([0.0, -1e9, -1e9, -1e9], np.float32), 2)
    gs, gt, gb = compare_beam(w, 4, bs)
    assert (gb == 0).all()


def test_bf16_benchmark_rows_small():
    w = W.beam_workload(prompts=6, beams=4)
    compare_beam(w, 4, w.extra["beam_scores"])


def test_bf16_benchmark_rows_full_sampled():
    w = W.beam_workload()
    gs, gt, gb, keep = gpu_beam(w, 4, w.extra["beam_scores"])
    # the same result on a second run (no order-dependent arithmetic or races)
    gs2, gt2, gb2, _ = gpu_beam(w, 4, w.extra["beam_scores"])
    assert (gs == gs2).all() and (gt == gt2).all() and (gb == gb2).all()
    # the oracle on every eighth prompt
    p = O.Params(**w.params)
    sub = [i for i in range(w.B // 4) if i % 8 == 0]
    rows = [4 * i + j for i in sub for j in range(4)]
    ids = [w.history(r) for r in rows]
    off = np.concatenate([[0], np.cumsum([len(h) for h in ids])]).astype(np.int64)
    ws = W.Workload("sub", w.params, w.logits[rows], np.concatenate(ids).astype(np.int32), off,
                    w.prompt_lens[rows], w.uniforms[rows])
    bs = w.extra["beam_scores"][rows]
    s2, t2, b2 = compare_beam(ws, 4, bs)
    for k, i in enumerate(sub):
        assert (gt[i] == t2[k]).all() and (gb[i] == b2[k]).all() and (gs[i] == s2[k]).all()


def test_forced_and_empty_rows():
    V = 3000
    rng = np.random.default_rng(8)
    # 2 prompts x 3 beams: forced eos (L == P + 3), empty row, ordinary, forced bos (L == 1), ...
    hists = [[1, 2, 3, 4, 5], [], [4, 5, 6], [11], [9, 9, 9], [5, 6, 7, 8]]
    plens = [2, 0, 1, 1, 2, 1]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (6, V)).astype(np.float32)
    params = dict(vocab=V, logits_dtype="f32", mode="greedy", eos_token_ids=[2], forced_eos_token_ids=[2, 5],
                  max_new_tokens=4, forced_bos_token_id=7, suppress_tokens=[5], repetition_penalty=1.2)
    w = W.Workload("forced", params, logits, ids, off, np.array(plens, np.int32), rng.random(6, dtype=np.float32))
    compare_beam(w, 3, np.array([-1.0, -2.0, -3.0, -0.5, -9.0, -2.5], np.float32))


def test_all_empty_prompt_and_unaligned_rows():
    # V odd with f32: rows are not 16-byte aligned (the element-wise path)
    w = W.random_case(77, B=6, V=1001, dtype="f32", mode="greedy", L_max=9)
    w.hist_offsets = w.hist_offsets.copy()
    # prompt 1 (rows 3..5) empty
    L3 = int(w.hist_offsets[3])
    w.hist_offsets[4:] = L3
    w.hist_ids = w.hist_ids[:L3].copy()
    w.prompt_lens = w.prompt_lens.copy()
    w.prompt_lens[3:] = 0
    gs, gt, gb = compare_beam(w, 3, np.zeros(6, np.float32))
    assert (gt[1] == -1).all() and (gb[1] == -1).all()


def test_ties_and_all_removed_rows():
    # few distinct logits: ties at the kept boundary (the exact tie rules)
    V = 500
    rng = np.random.default_rng(19)
    ids, off = W._pack([rng.integers(0, V, 4).astype(np.int32) for _ in range(6)])
    logits = rng.integers(0, 3, (6, V)).astype(np.float32)
    w = W.Workload("ties", dict(vocab=V, logits_dtype="f32", eos_token_ids=[1], repetition_penalty=1.5),
                   logits, ids, off, np.ones(6, np.int32), rng.random(6, dtype=np.float32))
    compare_beam(w, 2, np.array([-1.0, -1.0, 0.0, -2.0, -0.5, -0.5], np.float32))
    # every token suppressed
    w2 = W.Workload("removed", dict(vocab=V, logits_dtype="f32", suppress_tokens=list(range(V))),
                    logits, ids, off, np.ones(6, np.int32), rng.random(6, dtype=np.float32))
    compare_beam(w2, 3, np.zeros(6, np.float32))


@pytest.mark.parametrize("nb", [2, 4])
def test_renormalize_logits(nb):
    """Each beam row's processed log-probabilities less their own log-sum-exp,
    then the beam's score; forced rows share their mass, an all-removed row
    scores -ln V everywhere."""
    w = W.random_case(81 + nb, B=3 * nb, V=1000, dtype="f32", mode="greedy", L_max=40, repetition_penalty=1.6,
                      no_repeat_ngram_size=2, suppress_tokens=list(range(40)), renormalize_logits=True)
    bs = np.random.default_rng(nb).normal(-3, 1, w.B).astype(np.float32)
    compare_beam(w, nb, bs)
    V = 3000
    rng = np.random.default_rng(8)
    hists = [[1, 2, 3, 4, 5], [7], [4, 5, 6], [11], [9, 9, 9], [5, 6, 7, 8]]
    plens = [2, 1, 1, 1, 2, 1]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (6, V)).astype(np.float32)
    params = dict(vocab=V, logits_dtype="f32", mode="greedy", eos_token_ids=[2], forced_eos_token_ids=[2, 5],
                  max_new_tokens=4, forced_bos_token_id=7, suppress_tokens=[5], repetition_penalty=1.2,
                  renormalize_logits=True)
    w2 = W.Workload("forced", params, logits, ids, off, np.array(plens, np.int32), rng.random(6, dtype=np.float32))
    compare_beam(w2, 3, np.array([-1.0, -2.0, -3.0, -0.5, -9.0, -2.5], np.float32))
    w3 = W.Workload("removed", dict(vocab=V, logits_dtype="f32", suppress_tokens=list(range(V)), renormalize_logits=True),
                    logits, ids, off, np.ones(6, np.int32), rng.random(6, dtype=np.float32))
    compare_beam(w3, 2, np.zeros(6, np.float32))
