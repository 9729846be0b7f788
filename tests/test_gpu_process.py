"""tg_process (diagnostic) against the oracle: processed scores bit-exact
(0 ULP), ban bits bit-exact, final probabilities within 1e-6 relative plus
one fixed-point quantum (2^-44) absolute."""
import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

from .gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def run_process(w):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params)
    d = to_device(w)
    nw = (w.V + 31) // 32
    sc = torch.full((w.B, w.V), 123.0, device="cuda")
    bb = torch.zeros((w.B, nw), dtype=torch.int32, device="cuda")
    pr = torch.zeros((w.B, w.V), device="cuda")
    tg.tg_process(d["logits"], d["hist_ids"], d["hist_offsets"], d["prompt_lens"], cfg, sc, bb, pr)
    torch.cuda.synchronize()
    return sc.cpu().numpy(), bb.cpu().numpy().view(np.uint32), pr.cpu().numpy()


def check(w, rows=None):
    sc, bb, pr = run_process(w)
    p = O.Params(**w.params)
    rows = range(w.B) if rows is None else rows
    for b in rows:
        h = list(w.history(b))
        if not h:
            assert np.all(sc[b] == 123.0)
            continue
        x = O.upcast_row(w.logits[b], p.logits_dtype)
        s_ref, banned = O.processed_scores(x, h, int(w.prompt_lens[b]), p)
        assert np.array_equal(sc[b].view(np.uint32) & 0x7fffffff, s_ref.view(np.uint32) & 0x7fffffff), b
        assert np.array_equal(sc[b], s_ref), b
        bits = np.unpackbits(bb[b].view(np.uint8), bitorder="little")[:w.V].astype(bool)
        assert np.array_equal(bits, banned), b
        if p.mode == "sample":
            _, _, _, _, info = O.sample_distribution(s_ref, p)
            if info.topp_boundary:
                continue
            ref = O.final_distribution(s_ref, p)
        else:
            ref = O.softmax64(s_ref)
        tol = 1e-6 * ref + 2.0 ** -44
        assert np.all(np.abs(pr[b].astype(np.float64) - ref) <= tol), (b, np.max(np.abs(pr[b] - ref) - tol))


def test_process_config2():
    check(W.config2(B=16))


def test_process_config3():
    check(W.config3(B=16))


def test_process_config5():
    check(W.config5(B=4, L_max=2048))


def test_process_config1():
    check(W.config1())


@pytest.mark.parametrize("seed", range(4))
def test_process_random(seed):
    w = W.random_case(seed, B=8, V=997, dtype="bf16" if seed % 2 else "f32", mode="sample",
                      repetition_penalty=1.4, no_repeat_ngram_size=2, temperature=0.6, top_k=50, top_p=0.8,
                      eos_token_ids=[1], min_new_tokens=3, suppress_tokens=[4, 5])
    check(w)


@pytest.mark.parametrize("seed", range(3))
def test_process_multi_token_bad_words(seed):
    # the rows' ids come from a six-id alphabet, so the words' prefixes match often
    a = [0, 166, 332, 498, 664, 830]
    words = [[a[0], a[1], 5], [a[2], 7], [a[5], a[5], a[5], 11], [13], [a[3], a[4], a[0], a[1], 17]]
    w = W.random_case(40 + seed, B=12, V=997, dtype="f32", mode="sample", L_max=30,
                      repetition_penalty=1.2, bad_word_seqs=words, bad_words_ids=[19])
    check(w)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_process_renormalize_logits(mode):
    """renormalize_logits: the scores after the processors less their
    log-sum-exp (before temperature).  The kernel forms s - lse with lse as a
    two-float pair, the oracle rounds s - lse once from fp64: a few ulp apart,
    2e-6 * max(1, |s|); removed tokens stay at the filter value bit for bit."""
    w = W.random_case(70, B=8, V=997, dtype="f32", mode=mode, repetition_penalty=1.3, suppress_tokens=[4, 5],
                      temperature=0.7, renormalize_logits=True)
    sc, bb, pr = run_process(w)
    p = O.Params(**w.params)
    for b in range(w.B):
        h = list(w.history(b))
        if not h:
            continue
        x = O.upcast_row(w.logits[b], p.logits_dtype)
        s_ref, banned = O.processed_scores(x, h, int(w.prompt_lens[b]), p)
        d = np.abs(sc[b].astype(np.float64) - s_ref.astype(np.float64))
        assert np.all(d <= 2e-6 * np.maximum(1.0, np.abs(s_ref.astype(np.float64)))), (b, d.max())
        assert np.array_equal(sc[b][banned], s_ref[banned])


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_process_renormalize_degenerate_rows(mode):
    """renormalize_logits on a row with every token removed (-ln V everywhere,
    before temperature) and on rows forced to one token (0 there)."""
    V = 3000
    rng = np.random.default_rng(71)
    logits = rng.normal(0, 2, (3, V)).astype(np.float32)
    ids, off = W._pack([np.array(h, np.int32) for h in ([1, 2, 3], [4], [5, 6])])
    uni = rng.random(3, dtype=np.float32)
    for params in (dict(suppress_tokens=list(range(V))),
                   dict(forced_bos_token_id=7, forced_eos_token_ids=[9], max_new_tokens=1)):
        w = W.Workload("degenerate", dict(vocab=V, logits_dtype="f32", mode=mode, temperature=0.5,
                                          renormalize_logits=True, **params),
                       logits, ids, off, np.array([1, 1, 1], np.int32), uni)
        sc, _, _ = run_process(w)
        p = O.Params(**w.params)
        for b in range(3):
            x = O.upcast_row(w.logits[b], p.logits_dtype)
            s_ref, _ = O.processed_scores(x, list(w.history(b)), 1, p)
            d = np.abs(sc[b].astype(np.float64) - s_ref.astype(np.float64))
            assert np.all(d <= 2e-6 * np.maximum(1.0, np.abs(s_ref.astype(np.float64)))), (b, d.max())
