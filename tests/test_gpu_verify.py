"""tg_verify on the GPU against the oracle's verify (Assisted Generation,
steps 3-5), for B in {1, 8, 32} and K from 1 to 16, greedy and sampling."""
import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def make_case(B, K, mode, **ov):
    w = W.config4(B=B, K=K, mode=mode)
    w.params.update(ov)
    tgt = w.extra["target"]
    p = O.Params(**w.params)
    # the agreeing candidates copy the target's greedy token (oracle argmax)
    greedy = np.array([[O.select_row(tgt[b, j], [0], 1, O.Params(vocab=w.V), 0.0)[0] for j in range(K)]
                       for b in range(B)])
    cand = W.make_candidates(greedy, w.extra["agree"], w.extra["offsets"], w.V)
    return w, tgt, cand, p


def run_gpu(w, tgt, cand, K):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params, max_batch=64)
    t = torch.from_numpy(np.ascontiguousarray(tgt)).cuda()
    c = torch.from_numpy(cand).cuda()
    u = torch.from_numpy(np.ascontiguousarray(w.uniforms)).cuda()
    om = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    on = torch.full((w.B, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify(t, c, K, cfg, u, om, on)
    torch.cuda.synchronize()
    return om.cpu().numpy(), on.cpu().numpy(), cfg


@pytest.mark.parametrize("B", [1, 8, 32])
@pytest.mark.parametrize("K", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_verify_parity(B, K, mode):
    w, tgt, cand, p = make_case(B, K, mode)
    om, on, _ = run_gpu(w, tgt, cand, K)
    m_ref, n_ref, infos = O.verify(tgt, cand, K, p, w.uniforms)
    for b in range(B):
        nxt, row_infos = infos[b]
        # a row is decided once every position up to its first mismatch is off any CDF boundary
        upto = int(m_ref[b])
        if any(ri.u_boundary or ri.topp_boundary for ri in row_infos[:upto + 1]):
            continue
        assert om[b] == m_ref[b], (b, om[b], m_ref[b])
        assert list(on[b]) == list(n_ref[b]), (b, on[b], n_ref[b])


def test_verify_warpers_and_repeat():
    # temperature/top_k/top_p apply per position; repeated calls reuse the tickets
    w, tgt, cand, p = make_case(8, 4, "sample", temperature=0.7, top_k=40, top_p=0.9)
    om1, on1, cfg = run_gpu(w, tgt, cand, 4)
    om2, on2, _ = run_gpu(w, tgt, cand, 4)
    assert np.array_equal(om1, om2) and np.array_equal(on1, on2)
    m_ref, n_ref, infos = O.verify(tgt, cand, 4, p, w.uniforms)
    for b in range(8):
        if any(ri.u_boundary or ri.topp_boundary for ri in infos[b][1]):
            continue
        assert om1[b] == m_ref[b] and list(on1[b]) == list(n_ref[b])


def test_candidate_heuristic_trace():
    import logits_processing_token_gb300 as tg
    K = O.INITIAL_NUM_CANDIDATES
    trace = []
    for n in (5, 7, 3, 0, 6, 6):
        K2 = tg.tg_next_num_candidates(K, min(n, K), 16)
        assert K2 == O.next_num_candidates(K, min(n, K), 16)
        trace.append(K2)
        K = K2
    assert trace[:2] == [7, 9]


def run_gpu_history(w, tgt, cand, K, hists, plens):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params, max_batch=64)
    ids, off = W._pack([np.asarray(h, np.int32) for h in hists])
    t = torch.from_numpy(np.ascontiguousarray(tgt)).cuda()
    c = torch.from_numpy(cand).cuda()
    u = torch.from_numpy(np.ascontiguousarray(w.uniforms)).cuda()
    om = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    on = torch.full((w.B, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify_history(t, c, K, torch.from_numpy(ids).cuda(), torch.from_numpy(off).cuda(),
                         torch.from_numpy(np.asarray(plens, np.int32)).cuda(), cfg, u, om, on)
    torch.cuda.synchronize()
    return om.cpu().numpy(), on.cpu().numpy(), ids, off


@pytest.mark.parametrize("mode", ["greedy", "sample"])
@pytest.mark.parametrize("K", [1, 2, 5, 8, 16])
def test_verify_history_parity(mode, K):
    """Processors at every position with the candidates as history: repetition
    penalty, 3-gram bans, bad words of several tokens, min_new_tokens, forced
    eos, against the oracle's verify_history."""
    B = 12
    w, tgt, cand, _ = make_case(B, K, mode, repetition_penalty=1.5, no_repeat_ngram_size=3,
                                eos_token_ids=[2], min_new_tokens=4, forced_eos_token_ids=[2], max_new_tokens=9,
                                bad_word_seqs=[[5, 9], [17, 23, 31]])
    rng = np.random.default_rng(100 + K)
    hists, plens = [], []
    for b in range(B):
        if b == 3:
            hists.append([])          # a padding row
            plens.append(0)
            continue
        L = int(rng.integers(1, 40))
        h = list(rng.integers(0, 50, L))
        # repeat the first candidates inside the history so penalties and n-grams fire
        h[:2] = [int(cand[b, 0]), int(cand[b, min(1, K - 1)])]
        hists.append(h)
        plens.append(int(rng.integers(1, L + 1)))
    om, on, ids, off = run_gpu_history(w, tgt, cand, K, hists, plens)
    p = O.Params(**w.params)
    m_ref, n_ref, infos = O.verify_history(tgt, cand, K, ids, off, np.asarray(plens, np.int32), p, w.uniforms)
    checked = 0
    for b in range(B):
        nxt, row_infos = infos[b]
        upto = int(m_ref[b])
        if any(ri.u_boundary or ri.topp_boundary for ri in row_infos[:upto + 1]):
            continue
        assert om[b] == m_ref[b], (b, om[b], m_ref[b])
        assert list(on[b]) == list(n_ref[b]), (b, on[b], n_ref[b])
        checked += 1
    assert checked >= B - 3
    assert om[3] == 0 and list(on[3]) == [-1] * (K + 1)


@pytest.mark.parametrize("B,K", [(1, 1), (1, 5), (2, 2), (1, 8), (2, 5)])
def test_verify_greedy_split_rows(B, K):
    # Greedy verify of a batch this small splits each position's row over
    # several CTAs (all but B=2, K=5: 12 positions of 13 slices do not fit one
    # wave); the same sequences repeated into a batch of 64 (the config's
    # max_batch) take one CTA per row.  Both, and a second call on the same
    # config, give the same results.
    import torch
    import logits_processing_token_gb300 as tg
    w, tgt, cand, p = make_case(B, K, "greedy")
    om, on, cfg = run_gpu(w, tgt, cand, K)
    t = torch.from_numpy(np.ascontiguousarray(tgt)).cuda()
    c = torch.from_numpy(cand).cuda()
    u = torch.from_numpy(np.ascontiguousarray(w.uniforms)).cuda()
    om2 = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    on2 = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify(t, c, K, cfg, u, om2, on2)
    torch.cuda.synchronize()
    assert np.array_equal(om2.cpu().numpy(), om) and np.array_equal(on2.cpu().numpy(), on)
    reps = 64 // B
    tb = torch.from_numpy(np.ascontiguousarray(np.tile(tgt, (reps, 1, 1)))).cuda()
    cb = torch.from_numpy(np.ascontiguousarray(np.tile(cand, (reps, 1)))).cuda()
    ub = torch.from_numpy(np.ascontiguousarray(np.tile(w.uniforms, (reps, 1)))).cuda()
    omb = torch.full((B * reps,), -9, dtype=torch.int32, device="cuda")
    onb = torch.full((B * reps, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify(tb, cb, K, cfg, ub, omb, onb)
    torch.cuda.synchronize()
    assert np.array_equal(omb.cpu().numpy()[:B], om) and np.array_equal(onb.cpu().numpy()[:B], on)
    m_ref, n_ref, _ = O.verify(tgt, cand, K, p, w.uniforms)
    assert list(om) == [int(x) for x in m_ref]
    assert [list(r) for r in on] == [[int(x) for x in r] for r in n_ref]
