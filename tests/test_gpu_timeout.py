"""A bounded wait that runs out (its limit shortened to a few cycles through
tg_set_wait_limit, so the copies it waits on are still in flight): the
launch raises TG_FLAG_TIMEOUT, its unfinished rows give -1 (verify: out_match
-1), and the next normal call on the same config matches the oracle."""
import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O
from tests.test_gpu_verify import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def _verify(cfg, tgt, cand, u, B, K):
    import torch
    import logits_processing_token_gb300 as tg
    t = torch.from_numpy(np.ascontiguousarray(tgt)).cuda()
    c = torch.from_numpy(cand).cuda()
    uu = torch.from_numpy(np.ascontiguousarray(u)).cuda()
    om = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    on = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify(t, c, K, cfg, uu, om, on)
    torch.cuda.synchronize()
    return om.cpu().numpy(), on.cpu().numpy()


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_verify_after_timeout(mode):
    import logits_processing_token_gb300 as tg
    B, K = 8, 4
    w, tgt, cand, p = make_case(B, K, mode)
    cfg = tg.Config(**w.params, max_batch=64)
    tg.tg_set_wait_limit(1)
    try:
        om, on = _verify(cfg, tgt, cand, w.uniforms, B, K)
    finally:
        tg.tg_set_wait_limit(0)
    flags, _ = tg.tg_query_status(cfg)
    assert flags & tg.TG_FLAG_TIMEOUT
    assert (om == -1).any()
    assert not (om == -9).any()          # every batch row was written: a count, or -1
    tg.tg_clear_status(cfg)
    om2, on2 = _verify(cfg, tgt, cand, w.uniforms, B, K)
    assert tg.tg_query_status(cfg)[0] & tg.TG_FLAG_TIMEOUT == 0
    m_ref, n_ref, infos = O.verify(tgt, cand, K, p, w.uniforms)
    for b in range(B):
        upto = int(m_ref[b])
        if any(ri.u_boundary or ri.topp_boundary for ri in infos[b][1][:upto + 1]):
            continue
        assert om2[b] == m_ref[b], (b, om2[b], m_ref[b])
        assert list(on2[b]) == list(n_ref[b])


def test_select_after_timeout():
    import torch
    import logits_processing_token_gb300 as tg
    from tests.gpu_util import compare_select
    w = W.config2(B=16)
    cfg = tg.Config(**w.params)
    lg = torch.from_numpy(w.logits).cuda()
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    u = torch.from_numpy(w.uniforms).cuda()
    out = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    tg.tg_set_wait_limit(1)
    try:
        tg.tg_select(lg, hid, off, pl, cfg, u, out)
        torch.cuda.synchronize()
    finally:
        tg.tg_set_wait_limit(0)
    o = out.cpu().numpy()
    assert tg.tg_query_status(cfg)[0] & tg.TG_FLAG_TIMEOUT
    assert (o == -1).any() and not (o == -9).any()
    compare_select(w)


def test_verify_history_after_timeout():
    import logits_processing_token_gb300 as tg
    from tests.test_gpu_verify import run_gpu_history
    B, K = 6, 4
    w, tgt, cand, p = make_case(B, K, "greedy", repetition_penalty=1.5, no_repeat_ngram_size=3)
    rng = np.random.default_rng(5)
    hists = [list(rng.integers(0, 50, int(rng.integers(2, 30)))) for _ in range(B)]
    plens = [1] * B
    tg.tg_set_wait_limit(1)
    try:
        om, _, _, _ = run_gpu_history(w, tgt, cand, K, hists, plens)
    finally:
        tg.tg_set_wait_limit(0)
    assert (om == -1).any() and not (om == -9).any()
    om2, on2, ids, off = run_gpu_history(w, tgt, cand, K, hists, plens)
    m_ref, n_ref, infos = O.verify_history(tgt, cand, K, ids, off, np.asarray(plens, np.int32), O.Params(**w.params),
                                           w.uniforms)
    assert np.array_equal(om2, m_ref) and np.array_equal(on2, n_ref)
