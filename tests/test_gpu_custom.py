"""A task processor compiled by the caller (include/tg_custom.cuh) against the
oracle with the same function as Params.custom: every token's score plus the
row's state entry of its bucket (Transmuter.Generation, section "Processors")."""
import ctypes

import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def task_lib(tmp_path_factory):
    from tests import custom_build
    path, _ = custom_build.build(tmp_path_factory.mktemp("task"))
    lib = ctypes.CDLL(path)
    lib.task_select.restype = ctypes.c_int
    return lib


def run(lib, w, state, logprobs):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params)
    if w.params.get("logits_dtype") == "bf16":
        lg = torch.from_numpy(w.logits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        lg = torch.from_numpy(w.logits).cuda()
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    u = torch.from_numpy(w.uniforms).cuda()
    st = torch.from_numpy(state).cuda()
    scores = torch.empty((w.B, w.V), dtype=torch.float32, device="cuda")
    out = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    lp = torch.empty(w.B, dtype=torch.float32, device="cuda") if logprobs else None
    p = ctypes.c_void_p
    rc = lib.task_select(p(lg.data_ptr()), w.B, w.V, p(hid.data_ptr()), p(off.data_ptr()), p(pl.data_ptr()),
                         cfg.handle, p(st.data_ptr()), state.shape[1], p(u.data_ptr()), p(scores.data_ptr()),
                         p(out.data_ptr()), p(lp.data_ptr()) if lp is not None else None,
                         p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return out.cpu().numpy(), (lp.cpu().numpy() if lp is not None else None), cfg


def bucket_bias(S, V):
    idx = np.arange(V) % S
    return lambda s, row: (s + row[idx]).astype(np.float32)


@pytest.mark.parametrize("case", ["config3", "config2", "greedy"])
def test_task_processor_matches_oracle(task_lib, case):
    if case == "config3":
        w = W.config3(B=24)
    elif case == "config2":
        w = W.config2(B=16)
    else:
        w = W.random_case(31, B=9, V=40_000, dtype="f32", mode="greedy", L_max=40, repetition_penalty=1.4,
                          suppress_tokens=[3, 9])
    S = 64
    state = np.random.default_rng(99).normal(0.0, 1.5, (w.B, S)).astype(np.float32)
    ids, lps, cfg = run(task_lib, w, state, logprobs=True)
    p = O.Params(**w.params, custom=bucket_bias(S, w.V))
    ref, infos = O.select(w.logits, w.hist_ids, w.hist_offsets, w.prompt_lens, p, w.uniforms, proc_state=state)
    boundary = 0
    for r in range(w.B):
        if infos[r].u_boundary or infos[r].topp_boundary:
            boundary += 1
            continue
        assert ids[r] == ref[r], (r, ids[r], ref[r])
        if ref[r] >= 0:
            assert abs(lps[r] - infos[r].logprob) <= 1e-6 + 1e-6 * abs(infos[r].logprob), (r, lps[r], infos[r].logprob)
    assert boundary <= max(1, w.B // 10)
    # ids without log-probabilities are the same ids
    ids2, _, _ = run(task_lib, w, state, logprobs=False)
    assert np.array_equal(ids, ids2)


def test_task_processor_zero_state_is_plain_select(task_lib):
    # a zero table changes no score: the same ids as tg_select
    from tests.gpu_util import gpu_select
    w = W.config2(B=8)
    ids, _, _ = run(task_lib, w, np.zeros((w.B, 16), np.float32), logprobs=False)
    plain, _ = gpu_select(w)
    assert np.array_equal(ids, plain)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_task_processor_in_verify(task_lib, mode):
    import torch
    import logits_processing_token_gb300 as tg
    B, K, S = 8, 5, 32
    w = W.config4(B=B, K=K, mode=mode)
    if mode == "sample":
        w.params.update(temperature=0.8, top_p=0.9)
    tgt = np.ascontiguousarray(w.extra["target"])
    greedy = tgt.argmax(axis=-1)[:, :K]
    cand = W.make_candidates(greedy, w.extra["agree"], w.extra["offsets"], w.V)
    state = np.random.default_rng(98).normal(0.0, 1.0, (B * (K + 1), S)).astype(np.float32)
    cfg = tg.Config(**w.params)
    t = torch.from_numpy(tgt).cuda()
    c = torch.from_numpy(cand).cuda()
    u = torch.from_numpy(np.ascontiguousarray(w.uniforms)).cuda()
    st = torch.from_numpy(state).cuda()
    scores = torch.empty((B * (K + 1), w.V), dtype=torch.float32, device="cuda")
    om = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    on = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p
    rc = task_lib.task_verify(p(t.data_ptr()), B, w.V, p(c.data_ptr()), K, cfg.handle, p(st.data_ptr()), S,
                              p(u.data_ptr()), p(scores.data_ptr()), p(om.data_ptr()), p(on.data_ptr()),
                              p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    om, on = om.cpu().numpy(), on.cpu().numpy()
    po = O.Params(**w.params, custom=bucket_bias(S, w.V))
    m_ref, n_ref, infos = O.verify(tgt, cand, K, po, w.uniforms, proc_state=state)
    for b in range(B):
        upto = int(m_ref[b])
        if any(ri.u_boundary or ri.topp_boundary for ri in infos[b][1][:upto + 1]):
            continue
        assert om[b] == m_ref[b], (b, om[b], m_ref[b])
        assert list(on[b]) == list(n_ref[b])
