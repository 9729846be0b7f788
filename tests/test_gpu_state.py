"""tg_select_state and tg_process_state (the task's processors) on the GPU
against the CPU oracle.

The processors (Transmuter.Generation, section "Processors") run after
begin_suppress_tokens: "bias" adds its value to a listed token's score, "set"
replaces it.  Processed scores are compared bit for bit (0 ULP), ban bits bit
for bit, ids exactly except on rows the oracle flags as lying within 1e-6 of
a top-p cut or a CDF step (counted, bounded), and log-probabilities within
1e-6 + 1e-7 |lp| as for tg_select_logprobs.
"""
import math

import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

from .gpu_util import to_device

pytestmark = pytest.mark.gpu

PROCS = (("bias", 24), ("set", 8))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def with_state(w, procs=PROCS, seed=0, **kw):
    """w with the processors in its params and a seeded state (half of a
    row's ids drawn from its history) in w.extra["state"]."""
    w.params["processors"] = tuple(procs)
    hot = [np.asarray(w.history(b)) for b in range(w.B)]
    w.extra["state"] = W.processor_state(seed, w.B, int(w.params["vocab"]), procs, hot=hot, **kw)
    return w


def state_dev(w):
    import torch
    ids, vals = w.extra["state"]
    return (torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(vals, np.float32)).cuda())


def gpu_select_state(w, logprobs=True):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params)
    dev = to_device(w)
    sid, sval = state_dev(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    lp = torch.full((w.B,), 123.0, dtype=torch.float32, device="cuda") if logprobs else None
    tg.tg_select_state(dev["logits"], dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg, sid, sval,
                       dev["uniforms"], out, out_logprobs=lp)
    torch.cuda.synchronize()
    flags, _ = tg.tg_query_status(cfg)
    return out.cpu().numpy(), (lp.cpu().numpy() if logprobs else None), flags


def oracle_rows(w, rows):
    p = O.Params(**w.params)
    return O.select(w.logits, w.hist_ids, w.hist_offsets, w.prompt_lens, p, w.uniforms, rows=rows,
                    proc_state=w.extra["state"])


def acceptable_tokens(w, b):
    """The draw with the top-p cut moved by one token either way and u moved
    by 2e-6 either way (rows within 1e-6 of a boundary)."""
    p = O.Params(**w.params)
    ids, vals = w.extra["state"]
    x = O.upcast_row(w.logits[b], p.logits_dtype)
    s, _, _ = O.process_row(x, list(w.history(b)), int(w.prompt_lens[b]), p, (ids[b], vals[b]))
    s_t = O.apply_temperature(s, p)
    order, n_kept, probs, _, _ = O.sample_distribution(s_t, p)
    u = float(w.uniforms[b])
    out = set()
    for n in (n_kept - 1, n_kept, n_kept + 1):
        if 1 <= n <= s_t.size:
            for du in (-2e-6, 0.0, 2e-6):
                uu = min(max(u + du, 0.0), np.nextafter(1.0, 0.0))
                out.add(O.draw(order, n, probs, uu)[0])
    return out


def compare_state(w, rows=None, max_boundary_frac=0.06, logprobs=True):
    ids, lps, flags = gpu_select_state(w, logprobs)
    rows = list(range(w.B)) if rows is None else list(rows)
    ora, infos = oracle_rows(w, rows)
    bad, boundary, compared = [], 0, 0
    for r, o, info in zip(rows, ora, infos):
        if int(o) < 0:
            if int(ids[r]) != -1 or (logprobs and not math.isnan(float(lps[r]))):
                bad.append((r, "padding", int(ids[r])))
            continue
        if info.topp_boundary or info.u_boundary:
            boundary += 1
            if int(ids[r]) != int(o) and int(ids[r]) not in acceptable_tokens(w, r):
                bad.append((r, "boundary", int(ids[r]), int(o)))
            continue
        if int(ids[r]) != int(o):
            bad.append((r, "id", int(ids[r]), int(o)))
            continue
        if logprobs:
            tol = 1e-6 + 1e-7 * abs(info.logprob)
            if not abs(float(lps[r]) - info.logprob) <= tol:
                bad.append((r, "logprob", float(lps[r]), info.logprob))
        compared += 1
    assert not bad, "mismatching rows: %s" % bad[:10]
    assert boundary <= max(3, max_boundary_frac * len(rows)), boundary
    return ids, flags, infos, compared


CASES = [
    # (V, dtype, mode, overrides)
    (1, "f32", "greedy", {}),
    (7, "bf16", "sample", dict(top_k=3)),
    (33, "f32", "greedy", dict(repetition_penalty=1.5, no_repeat_ngram_size=2)),
    (1000, "f32", "sample", dict(temperature=0.5, top_k=10, top_p=0.8, repetition_penalty=1.3)),
    (1000, "bf16", "sample", dict(no_repeat_ngram_size=1, eos_token_ids=[3], min_length=40)),
    (4100, "f32", "sample", dict(top_p=0.7, repetition_penalty=0.8, no_repeat_ngram_size=3)),
    (8193, "bf16", "greedy", dict(repetition_penalty=2.0, no_repeat_ngram_size=2)),
    (20001, "f32", "sample", dict(top_k=0, top_p=1.0)),
    (50257, "f32", "sample", dict(top_p=0.9, repetition_penalty=1.2, suppress_tokens=[5, 77])),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_cases(case):
    V, dtype, mode, ov = CASES[case]
    for seed in range(2):
        w = W.random_case(900 + 10 * case + seed, B=9, V=V, dtype=dtype, mode=mode, L_max=40, **ov)
        # values on the quarter grid of the scores (ties across processed tokens)
        with_state(w, procs=(("bias", min(V, 6)), ("set", min(V, 4)), ("bias", 3)), seed=seed, sigma=2.0)
        ids, vals = w.extra["state"]
        keep = vals == np.float32(-np.finfo(np.float32).max)
        vals[~keep] = np.round(vals[~keep] * 4) / 4
        compare_state(w, max_boundary_frac=0.34)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_forced_and_padding_rows(mode):
    """Forced rows: the processors see 0 at the forced ids and the filter
    value elsewhere; a set raises a token, a bias on the filter value keeps
    it there, a bias on a forced id shifts it."""
    V = 3000
    rng = np.random.default_rng(41)
    hists = [[], [11], [1, 2, 3, 4, 5], [9, 9, 9], [4, 5, 6, 7], [3, 1]]
    plens = [0, 1, 2, 3, 1, 2]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (len(hists), V)).astype(np.float32)
    params = dict(vocab=V, logits_dtype="f32", mode=mode, top_p=0.9, eos_token_ids=[2],
                  forced_eos_token_ids=[2, 5, 8], max_new_tokens=4, forced_bos_token_id=7,
                  suppress_tokens=[5], begin_suppress_tokens=[7], processors=(("bias", 3), ("set", 2)))
    w = W.Workload("forced", params, logits, ids, off, np.array(plens, np.int32),
                   rng.random(len(hists), dtype=np.float32))
    F = -np.finfo(np.float32).max
    st_ids = np.array([[-1, -1, -1, -1, -1],
                       [7, 100, -1, 7, -1],        # bos row: bias bos, set bos again
                       [2, 8, -1, 2999, -1],        # forced eos row: shift 2 and 8, raise 2999
                       [0, -1, -1, -1, -1],
                       [2, 5, 9, 5, 9],             # set raises a suppressed id
                       [-1, -1, -1, 3, -1]], np.int32)
    st_vals = np.array([[0, 0, 0, 0, 0],
                        [1.5, 4.0, 0, -0.5, 0],
                        [np.log(3.0), 0.25, 0, -1.0, 0],
                        [2.0, 0, 0, 0, 0],
                        [1.0, 2.0, 3.0, 0.5, F],
                        [0, 0, 0, 1.0, 0]], np.float32)
    w.extra["state"] = (st_ids, st_vals)
    got, _, _, n = compare_state(w, max_boundary_frac=1.0)
    assert got[0] == -1 and n >= 4


def test_invalid_states_are_dropped_and_flagged():
    import logits_processing_token_gb300 as tg
    w = W.random_case(77, B=6, V=500, mode="sample", top_p=0.8, repetition_penalty=1.3, L_max=30)
    with_state(w, procs=(("bias", 4), ("set", 3)), seed=3)
    ids, vals = w.extra["state"]
    ids[1, :4] = [9, 5, -1, -1]      # not ascending
    ids[2, :4] = [-1, 5, -1, -1]     # padding before an id
    ids[3, 4:] = [1, 500, -1]        # id out of range
    ids[4, 4:] = [-2, -1, -1]        # negative id other than -1
    got, flags, infos, _ = compare_state(w, max_boundary_frac=0.5)
    assert flags & tg.TG_FLAG_BAD_STATE
    assert [bool(i.bad_state) for i in infos] == [False, True, True, True, True, False]


def test_no_entries_matches_tg_select():
    """A state with no entries in use changes nothing: tg_select_state gives
    tg_select's ids on the same config without processors."""
    import torch
    import logits_processing_token_gb300 as tg
    from .gpu_util import gpu_select
    w = W.config3(B=24)
    gpu_plain, _ = gpu_select(w)
    with_state(w, procs=(("bias", 16),), fill=0.0)
    assert (w.extra["state"][0] == -1).all()
    got, _, infos, _ = compare_state(w)
    for r, info in enumerate(infos):
        if not (info.topp_boundary or info.u_boundary):
            assert int(got[r]) == int(gpu_plain[r]), r


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_process_state_scores_and_banbits(mode):
    """tg_process_state: processed scores bit for bit, ban bits bit for bit."""
    import torch
    import logits_processing_token_gb300 as tg
    for seed, (V, dtype) in enumerate([(1000, "f32"), (4099, "bf16"), (33, "f32")]):
        ov = dict(repetition_penalty=1.3, no_repeat_ngram_size=2, suppress_tokens=[1, 4], eos_token_ids=[3],
                  min_new_tokens=5, temperature=0.7 if mode == "sample" else 1.0,
                  forced_eos_token_ids=[3], max_new_tokens=6)
        w = W.random_case(300 + seed, B=10, V=V, dtype=dtype, mode=mode, L_max=24, **ov)
        with_state(w, procs=(("set", 5), ("bias", 7)), seed=seed)
        cfg = tg.Config(**w.params)
        dev = to_device(w)
        sid, sval = state_dev(w)
        nw = (V + 31) // 32
        sc = torch.full((w.B, V), 7.0, dtype=torch.float32, device="cuda")
        bb = torch.zeros((w.B, nw), dtype=torch.int32, device="cuda")
        tg.tg_process_state(dev["logits"], dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg, sid, sval,
                            sc, bb)
        torch.cuda.synchronize()
        sc, bb = sc.cpu().numpy(), bb.cpu().numpy().view(np.uint32)
        p = O.Params(**w.params)
        st_ids, st_vals = w.extra["state"]
        for b in range(w.B):
            h = list(w.history(b))
            if not h:
                continue
            x = O.upcast_row(w.logits[b], p.logits_dtype)
            s, banned = O.processed_scores(x, h, int(w.prompt_lens[b]), p, (st_ids[b], st_vals[b]))
            assert np.array_equal(sc[b].view(np.uint32), s.astype(np.float32).view(np.uint32)), (seed, b)
            bits = np.zeros(nw * 32, bool)
            bits[:V] = banned
            words = (bits.reshape(nw, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1)
            assert np.array_equal(bb[b].astype(np.uint64), words), (seed, b)


def test_benchmark_rows_with_processors():
    """The benchmark rows (B=256, V=151,936 bf16, full chain, top_p 0.95)
    with a bias of 64 and a set of 32 columns per row: every eighth row
    against the oracle, and ids and log-probabilities bit-identical on a
    second call."""
    w = with_state(W.config3(), procs=(("bias", 64), ("set", 32)), seed=5)
    rows = list(range(0, w.B, 8))
    ids, flags, _, n = compare_state(w, rows=rows)
    assert n >= 24
    ids2, lps2, _ = gpu_select_state(w)
    ids3, lps3, _ = gpu_select_state(w)
    assert np.array_equal(ids2, ids3) and np.array_equal(lps2.view(np.uint32), lps3.view(np.uint32))


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_rows_left_to_the_exact_path(mode):
    """Rows select_kernel hands to state_kernel: histories too long to stage
    (9,000 ids), forced rows under top_k (more and fewer tokens above the
    filter value than k), and a draw without top_p (the exact path)."""
    V = 5000
    rng = np.random.default_rng(12)
    hists = [rng.integers(0, V, 9000).astype(np.int32), rng.integers(0, V, 20).astype(np.int32),
             np.arange(3, dtype=np.int32), np.arange(3, dtype=np.int32), rng.integers(0, V, 40).astype(np.int32)]
    plens = [100, 5, 1, 1, 40]
    ids, off = W._pack(hists)
    logits = rng.normal(0, 2, (len(hists), V)).astype(np.float32)
    params = dict(vocab=V, logits_dtype="f32", mode=mode, top_k=2, top_p=1.0, repetition_penalty=1.3,
                  no_repeat_ngram_size=2, forced_eos_token_ids=[2, 8], max_new_tokens=3,
                  processors=(("bias", 4), ("set", 3)))
    w = W.Workload("deferred", params, logits, ids, off, np.array(plens, np.int32),
                   rng.random(len(hists), dtype=np.float32))
    st_ids = np.array([[int(hists[0][0]), 4000, -1, -1, 7, 9, -1],
                       [-1, -1, -1, -1, int(hists[1][3]), -1, -1],
                       [2, -1, -1, -1, 11, 12, 13],       # forced: 2, 8 and three set tokens above F
                       [8, -1, -1, -1, -1, -1, -1],       # forced: only 2 and 8
                       [5, 6, -1, -1, 5, -1, -1]], np.int32)
    st_vals = np.array([[1.0, 2.0, 0, 0, 3.5, -1.0, 0],
                        [0, 0, 0, 0, 6.0, 0, 0],
                        [0.5, 0, 0, 0, 0.25, 1.0, -0.5],
                        [-0.75, 0, 0, 0, 0, 0, 0],
                        [0.5, 0.5, 0, 0, -2.0, 0, 0]], np.float32)
    w.extra["state"] = (st_ids, st_vals)
    compare_state(w, max_boundary_frac=1.0)


def test_largest_workload_sampled_rows():
    """B=1,024, V=262,144 f32 Student-t rows (histories up to 4,096 Zipf ids,
    repetition penalty, 4-gram bans, top_p 0.9) with a bias of 48 and a set
    of 16 columns per row: every 32nd row against the oracle."""
    w = with_state(W.config5(), procs=(("bias", 48), ("set", 16)), seed=8)
    rows = list(range(0, w.B, 32))
    _, _, _, n = compare_state(w, rows=rows)
    assert n >= 28


def test_benchmark_rows_greedy_with_processors():
    w = W.config3(B=64)
    w.params["mode"] = "greedy"
    with_state(w, procs=(("set", 16), ("bias", 16)), seed=6)
    compare_state(w)
