"""tg_select_logprobs on the GPU against the CPU oracle.

Per row: the id must equal tg_select's id and the oracle's (rows the oracle
flags as lying within 1e-6 of a top-p cut or a CDF step are skipped), and the
log-probability must match the oracle's fp64 value within 1e-6 + 1e-7 |lp|:
the kernel takes it from the token's f32 score and the kept set's 44-bit
fixed-point mass, whose weights carry at most 2^-22 relative error each
(ex2.approx), then rounds it to f32.  Padding rows give NaN.
"""
import math

import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

from .gpu_util import gpu_select, oracle_select, to_device

pytestmark = pytest.mark.gpu

ABS_TOL = 1e-6
REL_TOL = 1e-7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def gpu_select_logprobs(w):
    import torch
    import logits_processing_token_gb300 as tg
    cfg = tg.Config(**w.params)
    dev = to_device(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    lp = torch.full((w.B,), 123.0, dtype=torch.float32, device="cuda")
    tg.tg_select(dev["logits"], dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg,
                 dev["uniforms"], out, out_logprobs=lp)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lp.cpu().numpy()


def compare_logprobs(w, rows=None, max_skipped_frac=0.06):
    ids, lps = gpu_select_logprobs(w)
    plain, _ = gpu_select(w)
    rows = list(range(w.B)) if rows is None else list(rows)
    ora, infos = oracle_select(w, rows)
    bad, skipped, compared = [], 0, 0
    for r, o, info in zip(rows, ora, infos):
        if int(o) < 0:
            if not (int(ids[r]) == -1 and math.isnan(float(lps[r]))):
                bad.append((r, "padding", int(ids[r]), float(lps[r])))
            continue
        if info.topp_boundary or info.u_boundary:
            skipped += 1
            continue
        if int(ids[r]) != int(o) or int(plain[r]) != int(o):
            bad.append((r, "id", int(ids[r]), int(plain[r]), int(o)))
            continue
        tol = ABS_TOL + REL_TOL * abs(info.logprob)
        if not abs(float(lps[r]) - info.logprob) <= tol:
            bad.append((r, "logprob", float(lps[r]), info.logprob))
        compared += 1
    assert not bad, "mismatching rows: %s" % bad[:10]
    assert skipped <= max(3, max_skipped_frac * len(rows)), skipped
    return ids, lps, compared


def test_config1_greedy():
    _, lps, n = compare_logprobs(W.config1())
    assert n == 1 and lps[0] <= 0.0


def test_config2_sampling():
    compare_logprobs(W.config2())


def test_config3_sampling_small():
    compare_logprobs(W.config3(B=24))


def test_config3_sampling_full():
    _, _, n = compare_logprobs(W.config3())
    assert n >= 200


def test_config3_greedy():
    w = W.config3(B=16)
    w.params["mode"] = "greedy"
    compare_logprobs(w)


def test_config5_small():
    compare_logprobs(W.config5(B=12, L_max=1024))


CASES = [
    # (V, dtype, mode, overrides): the one-pass finish, top_k ties, the exact
    # path (a draw without top_k / top_p), temperature, ragged vocabularies
    (1, "f32", "sample", {}),
    (7, "bf16", "sample", dict(top_k=3)),
    (1000, "f32", "sample", dict(temperature=0.5, top_k=10, top_p=0.8, repetition_penalty=1.3)),
    (8200, "bf16", "sample", dict(temperature=1.7, top_p=0.95)),
    (20001, "f32", "sample", dict(top_k=0, top_p=1.0)),
    (16384, "f32", "sample", dict(top_k=200, temperature=0.8)),
    (50257, "bf16", "greedy", dict(repetition_penalty=1.2, no_repeat_ngram_size=3)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_cases(case):
    V, dtype, mode, ov = CASES[case]
    for seed in range(2):
        w = W.random_case(700 + 10 * case + seed, B=9, V=V, dtype=dtype, mode=mode, L_max=40, **ov)
        compare_logprobs(w, max_skipped_frac=0.34)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_forced_padding_and_all_removed_rows(mode):
    V = 3000
    rng = np.random.default_rng(4)
    hists = [[], [11], [1, 2, 3, 4, 5], [9, 9, 9], [4, 5, 6, 7]]
    plens = [0, 1, 2, 3, 1]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (len(hists), V)).astype(np.float32)
    params = dict(vocab=V, logits_dtype="f32", mode=mode, top_p=0.9, eos_token_ids=[2],
                  forced_eos_token_ids=[2, 5, 8], max_new_tokens=4, forced_bos_token_id=7,
                  suppress_tokens=[5], begin_suppress_tokens=[7])
    w = W.Workload("forced", params, logits, ids, off, np.array(plens, np.int32),
                   rng.random(len(hists), dtype=np.float32))
    got, lps, _ = compare_logprobs(w, max_skipped_frac=1.0)
    assert got[0] == -1 and math.isnan(float(lps[0]))
    # every token suppressed: all scores equal
    w2 = W.random_case(5, B=4, V=40, mode=mode, suppress_tokens=list(range(40)))
    compare_logprobs(w2, max_skipped_frac=1.0)


def test_flat_rows_on_the_exact_path():
    import logits_processing_token_gb300 as tg
    rng = np.random.default_rng(12)
    B, V = 6, 30000
    logits = (rng.random((B, V)) * 0.01).astype(np.float32)
    ids, off = W._pack([np.array([1, 2, 3], np.int32)] * B)
    w = W.Workload("flat", dict(vocab=V, logits_dtype="f32", mode="sample", top_p=0.9), logits, ids, off,
                   np.full(B, 1, np.int32), rng.random(B, dtype=np.float32))
    compare_logprobs(w, max_skipped_frac=0.5)
