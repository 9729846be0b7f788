"""tg_select on the GPU against the CPU oracle, element by element.

Ids are compared bit-exactly except on rows the oracle flags as lying within
1e-6 of a top-p cut or a CDF step (counted, bounded).  Sizes: every workload
at its full size (sampled rows where the oracle would take long) plus smaller
cases that still span many 16 KB sub-chunks and ragged tails.
"""
import numpy as np
import pytest

from logits_processing_token_gb300 import workloads as W
from oracle import tg_oracle as O

from .gpu_util import compare_select, gpu_select, oracle_select, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from logits_processing_token_gb300 import _build
    _build.build()


def test_config1_greedy_full():
    gpu, cfg, _ = compare_select(W.config1())
    assert gpu[0] >= 0


def test_config2_sampling_full():
    w = W.config2()
    gpu, cfg, nb = compare_select(w)
    # the planted 3-gram's continuation is banned in every row
    for b in range(w.B):
        h = w.history(b)
        assert O.ngram_banned_tokens(list(h), 3)


def test_config3_small():
    compare_select(W.config3(B=24))


def test_config3_full():
    compare_select(W.config3())


def test_config5_small():
    compare_select(W.config5(B=12, L_max=1024))


def test_config5_full_sampled_rows():
    w = W.config5()
    rows = list(range(0, w.B, 16))
    compare_select(w, rows=rows)


@pytest.mark.parametrize("maker", [W.config2, W.config3, W.config5])
def test_greedy_variants(maker):
    w = maker(B=16) if maker is not W.config5 else maker(B=8, L_max=1024)
    w.params["mode"] = "greedy"
    compare_select(w)


CASES = [
    # (V, dtype, mode, overrides)
    (1, "f32", "greedy", {}),
    (1, "bf16", "sample", {}),
    (2, "f32", "sample", dict(top_p=0.5)),
    (7, "bf16", "sample", dict(top_k=3)),
    (33, "f32", "greedy", dict(repetition_penalty=1.5, no_repeat_ngram_size=2)),
    (1000, "f32", "sample", dict(temperature=0.5, top_k=10, top_p=0.8, repetition_penalty=1.3)),
    (1000, "bf16", "sample", dict(no_repeat_ngram_size=1, eos_token_ids=[3], min_length=40)),
    (4100, "f32", "sample", dict(top_p=0.7, repetition_penalty=0.8, no_repeat_ngram_size=3)),
    (8193, "bf16", "greedy", dict(repetition_penalty=2.0, no_repeat_ngram_size=2)),
    (8200, "bf16", "sample", dict(temperature=1.7, top_p=0.95)),
    (20001, "f32", "sample", dict(top_k=0, top_p=1.0)),
    (50257, "f32", "sample", dict(top_p=0.9, repetition_penalty=1.2)),
    (50257, "bf16", "greedy", dict(repetition_penalty=1.2, no_repeat_ngram_size=3)),
    (16384, "f32", "sample", dict(top_k=200, temperature=0.8)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_cases(case):
    V, dtype, mode, ov = CASES[case]
    for seed in range(3):
        w = W.random_case(100 * case + seed, B=9, V=V, dtype=dtype, mode=mode, L_max=40, **ov)
        compare_select(w, max_boundary_frac=0.34)


def _forced_params(V, **kw):
    base = dict(vocab=V, logits_dtype="f32", eos_token_ids=[2], forced_eos_token_ids=[2, 5],
                max_new_tokens=4, forced_bos_token_id=7, suppress_tokens=[5], begin_suppress_tokens=[7])
    base.update(kw)
    return base


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_forced_padding_and_begin_rows(mode):
    V = 3000
    rng = np.random.default_rng(4)
    # rows: padding, L==1 (forced bos; begin index shifted), forced eos (L == P+3),
    # begin suppress at L == P, ordinary
    hists = [[], [11], [1, 2, 3, 4, 5], [9, 9, 9], [4, 5, 6, 7]]
    plens = [0, 1, 2, 3, 1]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (len(hists), V)).astype(np.float32)
    w = W.Workload("forced", _forced_params(V, mode=mode, top_p=0.9), logits, ids, off,
                   np.array(plens, np.int32), rng.random(len(hists), dtype=np.float32))
    gpu, _, _ = compare_select(w, max_boundary_frac=1.0)
    assert gpu[0] == -1


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_all_removed_row(mode):
    # every token suppressed: all scores are the filter value
    V = 40
    w = W.random_case(5, B=6, V=V, mode=mode, suppress_tokens=list(range(V)), top_p=0.6)
    gpu, _, _ = compare_select(w, max_boundary_frac=1.0)
    if mode == "greedy":
        assert all(g in (-1, 0) for g in gpu)


def test_out_of_range_history_ids_flagged():
    import logits_processing_token_gb300 as tg
    w = W.random_case(8, B=4, V=500, mode="greedy", repetition_penalty=3.0)
    w.hist_ids = w.hist_ids.copy()
    if w.hist_ids.size:
        w.hist_ids[::3] = np.where(np.arange(w.hist_ids[::3].size) % 2, -5, 500)
    gpu, cfg, _ = compare_select(w)
    flags, _ = tg.tg_query_status(cfg)
    assert tg.tg_status_word(cfg) == flags
    assert flags & tg.TG_FLAG_HISTORY_ID_OUT_OF_RANGE


def test_bad_rows_give_minus_one():
    import logits_processing_token_gb300 as tg
    w = W.random_case(9, B=3, V=100, mode="greedy", L_max=10)
    w.prompt_lens = np.array([int(w.hist_offsets[b + 1] - w.hist_offsets[b]) + 1 for b in range(3)], np.int32)
    gpu, cfg = gpu_select(w)
    assert list(gpu) == [-1, -1, -1]
    flags, _ = tg.tg_query_status(cfg)
    assert flags & tg.TG_FLAG_BAD_ROW


def test_flat_rows_take_exact_multipass_path():
    import logits_processing_token_gb300 as tg
    # nearly flat scores: top_p keeps most of the row, beyond the candidate list
    rng = np.random.default_rng(12)
    B, V = 6, 30000
    logits = (rng.random((B, V)) * 0.01).astype(np.float32)
    ids, off = W._pack([np.array([1, 2, 3], np.int32)] * B)
    w = W.Workload("flat", dict(vocab=V, logits_dtype="f32", mode="sample", top_p=0.9), logits, ids, off,
                   np.full(B, 1, np.int32), rng.random(B, dtype=np.float32))
    gpu, cfg, _ = compare_select(w, max_boundary_frac=0.5)
    flags, slow = tg.tg_query_status(cfg)
    assert slow >= 1 and (flags & tg.TG_FLAG_SLOW_PATH)


def test_nondefault_stream_and_repeat():
    import torch
    import logits_processing_token_gb300 as tg
    w = W.config2(B=16)
    dev = to_device(w)
    cfg = tg.Config(**w.params)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            o = torch.empty(w.B, dtype=torch.int32, device="cuda")
            tg.tg_select(dev["logits"], dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg,
                         dev["uniforms"], o, stream=s)
            outs.append(o)
    s.synchronize()
    ref = outs[0].cpu().numpy()
    for o in outs[1:]:
        assert np.array_equal(o.cpu().numpy(), ref)
    ora, infos = oracle_select(w)
    for r in range(w.B):
        if not (infos[r].topp_boundary or infos[r].u_boundary):
            assert ref[r] == ora[r]


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_multi_token_bad_words(mode):
    a = [0, 166, 332, 498, 664, 830]
    # the banned last ids score high, so a missed ban changes the selection
    words = [[a[0], a[1], 5], [a[2], 7], [a[5], a[5], a[5], 11], [13], [a[3], a[4], a[0], 17]]
    for seed in range(3):
        w = W.random_case(60 + seed, B=16, V=997, dtype="f32", mode=mode, L_max=30,
                          repetition_penalty=1.2, bad_word_seqs=words, top_p=0.7)
        w.logits = w.logits.copy()
        w.logits[:, [5, 7, 11, 13, 17]] = 30.0
        compare_select(w, max_boundary_frac=0.34)


# Greedy ids of a batch too small to fill the GPU run with each row split over
# several CTAs (when batch x slices fits one wave of CTAs); the same rows in a
# batch too large for that split run one row per CTA.  Both must give the
# oracle's ids, and a second call on the same config the same ids again.
SPLIT_CASES = [
    # (V, dtype, B, overrides)
    (50272, "f32", 1, dict(repetition_penalty=1.3, no_repeat_ngram_size=2)),
    (50257, "bf16", 5, dict(repetition_penalty=1.2, no_repeat_ngram_size=3)),   # rows not on 16-byte boundaries
    (151936, "bf16", 4, dict(suppress_tokens=list(range(0, 151936, 7)), repetition_penalty=0.9)),
    (262144, "f32", 2, dict(repetition_penalty=0.7, eos_token_ids=[3], min_length=30)),
    (20000, "f32", 7, {}),                                                        # no processors
    (4104, "bf16", 9, dict(repetition_penalty=2.0)),                              # two slices of 2,056 tokens
]


def _replicated(w, B2):
    hists = [np.asarray(w.history(b % w.B), np.int32) for b in range(B2)]
    ids, off = W._pack(hists)
    reps = (B2 + w.B - 1) // w.B
    return W.Workload("replicated", dict(w.params), np.tile(w.logits, (reps, 1))[:B2], ids, off,
                      np.tile(w.prompt_lens, reps)[:B2], np.tile(w.uniforms, reps)[:B2])


@pytest.mark.parametrize("case", range(len(SPLIT_CASES)))
def test_split_greedy_rows(case):
    V, dtype, B, ov = SPLIT_CASES[case]
    w = W.random_case(700 + case, B=B, V=V, dtype=dtype, mode="greedy", L_max=60, **ov)
    gpu, cfg, _ = compare_select(w)
    again, _ = gpu_select(w, cfg=cfg)
    assert np.array_equal(again, gpu)
    big, _ = gpu_select(_replicated(w, 160))
    assert np.array_equal(big[:B], gpu)


def test_split_greedy_forced_and_removed_rows():
    # padding, forced bos, forced eos, begin-suppress and ordinary rows on a vocabulary that is split
    V = 20000
    rng = np.random.default_rng(14)
    hists = [[], [11], [1, 2, 3, 4, 5], [9, 9, 9], [4, 5, 6, 7]]
    plens = [0, 1, 2, 3, 1]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    logits = rng.normal(0, 2, (len(hists), V)).astype(np.float32)
    w = W.Workload("forced", _forced_params(V, mode="greedy"), logits, ids, off, np.array(plens, np.int32),
                   rng.random(len(hists), dtype=np.float32))
    gpu, _, _ = compare_select(w)
    assert gpu[0] == -1
    # every token suppressed: the filter value everywhere
    w2 = W.random_case(15, B=4, V=10000, mode="greedy", suppress_tokens=list(range(10000)))
    gpu2, _, _ = compare_select(w2)
    assert all(g == 0 for g in gpu2 if g != -1)


def test_split_greedy_unaligned_rows():
    # logits that start 4 bytes past a 16-byte boundary: the split reads element by element
    import torch
    import logits_processing_token_gb300 as tg
    w = W.random_case(16, B=3, V=50272, dtype="f32", mode="greedy", L_max=40, repetition_penalty=1.4)
    dev = to_device(w)
    buf = torch.empty(w.B * w.V + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(dev["logits"].reshape(-1))
    shifted = buf[1:].view(w.B, w.V)
    assert shifted.data_ptr() % 16 == 4
    cfg = tg.Config(**w.params)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    tg.tg_select(shifted, dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg, dev["uniforms"], out)
    torch.cuda.synchronize()
    ora, _ = oracle_select(w)
    assert [int(x) for x in out.cpu().numpy()] == [int(x) for x in ora]
