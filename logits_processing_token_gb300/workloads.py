"""Seeded synthetic workloads for token selection and verify.

Only input generation lives here: random logits, ragged histories, prompt
lengths, uniforms and the generation settings of each workload.  None of the
selection arithmetic is here; where a workload needs a selected token (the
verify candidates that agree with the target's greedy choice), the caller
passes it in.

Workloads (numpy ``default_rng(seed)``, seed = 1000 + workload number):

1. greedy, B=1, V=50,272 fp32 N(0, 2^2); a 64-token history (uniform ids),
   prompt 48; repetition_penalty 1.2, no_repeat_ngram_size 3, eos 2,
   min_new_tokens 20.
2. sampling, B=64, V=32,000 fp32 N(0, 3^2); histories of 16..512 tokens with
   prompts of 8..min(256, L-1); each row repeats a planted 3-gram (a, b, c)
   and ends with (a, b); temperature 0.7, top_k 50, top_p 0.9,
   no_repeat_ngram_size 3.
3. sampling, B=256, V=151,936 bf16 N(0, 2^2) plus 8 on 1% of entries;
   histories of 1..2048 tokens with 0..255 new tokens; the full processor
   chain (repetition_penalty 1.1, no_repeat_ngram_size 4, 50 bad words, 100
   suppressed ids, begin_suppress [eos], min_length 64, forced eos at
   prompt + 256 - 1), top_p 0.95.  Rows b % 8 == 0..4 force the begin-suppress,
   forced-eos, min-length, one-token and planted-4-gram cases.
4. verify, B in {1, 8, 32}, K in 1..16, target fp32 N(0, 2^2)
   [B, K+1, 50,272]; candidate j agrees with the target's greedy token with
   probability 0.6, else is another random id.
5. sampling, B=1024, V=262,144 fp32 Student-t (nu=3) times 2; histories of
   256..4096 tokens drawn Zipf(1.1) over a seeded permutation of the
   vocabulary; repetition_penalty 1.3, no_repeat_ngram_size 4,
   min_new_tokens 8, top_p 0.9.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

EOS = 2


@dataclass
class Workload:
    name: str
    params: dict
    logits: np.ndarray            # [B, V] float32, or uint16 bf16 bits
    hist_ids: np.ndarray          # int32, all rows' histories back to back
    hist_offsets: np.ndarray      # int64 [B+1]
    prompt_lens: np.ndarray       # int32 [B]
    uniforms: np.ndarray          # float32 [B]
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.prompt_lens.shape[0])

    @property
    def V(self) -> int:
        return int(self.params["vocab"])

    def history(self, b: int) -> np.ndarray:
        return self.hist_ids[int(self.hist_offsets[b]):int(self.hist_offsets[b + 1])]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to the nearest bfloat16 (ties to even); bits out."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _pack(histories):
    lens = np.array([len(h) for h in histories], dtype=np.int64)
    off = np.zeros(len(histories) + 1, dtype=np.int64)
    np.cumsum(lens, out=off[1:])
    ids = (np.concatenate([np.asarray(h, np.int32) for h in histories])
           if len(histories) and off[-1] > 0 else np.zeros(0, np.int32))
    return ids.astype(np.int32), off


def _normal(rng, shape, sigma):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def config1(B: int = 1, V: int = 50_272, seed: int = 1001) -> Workload:
    rng = np.random.default_rng(seed)
    logits = _normal(rng, (B, V), 2.0)
    hists = [rng.integers(0, V, 64).astype(np.int32) for _ in range(B)]
    ids, off = _pack(hists)
    params = dict(vocab=V, logits_dtype="f32", mode="greedy", repetition_penalty=1.2,
                  no_repeat_ngram_size=3, eos_token_ids=[EOS], min_new_tokens=20)
    return Workload("greedy B=%d V=%d fp32" % (B, V), params, logits, ids, off,
                    np.full(B, 48, np.int32), np.zeros(B, np.float32))


def config2(B: int = 64, V: int = 32_000, seed: int = 1002) -> Workload:
    rng = np.random.default_rng(seed)
    logits = _normal(rng, (B, V), 3.0)
    hists, plens = [], []
    for _ in range(B):
        L = int(rng.integers(16, 513))
        P = int(rng.integers(8, min(256, L - 1) + 1))
        h = rng.integers(0, V, L).astype(np.int32)
        a, b, c = (int(t) for t in rng.integers(0, V, 3))
        j = int(rng.integers(0, L - 4))           # planted (a, b, c) ends before L-2
        h[j:j + 3] = (a, b, c)
        h[L - 2:] = (a, b)
        hists.append(h)
        plens.append(P)
    ids, off = _pack(hists)
    params = dict(vocab=V, logits_dtype="f32", mode="sample", temperature=0.7, top_k=50,
                  top_p=0.9, no_repeat_ngram_size=3, eos_token_ids=[EOS])
    return Workload("sample T=0.7 k=50 p=0.9 B=%d V=%d fp32" % (B, V), params, logits, ids,
                    off, np.array(plens, np.int32), rng.random(B, dtype=np.float32))


def config3(B: int = 256, V: int = 151_936, seed: int = 1003, L_max: int = 2048) -> Workload:
    rng = np.random.default_rng(seed)
    x = _normal(rng, (B, V), 2.0)
    x += np.float32(8.0) * (rng.random((B, V), dtype=np.float32) < np.float32(0.01))
    logits = f32_to_bf16_bits(x)
    del x
    pool = rng.permutation(np.arange(V, dtype=np.int32)[np.arange(V) != EOS])
    bad, sup = pool[:50].copy(), pool[50:150].copy()
    max_new = 256
    hists, plens = [], []
    for b in range(B):
        kind = b % 8
        if kind == 1:                                  # forced eos: new = max_new - 1
            P = int(rng.integers(1, max(2, L_max - max_new + 2)))
            L = P + max_new - 1
        elif kind == 2:                                # below min_length
            L = int(rng.integers(1, 64))
            P = L - int(rng.integers(0, min(255, L - 1) + 1))
        elif kind == 3:                                # a one-token row
            L, P = 1, 1
        else:
            L = int(rng.integers(1, L_max + 1))
            new = 0 if kind == 0 else int(rng.integers(0, min(255, L - 1) + 1))
            P = L - new
        h = rng.integers(0, V, L).astype(np.int32)
        if kind == 4 and L >= 9:                       # planted 4-gram that bans its 4th token
            g = rng.integers(0, V, 4).astype(np.int32)
            j = int(rng.integers(0, L - 7))
            h[j:j + 4] = g
            h[L - 3:] = g[:3]
        hists.append(h)
        plens.append(P)
    ids, off = _pack(hists)
    params = dict(vocab=V, logits_dtype="bf16", mode="sample", repetition_penalty=1.1,
                  no_repeat_ngram_size=4, bad_words_ids=bad.tolist(),
                  suppress_tokens=sup.tolist(), begin_suppress_tokens=[EOS],
                  eos_token_ids=[EOS], min_length=64, forced_eos_token_ids=[EOS],
                  max_new_tokens=max_new, top_p=0.95)
    return Workload("full chain top_p=0.95 B=%d V=%d bf16" % (B, V), params, logits, ids,
                    off, np.array(plens, np.int32), rng.random(B, dtype=np.float32))


def config4(B: int = 8, K: int = 5, V: int = 50_272, mode: str = "greedy",
            seed: int = 1004) -> Workload:
    """Verify inputs.  ``extra`` holds target [B, K+1, V], the agree mask and the
    random offsets that make a disagreeing candidate; build the candidates with
    :func:`make_candidates` once the target's greedy tokens are known."""
    rng = np.random.default_rng(seed + 97 * B + K)
    target = _normal(rng, (B, K + 1, V), 2.0)
    agree = rng.random((B, K)) < 0.6
    offs = rng.integers(0, V - 1, (B, K)).astype(np.int64)
    params = dict(vocab=V, logits_dtype="f32", mode=mode)
    w = Workload("verify %s B=%d K=%d V=%d fp32" % (mode, B, K, V), params,
                 target.reshape(B * (K + 1), V), np.zeros(0, np.int32),
                 np.zeros(B + 1, np.int64), np.zeros(B, np.int32),
                 rng.random((B, K + 1), dtype=np.float32))
    w.extra = dict(target=target, K=K, agree=agree, offsets=offs)
    return w


def make_candidates(greedy_ids: np.ndarray, agree: np.ndarray, offsets: np.ndarray,
                    V: int) -> np.ndarray:
    """Candidate j is the target's greedy token where ``agree``, else a
    different token (the greedy token shifted by 1 + offset, modulo V)."""
    g = np.asarray(greedy_ids, np.int64)
    other = (g + 1 + offsets) % V
    return np.where(agree, g, other).astype(np.int32)


def _zipf_ranks(rng, n, V, s=1.1):
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    return np.minimum(np.searchsorted(cdf, rng.random(n), side="right"), V - 1)


def config5(B: int = 1024, V: int = 262_144, seed: int = 1005, L_min: int = 256,
            L_max: int = 4096) -> Workload:
    rng = np.random.default_rng(seed)
    logits = np.empty((B, V), np.float32)
    step = 64
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        logits[b0:b1] = rng.standard_t(3, size=(b1 - b0, V)).astype(np.float32) * np.float32(2.0)
    perm = rng.permutation(V).astype(np.int32)
    hists, plens = [], []
    for _ in range(B):
        L = int(rng.integers(L_min, L_max + 1))
        P = int(rng.integers(1, L + 1))
        hists.append(perm[_zipf_ranks(rng, L, V)])
        plens.append(P)
    ids, off = _pack(hists)
    params = dict(vocab=V, logits_dtype="f32", mode="sample", repetition_penalty=1.3,
                  no_repeat_ngram_size=4, eos_token_ids=[EOS], min_new_tokens=8,
                  temperature=1.0, top_k=0, top_p=0.9)
    return Workload("top_p=0.9 B=%d V=%d fp32 student-t" % (B, V), params, logits, ids, off,
                    np.array(plens, np.int32), rng.random(B, dtype=np.float32))


def random_case(seed: int, B: int, V: int, dtype: str = "f32", mode: str = "sample",
                L_max: int = 64, **overrides) -> Workload:
    """A small random case for edge coverage: ragged histories (some empty),
    ids that repeat often (so n-gram bans fire), scores with ties."""
    rng = np.random.default_rng(seed)
    x = (rng.integers(-40, 40, (B, V)) * 0.25).astype(np.float32)
    logits = f32_to_bf16_bits(x) if dtype == "bf16" else x
    hists, plens = [], []
    alpha = max(2, min(V, 6))
    for _ in range(B):
        L = int(rng.integers(0, L_max + 1))
        h = rng.integers(0, alpha, L).astype(np.int32) * max(1, V // alpha)
        hists.append(np.minimum(h, V - 1).astype(np.int32))
        plens.append(int(rng.integers(0, L + 1)) if L else 0)
    ids, off = _pack(hists)
    params = dict(vocab=V, logits_dtype=dtype, mode=mode)
    params.update(overrides)
    return Workload("random seed=%d B=%d V=%d %s" % (seed, B, V, dtype), params, logits, ids,
                    off, np.array(plens, np.int32), rng.random(B, dtype=np.float32))


def beam_workload(prompts: int = 64, beams: int = 4, V: int = 151_936, seed: int = 1006, L_max: int = 2048,
                  first_step: bool = False) -> Workload:
    """A beam-search step over the benchmark workload's rows: prompts * beams
    rows of its logits, histories and processors (temperature, top_k and top_p
    do not apply to beam search).  Beam scores are running sums of
    log-probabilities: N(-12, 3^2) per beam, or (first step) 0 for beam 0 and
    -1e9 for the others; they and the beam count are in ``extra``."""
    w = config3(B=prompts * beams, V=V, seed=seed, L_max=L_max)
    rng = np.random.default_rng(seed + 1)
    if first_step:
        bs = np.tile(np.array([0.0] + [-1e9] * (beams - 1), np.float32), prompts)
    else:
        bs = (rng.standard_normal(prompts * beams) * 3.0 - 12.0).astype(np.float32)
    w.name = "beam step %d prompts x %d beams V=%d bf16" % (prompts, beams, V)
    w.extra["beam_scores"] = bs
    w.extra["beams"] = beams
    return w


def processor_state(seed: int, rows: int, V: int, processors, fill: float = 0.6, hot=None,
                    set_removed: float = 0.3, sigma: float = 3.0):
    """A state for the task's processors, one row per logits row: for each
    (kind, size) processor, about fill * size distinct ids per row in
    ascending order followed by -1 padding, half of them (when ``hot`` gives
    each row's preferred ids) drawn from hot[r], the rest uniform over
    [0, V).  Values are N(0, sigma^2); a "set" entry is the filter value
    (-FLT_MAX, a removal) with probability ``set_removed``.  Returns
    (ids int32 [rows, S], values f32 [rows, S])."""
    rng = np.random.default_rng(seed)
    S = sum(int(n) for _, n in processors)
    ids = np.full((rows, S), -1, np.int32)
    vals = np.zeros((rows, S), np.float32)
    neg_max = -np.finfo(np.float32).max
    for r in range(rows):
        col = 0
        for kind, size in processors:
            size = int(size)
            m = min(int(rng.binomial(size, fill)), V)
            pool = set()
            if hot is not None and len(hot[r]):
                hr = np.asarray(hot[r])
                take = rng.choice(hr.size, size=min(hr.size, m // 2 + 1), replace=False)
                pool.update(int(hr[q]) for q in take)
            while len(pool) < m:
                pool.add(int(rng.integers(0, V)))
            chosen = sorted(int(t) for t in rng.permutation(sorted(pool))[:m])
            ids[r, col:col + len(chosen)] = chosen
            v = (rng.standard_normal(len(chosen)) * sigma).astype(np.float32)
            if kind in ("set", 1):
                v[rng.random(len(chosen)) < set_removed] = neg_max
            vals[r, col:col + len(chosen)] = v
            col += size
    return ids, vals
