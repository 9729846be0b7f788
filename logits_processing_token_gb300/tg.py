"""Python binding of libtg (include/tg.h): argument marshalling only.

Every step of the computation runs in the CUDA kernels of libtg.so.  This
module turns torch CUDA tensors into device pointers, passes the current
stream, and raises :class:`TGError` on a non-zero status.  It never computes
a result itself; if the library is missing it raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_uint32, c_uint64, c_void_p

from . import _build

TG_OK = 0
TG_ERR_INVALID_ARGUMENT = -1
TG_ERR_UNSUPPORTED = -2
TG_ERR_CUDA = -3
TG_ERR_OUT_OF_MEMORY = -4

TG_DTYPE_F32, TG_DTYPE_BF16 = 0, 1
TG_GREEDY, TG_SAMPLE = 0, 1

TG_FLAG_HISTORY_ID_OUT_OF_RANGE = 0x1
TG_FLAG_BAD_ROW = 0x2
TG_FLAG_SLOW_PATH = 0x4
TG_FLAG_TIMEOUT = 0x8
TG_FLAG_BAD_STATE = 0x10
TG_MAX_VOCAB = 1 << 18
TG_PROC_BIAS, TG_PROC_SET = 0, 1
TG_MAX_PROCESSORS = 8
TG_MAX_STATE_COLS = 4096

# Names of every entry point declared in include/tg.h.
EXPORTS = ("tg_params_init", "tg_config_create", "tg_config_destroy", "tg_select", "tg_select_logprobs", "tg_verify",
           "tg_process", "tg_query_status", "tg_clear_status", "tg_next_num_candidates",
           "tg_status_string", "tg_verify_noalloc", "tg_beam_step", "tg_beam_keep",
           "tg_verify_history", "tg_select_state", "tg_process_state", "tg_set_wait_limit", "tg_status_word",
           "tg_config_view", "tg_config_selection")
TG_NOALLOC_MAX_BATCH = 1024


class TGError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


class tg_params(ctypes.Structure):
    _fields_ = [
        ("vocab", c_int32),
        ("logits_dtype", c_int),
        ("mode", c_int),
        ("repetition_penalty", c_float),
        ("no_repeat_ngram_size", c_int32),
        ("bad_words_ids", POINTER(c_int32)),
        ("n_bad_words_ids", c_int32),
        ("suppress_tokens", POINTER(c_int32)),
        ("n_suppress_tokens", c_int32),
        ("begin_suppress_tokens", POINTER(c_int32)),
        ("n_begin_suppress_tokens", c_int32),
        ("eos_token_ids", POINTER(c_int32)),
        ("n_eos_token_ids", c_int32),
        ("min_length", c_int32),
        ("min_new_tokens", c_int32),
        ("forced_bos_token_id", c_int32),
        ("forced_eos_token_ids", POINTER(c_int32)),
        ("n_forced_eos_token_ids", c_int32),
        ("max_new_tokens", c_int32),
        ("temperature", c_float),
        ("top_k", c_int32),
        ("top_p", c_float),
        ("max_batch", c_int32),
        ("bad_word_seq_ids", POINTER(c_int32)),
        ("bad_word_seq_offsets", POINTER(c_int32)),
        ("n_bad_word_seqs", c_int32),
        ("renormalize_logits", c_int32),
        ("processor_kinds", POINTER(c_int32)),
        ("processor_sizes", POINTER(c_int32)),
        ("n_processors", c_int32),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None):
    """Load libtg.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError("libtg.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    lib.tg_params_init.argtypes = [POINTER(tg_params), c_int32]
    lib.tg_params_init.restype = None
    lib.tg_config_create.argtypes = [POINTER(tg_params), POINTER(c_void_p), c_void_p]
    lib.tg_status_word.argtypes = [c_void_p, POINTER(c_uint32)]
    lib.tg_status_word.restype = c_int
    lib.tg_config_destroy.argtypes = [c_void_p]
    lib.tg_select.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p]
    lib.tg_select_logprobs.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p]
    lib.tg_verify.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p]
    lib.tg_verify_history.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.tg_verify_history.restype = c_int
    lib.tg_verify_noalloc.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_int32, POINTER(tg_params), c_void_p,
                                      c_void_p, c_void_p, c_void_p]
    lib.tg_verify_noalloc.restype = c_int
    lib.tg_set_wait_limit.argtypes = [c_uint64]
    lib.tg_set_wait_limit.restype = c_int
    lib.tg_process.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_void_p, c_void_p]
    lib.tg_select_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.tg_select_state.restype = c_int
    lib.tg_process_state.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.tg_process_state.restype = c_int
    lib.tg_query_status.argtypes = [c_void_p, POINTER(c_uint32), POINTER(c_uint64)]
    lib.tg_clear_status.argtypes = [c_void_p]
    lib.tg_beam_step.argtypes = [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.tg_beam_step.restype = c_int
    lib.tg_beam_keep.argtypes = [c_void_p, c_int32]
    lib.tg_beam_keep.restype = c_int32
    lib.tg_next_num_candidates.argtypes = [c_int32, c_int32, c_int32]
    lib.tg_next_num_candidates.restype = c_int32
    lib.tg_status_string.argtypes = [c_int]
    lib.tg_status_string.restype = c_char_p
    for fn in ("tg_config_create", "tg_config_destroy", "tg_select", "tg_select_logprobs", "tg_verify", "tg_process",
               "tg_query_status", "tg_clear_status"):
        getattr(lib, fn).restype = c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().tg_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != TG_OK:
        raise TGError(fn, status)


def _ids(seq):
    seq = [int(t) for t in (seq or ())]
    arr = (c_int32 * max(1, len(seq)))(*seq) if seq else None
    return arr, len(seq)


def make_params(vocab: int, logits_dtype="f32", mode="greedy", repetition_penalty=1.0,
                no_repeat_ngram_size=0, bad_words_ids=(), suppress_tokens=(), begin_suppress_tokens=(),
                eos_token_ids=(), min_length=0, min_new_tokens=0, forced_bos_token_id=-1,
                forced_eos_token_ids=(), max_new_tokens=0, temperature=1.0, top_k=0, top_p=1.0,
                max_batch=0, bad_word_seqs=(), renormalize_logits=False, processors=()):
    """A filled tg_params plus the ctypes arrays its pointers refer to."""
    lib = load_library()
    p = tg_params()
    lib.tg_params_init(ctypes.byref(p), int(vocab))
    p.logits_dtype = {"f32": TG_DTYPE_F32, "bf16": TG_DTYPE_BF16}[logits_dtype] if isinstance(logits_dtype, str) else int(logits_dtype)
    p.mode = {"greedy": TG_GREEDY, "sample": TG_SAMPLE}[mode] if isinstance(mode, str) else int(mode)
    p.repetition_penalty = float(repetition_penalty)
    p.no_repeat_ngram_size = int(no_repeat_ngram_size)
    keep = []
    for name, seq in (("bad_words_ids", bad_words_ids), ("suppress_tokens", suppress_tokens),
                      ("begin_suppress_tokens", begin_suppress_tokens), ("eos_token_ids", eos_token_ids),
                      ("forced_eos_token_ids", forced_eos_token_ids)):
        arr, n = _ids(seq)
        keep.append(arr)
        setattr(p, name, ctypes.cast(arr, POINTER(c_int32)) if arr is not None else None)
        setattr(p, "n_" + name, n)
    p.min_length = int(min_length)
    p.min_new_tokens = int(min_new_tokens)
    p.forced_bos_token_id = int(forced_bos_token_id)
    p.max_new_tokens = int(max_new_tokens)
    p.temperature = float(temperature)
    p.top_k = int(top_k)
    p.top_p = float(top_p)
    p.max_batch = int(max_batch)
    p.renormalize_logits = 1 if renormalize_logits else 0
    # bad words of one or more tokens: ids back to back, then n + 1 offsets
    seqs = [list(map(int, s)) for s in bad_word_seqs]
    if seqs:
        flat = [t for s in seqs for t in s]
        offs = [0]
        for s in seqs:
            offs.append(offs[-1] + len(s))
        ids_arr, _ = _ids(flat)
        off_arr, _ = _ids(offs)
        keep += [ids_arr, off_arr]
        p.bad_word_seq_ids = ctypes.cast(ids_arr, POINTER(c_int32))
        p.bad_word_seq_offsets = ctypes.cast(off_arr, POINTER(c_int32))
        p.n_bad_word_seqs = len(seqs)
    # the task's processors: (kind, size) pairs, kind "bias" / "set" or TG_PROC_*
    procs = [(({"bias": TG_PROC_BIAS, "set": TG_PROC_SET}[k] if isinstance(k, str) else int(k)), int(n))
             for k, n in processors]
    if procs:
        kinds_arr, _ = _ids([k for k, _ in procs])
        sizes_arr, _ = _ids([n for _, n in procs])
        keep += [kinds_arr, sizes_arr]
        p.processor_kinds = ctypes.cast(kinds_arr, POINTER(c_int32))
        p.processor_sizes = ctypes.cast(sizes_arr, POINTER(c_int32))
        p.n_processors = len(procs)
    return p, keep


class Config:
    """Owns a tg_config* (tg_config_create / tg_config_destroy)."""

    def __init__(self, stream=None, **params):
        lib = load_library()
        p, keep = make_params(**params)
        h = c_void_p()
        # the uploads go on `stream` (a torch stream), or on the default stream
        st = c_void_p(stream.cuda_stream) if stream is not None else None
        _check("tg_config_create", lib.tg_config_create(ctypes.byref(p), ctypes.byref(h), st))
        self.handle = h
        self.params = dict(params)
        del keep

    def close(self):
        if self.handle:
            load_library().tg_config_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr(t, name, dtypes=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError("%s is required" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    return c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def _logit_dtypes():
    import torch
    return (torch.float32, torch.bfloat16, torch.int16, torch.uint16)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _check_logits(t, cfg, name):
    """The library reads rows of cfg's element type through a raw pointer:
    the tensor's element size must match it and its last dimension must be V."""
    want = 2 if cfg.params.get("logits_dtype", "f32") in ("bf16", 1) else 4
    _need(t.element_size() == want, "%s has %d-byte elements; the config expects %d-byte logits"
          % (name, t.element_size(), want))
    _need(int(t.shape[-1]) == int(cfg.params["vocab"]), "%s has %d columns; the config's vocab is %d"
          % (name, int(t.shape[-1]), int(cfg.params["vocab"])))


def _check_len(t, n, name):
    if t is not None:
        _need(t.numel() >= n, "%s holds %d elements; the call needs %d" % (name, t.numel(), n))


def tg_select(logits, hist_ids, hist_offsets, prompt_lens, cfg: Config, uniforms, out_ids, stream=None,
              out_logprobs=None):
    """logits [B, V]; hist_offsets [B+1]; prompt_lens [B]; uniforms [B] (sampling); out_ids [B];
    out_logprobs [B] f32 or None (given: tg_select_logprobs, the token's log-probability per row).
    The history ids that hist_offsets point at are not bounds-checked here: they live on the device."""
    import torch
    _need(logits.dim() == 2, "logits must be [B, V]")
    _check_logits(logits, cfg, "logits")
    B, V = int(logits.shape[0]), int(logits.shape[-1])
    _check_len(hist_offsets, B + 1, "hist_offsets")
    _check_len(prompt_lens, B, "prompt_lens")
    _check_len(uniforms, B, "uniforms")
    _check_len(out_ids, B, "out_ids")
    _check_len(out_logprobs, B, "out_logprobs")
    args = [_ptr(logits, "logits", _logit_dtypes()), B, V,
            _ptr(hist_ids, "hist_ids", (torch.int32,), allow_none=True) if hist_ids is not None and hist_ids.numel() else None,
            _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
            cfg.handle, _ptr(uniforms, "uniforms", (torch.float32,), allow_none=True),
            _ptr(out_ids, "out_ids", (torch.int32,))]
    lib = load_library()
    if out_logprobs is None:
        st = lib.tg_select(*args, _stream(stream))
        _check("tg_select", st)
    else:
        st = lib.tg_select_logprobs(*args, _ptr(out_logprobs, "out_logprobs", (torch.float32,)), _stream(stream))
        _check("tg_select_logprobs", st)
    return out_ids


def _state_cols(cfg):
    return sum(int(n) for _, n in cfg.params.get("processors", ()))


def tg_select_state(logits, hist_ids, hist_offsets, prompt_lens, cfg: Config, state_ids, state_values, uniforms,
                    out_ids, out_logprobs=None, stream=None):
    """tg_select with the config's task processors: state_ids int32 [B, S] and state_values f32
    [B, S] (S = the processors' columns); out_logprobs [B] f32 or None."""
    import torch
    _need(logits.dim() == 2, "logits must be [B, V]")
    _check_logits(logits, cfg, "logits")
    B, V = int(logits.shape[0]), int(logits.shape[-1])
    S = _state_cols(cfg)
    _check_len(hist_offsets, B + 1, "hist_offsets")
    _check_len(prompt_lens, B, "prompt_lens")
    _check_len(state_ids, B * S, "state_ids")
    _check_len(state_values, B * S, "state_values")
    _check_len(uniforms, B, "uniforms")
    _check_len(out_ids, B, "out_ids")
    _check_len(out_logprobs, B, "out_logprobs")
    st = load_library().tg_select_state(
        _ptr(logits, "logits", _logit_dtypes()), B, V,
        _ptr(hist_ids, "hist_ids", (torch.int32,), allow_none=True) if hist_ids is not None and hist_ids.numel() else None,
        _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
        cfg.handle, _ptr(state_ids, "state_ids", (torch.int32,)), _ptr(state_values, "state_values", (torch.float32,)),
        _ptr(uniforms, "uniforms", (torch.float32,), allow_none=True), _ptr(out_ids, "out_ids", (torch.int32,)),
        _ptr(out_logprobs, "out_logprobs", (torch.float32,), allow_none=True), _stream(stream))
    _check("tg_select_state", st)
    return out_ids


def tg_process_state(logits, hist_ids, hist_offsets, prompt_lens, cfg: Config, state_ids, state_values, out_scores,
                     out_banbits=None, out_probs=None, stream=None):
    """tg_process with the config's task processors (state as tg_select_state)."""
    import torch
    _need(logits.dim() == 2, "logits must be [B, V]")
    _check_logits(logits, cfg, "logits")
    B, V = int(logits.shape[0]), int(logits.shape[-1])
    S = _state_cols(cfg)
    _check_len(hist_offsets, B + 1, "hist_offsets")
    _check_len(prompt_lens, B, "prompt_lens")
    _check_len(state_ids, B * S, "state_ids")
    _check_len(state_values, B * S, "state_values")
    _check_len(out_scores, B * V, "out_scores")
    _check_len(out_banbits, B * ((V + 31) // 32), "out_banbits")
    _check_len(out_probs, B * V, "out_probs")
    st = load_library().tg_process_state(
        _ptr(logits, "logits", _logit_dtypes()), B, V,
        _ptr(hist_ids, "hist_ids", (torch.int32,)) if hist_ids is not None and hist_ids.numel() else None,
        _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
        cfg.handle, _ptr(state_ids, "state_ids", (torch.int32,)), _ptr(state_values, "state_values", (torch.float32,)),
        _ptr(out_scores, "out_scores", (torch.float32,)),
        _ptr(out_banbits, "out_banbits", (torch.int32, torch.uint32), allow_none=True),
        _ptr(out_probs, "out_probs", (torch.float32,), allow_none=True), _stream(stream))
    _check("tg_process_state", st)


def tg_beam_keep(cfg: Config, num_beams: int) -> int:
    """Candidates a prompt keeps per beam step: max(2, 1 + eos ids) * num_beams."""
    n = load_library().tg_beam_keep(cfg.handle, int(num_beams))
    _need(n > 0, "num_beams must be >= 1")
    return int(n)


def tg_beam_step(logits, beam_scores, hist_ids, hist_offsets, prompt_lens, cfg: Config, num_beams: int,
                 out_scores, out_tokens, out_beams, stream=None):
    """logits [P * num_beams, V]; beam_scores [P * num_beams] f32; hist_offsets [P * num_beams + 1];
    prompt_lens [P * num_beams]; out_scores f32, out_tokens and out_beams int32, each [P, keep]."""
    import torch
    _need(logits.dim() == 2, "logits must be [P * num_beams, V]")
    _check_logits(logits, cfg, "logits")
    R, V = int(logits.shape[0]), int(logits.shape[-1])
    nb = int(num_beams)
    _need(nb >= 1 and R % nb == 0, "the rows must be num_beams per prompt")
    P = R // nb
    keep = tg_beam_keep(cfg, nb)
    _check_len(beam_scores, R, "beam_scores")
    _check_len(hist_offsets, R + 1, "hist_offsets")
    _check_len(prompt_lens, R, "prompt_lens")
    for t, name in ((out_scores, "out_scores"), (out_tokens, "out_tokens"), (out_beams, "out_beams")):
        _check_len(t, P * keep, name)
    st = load_library().tg_beam_step(
        _ptr(logits, "logits", _logit_dtypes()), P, nb, V, _ptr(beam_scores, "beam_scores", (torch.float32,)),
        _ptr(hist_ids, "hist_ids", (torch.int32,), allow_none=True) if hist_ids is not None and hist_ids.numel() else None,
        _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
        cfg.handle, _ptr(out_scores, "out_scores", (torch.float32,)), _ptr(out_tokens, "out_tokens", (torch.int32,)),
        _ptr(out_beams, "out_beams", (torch.int32,)), _stream(stream))
    _check("tg_beam_step", st)
    return out_scores, out_tokens, out_beams


def tg_verify(target_logits, cand_ids, K: int, cfg: Config, uniforms, out_match, out_next, stream=None):
    """target_logits [B, K+1, V]; cand_ids [B, K]; uniforms [B, K+1] (sampling);
    out_match [B]; out_next [B, K+1]."""
    import torch
    _need(target_logits.dim() == 3 and int(target_logits.shape[1]) == int(K) + 1,
          "target_logits must be [B, K+1, V]")
    _check_logits(target_logits, cfg, "target_logits")
    B, V = int(target_logits.shape[0]), int(target_logits.shape[-1])
    _check_len(cand_ids, B * int(K), "cand_ids")
    _check_len(uniforms, B * (int(K) + 1), "uniforms")
    _check_len(out_match, B, "out_match")
    _check_len(out_next, B * (int(K) + 1), "out_next")
    st = load_library().tg_verify(
        _ptr(target_logits, "target_logits", _logit_dtypes()), B, V, _ptr(cand_ids, "cand_ids", (torch.int32,)),
        int(K), cfg.handle, _ptr(uniforms, "uniforms", (torch.float32,), allow_none=True),
        _ptr(out_match, "out_match", (torch.int32,)), _ptr(out_next, "out_next", (torch.int32,)), _stream(stream))
    _check("tg_verify", st)
    return out_match, out_next


def tg_verify_history(target_logits, cand_ids, K: int, hist_ids, hist_offsets, prompt_lens, cfg: Config, uniforms,
                      out_match, out_next, stream=None):
    """tg_verify with the processors at every position: position j of row b sees
    the row's history (hist_offsets [B+1], prompt_lens [B]) and its first j candidates."""
    import torch
    _need(target_logits.dim() == 3 and int(target_logits.shape[1]) == int(K) + 1,
          "target_logits must be [B, K+1, V]")
    _check_logits(target_logits, cfg, "target_logits")
    B, V = int(target_logits.shape[0]), int(target_logits.shape[-1])
    _check_len(cand_ids, B * int(K), "cand_ids")
    _check_len(hist_offsets, B + 1, "hist_offsets")
    _check_len(prompt_lens, B, "prompt_lens")
    _check_len(uniforms, B * (int(K) + 1), "uniforms")
    _check_len(out_match, B, "out_match")
    _check_len(out_next, B * (int(K) + 1), "out_next")
    st = load_library().tg_verify_history(
        _ptr(target_logits, "target_logits", _logit_dtypes()), B, V, _ptr(cand_ids, "cand_ids", (torch.int32,)),
        int(K),
        _ptr(hist_ids, "hist_ids", (torch.int32,), allow_none=True) if hist_ids is not None and hist_ids.numel() else None,
        _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
        cfg.handle, _ptr(uniforms, "uniforms", (torch.float32,), allow_none=True),
        _ptr(out_match, "out_match", (torch.int32,)), _ptr(out_next, "out_next", (torch.int32,)), _stream(stream))
    _check("tg_verify_history", st)
    return out_match, out_next


def tg_process(logits, hist_ids, hist_offsets, prompt_lens, cfg: Config, out_scores, out_banbits=None,
               out_probs=None, stream=None):
    import torch
    _need(logits.dim() == 2, "logits must be [B, V]")
    _check_logits(logits, cfg, "logits")
    B, V = int(logits.shape[0]), int(logits.shape[-1])
    _check_len(hist_offsets, B + 1, "hist_offsets")
    _check_len(prompt_lens, B, "prompt_lens")
    _check_len(out_scores, B * V, "out_scores")
    _check_len(out_banbits, B * ((V + 31) // 32), "out_banbits")
    _check_len(out_probs, B * V, "out_probs")
    st = load_library().tg_process(
        _ptr(logits, "logits", _logit_dtypes()), B, V,
        _ptr(hist_ids, "hist_ids", (torch.int32,)) if hist_ids is not None and hist_ids.numel() else None,
        _ptr(hist_offsets, "hist_offsets", (torch.int64,)), _ptr(prompt_lens, "prompt_lens", (torch.int32,)),
        cfg.handle, _ptr(out_scores, "out_scores", (torch.float32,)),
        _ptr(out_banbits, "out_banbits", (torch.int32, torch.uint32), allow_none=True),
        _ptr(out_probs, "out_probs", (torch.float32,), allow_none=True), _stream(stream))
    _check("tg_process", st)


def tg_query_status(cfg: Config):
    f, s = c_uint32(), c_uint64()
    _check("tg_query_status", load_library().tg_query_status(cfg.handle, ctypes.byref(f), ctypes.byref(s)))
    return int(f.value), int(s.value)


def tg_status_word(cfg: Config) -> int:
    """The sticky status bits (synchronous)."""
    f = c_uint32()
    _check("tg_status_word", load_library().tg_status_word(cfg.handle, ctypes.byref(f)))
    return int(f.value)


def tg_clear_status(cfg: Config):
    _check("tg_clear_status", load_library().tg_clear_status(cfg.handle))


def tg_set_wait_limit(cycles: int):
    """Testing: the select/verify kernels give up a bulk-copy wait after
    ``cycles`` SM cycles (0 restores the default of about one second)."""
    lib = load_library()
    _check("tg_set_wait_limit", lib.tg_set_wait_limit(int(cycles)))


def tg_next_num_candidates(K: int, n_match: int, K_max: int) -> int:
    return int(load_library().tg_next_num_candidates(int(K), int(n_match), int(K_max)))


def tg_status_string(status: int) -> str:
    return status_string(status)
