"""tg_verify_noalloc: the verify step for callers that may not allocate device
memory (for example a serving engine whose memory pool owns all of HBM, or a
pipelined decode step where cudaMalloc would synchronise the device).

It must give the same outputs as tg_verify on the same inputs, on two calls
in a row (its device-side tickets are shared between calls and cleared by
each call).  Called through the C ABI with ctypes.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from logits_processing_token_gb300 import _build
    _build.build()
    import logits_processing_token_gb300 as tg
    return tg.load_library()


def _case(B, K, V, mode, seed):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    greedy = tgt.argmax(-1)[:, :K]
    agree = rng.random((B, K)) < 0.6
    cand = np.where(agree, greedy, (greedy + 1 + rng.integers(0, V - 1, (B, K))) % V).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    return tgt, cand, u


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_noalloc_matches_tg_verify_twice(lib, mode):
    import torch
    import logits_processing_token_gb300 as tg
    B, K, V = 8, 5, 50_272
    settings = dict(vocab=V, mode=mode, temperature=0.8 if mode == "sample" else 1.0, top_p=0.9)
    cfg = tg.Config(**settings, max_batch=64)
    params, keep = tg.make_params(**settings)
    for call in range(2):
        tgt, cand, u = _case(B, K, V, mode, 100 + call)
        t = torch.from_numpy(tgt).cuda()
        c = torch.from_numpy(cand).cuda()
        uu = torch.from_numpy(u).cuda()
        ref_m = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        ref_n = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
        tg.tg_verify(t, c, K, cfg, uu, ref_m, ref_n)
        out_m = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        out_n = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.tg_verify_noalloc(ctypes.c_void_p(t.data_ptr()), B, V, ctypes.c_void_p(c.data_ptr()), K,
                                   ctypes.byref(params), ctypes.c_void_p(uu.data_ptr()),
                                   ctypes.c_void_p(out_m.data_ptr()), ctypes.c_void_p(out_n.data_ptr()), stream)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        torch.cuda.synchronize()
        # integer outputs: the tolerance is exact equality
        assert np.array_equal(out_m.cpu().numpy(), ref_m.cpu().numpy()), call
        assert np.array_equal(out_n.cpu().numpy(), ref_n.cpu().numpy()), call


def test_noalloc_rejects_batch_above_maximum(lib):
    import torch
    import logits_processing_token_gb300 as tg
    B, K, V = tg.TG_NOALLOC_MAX_BATCH + 1, 1, 64
    params, keep = tg.make_params(vocab=V)
    t = torch.zeros((B, K + 1, V), device="cuda")
    c = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    om = torch.zeros(B, dtype=torch.int32, device="cuda")
    on = torch.zeros((B, K + 1), dtype=torch.int32, device="cuda")
    st = lib.tg_verify_noalloc(ctypes.c_void_p(t.data_ptr()), B, V, ctypes.c_void_p(c.data_ptr()), K,
                               ctypes.byref(params), None, ctypes.c_void_p(om.data_ptr()),
                               ctypes.c_void_p(on.data_ptr()), None)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_noalloc_after_timeout(lib):
    # a launch whose bounded wait ran out writes -1 to the batch rows it did not
    # finish (no status word is reported here); the next call is exact again
    import torch
    import logits_processing_token_gb300 as tg
    B, K, V = 8, 5, 50_272
    settings = dict(vocab=V, mode="greedy")
    cfg = tg.Config(**settings, max_batch=64)
    params, keep = tg.make_params(**settings)
    tgt, cand, u = _case(B, K, V, "greedy", 7)
    t = torch.from_numpy(tgt).cuda()
    c = torch.from_numpy(cand).cuda()
    uu = torch.from_numpy(u).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        om = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        on = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
        st = lib.tg_verify_noalloc(ctypes.c_void_p(t.data_ptr()), B, V, ctypes.c_void_p(c.data_ptr()), K,
                                   ctypes.byref(params), ctypes.c_void_p(uu.data_ptr()),
                                   ctypes.c_void_p(om.data_ptr()), ctypes.c_void_p(on.data_ptr()), stream)
        assert st == tg.TG_OK
        torch.cuda.synchronize()
        return om.cpu().numpy(), on.cpu().numpy()

    tg.tg_set_wait_limit(1)
    try:
        om, _ = call()
    finally:
        tg.tg_set_wait_limit(0)
    assert (om == -1).any() and not (om == -9).any()
    om2, on2 = call()
    ref_m = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ref_n = torch.full((B, K + 1), -9, dtype=torch.int32, device="cuda")
    tg.tg_verify(t, c, K, cfg, uu, ref_m, ref_n)
    torch.cuda.synchronize()
    assert np.array_equal(om2, ref_m.cpu().numpy()) and np.array_equal(on2, ref_n.cpu().numpy())
