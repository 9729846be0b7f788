"""The roofline numerator of bench.py on CPU: the algorithmic bytes of one
step are the logits of every row whose token depends on them (not empty, not
forced by forced_bos / forced_eos), each row's history, and 20 bytes per row
of offsets, prompt length, uniform and output id (plus the closing offset)."""
import numpy as np

import bench
from logits_processing_token_gb300 import workloads as W


def test_required_bytes_by_hand():
    V = 1000
    hists = [[], [5], [1, 2, 3], [4, 5, 6, 7], [8, 9]]
    plens = [0, 1, 1, 3, 2]
    ids, off = W._pack([np.array(h, np.int32) for h in hists])
    params = dict(vocab=V, logits_dtype="f32", mode="sample", forced_bos_token_id=3,
                  forced_eos_token_ids=[2], max_new_tokens=3)
    w = W.Workload("t", params, np.zeros((5, V), np.float32), ids, off, np.array(plens, np.int32),
                   np.zeros(5, np.float32))
    # row 0 empty; row 1 L == 1 (forced bos); row 2 L == P + max_new - 1 == 3 (forced eos);
    # rows 3 (L 4, P 3) and 4 (L 2, P 2) are not forced and read their logits
    got, n_read = bench.required_bytes(w)
    assert n_read == 2
    assert got == 2 * V * 4 + 4 * (0 + 1 + 3 + 4 + 2) + 5 * 20 + 8


def test_required_bytes_of_the_benchmark_step():
    w = W.config3()
    got, n_read = bench.required_bytes(w)
    # 32 of the 256 rows are forced-eos rows (b % 8 == 1): 224 rows read 151,936 bf16 logits each
    assert n_read == 224
    assert got == 224 * 151_936 * 2 + 4 * int(w.hist_offsets[-1]) + 256 * 20 + 8 == 68_867_928


def test_graph_timing_reports_a_failure_instead_of_raising():
    # without a usable GPU the capture cannot start: the line gets the reason
    import torch
    if torch.cuda.is_available():
        import pytest
        pytest.skip("a GPU is present: the failure path is not reachable this way")
    got = bench.graph_timing(lambda i: None, 256, 10)
    assert set(got) == {"unavailable"} and got["unavailable"]
