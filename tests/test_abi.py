"""The C-ABI library builds, loads and exports what include/tg.h declares.
No GPU needed: only host-side entry points are called."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import logits_processing_token_gb300 as tg
from logits_processing_token_gb300 import _build
from oracle import tg_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tg.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(tg.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(r"\sT\s%s$" % n, out, re.M), n


def test_params_layout_matches_c(lib):
    # compile the header as plain C and compare sizeof/offsetof with ctypes
    fields = [f for f, _ in tg.tg_params._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"tg.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(tg_params));\n'
    for f in fields:
        src += 'printf("%%zu\\n", offsetof(tg_params, %s));\n' % f
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), c, "-o", exe])
        vals = [int(x) for x in subprocess.check_output([exe]).split()]
    assert vals[0] == ctypes.sizeof(tg.tg_params)
    for f, off in zip(fields, vals[1:]):
        assert getattr(tg.tg_params, f).offset == off, f


def test_params_init_defaults(lib):
    p = tg.tg_params()
    lib.tg_params_init(ctypes.byref(p), 1234)
    assert p.vocab == 1234 and p.repetition_penalty == 1.0 and p.temperature == 1.0
    assert p.top_p == 1.0 and p.top_k == 0 and p.forced_bos_token_id == -1 and p.mode == tg.TG_GREEDY


def test_next_num_candidates_matches_oracle(lib):
    for K in range(1, 20):
        for n in range(0, K + 1):
            for kmax in (1, 8, 16, 64):
                assert tg.tg_next_num_candidates(K, n, kmax) == O.next_num_candidates(K, n, kmax)


def test_status_strings(lib):
    for s, name in ((0, "TG_OK"), (-1, "TG_ERR_INVALID_ARGUMENT"), (-2, "TG_ERR_UNSUPPORTED"),
                    (-3, "TG_ERR_CUDA"), (-4, "TG_ERR_OUT_OF_MEMORY")):
        assert tg.tg_status_string(s) == name


def test_config_create_rejects_bad_params_on_host(lib):
    # argument errors are caught before any device work
    bad = [dict(vocab=0), dict(vocab=tg.TG_MAX_VOCAB + 1), dict(vocab=10, top_p=0.0),
           dict(vocab=10, top_p=1.5), dict(vocab=10, temperature=0.0), dict(vocab=10, repetition_penalty=0.0),
           dict(vocab=10, suppress_tokens=[10]), dict(vocab=10, eos_token_ids=[-1]),
           dict(vocab=10, forced_bos_token_id=10), dict(vocab=10, forced_eos_token_ids=[1]),
           dict(vocab=10, top_k=-1), dict(vocab=10, eos_token_ids=list(range(9)))]
    for kw in bad:
        p, keep = tg.make_params(**kw)
        h = ctypes.c_void_p()
        st = lib.tg_config_create(ctypes.byref(p), ctypes.byref(h), None)
        want = tg.TG_ERR_UNSUPPORTED if kw.get("vocab", 0) > tg.TG_MAX_VOCAB else tg.TG_ERR_INVALID_ARGUMENT
        assert st == want, kw


def test_null_arguments_rejected(lib):
    assert lib.tg_select(None, 1, 10, None, None, None, None, None, None, None) == tg.TG_ERR_INVALID_ARGUMENT
    assert lib.tg_verify(None, 1, 10, None, 1, None, None, None, None, None) == tg.TG_ERR_INVALID_ARGUMENT
    assert lib.tg_config_destroy(None) == tg.TG_ERR_INVALID_ARGUMENT


def test_binding_rejects_mis_shaped_tensors():
    """The C ABI takes raw pointers and cannot see buffer extents, so the
    binding checks shapes and element sizes before any call."""
    import types
    import torch
    import logits_processing_token_gb300 as tg
    cfg32 = types.SimpleNamespace(params=dict(vocab=64, logits_dtype="f32"), handle=None)
    cfg16 = types.SimpleNamespace(params=dict(vocab=64, logits_dtype="bf16"), handle=None)
    i32 = torch.int32
    # verify targets must be [B, K+1, V]: a flattened [B*(K+1), V] would make B too large
    with pytest.raises(ValueError, match=r"\[B, K\+1, V\]"):
        tg.tg_verify(torch.zeros(3 * 5, 64), torch.zeros(3, 4, dtype=i32), 4, cfg32, None,
                     torch.zeros(3, dtype=i32), torch.zeros(3, 5, dtype=i32))
    with pytest.raises(ValueError, match="out_next"):
        tg.tg_verify(torch.zeros(3, 5, 64), torch.zeros(3, 4, dtype=i32), 4, cfg32, None,
                     torch.zeros(3, dtype=i32), torch.zeros(3, 4, dtype=i32))
    with pytest.raises(ValueError, match="cand_ids"):
        tg.tg_verify(torch.zeros(3, 5, 64), torch.zeros(3, 3, dtype=i32), 4, cfg32, None,
                     torch.zeros(3, dtype=i32), torch.zeros(3, 5, dtype=i32))
    # element size and vocabulary must match the config
    with pytest.raises(ValueError, match="2-byte"):
        tg.tg_select(torch.zeros(2, 64), None, torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=i32),
                     cfg16, None, torch.zeros(2, dtype=i32))
    with pytest.raises(ValueError, match="vocab"):
        tg.tg_select(torch.zeros(2, 63), None, torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=i32),
                     cfg32, None, torch.zeros(2, dtype=i32))
    with pytest.raises(ValueError, match="hist_offsets"):
        tg.tg_select(torch.zeros(2, 64), None, torch.zeros(2, dtype=torch.int64), torch.zeros(2, dtype=i32),
                     cfg32, None, torch.zeros(2, dtype=i32))
    with pytest.raises(ValueError, match="out_ids"):
        tg.tg_select(torch.zeros(2, 64), None, torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=i32),
                     cfg32, None, torch.zeros(1, dtype=i32))
    with pytest.raises(ValueError, match="out_scores"):
        tg.tg_process(torch.zeros(2, 64), None, torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=i32),
                      cfg32, torch.zeros(2, 63))


def test_config_create_rejects_bad_processors_on_host(lib):
    # the task's processors: kind bias/set, sizes >= 1, at most 8 of them and 4,096 columns in all
    bad = [dict(processors=[(2, 4)]), dict(processors=[("bias", 0)]),
           dict(processors=[("bias", 1)] * (tg.TG_MAX_PROCESSORS + 1)),
           dict(processors=[("bias", tg.TG_MAX_STATE_COLS), ("set", 1)])]
    for kw in bad:
        p, keep = tg.make_params(vocab=10, **kw)
        h = ctypes.c_void_p()
        assert lib.tg_config_create(ctypes.byref(p), ctypes.byref(h), None) == tg.TG_ERR_INVALID_ARGUMENT, kw


def test_state_entry_points_reject_null_arguments(lib):
    assert lib.tg_select_state(None, 1, 10, None, None, None, None, None, None, None, None, None,
                               None) == tg.TG_ERR_INVALID_ARGUMENT
    assert lib.tg_process_state(None, 1, 10, None, None, None, None, None, None, None, None, None,
                                None) == tg.TG_ERR_INVALID_ARGUMENT


def test_binding_checks_the_state_shape():
    import types
    import torch
    cfg = types.SimpleNamespace(params=dict(vocab=64, logits_dtype="f32", processors=[("bias", 3), ("set", 2)]),
                                handle=None)
    i32 = torch.int32
    args = (torch.zeros(2, 64), None, torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=i32), cfg)
    with pytest.raises(ValueError, match="state_ids"):
        tg.tg_select_state(*args, torch.zeros(2, 4, dtype=i32), torch.zeros(2, 5), None, torch.zeros(2, dtype=i32))
    with pytest.raises(ValueError, match="state_values"):
        tg.tg_process_state(*args, torch.zeros(2, 5, dtype=i32), torch.zeros(2, 4), torch.zeros(2, 64))


def test_status_flags_agree_across_header_binding_and_kernels():
    # every status bit the kernels raise is declared in include/tg.h, with the
    # same value in the binding
    import re
    from logits_processing_token_gb300 import tg as T
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "tg.h")).read()
    declared = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define TG_FLAG_(\w+) (0x[0-9a-fA-F]+)u", hdr)}
    dev = open(os.path.join(root, "logits_processing_token_gb300", "csrc", "tg_device.cuh")).read()
    raised = {int(m.group(1), 16) for m in re.finditer(r"constexpr unsigned kFlag\w+ = (0x[0-9a-fA-F]+)u", dev)}
    assert raised == set(declared.values())
    for name, value in declared.items():
        assert getattr(T, "TG_FLAG_" + name) == value


def test_task_processor_header_compiles(tmp_path):
    # include/tg_custom.cuh instantiated with a functor, as a caller would build it
    from tests import custom_build
    out = os.path.join(str(tmp_path), "task_processor.o")
    r = subprocess.run(custom_build.nvcc_cmd(out, shared=False), capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
