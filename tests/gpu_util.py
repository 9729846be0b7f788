"""Helpers for the GPU parity tests: move a workload to the device, run the
C-ABI entry points, and compare with the CPU oracle."""
import numpy as np

from oracle import tg_oracle as O


def torch_mod():
    import torch
    return torch


def to_device(w):
    torch = torch_mod()
    if w.params.get("logits_dtype", "f32") == "bf16":
        logits = torch.from_numpy(np.ascontiguousarray(w.logits).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        logits = torch.from_numpy(np.ascontiguousarray(w.logits)).cuda()
    d = dict(
        logits=logits,
        hist_ids=torch.from_numpy(np.ascontiguousarray(w.hist_ids, np.int32)).cuda(),
        hist_offsets=torch.from_numpy(np.ascontiguousarray(w.hist_offsets, np.int64)).cuda(),
        prompt_lens=torch.from_numpy(np.ascontiguousarray(w.prompt_lens, np.int32)).cuda(),
        uniforms=torch.from_numpy(np.ascontiguousarray(w.uniforms, np.float32)).cuda(),
    )
    return d


def gpu_select(w, cfg=None, dev=None):
    import logits_processing_token_gb300 as tg
    torch = torch_mod()
    cfg = cfg or tg.Config(**w.params)
    dev = dev or to_device(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    tg.tg_select(dev["logits"], dev["hist_ids"], dev["hist_offsets"], dev["prompt_lens"], cfg,
                 dev["uniforms"], out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), cfg


def oracle_select(w, rows=None):
    p = O.Params(**w.params)
    return O.select(w.logits, w.hist_ids, w.hist_offsets, w.prompt_lens, p, w.uniforms, rows=rows)


def acceptable_tokens(w, b):
    """Tokens a correct implementation may return on a row the oracle flags
    as a boundary row: the draw with the top-p cut moved by one token either
    way, and with u moved by 2e-6 either way."""
    p = O.Params(**w.params)
    h = list(w.history(b))
    x = O.upcast_row(w.logits[b], p.logits_dtype)
    s, _, _ = O.process_row(x, h, int(w.prompt_lens[b]), p)
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


def compare_select(w, rows=None, max_boundary_frac=0.06):
    """GPU vs oracle on the listed rows (all by default).  Ids must be equal,
    except on rows the oracle flags as within 1e-6 of a top-p cut or a CDF
    step; there the GPU's id must be one the oracle gives with the cut or u
    nudged across that boundary.  Flagged rows are counted and bounded."""
    gpu, cfg = gpu_select(w)
    rows = list(range(w.B)) if rows is None else list(rows)
    ora, infos = oracle_select(w, rows)
    boundary = 0
    bad = []
    for r, o, info in zip(rows, ora, infos):
        if info.topp_boundary or info.u_boundary:
            boundary += 1
            if int(gpu[r]) != int(o) and int(gpu[r]) not in acceptable_tokens(w, r):
                bad.append((r, int(gpu[r]), int(o), "boundary"))
            continue
        if int(gpu[r]) != int(o):
            bad.append((r, int(gpu[r]), int(o)))
    assert not bad, "mismatching rows (row, gpu, oracle): %s" % bad[:10]
    assert boundary <= max(3, max_boundary_frac * len(rows)), boundary
    return gpu, cfg, boundary
