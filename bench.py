#!/usr/bin/env python
"""Benchmark of one token-selection step: tg_select over B=256 rows of
V=151,936 bf16 logits with the full processor chain (repetition penalty,
4-gram ban, 50 bad words, 100 suppressed ids, begin-suppress, min_length,
forced eos) and top_p 0.95 sampling.

One JSON line on stdout (rank 0).  ``value`` is whole-job rows/s with the
inputs resident in HBM; ``e2e`` is the same metric with host->device copies of
the inputs and the device->host read of the ids inside the timed region.
``--impl reference`` times the CPU oracle instead (the reference arm).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rows/s and logits GB/s (% of GB300 HBM peak) at B=256, V=151,936"
WORKLOAD = "tg_select: full processor chain + top_p=0.95 sampling, B=256, V=151,936 bf16 logits (synthetic N(0,2^2) + 8 on 1%), histories 1..2048"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph-captured timing")
    ap.add_argument("--beam", action="store_true",
                    help="time tg_beam_step (64 prompts x 4 beams over the same rows) instead of tg_select")
    ap.add_argument("--state", action="store_true",
                    help="time tg_select_state (the benchmark rows with a bias of 64 and a set of 32 state columns "
                         "per row) instead of tg_select")
    ap.add_argument("--logprobs", action="store_true",
                    help="time tg_select_logprobs (ids plus each token's log-probability) instead of tg_select")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device):
    """The largest of one float over all ranks (every rank gets it); the step
    time of a multi-GPU run is the slowest rank's."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, rows_per_rank, ms_per_step):
    """Rows per second over all ranks: every rank selects its own rows."""
    return world * rows_per_rank / (ms_per_step / 1000.0)


CSRC = os.path.join(ROOT, "logits_processing_token_gb300", "csrc")
PROFILE = os.path.join(ROOT, "profiles", "select_kernel_bf16_workload3.md")


def source_digest():
    """sha256 over the CUDA sources and the C header: names a kernel build."""
    import hashlib
    h = hashlib.sha256()
    files = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))
    for f in files + ["../../include/tg.h"]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch (read + write) from the committed ncu summary of
    this workload, if it was taken on the current sources; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None, None
    import re
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_traf = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_hash and m_traf):
        return None, None
    if m_hash.group(1) != source_digest():
        return None, "stale (sources changed since the capture)"
    return int(m_traf.group(1)), os.path.relpath(PROFILE, ROOT)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def required_bytes(w):
    """Bytes the method must move for one step: the logits of every row whose
    result depends on them (non-empty, not forced to a fixed token by
    forced_bos/forced_eos), plus each row's history, offsets, prompt length,
    uniform and output id."""
    p = w.params
    elt = 2 if p["logits_dtype"] == "bf16" else 4
    n_read = 0
    hist = 0
    for b in range(w.B):
        L = int(w.hist_offsets[b + 1] - w.hist_offsets[b])
        P = int(w.prompt_lens[b])
        hist += 4 * L
        forced = (p.get("forced_bos_token_id", -1) >= 0 and L == 1) or (
            len(p.get("forced_eos_token_ids", ())) > 0 and L == P + p.get("max_new_tokens", 0) - 1)
        if L > 0 and not forced:
            n_read += 1
    return n_read * w.V * elt + hist + w.B * 20 + 8, n_read


def graph_timing(launch, rows, steps):
    """The same step launched from a CUDA graph: `launch(i)` issues step i on
    the current stream; up to 20 consecutive steps (rotating over the logits
    copies) are captured once and the graph is replayed until about `steps`
    steps ran.  Any failure to capture or replay is reported, not raised."""
    import torch
    try:
        n_cap = max(1, min(20, steps))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(2):
                launch(i)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for i in range(n_cap):
                launch(i)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // n_cap)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * n_cap)
        return {"value": whole_job_rate(1, rows, ms), "unit": "rows/s", "ms_per_step": ms,
                "steps_per_graph": n_cap, "replays": reps}
    except Exception as e:  # reported in the line instead of ending the run
        return {"unavailable": "%s: %s" % (type(e).__name__, str(e)[:200])}


def cpu_baseline(w, seconds):
    """The oracle as it stands, timed on host cores over a bounded sample of rows."""
    from oracle import tg_oracle as O
    p = O.Params(**w.params)
    t0 = time.perf_counter()
    n = 0
    b = 0
    while True:
        O.select(w.logits, w.hist_ids, w.hist_offsets, w.prompt_lens, p, w.uniforms, rows=[b])
        n += 1
        b = (b + 1) % w.B
        el = time.perf_counter() - t0
        if el >= seconds or n >= 4 * w.B:
            break
    return {"value": n / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": "%d rows of the same workload (row-by-row numpy oracle, one thread), %.1f s" % (n, el)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from logits_processing_token_gb300 import workloads as W
    w = W.config3()
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    base = cpu_baseline(w, per_step * args.steps)
    val = base["value"]
    line = {"metric": METRIC, "value": val, "unit": "rows/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * w.B / val,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "B": w.B, "V": w.V, "logits_dtype": "bf16"},
            "cpu_baseline": base,
            "e2e": {"value": val, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from logits_processing_token_gb300 import _build
    _build.build()
    import logits_processing_token_gb300 as tg
    from logits_processing_token_gb300 import workloads as W

    w = W.config3(seed=1003 + 7919 * rank)
    B, V = w.B, w.V
    cfg = tg.Config(**w.params)
    # Enough distinct copies of the logits that consecutive steps never hit L2.
    row_bytes = B * V * 2
    n_sets = max(2, int(np.ceil(2.5 * L2_BYTES / row_bytes)))
    host_logits = torch.from_numpy(w.logits.view(np.int16))
    sets = [host_logits.cuda().view(torch.bfloat16) for _ in range(n_sets)]
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    u = torch.from_numpy(w.uniforms).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    lp = torch.empty(B, dtype=torch.float32, device="cuda") if args.logprobs else None
    stream = torch.cuda.current_stream()

    def step(i):
        tg.tg_select(sets[i % n_sets], hid, off, pl, cfg, u, out, stream=stream, out_logprobs=lp)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    tg.tg_clear_status(cfg)
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local, enabled=not args.no_clocks)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3 if clocks.proc else 0.0)
    # back to back, as a decode loop issues them (each launch may overlap the
    # previous one's tail through programmatic dependent launch)
    t_start.record(stream)
    for i in range(K):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    flags, slow_rows = tg.tg_query_status(cfg)
    total_ms = max_over_ranks(total_ms, world, "cuda")
    ms_per_step = total_ms / K
    value = whole_job_rate(world, B, ms_per_step)

    alg_bytes, n_read = required_bytes(w)
    # one select_kernel launch per step (B <= 512 rows per CTA): its average
    # duration over the timed region
    mean_launch_s = t_start.elapsed_time(t_end) / K / 1000.0
    traffic, traffic_src = profiled_traffic()
    peak, peak_kind = measured_peak()
    achieved = alg_bytes / mean_launch_s / 1e9
    nominal_gbs = B * V * 2 / (ms_per_step / 1000.0) / 1e9

    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "V": V, "logits_dtype": "bf16", "rows_per_gpu": B,
                       "parallelism": "replicas (rows independent, no collective)",
                       "l2": "inputs rotate over %d copies of the logits (%.0f MB) > L2" %
                             (n_sets, n_sets * row_bytes / 1e6),
                       "logprobs": bool(args.logprobs)},
            "logits_gbs": nominal_gbs, "logits_hbm_frac": nominal_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                         "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "bytes_per_launch": alg_bytes, "rows_reading_logits": n_read,
                         "kernel": "select_kernel<bf16>", "mean_launch_us": mean_launch_s * 1e6},
            "gpu_launches": K, "slow_path_rows": slow_rows, "status_flags": flags}
    if clk:
        line["clocks"] = clk

    if not args.no_e2e:
        # the public API from host buffers: H2D of every input, the call, D2H of the ids
        h_logits = host_logits.pin_memory()
        h_hid = torch.from_numpy(w.hist_ids).pin_memory()
        h_off = torch.from_numpy(w.hist_offsets).pin_memory()
        h_pl = torch.from_numpy(w.prompt_lens).pin_memory()
        h_u = torch.from_numpy(w.uniforms).pin_memory()
        h_out = torch.empty(B, dtype=torch.int32).pin_memory()
        h_lp = torch.empty(B, dtype=torch.float32).pin_memory() if lp is not None else None
        d_logits = torch.empty_like(h_logits, device="cuda")
        bi = sum(t.numel() * t.element_size() for t in (h_logits, h_hid, h_off, h_pl, h_u))
        bo = h_out.numel() * 4 + (h_lp.numel() * 4 if h_lp is not None else 0)

        def e2e_step():
            d_logits.copy_(h_logits, non_blocking=True)
            hid.copy_(h_hid, non_blocking=True)
            off.copy_(h_off, non_blocking=True)
            pl.copy_(h_pl, non_blocking=True)
            u.copy_(h_u, non_blocking=True)
            tg.tg_select(d_logits.view(torch.bfloat16), hid, off, pl, cfg, u, out, stream=stream, out_logprobs=lp)
            h_out.copy_(out, non_blocking=True)
            if lp is not None:
                h_lp.copy_(lp, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / args.e2e_steps
        e_ms = max_over_ranks(e_ms, world, "cuda")
        line["e2e"] = {"value": whole_job_rate(world, B, e_ms), "unit": "rows/s", "h2d_bytes_per_step": bi,
                       "d2h_bytes_per_step": bo, "ms_per_step": e_ms}

    if not args.no_graph and world == 1:
        # (at N = 1 only: a rank whose capture failed would leave the others in the max-over-ranks collective)
        line["graph"] = graph_timing(
            lambda i: tg.tg_select(sets[i % n_sets], hid, off, pl, cfg, u, out, out_logprobs=lp), B, K)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_beam(args):
    """One beam-search device step over the benchmark rows: 64 prompts x 4 beams."""
    import numpy as np
    import torch
    from logits_processing_token_gb300 import _build
    _build.build()
    import logits_processing_token_gb300 as tg
    from logits_processing_token_gb300 import workloads as W

    w = W.beam_workload()
    nb = w.extra["beams"]
    cfg = tg.Config(**w.params)
    row_bytes = w.B * w.V * 2
    n_sets = max(2, int(np.ceil(2.5 * L2_BYTES / row_bytes)))
    host_logits = torch.from_numpy(w.logits.view(np.int16))
    sets = [host_logits.cuda().view(torch.bfloat16) for _ in range(n_sets)]
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    bs = torch.from_numpy(w.extra["beam_scores"]).cuda()
    keep = tg.tg_beam_keep(cfg, nb)
    P = w.B // nb
    out_s = torch.empty((P, keep), dtype=torch.float32, device="cuda")
    out_t = torch.empty((P, keep), dtype=torch.int32, device="cuda")
    out_b = torch.empty((P, keep), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        tg.tg_beam_step(sets[i % n_sets], bs, hid, off, pl, cfg, nb, out_s, out_t, out_b, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    peak, peak_kind = measured_peak()
    alg = w.B * w.V * 2 + int(w.hist_ids.size) * 4 + w.B * 20
    achieved = alg / (ms / 1000.0) / 1e9
    line = {"metric": "beam rows/s (one beam-search device step)", "value": w.B / (ms / 1000.0), "unit": "rows/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "tg_beam_step: %d prompts x %d beams over the benchmark rows, V=151,936 bf16, "
                                   "full processor chain, keep %d per prompt" % (P, nb, keep),
                       "l2": "inputs rotate over %d copies of the logits > L2" % n_sets},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "bytes_per_launch": alg, "kernel": "beam_kernel<bf16>", "traffic": None},
            "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def run_state(args):
    """tg_select_state over the benchmark rows with the task's processors: a
    bias of 64 and a set of 32 state columns per row (half of a row's ids from
    its history)."""
    import numpy as np
    import torch
    from logits_processing_token_gb300 import _build
    _build.build()
    import logits_processing_token_gb300 as tg
    from logits_processing_token_gb300 import workloads as W

    procs = (("bias", 64), ("set", 32))
    w = W.config3()
    w.params["processors"] = procs
    hot = [np.asarray(w.history(b)) for b in range(w.B)]
    st_ids, st_vals = W.processor_state(5, w.B, w.V, procs, hot=hot)
    cfg = tg.Config(**w.params)
    row_bytes = w.B * w.V * 2
    n_sets = max(2, int(np.ceil(2.5 * L2_BYTES / row_bytes)))
    host_logits = torch.from_numpy(w.logits.view(np.int16))
    sets = [host_logits.cuda().view(torch.bfloat16) for _ in range(n_sets)]
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    u = torch.from_numpy(w.uniforms).cuda()
    sid = torch.from_numpy(st_ids).cuda()
    sval = torch.from_numpy(st_vals).cuda()
    out = torch.empty(w.B, dtype=torch.int32, device="cuda")
    lp = torch.empty(w.B, dtype=torch.float32, device="cuda") if args.logprobs else None
    stream = torch.cuda.current_stream()

    def step(i):
        tg.tg_select_state(sets[i % n_sets], hid, off, pl, cfg, sid, sval, u, out, out_logprobs=lp, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    tg.tg_clear_status(cfg)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    flags, slow_rows = tg.tg_query_status(cfg)
    peak, peak_kind = measured_peak()
    alg, _ = required_bytes(w)
    alg += int(st_ids.size) * 8
    achieved = alg / (ms / 1000.0) / 1e9
    line = {"metric": "rows/s with the task's processors (tg_select_state)", "value": w.B / (ms / 1000.0),
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD + "; processors bias 64 + set 32 state columns per row",
                       "logprobs": bool(args.logprobs),
                       "l2": "inputs rotate over %d copies of the logits > L2" % n_sets},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "bytes_per_step": alg,
                         "kernel": "select_kernel<bf16> (state ids marked), then state_kernel<bf16> on the rows it "
                                   "defers (forced rows here)", "traffic": None},
            "gpu_launches": 2 * args.steps, "slow_path_rows": slow_rows, "status_flags": flags}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.beam:
        run_beam(args)
    elif args.state:
        run_state(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
