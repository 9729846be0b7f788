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
    ap.add_argument("--cpu-seconds", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph-captured timing")
    ap.add_argument("--quick", action="store_true", help="the headline workload only (no other configurations)")
    ap.add_argument("--config", type=int, choices=[3, 5], default=3,
                    help="5: time config 5 (B=1,024, V=262,144 f32, top_p 0.9) as the line's workload instead")
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


def cpu_baseline_1core(w, seconds):
    """The oracle as it stands, on one host core, over a bounded sample of rows."""
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
            "sample": "%d rows of the same workload (row-by-row numpy oracle, one process), %.1f s" % (n, el)}


_OW = None


def _oracle_init(shm_name, shape, dtype, hist_ids, hist_offsets, prompt_lens, params, uniforms):
    global _OW
    import numpy as np
    from multiprocessing import shared_memory
    from oracle import tg_oracle as O
    shm = shared_memory.SharedMemory(name=shm_name)
    logits = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    _OW = (shm, logits, hist_ids, hist_offsets, prompt_lens, O.Params(**params), uniforms)


def _oracle_rows(rows):
    from oracle import tg_oracle as O
    _, logits, hid, off, pl, p, u = _OW
    ids, infos = O.select(logits, hid, off, pl, p, u, rows=rows)
    return [(int(r), int(i), bool(f.u_boundary or f.topp_boundary)) for r, i, f in zip(rows, ids, infos)]


class OraclePool:
    """The oracle as it stands on every host core the process may use: one
    spawned worker per core, the logits shared (not copied) between them."""

    def __init__(self, w):
        import multiprocessing as mp
        import numpy as np
        from multiprocessing import shared_memory
        self.cores = len(os.sched_getaffinity(0))
        self.shm = shared_memory.SharedMemory(create=True, size=w.logits.nbytes)
        np.ndarray(w.logits.shape, dtype=w.logits.dtype, buffer=self.shm.buf)[:] = w.logits
        self.pool = mp.get_context("spawn").Pool(
            self.cores, initializer=_oracle_init,
            initargs=(self.shm.name, w.logits.shape, w.logits.dtype.str, w.hist_ids, w.hist_offsets, w.prompt_lens,
                      w.params, w.uniforms))
        self.pool.map_async(_oracle_rows, [[] for _ in range(self.cores)]).get(timeout=300)   # workers up first

    def run(self, rows):
        """(seconds, [(row, id, on_boundary)]) for the listed rows."""
        rows = list(rows)
        parts = [rows[i::self.cores] for i in range(self.cores)]
        t0 = time.perf_counter()
        res = self.pool.map_async(_oracle_rows, parts).get(timeout=600)
        el = time.perf_counter() - t0
        return el, sorted(x for part in res for x in part)

    def close(self):
        self.pool.close()
        self.pool.join()
        self.shm.close()
        self.shm.unlink()


def oracle_check(w, gpu_ids, pool=None):
    """The oracle on all cores over every row of w: its rate, the rows whose
    uniform or top-p cut lies within 1e-6 of a boundary, and how many of the
    GPU's ids equal the oracle's (all rows, and off the boundaries)."""
    own = pool is None
    pool = pool or OraclePool(w)
    try:
        el, res = pool.run(range(w.B))
    finally:
        if own:
            pool.close()
    boundary = sum(1 for _, _, bnd in res if bnd)
    equal = sum(1 for r, i, _ in res if int(gpu_ids[r]) == i)
    equal_off = sum(1 for r, i, bnd in res if not bnd and int(gpu_ids[r]) == i)
    return {"value": w.B / el, "unit": "rows/s", "cores": pool.cores, "kind": "oracle",
            "sample": "all %d rows of the workload, one spawned process per core, %.2f s" % (w.B, el),
            "seconds": el, "boundary_rows": boundary, "ids_equal": equal, "ids_equal_off_boundary": equal_off,
            "rows_off_boundary": w.B - boundary}


def time_select(w, steps, warmup, gpu_index, clocks=True, logprobs=False):
    """tg_select on workload w, inputs resident in HBM (rotating over enough
    copies of the logits to exceed L2): stream and CUDA-graph timings, the
    roofline of the launch, and the ids of the last step."""
    import numpy as np
    import torch
    import logits_processing_token_gb300 as tg
    bf16 = w.params["logits_dtype"] == "bf16"
    cfg = tg.Config(**w.params)
    elt = 2 if bf16 else 4
    nbytes = w.B * w.V * elt
    n_sets = max(1, int(np.ceil(2.5 * L2_BYTES / nbytes)))
    host = torch.from_numpy(w.logits.view(np.int16) if bf16 else w.logits)
    sets = [host.cuda().view(torch.bfloat16) if bf16 else host.cuda() for _ in range(n_sets)]
    hid = torch.from_numpy(w.hist_ids).cuda()
    off = torch.from_numpy(w.hist_offsets).cuda()
    pl = torch.from_numpy(w.prompt_lens).cuda()
    u = torch.from_numpy(w.uniforms).cuda()
    out = torch.empty(w.B, dtype=torch.int32, device="cuda")
    lp = torch.empty(w.B, dtype=torch.float32, device="cuda") if logprobs else None
    stream = torch.cuda.current_stream()

    def step(i):
        tg.tg_select(sets[i % n_sets], hid, off, pl, cfg, u, out, stream=stream, out_logprobs=lp)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    tg.tg_clear_status(cfg)
    ck = Clocks(gpu_index, enabled=clocks)
    ck.start()
    time.sleep(0.3 if ck.proc else 0.0)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = ck.stop()
    ms = e0.elapsed_time(e1) / steps
    flags, slow_rows = tg.tg_query_status(cfg)
    ids = out.cpu().numpy()
    graph = graph_timing(lambda i: tg.tg_select(sets[i % n_sets], hid, off, pl, cfg, u, out, out_logprobs=lp), w.B,
                         steps)
    peak, peak_kind = measured_peak()
    alg, n_read = required_bytes(w)
    achieved = alg / (ms / 1000.0) / 1e9
    res = {"workload": w.name, "B": w.B, "V": w.V, "logits_dtype": w.params["logits_dtype"],
           "us_per_step": ms * 1000.0, "rows_per_s": w.B / (ms / 1000.0),
           "logits_gbs": nbytes / (ms / 1000.0) / 1e9,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                        "peak_source": "%s hbm_gbs (copy)" % peak_kind, "bytes_per_launch": alg,
                        "rows_reading_logits": n_read, "traffic": None},
           "graph": graph, "slow_path_rows": slow_rows, "status_flags": flags, "steps": steps, "warmup": warmup,
           "l2": "inputs rotate over %d copies of the logits (%.0f MB)" % (n_sets, n_sets * nbytes / 1e6)}
    if clk:
        res["clocks"] = clk
    del sets
    torch.cuda.empty_cache()
    return res, ids


def time_verify(B, K, mode, steps, warmup):
    """tg_verify on config 4's inputs (candidates agree with the target's
    argmax at the seeded positions): microseconds per call."""
    import numpy as np
    import torch
    import logits_processing_token_gb300 as tg
    from logits_processing_token_gb300 import workloads as W
    w = W.config4(B=B, K=K, mode=mode)
    tgt = torch.from_numpy(np.ascontiguousarray(w.extra["target"])).cuda()
    greedy = tgt.argmax(dim=-1)[:, :K].cpu().numpy()
    cand = torch.from_numpy(W.make_candidates(greedy, w.extra["agree"], w.extra["offsets"], w.V)).cuda()
    cfg = tg.Config(**w.params, max_batch=max(64, B))
    u = torch.from_numpy(np.ascontiguousarray(w.uniforms)).cuda()
    om = torch.empty(B, dtype=torch.int32, device="cuda")
    on = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    for _ in range(warmup):
        tg.tg_verify(tgt, cand, K, cfg, u, om, on)
    torch.cuda.synchronize()
    tg.tg_clear_status(cfg)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        tg.tg_verify(tgt, cand, K, cfg, u, om, on)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flags, slow_rows = tg.tg_query_status(cfg)
    nbytes = B * (K + 1) * w.V * 4
    peak, _ = measured_peak()
    return {"B": B, "K": K, "mode": mode, "us_per_call": ms * 1000.0, "logits_gbs": nbytes / (ms / 1000.0) / 1e9,
            "hbm_frac": nbytes / (ms / 1000.0) / 1e9 / peak, "slow_path_rows": slow_rows, "status_flags": flags,
            "l2": "target logits %.0f MB, not rotated (smaller calls run from L2)" % (nbytes / 1e6)}


def main_config(w, n_sets, logprobs=False):
    """The config dict both arms print for the headline workload."""
    return {"workload": WORKLOAD, "B": w.B, "V": w.V, "logits_dtype": "bf16", "rows_per_gpu": w.B,
            "parallelism": "replicas (rows independent, no collective)",
            "l2": "inputs rotate over %d copies of the logits (%.0f MB) > L2" % (n_sets, n_sets * w.B * w.V * 2 / 1e6),
            "logprobs": bool(logprobs)}


def headline_sets(w):
    import numpy as np
    return max(2, int(np.ceil(2.5 * L2_BYTES / (w.B * w.V * 2))))


def run_reference(args):
    """The oracle as it stands, on all host cores: each step selects a
    rotating sample of the workload's rows (four per core)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from logits_processing_token_gb300 import workloads as W
    w = W.config3()
    pool = OraclePool(w)
    per = min(w.B, 4 * pool.cores)
    try:
        def step(i):
            start = (i * per) % w.B
            return pool.run([(start + k) % w.B for k in range(per)])[0]
        for i in range(args.warmup):
            step(i)
        total = sum(step(args.warmup + i) for i in range(args.steps))
    finally:
        pool.close()
    ms = 1000.0 * total / args.steps
    val = per / (ms / 1000.0)
    line = {"metric": METRIC, "value": val, "unit": "rows/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": main_config(w, headline_sets(w), args.logprobs),
            "cpu_baseline": {"value": val, "unit": "rows/s", "cores": pool.cores, "kind": "oracle",
                             "sample": "each step: %d of the %d rows (rotating), one spawned process per core" %
                                       (per, w.B)},
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
    n_sets = headline_sets(w)
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
            "config": main_config(w, n_sets, args.logprobs),
            "logits_gbs": nominal_gbs, "logits_hbm_frac": nominal_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                         "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                         "bytes_per_launch": alg_bytes, "rows_reading_logits": n_read,
                         "kernel": "select_kernel<bf16>", "mean_launch_us": mean_launch_s * 1e6},
            "gpu_launches": K, "slow_path_rows": slow_rows, "status_flags": flags}
    if clk:
        line["clocks"] = clk

    ids_main = out.cpu().numpy()
    if not args.no_e2e:
        # The public API from host buffers: every step copies all of its inputs
        # from pinned host memory and reads its ids back.  Step i+1's copies run
        # on a second stream while step i's kernel runs (two sets of device
        # buffers); the kernel of a step waits for its own copies.
        h_logits = host_logits.pin_memory()
        h_small = [torch.from_numpy(a).pin_memory() for a in (w.hist_ids, w.hist_offsets, w.prompt_lens, w.uniforms)]
        h_out = torch.empty((2, B), dtype=torch.int32).pin_memory()
        h_lp = torch.empty((2, B), dtype=torch.float32).pin_memory() if lp is not None else None
        d_logits = [torch.empty_like(h_logits, device="cuda") for _ in range(2)]
        d_small = [[torch.empty_like(t, device="cuda") for t in h_small] for _ in range(2)]
        d_out = [torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(2)]
        d_lp = [torch.empty(B, dtype=torch.float32, device="cuda") for _ in range(2)] if lp is not None else None
        bi = h_logits.numel() * h_logits.element_size() + sum(t.numel() * t.element_size() for t in h_small)
        bo = B * 4 + (B * 4 if lp is not None else 0)
        copy_stream = torch.cuda.Stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)

        def e2e_run(n):
            e0.record(stream)
            copy_stream.wait_event(e0)
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(copy_stream):
                    if i >= 2:
                        copy_stream.wait_event(used[b])
                    d_logits[b].copy_(h_logits, non_blocking=True)
                    for d, h in zip(d_small[b], h_small):
                        d.copy_(h, non_blocking=True)
                    copied[b].record(copy_stream)
                stream.wait_event(copied[b])
                hid_b, off_b, pl_b, u_b = d_small[b]
                tg.tg_select(d_logits[b].view(torch.bfloat16), hid_b, off_b, pl_b, cfg, u_b, d_out[b], stream=stream,
                             out_logprobs=d_lp[b] if d_lp is not None else None)
                used[b].record(stream)
                h_out[b].copy_(d_out[b], non_blocking=True)
                if h_lp is not None:
                    h_lp[b].copy_(d_lp[b], non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        e2e_run(3)
        e_ms = e2e_run(args.e2e_steps)
        e_ms = max_over_ranks(e_ms, world, "cuda")
        line["e2e"] = {"value": whole_job_rate(world, B, e_ms), "unit": "rows/s", "h2d_bytes_per_step": bi,
                       "d2h_bytes_per_step": bo, "ms_per_step": e_ms,
                       "overlap": "step i+1's host-to-device copies run on a second stream during step i's kernel"}

    if not args.no_graph and world == 1:
        # (at N = 1 only: a rank whose capture failed would leave the others in the max-over-ranks collective)
        line["graph"] = graph_timing(
            lambda i: tg.tg_select(sets[i % n_sets], hid, off, pl, cfg, u, out, out_logprobs=lp), B, K)

    if world == 1 and not args.quick:
        # the other configurations, each timed the same way (inputs resident, > L2)
        del sets
        torch.cuda.empty_cache()
        others = {}
        for name, wk, st in (("1", W.config1(), args.steps), ("2", W.config2(), args.steps)):
            others[name], _ = time_select(wk, st, args.warmup, local, clocks=False, logprobs=args.logprobs)
        others["4"] = [time_verify(b, k, m, args.steps, args.warmup)
                       for b, k, m in ((1, 5, "greedy"), (8, 5, "sample"), (32, 16, "greedy"), (32, 16, "sample"))]
        line["configs"] = others
        # config 5: B=1,024, V=262,144 f32 -- the second roofline target
        w5 = W.config5()
        c5, ids5 = time_select(w5, args.steps, args.warmup, local, clocks=not args.no_clocks, logprobs=args.logprobs)
        c5["gpu_launches"] = args.steps
        if not args.no_cpu_baseline:
            c5["oracle"] = oracle_check(w5, ids5)
        line["config5"] = c5

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = oracle_check(w, ids_main)
        base["single_core"] = cpu_baseline_1core(w, args.cpu_seconds)
        line["cpu_baseline"] = base
        line["boundary_rows"] = base["boundary_rows"]
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


def run_config5(args):
    """Config 5 as the line's workload: B=1,024 rows of V=262,144 f32 logits."""
    import torch
    from logits_processing_token_gb300 import _build
    _build.build()
    from logits_processing_token_gb300 import workloads as W
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    w = W.config5()
    res, ids = time_select(w, args.steps, args.warmup, local, clocks=not args.no_clocks, logprobs=args.logprobs)
    ms = res["us_per_step"] / 1000.0
    line = {"metric": "rows/s and logits GB/s (% of GB300 HBM peak) at B=1,024, V=262,144", "value": res["rows_per_s"],
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "tg_select: " + w.name + ", repetition penalty 1.3, 4-gram ban, min_new_tokens 8",
                       "B": w.B, "V": w.V, "logits_dtype": "f32", "l2": res["l2"], "logprobs": bool(args.logprobs)},
            "roofline": dict(res["roofline"], kernel="select_kernel<f32>", mean_launch_us=res["us_per_step"]),
            "graph": res["graph"], "gpu_launches": args.steps, "slow_path_rows": res["slow_path_rows"],
            "status_flags": res["status_flags"]}
    if "clocks" in res:
        line["clocks"] = res["clocks"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_check(w, ids)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.config == 5:
        run_config5(args)
    elif args.beam:
        run_beam(args)
    elif args.state:
        run_state(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
