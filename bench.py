#!/usr/bin/env python3
"""Benchmark of the fused indexer launch (idx_launch) on GB300.

Workload: two requests x four rows at 524,288 cached keys each, FP8 E4M3 cache
(the 512K-key configuration the metric is quoted on), seeded synthetic inputs
from workloads.make_config(3).  One step = one idx_launch: plan + query prep,
the scoring scan with the fused first-digit histogram, and the exact top-2048
selection of every row.

Timing: W untimed warm-up steps, then K timed steps.  Before every step a 256 MB
buffer (twice the L2) is written so that no step finds the keys in L2; each step
is timed on the launching stream with CUDA events around the launch alone.  Every
other step also times the scoring kernel through the library's event hook; an
event recorded between two kernels of the launch costs their programmatic
overlap, so the launch time is the mean of the other steps.  The
e2e figure times idx_launch_host: host->device copies of every input from
pinned memory, the launch, and the device->host copy of the indices.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
batch of requests (the work shards by request with no exchange), the timed
region is bracketed by a barrier and synchronisation on every rank, and the
maximum time over ranks is reported: weak scaling.

`--impl reference` times the CPU oracle (the slow reference implementation of
the same method) on the host cores instead; rank 0 alone runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per indexer launch and key·rows/s at 512K keys; % of HBM/FP8 roofline"
WORKLOAD = ("cfg3: 2 requests x 4 rows, 524,288 keys each (page 64, shuffled pages), FP8 E4M3 cache "
            "with per-token scale, sigma 1/4 mixture keys, bf16 q, fp32 w, top-k 2048")
L2_FLUSH_BYTES = 256 << 20
KERNELS_PER_LAUNCH = 4  # prep, score, collect, finish


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def profile_traffic(kernel_src: str):
    """DRAM bytes per launch of the scoring kernel from the committed ncu summary,
    or None if the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "score_kernel_cfg3.md")
    if not os.path.exists(path):
        return None
    sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    fields = {}
    for line in open(path):
        if line.startswith("- ") and ": " in line:
            k, v = line[2:].split(": ", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("score.cu sha256[:16]") != sha:
        return None
    try:
        return int(fields["dram bytes per launch"].replace(",", ""))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms from before the
    warm-up to the end; summary() keeps the samples read inside a given window."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []   # (host time read, line)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def wait_first(self, timeout_s: float = 5.0):
        """Blocks until the sampler has printed once (nvidia-smi takes a while to start)."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if not (t0 <= t <= t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _row_sample(prob, rows, bound):
    import workloads
    return workloads.Problem(name="sample", q=prob.q[rows], w=prob.w[rows], k_cache=prob.k_cache,
                             k_scale=prob.k_scale, page_table=prob.page_table, row_req=prob.row_req[rows],
                             row_bound=bound, kv_dtype=prob.kv_dtype, K=prob.K)


def _oracle_pass(orc, sub):
    import numpy as np
    t0 = time.perf_counter()
    s = orc.score(sub)
    orc.topk(s.astype(np.float32), sub.row_bound, sub.K)
    return time.perf_counter() - t0


def cpu_baseline(prob, orc, budget_s: float = 12.0, rate_hint=None):
    """The oracle (score + exact top-k) on a bounded sample of the workload.

    The sample takes the workload's rows in order, the last one cut to its first
    L keys (a multiple of the 64-key page), so that one pass takes about
    budget_s.  When the whole workload takes less than that, the sample is the
    whole workload, repeated until about budget_s of oracle work is done.  The
    rate is sized on a probe of the first row (up to 64K keys) unless a rate from
    an earlier call is given."""
    import numpy as np
    rows = list(range(prob.R))
    rate = rate_hint
    if rate is None:
        probe = _row_sample(prob, rows[:1], np.array([min(65536, int(prob.row_bound[rows[0]]))], dtype=np.int32))
        _oracle_pass(orc, probe)                                   # warm (thread pool, pages)
        rate = int(probe.row_bound.sum()) / _oracle_pass(orc, probe)
    want = max(1024, int(rate * budget_s))
    bounds, take = [], []
    for r in rows:
        b = int(prob.row_bound[r])
        cut = min(b, max(64, (want - sum(bounds)) // 64 * 64))
        bounds.append(cut)
        take.append(r)
        if sum(bounds) >= want or cut < b:
            break
    sub = _row_sample(prob, take, np.array(bounds, dtype=np.int32))
    keys = int(sum(bounds))
    passes, dt = 0, 0.0
    while True:
        dt += _oracle_pass(orc, sub)
        passes += 1
        if dt / passes * (passes + 1) > 1.15 * budget_s:     # the next pass would overrun
            break
    what = (f"{passes} pass(es) over the whole workload ({prob.R} rows, {keys} key-rows each)"
            if len(take) == prob.R and bounds[-1] == int(prob.row_bound[prob.R - 1])
            else f"{len(take)} of {prob.R} rows of the workload with bounds {bounds} ({keys} key-rows)")
    return {"value": keys * passes / dt, "unit": "key·rows/s", "cores": orc.num_threads(),
            "kind": "oracle", "seconds": round(dt, 3), "rate": keys * passes / dt,
            "sample": what + ": oracle scores in fp64 + exact top-2048 by sort"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import workloads
    orc = oracle.default()
    prob = workloads.make_config(3)
    # the whole run (warm-up + timed steps) is held to about --ref-budget seconds
    per_step = max(0.02, args.ref_budget / max(1, args.steps + args.warmup))
    first = cpu_baseline(prob, orc, budget_s=per_step)
    rate = first["rate"]
    for _ in range(max(0, args.warmup - 1)):
        cpu_baseline(prob, orc, budget_s=per_step, rate_hint=rate)
    vals = [cpu_baseline(prob, orc, budget_s=per_step, rate_hint=rate) for _ in range(args.steps)]
    v = statistics.median(x["value"] for x in vals)
    ms = prob.key_rows / v * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "key·rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": prob.R, "seq_len": prob.max_bound,
                   "parallelism": "host cores (oracle)", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "key·rows/s", "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": "per step: " + vals[0]["sample"]},
        "e2e": {"value": v, "unit": "key·rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- multi-rank host logic
def rank_problem(cfg, rank: int):
    """The workload of one rank: rank 0 runs the named configuration itself, rank
    r > 0 the same shapes drawn with seed offset 1000 * r, so every rank holds an
    independent batch (the path shards by request, with no exchange)."""
    import workloads
    return workloads.make_config(cfg, seed_offset=1000 * rank)


def max_over_ranks(values, device: str):
    """Elementwise maximum of per-rank timings over the process group (every rank
    gets the result)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def total_key_rows(key_rows_per_rank: int, world: int) -> int:
    """Whole-job units: every rank scores a batch of the same shape."""
    return int(key_rows_per_rank) * int(world)


def emit(line, rank: int):
    """Rank 0 prints the JSON line; the other ranks print nothing."""
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


def run_top1(args):
    """--op top1: the one-launch top-1 of R rows of V fp32 logits (the page's later
    draft_topk1_postprocess commit), timed like the indexer launch: L2 flushed
    before every step, CUDA events around the launch.  HBM-bound: R * V * 4 bytes."""
    import numpy as np
    import torch
    import sparse_attention_indexer_launch_gb300 as lib
    R, V = args.top1_rows, args.top1_vocab
    rng = np.random.default_rng(11)
    x = torch.from_numpy((rng.standard_normal((R, V)) * 4).astype(np.float32)).cuda()
    idx = torch.empty(R, dtype=torch.int32, device="cuda")
    state = torch.zeros(lib.top1_state_size(R), dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        lib.idx_top1(x, idx, state)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        lib.idx_top1(x, idx, state)
        b.record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    import oracle
    xh = x.cpu().numpy()
    ref, _ = oracle.top1(xh)
    if not np.array_equal(ref, idx.cpu().numpy()):
        raise SystemExit("idx_top1 result differs from the oracle")
    t0 = time.perf_counter()
    oracle.top1(xh)
    cpu_s = time.perf_counter() - t0
    hbm_gbs, _, peak_src = measured_peaks()
    nbytes = R * V * 4
    print(json.dumps({
        "metric": "µs per top-1 launch (R rows x V fp32 logits)", "op": "top1", "value": us, "unit": "µs",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "config": {"workload": f"{R} rows x {V} logits, N(0, 16) fp32", "l2": "flushed before every step (256 MB write)"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (us * 1e-6) / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": nbytes / (us * 1e-6) / 1e9 / hbm_gbs, "algorithmic_bytes": nbytes,
                     "peak_source": peak_src},
        "cpu_baseline": {"value": cpu_s * 1e6, "unit": "µs", "cores": 1, "kind": "oracle",
                         "sample": "the same rows, one pass of the oracle's loop"},
    }))
    return 0


def run_patch(args):
    """--op patch: idx_patch_new_keys on the benchmark workload (8 rows' new keys
    quantised and written into the paged cache), CUDA events around the call."""
    import numpy as np
    import torch
    import sparse_attention_indexer_launch_gb300 as lib
    import workloads
    prob = workloads.make_config(3)
    dp = lib.DeviceProblem(prob)
    rng = np.random.default_rng(12)
    k_new = torch.from_numpy(rng.standard_normal((prob.R, 128)).astype(np.float32)).to(torch.bfloat16).cuda()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        lib.idx_patch_new_keys(dp.problem, k_new)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        lib.idx_patch_new_keys(dp.problem, k_new)
        b.record(stream)
    torch.cuda.synchronize()
    us_call = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    # the same call replayed from a CUDA graph: the device time without the host's
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        lib.idx_patch_new_keys(dp.problem, k_new)
    stream.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.idx_patch_new_keys(dp.problem, k_new)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    # the launch with and without the new keys written by its own first kernel,
    # against the patch launch followed by the plain launch (L2 flushed before each)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")

    def timed(fn):
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3

    us_fused = timed(lambda: lib.idx_launch_new_keys(dp.problem, k_new, prob.K, out, dp.ws))
    us_split = timed(lambda: (lib.idx_patch_new_keys(dp.problem, k_new), dp.launch(out)))
    us_plain = timed(lambda: dp.launch(out))
    print(json.dumps({"metric": "µs per new-key patch (8 rows, E4M3 cache), CUDA-graph replay", "op": "patch",
                      "value": us, "us_per_call_from_python": us_call,
                      "launch_with_new_keys_us": us_fused, "patch_then_launch_us": us_split,
                      "launch_alone_us": us_plain,
                      "unit": "µs", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
                      "warmup": args.warmup, "config": {"workload": workloads.CONFIG_NAMES[3]}}))
    return 0


def time_config(lib, prob, steps, warmup, flush, stream):
    """One workload timed as the main line is: L2 flushed before every step, CUDA
    events around the launch on its stream, every other step also timing the
    scoring kernel.  Returns (launch ms, scoring-kernel ms)."""
    import torch
    dp = lib.DeviceProblem(prob)
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")
    for _ in range(warmup):
        flush.zero_()
        dp.launch(out)
    torch.cuda.synchronize()
    st = dp.status()
    if st != lib.IDX_OK:
        raise SystemExit(f"device status ({prob.name}): {lib.status_string(st)}")
    pairs = []
    for i in range(steps):
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        sev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in (*ev, *sev):
            e.record(stream)
        flush.zero_()
        if i % 2 == 1:
            lib.profile_next_score(sev[0], sev[1])
        ev[0].record(stream)
        dp.launch(out)
        ev[1].record(stream)
        pairs.append((i, ev, sev))
    torch.cuda.synchronize()
    launch = [ev[0].elapsed_time(ev[1]) for i, ev, _ in pairs if i % 2 == 0]
    score = [sev[0].elapsed_time(sev[1]) for i, _, sev in pairs if i % 2 == 1]
    return statistics.mean(launch), statistics.mean(score)


def roofline_terms(prob, hbm_gbs, bf16_tf):
    """(launch roofline s, bound, FP8 TF/s) of a workload: max(key bytes / HBM,
    MMA flops / FP8 peak), FP8 taken as twice the measured bf16 rate."""
    fp8_tf = 2.0 * bf16_tf
    t_hbm = prob.key_bytes / (hbm_gbs * 1e9)
    t_fp8 = prob.mma_flops / (fp8_tf * 1e12)
    return max(t_hbm, t_fp8), ("hbm" if t_hbm >= t_fp8 else "tensor"), fp8_tf


def run_split(args):
    """--op split: the indexer's two halves called apart on the benchmark workload,
    idx_score (prep and the scan, scores and first digit out) and idx_topk on those
    scores (its own 12-bit histogram pass, collect, finish), each timed like the
    fused launch (L2 flushed before every call, CUDA events around it).  The sum
    against idx_launch shows what fusing the histogram into the scan saves."""
    import numpy as np
    import torch
    import oracle
    import sparse_attention_indexer_launch_gb300 as lib
    import workloads
    orc = oracle.default()
    prob = workloads.make_config(3)
    dp = lib.DeviceProblem(prob)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    scores, hist = dp.score()
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")
    ld = scores.shape[1]

    def timed(fn):
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3

    # preallocated outputs: nothing but the library's kernels between the events
    score_us = timed(lambda: lib.idx_score(dp.problem, scores, ld, hist, dp.ws))
    topk_us = timed(lambda: lib.idx_topk(scores, ld, dp.row_bound, prob.R, dp.max_bound, prob.K, None, out,
                                         dp.ws))
    launch_us = timed(lambda: lib.idx_launch(dp.problem, prob.K, out, dp.ws))
    got = dp.topk(scores).cpu().numpy()
    if not np.array_equal(got, orc.topk(scores.cpu().numpy(), prob.row_bound, prob.K)):
        raise SystemExit("idx_topk differs from the oracle's selection on the same scores")
    if dp.status() != lib.IDX_OK:
        raise SystemExit("device status not clean")
    key_rows = int(prob.row_bound.astype(np.int64).sum())
    print(json.dumps({"metric": "µs per idx_score and per idx_topk on the benchmark workload", "op": "split",
                      "value": score_us + topk_us, "unit": "µs", "higher_is_better": False, "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "idx_score_us": score_us,
                      "idx_topk_us": topk_us, "idx_launch_us": launch_us,
                      "topk_key_rows_per_s": key_rows / (topk_us * 1e-6),
                      "config": {"workload": "cfg3: 2 requests x 4 rows, 524,288 keys each, E4M3",
                                 "l2": "flushed before every call (256 MB write)"}}))
    return 0


def run_merge(args):
    """--op merge: idx_merge_topk of S ranked parts of R rows x K (the key-sharded
    indexer's owner merge), S = 2, 4, 8; CUDA events around each call, L2 flushed
    before each.  The parts are every row's top-K of S disjoint ranges of 524,288
    normal scores, ranked by the oracle."""
    import numpy as np
    import torch
    import oracle
    import sparse_attention_indexer_launch_gb300 as lib
    orc = oracle.default()
    R, K, L = 8, 2048, 524288
    rng = np.random.default_rng(13)
    scores = rng.standard_normal((R, L)).astype(np.float32)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    res = {}
    for S in (2, 4, 8):
        cuts = [L * i // S for i in range(S + 1)]
        pi = np.full((S, R, K), -1, np.int32)
        ps = np.full((S, R, K), -np.inf, np.float32)
        for i in range(S):
            sub = np.ascontiguousarray(scores[:, cuts[i]:cuts[i + 1]])
            idx = orc.topk(sub, np.full(R, cuts[i + 1] - cuts[i], np.int32), K)
            pi[i] = idx
            ps[i] = np.take_along_axis(sub, np.maximum(idx, 0), axis=1)
        dpi, dps = torch.from_numpy(pi).cuda(), torch.from_numpy(ps).cuda()
        out = torch.empty((R, K), dtype=torch.int32, device="cuda")
        for _ in range(args.warmup):
            lib.idx_merge_topk(dpi, dps, cuts[:-1], K, out)
        torch.cuda.synchronize()
        want = orc.topk(scores, np.full(R, L, np.int32), K)
        if not np.array_equal(out.cpu().numpy(), want):
            raise SystemExit(f"idx_merge_topk of {S} parts differs from the unsharded selection")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            lib.idx_merge_topk(dpi, dps, cuts[:-1], K, out)
            b.record(stream)
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
        t0 = time.perf_counter()
        orc.merge_topk(pi, ps, np.array(cuts[:-1], np.int32), K)
        res[S] = {"us": us, "oracle_us": (time.perf_counter() - t0) * 1e6, "bytes_in": pi.nbytes + ps.nbytes}
    print(json.dumps({"metric": "µs per owner merge of S ranked parts (8 rows x top-2048)", "op": "merge",
                      "value": res[2]["us"], "unit": "µs", "higher_is_better": False, "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "parts": res,
                      "config": {"workload": "8 rows x 524,288 N(0,1) scores split into S ranges",
                                 "l2": "flushed before every call (256 MB write)"}}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="3", help="workload: 0..4, 3a or 3b (default 3)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--extra-configs", default="3a",
                    help="comma-separated workloads also timed (same protocol) and reported under "
                         "extra_configs; 'none' for none")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds for the whole --impl reference run")
    ap.add_argument("--op", default="indexer", choices=["indexer", "top1", "patch", "merge", "split"],
                    help="indexer: the fused indexer launch (the benchmark); top1: the one-launch top-1; "
                         "patch: the new-key patch; merge: the key-sharded owner merge; "
                         "split: idx_score and idx_topk called apart")
    ap.add_argument("--top1-rows", type=int, default=8)
    ap.add_argument("--top1-vocab", type=int, default=151552)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not os.environ.get("IDX_BENCH_ALLOW_SHORT"):
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "top1":
        return run_top1(args)
    if args.op == "patch":
        return run_patch(args)
    if args.op == "split":
        return run_split(args)
    if args.op == "merge":
        return run_merge(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    import sparse_attention_indexer_launch_gb300 as lib
    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    cfg = args.config if args.config in ("3a", "3b") else int(args.config)
    prob = rank_problem(cfg, rank)
    dp = lib.DeviceProblem(prob)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    out = torch.empty((prob.R, prob.K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(ev=None, sev=None):
        flush.zero_()
        if sev is not None:
            lib.profile_next_score(sev[0], sev[1])
        if ev is not None:
            ev[0].record(stream)
        dp.launch(out)
        if ev is not None:
            ev[1].record(stream)

    clocks = ClockSampler(local).__enter__()
    clocks.wait_first()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = dp.status()
    if st != lib.IDX_OK:
        raise SystemExit(f"device status after warm-up: {lib.status_string(st)}")

    def events(n):
        out = []
        for _ in range(n):
            pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for e in pair:
                e.record(stream)   # creates the CUDA event, so the library can record it too
            out.append(pair)
        return out

    # Odd-numbered steps also record events around the scoring kernel (the
    # roofline figure); recording an event between two kernels of the launch
    # costs their programmatic overlap, so the launch time comes from the
    # even-numbered steps alone.
    evs = events(args.steps)
    sevs = events(args.steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    for i in range(args.steps):
        step(evs[i], sevs[i] if (i % 2 == 1 or args.steps == 1) else None)
    torch.cuda.synchronize()
    t_end = time.perf_counter()
    t_wall = t_end - t_start
    time.sleep(0.15)   # the sample that covers the end of the timed region
    clocks.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    st = dp.status()
    if st != lib.IDX_OK:
        raise SystemExit(f"device status after the timed steps: {lib.status_string(st)}")
    step_ms = [a.elapsed_time(b) for i, (a, b) in enumerate(evs) if i % 2 == 0 or args.steps == 1]
    score_ms = [a.elapsed_time(b) for i, (a, b) in enumerate(sevs) if i % 2 == 1 or args.steps == 1]
    ms = statistics.mean(step_ms)
    score_mean_ms = statistics.mean(score_ms)

    # end to end through idx_launch_host (pinned host inputs, copies in the timed region)
    e2e_ms = None
    h2d = d2h = 0
    if not args.no_e2e:
        host = {k: torch.from_numpy(np.ascontiguousarray(getattr(prob, k))).pin_memory()
                for k in ("q", "w", "k_cache", "k_scale", "page_table", "row_req", "row_bound")
                if getattr(prob, k) is not None}
        kv = lib.IDX_KV_E4M3 if prob.kv_dtype == "e4m3" else lib.IDX_KV_BF16
        hp = lib.make_problem(host["q"], host["w"], host["k_cache"], host.get("k_scale"), host["page_table"],
                              host["row_req"], host["row_bound"], prob.max_bound, kv)
        arena = lib.alloc_bytes(lib.host_arena_size(hp, prob.K))
        hout = torch.empty((prob.R, prob.K), dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = hout.numel() * hout.element_size()
        for _ in range(3):
            lib.idx_launch_host(hp, prob.K, hout, arena)
        torch.cuda.synchronize()
        if not np.array_equal(hout.numpy(), out.cpu().numpy()):
            raise SystemExit("idx_launch_host result differs from idx_launch")
        n_e2e = max(3, min(args.steps, 10))
        e2e_ev = events(n_e2e)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for a, b in e2e_ev:
            flush.zero_()
            a.record(stream)
            lib.idx_launch_host(hp, prob.K, hout, arena)
            b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)

    # max over ranks
    if world > 1:
        ms, score_mean_ms, e2e_ms = max_over_ranks([ms, score_mean_ms, e2e_ms or 0.0], "cuda")
        e2e_ms = e2e_ms or None

    # the other workloads of the metric's target (same protocol, after the main
    # timed region; rank 0 reports them)
    hbm_gbs, bf16_tf, peak_src = measured_peaks()
    extra = []
    for name in [c.strip() for c in args.extra_configs.split(",") if c.strip() and c.strip() != "none"]:
        ecfg = name if name in ("3a", "3b") else int(name)
        if ecfg == cfg:
            continue
        eprob = rank_problem(ecfg, rank)
        e_ms, e_score_ms = time_config(lib, eprob, max(2, min(args.steps, 400)), args.warmup, flush, stream)
        e_roof, e_bound, _ = roofline_terms(eprob, hbm_gbs, bf16_tf)
        extra.append({"workload": workloads.CONFIG_NAMES[ecfg], "us_per_launch": e_ms * 1e3,
                      "value": eprob.key_rows / (e_ms * 1e-3), "unit": "key·rows/s",
                      "kernel_us": e_score_ms * 1e3, "launch_roofline_us": e_roof * 1e6, "bound": e_bound,
                      "launch_frac_of_roofline": e_roof / (e_ms * 1e-3),
                      "kernel_frac_hbm": eprob.key_bytes / (e_score_ms * 1e-3) / 1e9 / hbm_gbs,
                      "tensor_frac_bf16_precision_matched":
                          eprob.mma_flops / (e_score_ms * 1e-3) / 1e12 / bf16_tf})
        del eprob

    key_rows_total = total_key_rows(prob.key_rows, world)
    value = key_rows_total / (ms * 1e-3)
    key_bytes = prob.key_bytes
    flops = prob.mma_flops
    # The metric's roofline: max(key bytes / HBM, FP8 flops / FP8 peak).
    t_roof, bound, fp8_tf = roofline_terms(prob, hbm_gbs, bf16_tf)
    score_s = score_mean_ms * 1e-3
    if bound == "hbm":
        achieved, peak, unit = key_bytes / score_s / 1e9, hbm_gbs, "GB/s"
    else:
        achieved, peak, unit = flops / score_s / 1e12, fp8_tf, "TFLOP/s"
    traffic = profile_traffic(os.path.join(ROOT, "sparse_attention_indexer_launch_gb300", "csrc", "score.cu"))
    # The epilogue's ALU term: 128 lane operations per (key, row) (64 max + 64 FMA)
    # over every SM's 128 FP32 lanes at the sampled SM clock.
    clk = clocks.summary(t_start, t_end)
    sm_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz") or 0.0
    n_sms = torch.cuda.get_device_properties(local).multi_processor_count
    alu_floor_us = prob.key_rows * 128 / (n_sms * 128 * sm_mhz * 1e6) * 1e6 if sm_mhz else None

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "key·rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "us_per_launch": ms * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3 x (2-term e4m3 split of bf16 q), fp32 accumulate" if prob.kv_dtype == "e4m3" else "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD if cfg == 3 else workloads.CONFIG_NAMES[cfg],
                       "global_batch": prob.R * world, "seq_len": prob.max_bound,
                       "parallelism": f"replicas x{world} (independent requests per GPU)",
                       "l2": "flushed before every step (256 MB write)"},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic,
                         "frac_scope": "the scoring kernel alone (the dominant kernel); "
                                       "launch_frac_of_roofline is the whole launch",
                         "kernel": "score_kernel (scan + contraction + head reduction + histogram)",
                         "kernel_us": score_mean_ms * 1e3,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json; FP8 = 2 x bf16)",
                         "algorithmic_bytes": key_bytes, "algorithmic_flops": flops,
                         "launch_roofline_us": t_roof * 1e6,
                         "launch_frac_of_roofline": t_roof / (ms * 1e-3),
                         "tensor_frac_fp8": flops / score_s / 1e12 / fp8_tf,
                         "tensor_frac_bf16_precision_matched": flops / score_s / 1e12 / bf16_tf,
                         "alu_epilogue_floor_us": alu_floor_us},
            "clocks": clk,
            "gpu_launches": KERNELS_PER_LAUNCH * args.steps,
            "wall_s_timed_region": t_wall,
        }
        if extra:
            line["extra_configs"] = extra
        if e2e_ms is not None:
            line["e2e"] = {"value": key_rows_total / (e2e_ms * 1e-3), "unit": "key·rows/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        if not args.no_cpu_baseline:
            import oracle
            line["cpu_baseline"] = cpu_baseline(prob, oracle.default())
    emit(line if rank == 0 else None, rank)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
