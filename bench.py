"""Benchmark of the verify sampler on GB300: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (one "step" = one call over one batch): block verification of B = 64
streams, k = 5 drafts + 1 bonus slot each, V = 129,280, bf16 logits, per-stream draft noise
sigma ~ U[0.2, 2.0], T ~ U[0.3, 1.0], 5% greedy streams.  Metric: verified draft slots per
second (sum of k over the batch per call / time).  Three input sets of 182 MB each rotate, so
every call reads logits that are not in the 129 MB L2.

Legs:
  value     device time of K back-to-back calls (CUDA events on the launching stream), inputs
            resident in HBM;
  e2e       the same calls through the public API with the inputs in pinned host memory: every
            step copies its inputs host->device (into one of two device buffers, on a copy
            stream, so the next step's copy overlaps this step's kernels) and reads its
            results (accepted_len, out_tokens, n_emitted, status) back;
  roofline  algorithmic bytes (one read of every logit row) / mean per-launch kernel time,
            against the measured HBM copy bandwidth;
  cpu_baseline / --impl reference   the float64 oracle on the host cores (process pool), on a
            bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own batch (streams shard with no exchange), timing
is max over ranks, value sums all ranks' slots.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "batch64"
METRIC = "verified draft slots/sec and HBM GB/s (% of roofline), batch 64, k=5, V=129280"
UNIT = "verified draft slots/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rule", default="block", choices=["block", "tokenwise"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle leg (profiling runs)")
    ap.add_argument("--cpu-sample", type=int, default=512,
                    help="oracle stream-verifies for cpu_baseline (about 10-15 s of CPU work)")
    ap.add_argument("--ref-sample", type=int, default=16,
                    help="oracle stream-verifies per step of --impl reference")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------
# distributed plumbing (barrier and max-over-ranks only; no data-path collective)
# ---------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if _cuda_ok() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if self.pg.get_backend() == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if self.pg.get_backend() == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# ---------------------------------------------------------------------------------------
# oracle on the host cores
# ---------------------------------------------------------------------------------------
_ORACLE_INPUTS = {}


def _oracle_task(args):
    """One worker's share: stream b of the seeded batch (generated once per worker process)."""
    rule, seed, b, steps = args
    sys.path.insert(0, ROOT)
    import numpy as np

    from oracle import verify as ov
    from speculative_decoding_block_verify_gb300 import workloads
    if seed not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[seed] = workloads.make_verify_inputs(HEADLINE, seed, B=16)
    inp = _ORACLE_INPUTS[seed]
    cu = inp["cu_drafts"]
    n = cu[b + 1] - cu[b]
    q_rows = np.asarray(inp["draft_logits"][cu[b]:cu[b] + n])
    p_rows = np.asarray(inp["target_logits"][cu[b] + b:cu[b] + b + n + 1])
    x = np.asarray(inp["draft_tokens"][cu[b]:cu[b] + n])
    T = float(inp["temperature"][b])
    if T == 0.0:   # greedy streams are not part of the sample
        return 0.0, 0, 0, 0
    t0 = time.perf_counter()
    ties = 0
    for st in steps:
        ties += int(ov.verify_stream(rule, q_rows, p_rows, x, T, 0, st, b)["tie"])
    return time.perf_counter() - t0, len(steps) * len(x), ties, len(steps)


def oracle_pool():
    """A spawned process pool over the host cores (spawn: safe whether or not CUDA is up)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    return mp.get_context("spawn").Pool(processes=cores), cores


def oracle_sample(n_verifies, rule, seed=3000, pool=None):
    """Time the oracle on about n_verifies stream-verifies of the headline workload: the
    sampled (T > 0) streams among the first 16 of the seeded batch, steps split over the
    workers.  Input generation in the workers is outside the timed part."""
    streams = list(range(16))
    per = max(1, n_verifies // len(streams))
    own = pool is None
    if own:
        pool, cores = oracle_pool()
    else:
        cores = pool._processes
    r = 1 if rule == "block" else 0
    chunks = max(1, cores // len(streams))
    split = []
    for b in streams:
        for c in range(chunks):
            sub = list(range(per))[c::chunks]
            if sub:
                split.append((r, seed, b, sub))
    try:
        pool.map(_oracle_task, [(r, seed, b, []) for b in streams for _ in range(chunks)])   # warm the inputs
        t0 = time.perf_counter()
        res = pool.map(_oracle_task, split)
        wall = time.perf_counter() - t0
    finally:
        if own:
            pool.close()
            pool.join()
    cpu_s = sum(x[0] for x in res)
    slots = sum(x[1] for x in res)
    ties, verifies = sum(x[2] for x in res), sum(x[3] for x in res)
    return {"value": slots / wall, "unit": UNIT, "cores": min(cores, len(split)), "kind": "oracle",
            "sample": f"the sampled streams among 16 x {per} steps of the batch-64 workload (k=5, V=129280), "
                      f"{rule} rule, float64 NumPy, {cpu_s:.1f} s of CPU work in {wall:.1f} s wall",
            "near_tie_streams": ties, "stream_verifies": verifies}


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------------------
def traffic_from_profiles(kernel_tag):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on the current
    kernel source (its sha256 is recorded in the summary)."""
    import hashlib
    src = os.path.join(ROOT, "speculative_decoding_block_verify_gb300", "csrc", "verify.cu")
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            tok = v.split()
            vals[k.strip()] = tok[0].strip("`") if tok else ""   # the value is the first token
    if vals.get("source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(inp):
    """One read of every draft row and every target row (bonus row included) of the batch:
    (2 N_b + 1) rows of V logits per stream - 568,832 B per draft slot at k = 5, V = 129,280,
    bf16.  Per-stream scalars and outputs (< 0.01%) are left out."""
    cu = inp["cu_drafts"].cpu()
    V = inp["V"]
    es = 2 if inp["dtype"] == "bf16" else 4
    B = len(cu) - 1
    if "t2d" in inp:   # reduced draft vocabulary: draft rows of K logits, plus the column map
        return (int(cu[-1]) + B) * V * es + int(cu[-1]) * inp["K"] * es + V * 4
    rows = 2 * int(cu[-1]) + B
    return rows * V * es


def run_e2e(a, dist, fn, sets, outs, kmax, slots_per_step, stream):
    """The same calls through the public API with the inputs in pinned host memory."""
    import torch
    host = []
    for s in sets:
        h = {}
        for k in ("cu_drafts", "draft_logits", "target_logits", "draft_tokens", "temperature"):
            h[k] = s[k].cpu().pin_memory()
        host.append(h)
    # two device input buffers: step i + 1's host-to-device copy (on its own stream) overlaps
    # step i's kernels; each step still copies all of its inputs and reads back its results
    dbufs = [{k: torch.empty_like(sets[0][k]) for k in host[0]} for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    copy_stream = torch.cuda.Stream()
    results = ("accepted_len", "out_tokens", "n_emitted", "status")
    hout = {k: torch.empty(outs[0][k].shape, dtype=outs[0][k].dtype, pin_memory=True) for k in results}
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values())

    def e2e_step(i):
        h, j = host[i % 3], i % 2
        dbuf = dbufs[j]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(used[j])   # the kernels that last read this buffer are done
            for k in dbuf:
                dbuf[k].copy_(h[k], non_blocking=True)
            copied[j].record(copy_stream)
        stream.wait_event(copied[j])
        o = fn(dbuf["cu_drafts"], dbuf["draft_logits"], dbuf["target_logits"], dbuf["draft_tokens"],
               dbuf["temperature"], kmax, 0, i, out=outs[0])
        used[j].record(stream)
        for k in hout:
            hout[k].copy_(o[k], non_blocking=True)

    n_e2e = max(3, min(a.steps, 30))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_stream(stream)   # no copy of the timed steps starts before e0
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(stream)   # after the last step's results: the stream waited for every copy it used
    torch.cuda.synchronize()
    e2e_ms = dist.max(e0.elapsed_time(e1))
    e2e_value = dist.sum(slots_per_step * n_e2e) / (e2e_ms / 1e3)

    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_ours(a, dist):
    import torch

    import speculative_decoding_block_verify_gb300 as sv
    from speculative_decoding_block_verify_gb300 import workloads

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    sv.lib()
    fn = sv.spec_verify_block if a.rule == "block" else sv.spec_verify_tokenwise
    sets = [workloads.make_verify_inputs(HEADLINE, 3000 + 17 * i + 1000 * dist.rank, backend="torch",
                                         device=dev) for i in range(3)]
    B, kmax, V = sets[0]["B"], sets[0]["kmax"], sets[0]["V"]
    slots_per_step = int(sets[0]["cu_drafts"][-1].item())
    outs = [fn(s["cu_drafts"], s["draft_logits"], s["target_logits"], s["draft_tokens"],
               s["temperature"], kmax, 0, 0) for s in sets]
    stream = torch.cuda.current_stream()

    def step(i):
        s = sets[i % 3]
        fn(s["cu_drafts"], s["draft_logits"], s["target_logits"], s["draft_tokens"],
           s["temperature"], kmax, 0, i, out=outs[i % 3])

    for i in range(a.warmup):
        step(i)
    torch.cuda.synchronize()
    clocks = Clocks(dev.index)
    clocks.start()
    time.sleep(0.3)
    # the timed region: events at its two ends on the launching stream, the calls back to back
    # in between (an event recorded between two calls would put a gap between them), so the
    # average call is the region's time over the number of calls
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(a.steps):
        step(a.warmup + i)
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    local_ms = t0.elapsed_time(t1)
    elapsed_ms = dist.max(local_ms)
    clk = clocks.stop()
    mean_launch_ms = local_ms / a.steps
    total_slots = dist.sum(slots_per_step * a.steps)
    value = total_slots / (elapsed_ms / 1e3)
    alg = statistics.fmean(algorithmic_bytes(s) for s in sets)
    peak, peak_kind = measured_peak()
    achieved = alg / (mean_launch_ms * 1e-3) / 1e9
    traffic = traffic_from_profiles(f"verify_{a.rule}_batch64")
    status_ok = all(int((o["status"] != 0).sum()) == 0 for o in outs)

    e2e = None
    if not a.no_e2e:
        e2e = run_e2e(a, dist, fn, sets, outs, kmax, slots_per_step, stream)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": elapsed_ms / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accum_dtype": "f32",
        "data": "synthetic (seeded torch generator on the device; bf16 logits)",
        "config": {"workload": f"{HEADLINE}: B=64 streams, k=5 drafts + 1 bonus, V=129280, bf16 logits, "
                               f"{a.rule} verification",
                   "B": B, "k": 5, "V": V, "rule": a.rule, "logits": "bf16",
                   "l2": "inputs larger than L2: 3 rotating input sets of 182 MB",
                   "parallelism": f"streams sharded, {dist.world} independent batch(es)"},
        "gpu_launches": 4 * a.steps,   # stats, decide, sweep and finish kernels per call
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "one verify call: stats_kernel, decide_kernel, sweep_kernel, finish_kernel "
                               "on one stream (the logits are read by stats_kernel and sweep_kernel)",
                     "algorithmic_bytes_per_launch": alg, "mean_launch_us": mean_launch_ms * 1e3,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)"},
        "e2e": e2e,
        "clocks": clk,
        "all_status_ok": status_ok,
    }
    if not a.no_secondary and dist.rank == 0:
        result["secondary"] = secondary(sv, workloads, torch, dev)
        result["acceptance"] = [acceptance(sv, workloads, torch, dev, HEADLINE, 3000, a.rule),
                                acceptance(sv, workloads, torch, dev, "batch256_k9", 6000, "block", steps=5)]
    return result


def _time(fn, n, stream):
    import torch
    for _ in range(3):
        fn(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _time_graph(fn, n, stream, replays=5):
    """Device time per call of `fn` with the host's launch overhead taken out: n calls are
    captured in one CUDA graph and the graph is replayed (short kernels are otherwise timed at
    the rate the host can launch them)."""
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (n * replays)


def secondary(sv, workloads, torch, dev):
    """The other workloads, each timed on its own (device time per call, inputs in HBM)."""
    import numpy as np
    stream = torch.cuda.current_stream()
    res = {}
    # batch-64 token-wise
    # every timed call reuses its set's outputs and workspace (allocated by the first call), as
    # the headline does: a call without `out` would also time an allocation and a zero fill
    sets = [workloads.make_verify_inputs(HEADLINE, 5000 + i, backend="torch", device=dev) for i in range(3)]
    outs = {}

    def tw(i):
        s = sets[i % 3]
        outs[i % 3] = sv.spec_verify_tokenwise(s["cu_drafts"], s["draft_logits"], s["target_logits"],
                                               s["draft_tokens"], s["temperature"], 5, 0, i, out=outs.get(i % 3))
    ms = _time(tw, 50, stream)
    alg = algorithmic_bytes(sets[0])
    res["batch64_tokenwise"] = {"us_per_call": ms * 1e3, "slots_per_s": 320 / (ms / 1e3),
                                "GBps": alg / (ms / 1e3) / 1e9}
    del sets
    outs = {}
    # batch-256 k=9 fp32 block
    s = workloads.make_verify_inputs("batch256_k9", 6000, backend="torch", device=dev)

    def blk(i):
        outs[0] = sv.spec_verify_block(s["cu_drafts"], s["draft_logits"], s["target_logits"],
                                       s["draft_tokens"], s["temperature"], 9, 0, i, out=outs.get(0))
    ms = _time(blk, 30, stream)
    alg = algorithmic_bytes(s)
    res["batch256_k9_fp32_block"] = {"us_per_call": ms * 1e3, "slots_per_s": 2304 / (ms / 1e3),
                                     "GBps": alg / (ms / 1e3) / 1e9}
    del s
    outs = {}
    torch.cuda.empty_cache()
    # batch-64 block verify with a reduced draft vocabulary (K = 32,768 draft columns)
    sets = [workloads.make_verify_inputs("batch64_topk", 5100 + i, backend="torch", device=dev) for i in range(3)]

    def red(i):
        s = sets[i % 3]
        outs[i % 3] = sv.spec_verify_block_reduced(s["cu_drafts"], s["draft_logits"], s["t2d"], s["target_logits"],
                                                   s["draft_tokens"], s["temperature"], 5, 0, i, out=outs.get(i % 3))
    ms = _time(red, 50, stream)
    alg = algorithmic_bytes(sets[0])
    res["batch64_topk_block"] = {"us_per_call": ms * 1e3, "slots_per_s": 320 / (ms / 1e3),
                                 "algorithmic_bytes": alg, "GBps": alg / (ms / 1e3) / 1e9,
                                 "draft_vocab": sets[0]["K"]}
    del sets
    torch.cuda.empty_cache()
    # single stream: Markov bias (rank 256) then block verify
    inp = workloads.make_verify_inputs("single_bias", 7000)
    bias = workloads.make_bias_inputs("single_bias", 7000)
    bf = lambda a: torch.as_tensor(np.asarray(a, np.float32), device=dev).to(torch.bfloat16)  # noqa: E731
    dq, dp = bf(inp["draft_logits"]), bf(inp["target_logits"])
    w1, w2 = bf(bias["W1"]), bf(bias["W2"])
    prev = torch.as_tensor(bias["prev"], device=dev)
    cu = torch.as_tensor(inp["cu_drafts"], device=dev)
    x = torch.as_tensor(inp["draft_tokens"], device=dev)
    T = torch.as_tensor(inp["temperature"], device=dev)
    biased = torch.empty(dq.shape, dtype=torch.float32, device=dev)
    scrub = torch.empty(64 << 20, dtype=torch.float32, device=dev)

    def bias_only(i):
        sv.dspark_markov_bias(dq, prev, w1, w2, out=biased)
    ms_warm = _time_graph(bias_only, 50, stream)
    # cold: five copies of W2 (331 MB, more than L2) taken in turn, so that each call reads its
    # W2 from HBM; timed as graph replays so that the host's launch rate does not enter
    w2_set = [w2] + [w2.clone() for _ in range(4)]

    def bias_cold(i):
        sv.dspark_markov_bias(dq, prev, w1, w2_set[i % 5], out=biased)
    ms_cold = _time_graph(bias_cold, 50, stream)
    # the same after a 256 MB write between calls (its time subtracted): the call then also
    # pays for writing back the dirty lines that the scrub left in L2
    def scrub_only(i):
        scrub.fill_(float(i))
    ms_scrub = _time_graph(scrub_only, 20, stream)

    def bias_after_scrub(i):
        scrub.fill_(float(i))
        sv.dspark_markov_bias(dq, prev, w1, w2, out=biased)
    ms_after_scrub = _time_graph(bias_after_scrub, 20, stream) - ms_scrub
    del w2_set
    ms_eager = _time(bias_only, 50, stream)
    w2_bytes = w2.numel() * 2

    outs = {}

    def pipe(i):
        sv.dspark_markov_bias(dq, prev, w1, w2, out=biased)
        outs[0] = sv.spec_verify_block(cu, biased, dp, x, T, 5, 0, i, out=outs.get(0))
    ms_pipe = _time(pipe, 50, stream)
    res["single_bias_then_block"] = {"bias_us_warm_L2": ms_warm * 1e3, "bias_us_cold": ms_cold * 1e3,
                                     "bias_GBps_cold_W2": w2_bytes / (ms_cold / 1e3) / 1e9,
                                     "bias_cold": "5 rotating copies of W2 (331 MB > L2)",
                                     "bias_us_after_write_scrub": ms_after_scrub * 1e3,
                                     "bias_us_eager_launches": ms_eager * 1e3,
                                     "pipeline_us_per_step": ms_pipe * 1e3,
                                     "slots_per_s": 5 / (ms_pipe / 1e3)}
    # the same stream with the draft tokens sampled by the Markov walk (slot i biased by t_{i-1})
    anchor = prev[:1].contiguous()
    wo = sv.dspark_markov_walk(dq.view(1, 5, -1), anchor, w1, w2, T, 0, 0)

    def walk_only(i):
        sv.dspark_markov_walk(dq.view(1, 5, -1), anchor, w1, w2, T, 0, i, out=wo)
    ms_walk = _time(walk_only, 30, stream)

    def walk_then_verify(i):
        sv.dspark_markov_walk(dq.view(1, 5, -1), anchor, w1, w2, T, 0, i, out=wo)
        outs[0] = sv.spec_verify_block(cu, wo["logits"].view(5, -1), dp, wo["tokens"].view(-1), T, 5, 0, i,
                                       out=outs.get(0))
    ms_wv = _time(walk_then_verify, 30, stream)
    res["single_walk_then_block"] = {"walk_us": ms_walk * 1e3, "pipeline_us_per_step": ms_wv * 1e3,
                                     "slots_per_s": 5 / (ms_wv / 1e3)}
    del scrub, wo
    # adaptive: pick k (B=128, H=7168) then ragged block verify
    c = workloads.make_confidence_inputs(12)
    h = torch.as_tensor(c["hidden"], device=dev).to(torch.bfloat16)
    w = torch.as_tensor(c["w"], device=dev).to(torch.bfloat16)
    vm = torch.as_tensor(c["verify_ms"], device=dev)
    pk = sv.adaptive_pick_k(h, w, 0.0, vm)
    kk = pk["k"].cpu().numpy()
    vin = workloads.make_verify_inputs("adaptive128", 13, k=np.full(128, 5), backend="torch", device=dev)

    def pick_only(i):
        sv.adaptive_pick_k(h, w, 0.0, vm, out=pk)
    ms_pick = _time_graph(pick_only, 50, stream)

    outs = {}

    def adaptive(i):
        sv.adaptive_pick_k(h, w, 0.0, vm, out=pk)
        outs[0] = sv.spec_verify_block(pk["cu"], vin["draft_logits"], vin["target_logits"], vin["draft_tokens"],
                                       vin["temperature"], 5, 0, i, out=outs.get(0))
    ms_ad = _time(adaptive, 30, stream)
    res["adaptive128_pick_then_ragged_block"] = {
        "pick_us": ms_pick * 1e3, "pick_GBps": (h.numel() * 2) / (ms_pick / 1e3) / 1e9,
        "pipeline_us_per_step": ms_ad * 1e3, "drafts_verified_per_step": int(kk.sum()),
        "k_histogram": np.bincount(kk, minlength=6).tolist(),
        "slots_per_s": int(kk.sum()) / (ms_ad / 1e3)}
    del vin
    torch.cuda.empty_cache()
    # the same step as one CUDA graph (pick -> verify of each stream's first k_b drafts ->
    # acceptance counters -> step + 1), on the dense draft/target layout the drafter fills
    dn = workloads.make_verify_inputs("adaptive128", 13, backend="torch", device=dev)   # k = 5 everywhere
    B, K, V = 128, 5, dn["V"]
    pl = sv.SpecPipeline(h, w, 0.0, vm, dn["draft_logits"].view(B, K, V), dn["target_logits"].view(B, K + 1, V),
                         dn["draft_tokens"].view(B, K), dn["temperature"], rule=1)
    ms_graph = _time(lambda i: pl.launch(), 30, stream)
    a_p, marg, tps = sv.acceptance_rates(pl.counts, K)
    # the same graph with the online cost curve in the loop (P3): an event pair around every
    # step filed under B + cu_drafts_out[B] tokens, folded in without waiting, the rebuilt
    # table uploaded into the verify_ms the graph reads
    curve = sv.CostCurve(c["verify_ms"])

    def step_with_curve(i):
        curve.begin()
        pl.launch()
        curve.end(B, device_count=pl.out["cu"][B:B + 1])
        curve.poll()
        curve.upload(vm)
    ms_curve = _time(step_with_curve, 64, stream)
    torch.cuda.synchronize()
    curve.poll()
    table, cc = curve.table()
    n_tok = B + int(pl.out["cu"][B].item())
    res["adaptive128_graph"] = {
        "graph_us_per_step": ms_graph * 1e3,
        "eager_us_per_step": ms_ad * 1e3,
        "with_online_cost_curve_us_per_step": ms_curve * 1e3,
        "cost_curve": {"observations": cc["observations"], "rebuilds": cc["rebuilds"],
                       "tokens_last_step": n_tok, "boot_ms": float(c["verify_ms"][n_tok]),
                       "learned_ms": table[n_tok]},
        "drafts_verified_per_step": int(pl.out["k"].sum().item()),
        "a_p": a_p, "tokens_per_step": tps}
    curve.close()
    pl.close()
    del dn, pl
    torch.cuda.empty_cache()
    # the tiny configuration's latency (B = 1, k = 5, V = 1024, fp32)
    tiny = workloads.make_verify_inputs("tiny", 1000, backend="torch", device=dev)
    to = sv.spec_verify_block(tiny["cu_drafts"], tiny["draft_logits"], tiny["target_logits"], tiny["draft_tokens"],
                              tiny["temperature"], 5, 0, 0)

    def tiny_call(i):
        sv.spec_verify_block(tiny["cu_drafts"], tiny["draft_logits"], tiny["target_logits"], tiny["draft_tokens"],
                             tiny["temperature"], 5, 0, i, out=to)
    res["tiny_block_latency_us"] = _time(tiny_call, 200, stream) * 1e3
    res["tiny_block_device_us"] = _time_graph(tiny_call, 50, stream) * 1e3
    return res


def acceptance(sv, workloads, torch, dev, name, seed, rule, steps=30):
    """Per-position acceptance a_p, the marginal a_p / a_{p-1}, tokens per step = 1 + sum a_p
    (P1 §6) and the status counts of `steps` untimed calls on the workload."""
    import numpy as np
    inp = workloads.make_verify_inputs(name, seed, backend="torch", device=dev)
    k = inp["kmax"]
    fn = sv.spec_verify_block if rule == "block" else sv.spec_verify_tokenwise
    counts, status = None, np.zeros(8, np.int64)
    out = None
    for i in range(steps):
        out = fn(inp["cu_drafts"], inp["draft_logits"], inp["target_logits"], inp["draft_tokens"],
                 inp["temperature"], k, 0, i, out=out)
        counts = sv.spec_accept_counters(out["accepted_len"], out["status"], inp["cu_drafts"], k, counts)
        status += np.bincount(out["status"].cpu().numpy(), minlength=8)[:8]
    a_p, marg, tps = sv.acceptance_rates(counts, k)
    del inp
    torch.cuda.empty_cache()
    return {"workload": name, "rule": rule, "steps": steps, "a_p": a_p, "marginal": marg,
            "tokens_per_step": tps,
            "status_counts": {sv.STATUS_NAMES[j]: int(status[j]) for j in range(8) if status[j]}}


def run_reference(a, dist):
    """The oracle (float64 NumPy, host cores) on the headline workload, one bounded sample per
    step; rank 0 only."""
    res_steps = []
    pool, _ = oracle_pool()
    try:
        for i in range(a.warmup + a.steps):
            r = oracle_sample(a.ref_sample, a.rule, seed=3000 + i % 4, pool=pool)
            if i >= a.warmup:
                res_steps.append(r)
    finally:
        pool.close()
        pool.join()
    value = statistics.fmean(r["value"] for r in res_steps)
    cb = dict(res_steps[-1])
    cb["value"] = value
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: B=64 streams, k=5 drafts + 1 bonus, V=129280, bf16 logits, "
                               f"{a.rule} verification", "B": 64, "k": 5, "V": 129280, "rule": a.rule},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    a = parse()
    dist = Dist()
    try:
        if a.impl == "reference":
            if dist.rank != 0:
                return
            print(json.dumps(run_reference(a, dist)), flush=True)
            return
        cpu = None
        if dist.rank == 0 and not a.no_cpu_baseline:
            cpu = oracle_sample(a.cpu_sample, a.rule)   # before the first GPU call (spawned pool)
        res = run_ours(a, dist)
        if dist.rank == 0:
            res["cpu_baseline"] = cpu
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
