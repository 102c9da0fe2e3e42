"""Throughput of speculative-decoding verification on GB300.

One step = the whole hot path over one batch: the tree-attention mask, the vocabulary-streaming
row statistics over every (request, node) row, the per-request walk with rejection sampling,
the inverse-CDF bonus draw and the accepted-path compaction, on the large-tree workload
(B=256 requests, N=64-node random tries, V=152064 bf16 logits, temperature 1.0, point-mass
drafts, supplied uniforms). Inputs are synthetic and seeded.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank verifies its own batch (requests are independent: weak scaling, no
collective on the data path); the time is the max over ranks and rank 0 prints one JSON line.
``--impl reference`` times the float64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_tree_mask_gb300 import workloads as W  # noqa: E402

METRIC = "verified draft nodes/s and logit-read GB/s (% of HBM peak), B=256 N=64 V=152064"
UNIT = "draft nodes/s"
WORKLOAD = "large_tree"
FALLBACK_HBM_GBS = 6800.0
REF_BUDGET_S = 150.0   # wall time the reference arm's timed and warm-up steps may take


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def rank_seed(w: W.Workload, rank: int) -> int:
    """Every rank verifies its own batch of independent requests (weak scaling)."""
    return w.seed + rank


def aggregate_throughput(world: int, draft_nodes_per_rank: int, max_ms: float) -> float:
    """Whole-job draft nodes/s: all ranks' nodes over the slowest rank's step time."""
    return world * draft_nodes_per_rank / (max_ms / 1e3)


def config_of(w: W.Workload, world: int) -> dict:
    return {"workload": f"{w.name}: B={w.B} N={w.N} V={w.V} {w.dtype} T={w.temperature} "
                        f"point-mass drafts, random tries depth<={w.max_depth} "
                        f"branching 1-{w.max_branch}",
            "global_batch": w.B * world, "nodes_per_request": w.N, "vocab": w.V,
            "parallelism": f"independent requests x{world}",
            "l2": "inputs larger than L2 (logits %.2f GB per step)" % (w.B * w.N * w.V * 2 / 1e9)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace collapsed: what the compiler
    sees (the sources hold no string literal with a comment marker in it)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_sha(files) -> str:
    """Hash of the code of the kernel's source files (the .cu and every header it includes),
    comments left out: a comment edit does not change the kernel."""
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "speculative_decoding_tree_mask_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_record(kernel_file: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if none of the
    kernel's source files changed since the capture; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_file)
    if not rec:
        return None
    return rec["bytes_per_launch"] if rec.get("source_sha") == source_sha(rec["sources"]) \
        else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running. `mark()` brackets
    a timed region; `summary(region=True)` then takes the samples within one sampling
    interval of it (so even a region shorter than the interval has the samples on both
    sides of it), `summary()` every sample."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []          # (host time, line)
        self.region = None
        self.first = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def wait_first(self, timeout: float = 3.0):
        """Wait (bounded) until the sampler has produced its first sample."""
        if self.proc is not None:
            self.first.wait(timeout)

    def mark(self, start: float, end: float):
        self.region = (start, end)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))
            self.first.set()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, region: bool = False):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if region and self.region is not None:
            pad = self.interval_ms / 1e3
            a, z = self.region[0] - pad, self.region[1] + pad
            lines = [(t, ln) for t, ln in lines if a <= t <= z]
        for _, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "interval_ms": self.interval_ms}


def run_oracle_sample(x, w, nthreads: int, reps_target_s: float = 10.0, max_reps: int = 5):
    """The oracle over the whole batch, repeated for about reps_target_s: (draft nodes/s,
    repetitions, seconds, the oracle's outputs)."""
    from oracle import oracle as O
    orc = O.default()
    logits = W.host_logits(x["logits"])
    u = x["uniforms"].cpu().numpy()
    t0 = time.perf_counter()
    reps = 0
    while True:
        ref = orc.verify_sample(logits, x["tok_np"], x["parent_np"], w.temperature, u,
                                nthreads=nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= reps_target_s or reps >= max_reps:
            break
    return reps * w.draft_nodes / el, reps, el, ref


OUT_KEYS = ("accept_len", "out_tokens", "kv_commit", "bonus", "status")
MARGIN = 1e-6


def parity_summary(gpu: dict, ref: dict) -> dict:
    """Request-by-request agreement of the GPU's outputs with the oracle's on the same batch.
    A request whose accept decision lies within MARGIN of the oracle's threshold is counted
    apart (float32 against float64 may decide it either way). A request whose bonus draw lies
    within MARGIN of a CDF boundary must match in everything but the bonus, and its bonus must
    lie in the oracle's draw window [cdf_lo, cdf_hi]."""
    B = len(ref["accept_len"])
    excl = np.asarray(ref["decision_margin"]) < MARGIN
    near = (np.asarray(ref["cdf_margin"]) < MARGIN) & ~excl
    identical = np.ones(B, bool)
    for k in OUT_KEYS:
        identical &= np.asarray(gpu[k]).reshape(B, -1).__eq__(
            np.asarray(ref[k]).reshape(B, -1)).all(1)
    near_ok = np.zeros(B, bool)
    for i in np.nonzero(near & ~identical)[0]:
        L = int(ref["accept_len"][i])
        same = all(np.array_equal(np.asarray(gpu[k])[i], np.asarray(ref[k])[i])
                   for k in ("accept_len", "kv_commit", "status"))
        g_out, r_out = np.array(gpu["out_tokens"][i]), np.array(ref["out_tokens"][i])
        gb = int(gpu["bonus"][i])
        g_out[L] = r_out[L]
        near_ok[i] = (same and np.array_equal(g_out, r_out) and
                      int(ref["cdf_lo"][i]) <= gb <= int(ref["cdf_hi"][i]) and
                      int(gpu["out_tokens"][i][L]) == gb)
    agree = identical | near_ok
    return {"requests": B, "identical": int(identical.sum()),
            "near_boundary_in_window": int((near_ok & ~identical).sum()),
            "decision_margin_cases": int(excl.sum()),
            "decision_margin_differing": int((excl & ~agree).sum()),
            "mismatched": int((~agree & ~excl).sum()),
            "margin": MARGIN}


def greedy_parity(gpu: dict, ref: dict) -> dict:
    """Greedy results must equal the oracle's bit for bit, request by request."""
    B = len(ref["accept_len"])
    same = np.ones(B, bool)
    for k in OUT_KEYS:
        same &= np.asarray(gpu[k]).reshape(B, -1).__eq__(np.asarray(ref[k]).reshape(B, -1)).all(1)
    return {"requests": B, "identical": int(same.sum()), "mismatched": int((~same).sum())}


def snapshot(out: dict) -> dict:
    """Host copies of a call's outputs (taken right after the call's timed region)."""
    return {k: out[k].cpu().numpy() for k in OUT_KEYS}


def oracle_parity(x, w, results: dict, nthreads: int, ref: dict | None = None) -> dict:
    """Every request of the batch `x` verified by the oracle (sampling and greedy) and
    compared with the GPU's outputs in `results` (name -> (mode, outputs)). `ref` may hold
    the oracle's sampling result for `x` already."""
    from oracle import oracle as O
    orc = O.default()
    logits = W.host_logits(x["logits"])
    u = x["uniforms"].cpu().numpy()
    ref = dict(ref or {})
    if "sample" not in ref and any(m == "sample" for m, _ in results.values()):
        ref["sample"] = orc.verify_sample(logits, x["tok_np"], x["parent_np"], w.temperature, u,
                                          nthreads=nthreads)
    if any(m == "greedy" for m, _ in results.values()):
        ref["greedy"] = orc.verify_greedy(logits, x["tok_np"], x["parent_np"],
                                          nthreads=nthreads)
    del logits
    return {name: (parity_summary(g, ref["sample"]) if mode == "sample"
                   else greedy_parity(g, ref["greedy"]))
            for name, (mode, g) in results.items()}


def bench_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    w = W.WORKLOADS[WORKLOAD]
    if args.requests:
        w = w.scaled(B=args.requests)
    dev = f"cuda:{local}" if torch.cuda.is_available() else "cpu"
    x = W.make(w, device=dev)
    from oracle import oracle as O
    orc = O.default()
    nthreads = os.cpu_count() or 1
    logits = W.host_logits(x["logits"])
    u = x["uniforms"].cpu().numpy()
    tok, par = x["tok_np"], x["parent_np"]
    del x["logits"]
    # One untimed pass over the whole batch sizes the per-step sample: every step verifies the
    # first n requests, n chosen so that the whole run stays within about REF_BUDGET_S.
    t0 = time.perf_counter()
    orc.verify_sample(logits, tok, par, w.temperature, u, nthreads=nthreads)
    t_full = time.perf_counter() - t0
    calls = args.warmup + args.steps
    n = w.B
    if calls * t_full > REF_BUDGET_S:
        n = max(1, int(w.B * REF_BUDGET_S / (calls * t_full)))
    logits, tok, par, u = logits[:n], tok[:n], par[:n], u[:n]
    times = []
    for i in range(calls):
        t0 = time.perf_counter()
        orc.verify_sample(logits, tok, par, w.temperature, u, nthreads=nthreads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = n * (w.N - 1) / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random tries and N(0,3) logits)", "config": config_of(w, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": f"the first {n} of the {w.B} requests of the {WORKLOAD} "
                                       "batch per step, float64 C oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_ours(args):
    from speculative_decoding_tree_mask_gb300 import binding as G

    rank, world, local = dist_env()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    w = W.WORKLOADS[WORKLOAD]
    if args.requests:
        w = w.scaled(B=args.requests)
    run_clocks = ClockSampler(local).__enter__()   # the whole run, all legs
    x = W.make(w, device=dev, seed=rank_seed(w, rank))
    B, N, V, T = w.B, w.N, w.V, w.temperature
    h = G.Handle(B, N, V, local)
    mask = dict(anc_mask=torch.empty((B, N), dtype=torch.int64, device=dev),
                depth=torch.empty((B, N), dtype=torch.int32, device=dev),
                status=torch.empty(B, dtype=torch.int32, device=dev))
    out = G.alloc_outputs(B, N, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"], mask["status"],
                               stream)
        G.spec_verify_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"],
                             out["accept_len"], out["out_tokens"], out["kv_commit"],
                             out["bonus"], out["status"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        clocks.wait_first()
        t_start = time.perf_counter()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(t_start, time.perf_counter())
        time.sleep(clocks.interval_ms / 1e3 * 1.5)   # the sample after the region
    barrier(world)
    ms = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms, world, dev)
    value = aggregate_throughput(world, w.draft_nodes, ms)
    outs = {"eager_sample": ("sample", snapshot(out))}
    # Per-kernel durations: the same K steps again with CUDA events around every launch (on the
    # launching stream). The events sit between the kernels, so they also stop the stages from
    # overlapping their launches; that is why the headline region above runs without them.
    G.spec_profile_begin(h)
    torch.cuda.synchronize(dev)
    ps, pe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ps.record(stream)
    for _ in range(args.steps):
        step()
    pe.record(stream)
    torch.cuda.synchronize(dev)
    prof = G.spec_profile_end(h)
    ms_profiled = max_over_ranks(ps.elapsed_time(pe) / args.steps, world, dev)

    # dominant kernel: row statistics over all B*N rows
    rs_ms, rs_n = prof["row_stats"]
    rs_avg = rs_ms / max(rs_n, 1)
    alg_bytes = B * N * V * w.elem_bytes
    pk, pk_kind = peaks()
    achieved = alg_bytes / (rs_avg / 1e3) / 1e9
    # The committed DRAM-traffic record was captured on the full large-tree batch: it holds
    # only for a run of that batch (and only while the kernel's code is unchanged).
    full_batch = B == W.WORKLOADS[WORKLOAD].B
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic_record("row_stats.cu") if full_batch else None,
                "kernel": "row_stats_kernel<bf16, sample>", "peak_source": pk_kind,
                "algorithmic_bytes_per_launch": alg_bytes, "avg_launch_ms": rs_avg}
    if not full_batch:
        roofline["traffic_note"] = (f"null: the DRAM capture covers all {W.WORKLOADS[WORKLOAD].B}"
                                    f" requests, this run verified {B}")
    step_bytes = alg_bytes  # logits read once per step (bonus row and metadata excluded)
    # Secondary bound of the sampling stream: one exponential (ex2 on the special-function
    # unit) per logit. GB300's special-function units retire 32 ex2 per SM per clock (twice
    # the rate of the earlier Blackwell part), so the peak is SMs x 32 x max SM clock.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = pk.get("sm_max_mhz", 2070.0)
    ex2_peak = sms * 32 * sm_mhz * 1e6 / 1e12
    ex2_achieved = B * N * V / (rs_avg / 1e3) / 1e12
    sfu = {"bound": "sfu", "achieved": ex2_achieved, "peak": ex2_peak, "unit": "Tex2/s",
           "frac": ex2_achieved / ex2_peak, "kernel": "row_stats_kernel<bf16, sample>",
           "peak_source": f"derived: {sms} SMs x 32 ex2 per clock x {sm_mhz:.0f} MHz",
           "ex2_per_launch": B * N * V}
    kernels = {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]}
               for k, v in prof.items() if v[1]}

    # greedy verification of the same trees (argmax path, no exponentials)
    gout = G.alloc_outputs(B, N, dev)

    def greedy_step():
        G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"], mask["status"],
                               stream)
        G.spec_verify_greedy(h, x["logits"], x["draft_token"], x["parent"], gout["accept_len"],
                             gout["out_tokens"], gout["kv_commit"], gout["bonus"],
                             gout["status"], stream=stream)

    for _ in range(args.warmup):
        greedy_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gs.record(stream)
    for _ in range(args.steps):
        greedy_step()
    ge.record(stream)
    torch.cuda.synchronize(dev)
    gms = max_over_ranks(gs.elapsed_time(ge) / args.steps, world, dev)
    outs["eager_greedy"] = ("greedy", snapshot(gout))
    greedy = {"value": aggregate_throughput(world, w.draft_nodes, gms), "unit": UNIT,
              "ms_per_step": gms, "logit_GBps": alg_bytes / (gms / 1e3) / 1e9,
              "path": "tree mask + spec_verify_greedy (row statistics without exponentials, "
                      "warp-per-request walk)",
              "accept_len_mean": float(gout["accept_len"].float().mean().item())}

    # lazy verification: the same outputs, reading only the rows the walk visits
    lazy = None
    if not args.skip_lazy:
        lout = G.alloc_outputs(B, N, dev)

        def lazy_step():
            G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"],
                                   mask["status"], stream)
            G.spec_verify_sample_lazy(h, x["logits"], x["draft_token"], x["parent"], T,
                                      x["uniforms"], lout["accept_len"], lout["out_tokens"],
                                      lout["kv_commit"], lout["bonus"], lout["status"],
                                      stream=stream)

        for _ in range(args.warmup):
            lazy_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        s3, t3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        G.spec_profile_begin(h)
        s3.record(stream)
        for _ in range(args.steps):
            lazy_step()
        t3.record(stream)
        torch.cuda.synchronize(dev)
        lprof = G.spec_profile_end(h)
        direct_ms = max_over_ranks(s3.elapsed_time(t3) / args.steps, world, dev)
        # The lazy step is short enough that issuing two calls from Python per step can take
        # longer than the GPU work, so the step is also captured once in a CUDA graph and
        # replayed: that is the device throughput.
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            lazy_step_on = lambda: (  # noqa: E731
                G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"],
                                       mask["status"], side),
                G.spec_verify_sample_lazy(h, x["logits"], x["draft_token"], x["parent"], T,
                                          x["uniforms"], lout["accept_len"], lout["out_tokens"],
                                          lout["kv_commit"], lout["bonus"], lout["status"],
                                          stream=side))
            lazy_step_on()
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                lazy_step_on()
        stream.wait_stream(side)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        barrier(world)
        s4, t4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s4.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t4.record(stream)
        torch.cuda.synchronize(dev)
        lms = max_over_ranks(s4.elapsed_time(t4) / args.steps, world, dev)
        al = lout["accept_len"].cpu()
        outs["lazy_sample"] = ("sample", snapshot(lout))
        ndiff = int((lout["out_tokens"] != out["out_tokens"]).any(dim=1).sum().item())
        lazy = {"value": aggregate_throughput(world, w.draft_nodes, lms), "unit": UNIT,
                "ms_per_step": lms, "ms_per_step_direct_calls": direct_ms,
                "path": "tree mask + spec_verify_sample_lazy, one CUDA graph replayed per step",
                "rows_streamed_per_step": int(al.sum().item()) + B,
                "kernels": {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]}
                            for k, v in lprof.items() if v[1]},
                "requests_differing_from_eager": ndiff}
        # lazy greedy: the argmax path only, same trees, one graph per step
        lgout = G.alloc_outputs(B, N, dev)
        ggraph = torch.cuda.CUDAGraph()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            lazy_greedy_on = lambda: (  # noqa: E731
                G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"],
                                       mask["status"], side),
                G.spec_verify_greedy_lazy(h, x["logits"], x["draft_token"], x["parent"],
                                          lgout["accept_len"], lgout["out_tokens"],
                                          lgout["kv_commit"], lgout["bonus"], lgout["status"],
                                          stream=side))
            lazy_greedy_on()
            side.synchronize()
            with torch.cuda.graph(ggraph, stream=side):
                lazy_greedy_on()
        stream.wait_stream(side)
        for _ in range(args.warmup):
            ggraph.replay()
        torch.cuda.synchronize(dev)
        s5, t5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s5.record(stream)
        for _ in range(args.steps):
            ggraph.replay()
        t5.record(stream)
        torch.cuda.synchronize(dev)
        gl_ms = max_over_ranks(s5.elapsed_time(t5) / args.steps, world, dev)
        outs["lazy_greedy"] = ("greedy", snapshot(lgout))
        lazy["greedy"] = {"value": aggregate_throughput(world, w.draft_nodes, gl_ms),
                          "ms_per_step": gl_ms,
                          "rows_streamed_per_step":
                              int(lgout["accept_len"].sum().item()) + B,
                          "outputs_equal_eager_greedy": bool(
                              torch.equal(lgout["out_tokens"], gout["out_tokens"]) and
                              torch.equal(lgout["kv_commit"], gout["kv_commit"]))}

    # End to end, inputs in pinned host memory and results read back every step.
    # e2e: the lazy call reads the logits rows it needs straight from pinned host memory over
    # the host link (the small inputs are copied); e2e_copy: all logits are copied to the
    # device, then the eager call runs.
    e2e = e2e_copy = None
    if not args.skip_e2e:
        hl = torch.empty_like(x["logits"], device="cpu").pin_memory()
        hl.copy_(x["logits"])
        hsmall = {k: x[k].cpu().pin_memory() for k in ("draft_token", "parent", "uniforms")}
        hout = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in out.items()}
        hmask = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in mask.items()}
        small_h2d = sum(t.numel() * t.element_size() for t in hsmall.values())
        d2h = sum(t.numel() * t.element_size() for t in list(hout.values()) +
                  list(hmask.values()))
        row_bytes = V * w.elem_bytes

        def fetch_small():
            for k, t in hsmall.items():
                x[k].copy_(t, non_blocking=True)

        def read_back():
            for k, t in hout.items():
                t.copy_(out[k], non_blocking=True)
            for k, t in hmask.items():
                t.copy_(mask[k], non_blocking=True)

        # The zero-copy step moves its small inputs in one host-to-device copy and its results
        # in one device-to-host copy: the tensors are views into one buffer each way (eleven
        # small copies cost about 25 us per step).
        zin_h, zin_h_views = packed({k: x[k] for k in ("draft_token", "parent", "uniforms")},
                                    "cpu")
        zin_d, zin = packed({k: x[k] for k in ("draft_token", "parent", "uniforms")}, dev)
        for k, t in zin_h_views.items():
            t.copy_(x[k])
        zout_d, zout = packed({**out, **{"m_" + k: v for k, v in mask.items()}}, dev)
        zout_h, zout_h_views = packed(zout, "cpu")

        def zero_copy_step():
            zin_d.copy_(zin_h, non_blocking=True)
            G.spec_build_tree_mask(h, zin["parent"], zout["m_anc_mask"], zout["m_depth"],
                                   zout["m_status"], stream)
            G.spec_verify_sample_lazy(h, hl, zin["draft_token"], zin["parent"], T,
                                      zin["uniforms"], zout["accept_len"], zout["out_tokens"],
                                      zout["kv_commit"], zout["bonus"], zout["status"],
                                      stream=stream)
            zout_h.copy_(zout_d, non_blocking=True)

        def copy_step():
            x["logits"].copy_(hl, non_blocking=True)
            fetch_small()
            step()
            read_back()

        def timed_e2e(fn, k):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            barrier(world)
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(k):
                fn()
            z.record(stream)
            torch.cuda.synchronize(dev)
            return max_over_ranks(a.elapsed_time(z) / k, world, dev)

        zms = timed_e2e(zero_copy_step, args.e2e_steps * 10)
        # one statistics pass per visited node, then about 1/16 of the stop row for the bonus
        # (the chunk holding the draw, out of the 16 the lazy pass records)
        rows_read = int(zout_h_views["accept_len"].sum().item()) + B
        link_bytes = rows_read * row_bytes + B * (V // 16) * w.elem_bytes
        e2e = {"value": aggregate_throughput(world, w.draft_nodes, zms), "unit": UNIT,
               "h2d_bytes_per_step": int(small_h2d + link_bytes),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": zms,
               "steps": args.e2e_steps * 10, "host_link_GBps": link_bytes / zms / 1e6,
               "path": "spec_verify_sample_lazy reading pinned host logits over the host link "
                       "(one pass per visited row, one sixteenth of the stop row for the "
                       "bonus)"}
        cms = timed_e2e(copy_step, args.e2e_steps)
        e2e_copy = {"value": aggregate_throughput(world, w.draft_nodes, cms), "unit": UNIT,
                    "h2d_bytes_per_step": int(hl.numel() * hl.element_size() + small_h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": cms,
                    "steps": args.e2e_steps,
                    "h2d_GBps": (hl.numel() * hl.element_size() + small_h2d) / cms / 1e6,
                    "path": "all logits copied host to device, then spec_verify_sample"}

    # f2 and f1 on their own workloads: the KV commit after a verify call, and the dense chain
    check = rank == 0 and not args.skip_parity
    extra = {} if args.skip_extra else {"kv_commit": bench_kv_commit(dev, stream, args),
                                        "dense_chain": bench_dense_chain(dev, stream, args,
                                                                         check),
                                        "small_tries": bench_small_tries(dev, stream, args,
                                                                         check),
                                        "high_accept": bench_high_accept(h, w, mask, dev,
                                                                         stream, args, check),
                                        "adaptive_budget": bench_budget(h, x, w, dev, stream,
                                                                        args)}

    nthreads = os.cpu_count() or 1
    cpu = oref = None
    if rank == 0 and not args.skip_cpu_baseline:
        cval, reps, el, oref = run_oracle_sample(x, w, nthreads)
        cpu = {"value": cval, "unit": UNIT, "cores": nthreads, "kind": "oracle",
               "sample": f"the whole {WORKLOAD} batch ({w.B} requests) x{reps} "
                         f"({el:.1f} s), float64 C oracle, OpenMP over requests"}
    # Every request of the headline batch against the oracle: the outputs of the timed eager
    # steps, of the greedy leg and of the two lazy legs.
    parity = None
    if check:
        try:
            parity = oracle_parity(x, w, outs, nthreads, {"sample": oref} if oref else None)
            parity["margin"] = MARGIN
        except Exception as e:   # the line is printed whatever happens here
            parity = {"error": repr(e)[:200]}
        if lazy is not None and "lazy_sample" in parity:
            lazy["vs_oracle"] = parity["lazy_sample"]

    hist = np.bincount(out["accept_len"].cpu().numpy(), minlength=1).tolist()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic (seeded random tries and N(0,3) logits)",
                "config": config_of(w, world),
                "logit_GBps": step_bytes / (ms / 1e3) / 1e9,
                "logit_hbm_frac_of_measured": step_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                "rows_per_s": B * N * world / (ms / 1e3),
                "roofline": roofline, "secondary_bound": sfu,
                "cpu_baseline": cpu, "e2e": e2e, "e2e_copy": e2e_copy,
                "greedy": greedy, "lazy": lazy, "parity": parity, **extra,
                "gpu_launches": 3 * args.steps, "kernels": kernels,
                "ms_per_step_with_kernel_events": ms_profiled,
                "clocks": clocks.summary(region=True), "accept_len_hist": hist}
        run_clocks.__exit__(None, None, None)
        line["clocks_whole_run"] = dict(
            run_clocks.summary(),
            note="nvidia-smi every 50 ms over the whole run (all legs), beside the timed "
                 "region's own samples in clocks")
        print(json.dumps(line), flush=True)
    else:
        run_clocks.__exit__(None, None, None)
    h.close()
    if world > 1:
        torch.distributed.destroy_process_group()


SPIN_CYCLES = 400_000   # about 0.2 ms of GPU spin: longer than the host takes to issue a call


def _time_calls(fn, stream, steps, warmup, flush=None):
    """Mean device milliseconds of fn() over `steps` calls (events on `stream`), each call
    preceded by an L2 flush when `flush` (a device buffer larger than L2) is given: the buffer
    is read, so the flush leaves no dirty lines to be written back during the timed call.
    Between the flush and the start event the GPU spins for SPIN_CYCLES, so that every launch
    of the call is queued before the start event is reached: the timed region then holds the
    call's kernels only, not the host's time to issue them (which a single short call would
    otherwise expose as idle GPU time)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(steps):
        if flush is not None:
            flush.max()
        torch.cuda._sleep(SPIN_CYCLES)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        z.record(stream)
        torch.cuda.synchronize()
        total += a.elapsed_time(z)
    return total / steps


def call_floor(dev, stream, flush) -> dict:
    """The protocol's own floor: one tiny torch kernel timed like a verify call, with and
    without the spin before the start event."""
    e = torch.zeros(1, device=dev)
    with_spin = _time_calls(lambda: e.add_(1), stream, 50, 5, flush)
    tot = 0.0
    for _ in range(50):
        flush.max()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e.add_(1)
        z.record(stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(z)
    return {"tiny_kernel_us": with_spin * 1e3, "tiny_kernel_us_without_spin": tot / 50 * 1e3}


def _kernel_split(h, fn, stream, steps, flush):
    """Per-kernel device times of fn() (CUDA events around every launch, L2 flushed before
    each call): {kernel class: ms per launch}."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    G.spec_profile_begin(h)
    for _ in range(steps):
        flush.max()
        torch.cuda._sleep(SPIN_CYCLES)
        fn()
    torch.cuda.synchronize()
    prof = G.spec_profile_end(h)
    return {k: v[0] / v[1] for k, v in prof.items() if v[1]}


def packed(tensors: dict, device):
    """One byte buffer holding every tensor of `tensors` at 16-byte aligned offsets (pinned host
    memory for "cpu"), and views of it with the tensors' names, shapes and dtypes."""
    offs, total = {}, 0
    for k, t in tensors.items():
        total = (total + 15) // 16 * 16
        offs[k] = total
        total += t.numel() * t.element_size()
    if str(device) == "cpu":
        buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    else:
        buf = torch.empty(total, dtype=torch.uint8, device=device)
    views = {k: buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for (k, t), o in zip(tensors.items(), offs.values())}
    return buf, views


def _hbm(bytes_moved: int, ms: float) -> dict:
    pk, kind = peaks()
    gbs = bytes_moved / (ms / 1e3) / 1e9
    return {"GBps": gbs, "peak": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"],
            "peak_source": kind}


def bench_kv_commit(dev, stream, args):
    """KV commit of 8 slots per request (root + 7 accepted) for B=256, N=64, 32 heads x 128,
    bf16 sources, into an NHD paged cache of 16-token blocks: bf16 and fp8 (e4m3) caches. Its
    own handle, sized for this workload whatever the verify legs' batch."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    B, N, H, D, bs = 256, 64, 32, 128, 16
    with G.Handle(B, N, 1 << 10, dev.index if dev.index is not None else 0) as h:
        return _kv_commit_legs(h, dev, stream, B, N, H, D, bs)


def _kv_commit_legs(h, dev, stream, B, N, H, D, bs):
    from speculative_decoding_tree_mask_gb300 import binding as G
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    src_k = torch.randn((B, N, H, D), device=dev, generator=g).to(torch.bfloat16)
    src_v = torch.randn((B, N, H, D), device=dev, generator=g).to(torch.bfloat16)
    L = 7
    kv = torch.full((B, N), -1, dtype=torch.int32, device=dev)
    kv[:, :L + 1] = torch.arange(L + 1, dtype=torch.int32, device=dev) * 5   # root, then a path
    kv[:, 0] = 0
    al = torch.full((B,), L, dtype=torch.int32, device=dev)
    max_blocks = 8
    table = torch.randperm(B * max_blocks, device=dev, generator=g).to(torch.int32).view(
        B, max_blocks)
    pos = torch.full((B,), 37, dtype=torch.int32, device=dev)
    flush = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    # fp8 caches: a power-of-two scale (one multiply per element), and a scale that is not one
    # (the reciprocal route with its rounding-boundary test)
    for name, cache_kind, esz, sv in (("bf16", G.SPEC_CACHE_SAME, 2, None),
                                      ("fp8_e4m3", G.SPEC_CACHE_FP8_E4M3, 1, 0.5),
                                      ("fp8_e4m3_scale_0.0173", G.SPEC_CACHE_FP8_E4M3, 1, 0.0173)):
        cdt = torch.bfloat16 if esz == 2 else torch.uint8
        ck = torch.zeros((B * max_blocks, bs, H, D), dtype=cdt, device=dev)
        cv = torch.zeros_like(ck)
        scale = torch.tensor([sv], device=dev) if sv is not None else None

        def call():
            G.spec_kv_commit(h, src_k, src_v, kv, al, ck, cv, G.SPEC_KV_NHD, table, pos,
                             cache_kind=cache_kind, k_scale=scale, v_scale=scale, stream=stream)

        ms = _time_calls(call, stream, 50, 5, flush)
        moved = B * (L + 1) * 2 * H * D * (2 + esz)   # read K and V, write them into the cache
        out[name] = {"ms_per_call": ms, "bytes": moved, **_hbm(moved, ms)}
    out["config"] = ("B=256 N=64, 8 slots per request, H=32 D=128 bf16 sources, NHD cache of "
                     "16-token blocks; fp8 per-tensor scale 0.5 or 0.0173; L2 flushed before "
                     "every call")
    return out


def bench_dense_chain(dev, stream, args, check=False):
    """The dense-chain workload (B=64, k=5, V=128256, bf16 target and draft logits), one
    spec_verify_sample call with dense draft logits; L2 flushed before every call. The
    algorithmic bytes are the target rows and the draft rows of the inner nodes (the last
    draft row drafts nothing and is not read)."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    w = W.WORKLOADS["dense_chain"]
    x = W.make(w, device=dev, seed=w.seed)
    with G.Handle(w.B, w.N, w.V, dev.index if dev.index is not None else 0) as hd:
        out = G.alloc_outputs(w.B, w.N, dev)
        flush = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

        def call():
            G.verify_sample(hd, x["logits"], x["draft_token"], x["parent"], w.temperature,
                            x["uniforms"], draft=x["draft"], draft_kind=G.SPEC_DRAFT_LOGITS,
                            out=out, stream=stream)

        ms = _time_calls(call, stream, 50, 5, flush)
        row = w.V * x["logits"].element_size()
        moved = 2 * x["logits"].numel() * x["logits"].element_size()
        alg = w.B * (2 * w.N - 1) * row
        res = {"ms_per_call": ms, "value": w.B * (w.N - 1) / (ms / 1e3), "unit": UNIT,
               "logits_bytes": moved, "algorithmic_bytes": alg,
               "roofline": dict(_hbm(alg, ms), bound="hbm"),
               "kernels_ms": _kernel_split(hd, call, stream, 20, flush),
               "accept_len_mean": float(out["accept_len"].float().mean().item()),
               "config": "dense_chain: B=64, 5 drafts, V=128256, bf16 target and draft "
                         "logits, T=1; L2 flushed before every call"}
        if check:
            res["parity"] = dense_parity(x, w, snapshot(out))
        res["protocol_floor"] = call_floor(dev, stream, flush)
        return res


def dense_parity(x, w, got: dict) -> dict:
    from oracle import oracle as O
    ref = O.default().verify_sample(W.host_logits(x["logits"]), x["tok_np"], x["parent_np"],
                                    w.temperature, x["uniforms"].cpu().numpy(),
                                    draft=W.host_logits(x["draft"]),
                                    draft_kind=O.DRAFT_LOGITS, nthreads=os.cpu_count() or 1)
    return parity_summary(got, ref)


def bench_high_accept(h, w, mask, dev, stream, args, check=False):
    """The large-tree step on trees that the target mostly accepts: the same shapes with the
    grammar token boosted by 20 instead of 8 (p of a boosted child about 0.97 at T=1), so walks
    go several levels deep and a few requests reject a dominant token (the walk's full-row
    re-sums). Timed like the headline step, then once more with per-kernel events."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    wd = w.scaled(boost=20.0)
    xd = W.make(wd, device=dev, seed=wd.seed + 7919)
    out = G.alloc_outputs(wd.B, wd.N, dev)
    steps = min(args.steps, 500)

    def step():
        G.spec_build_tree_mask(h, xd["parent"], mask["anc_mask"], mask["depth"],
                               mask["status"], stream)
        G.spec_verify_sample(h, xd["logits"], xd["draft_token"], xd["parent"], wd.temperature,
                             xd["uniforms"], out["accept_len"], out["out_tokens"],
                             out["kv_commit"], out["bonus"], out["status"], stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    z.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / steps
    eager_out = snapshot(out)
    G.spec_profile_begin(h)
    for _ in range(steps):
        step()
    prof = G.spec_profile_end(h)
    # the lazy call on the same trees, one CUDA graph per step: deep walks stream more rows
    lout = G.alloc_outputs(wd.B, wd.N, dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        def lazy_on():
            G.spec_build_tree_mask(h, xd["parent"], mask["anc_mask"], mask["depth"],
                                   mask["status"], side)
            G.spec_verify_sample_lazy(h, xd["logits"], xd["draft_token"], xd["parent"],
                                      wd.temperature, xd["uniforms"], lout["accept_len"],
                                      lout["out_tokens"], lout["kv_commit"], lout["bonus"],
                                      lout["status"], stream=side)
        lazy_on()
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            lazy_on()
    stream.wait_stream(side)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize(dev)
    a2, z2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(stream)
    for _ in range(steps):
        graph.replay()
    z2.record(stream)
    torch.cuda.synchronize(dev)
    lms = a2.elapsed_time(z2) / steps
    al = out["accept_len"].cpu().numpy()
    res = {"ms_per_step": ms, "value": wd.draft_nodes / (ms / 1e3), "unit": UNIT,
           "accept_len_mean": float(al.mean()),
           "accept_len_hist": np.bincount(al, minlength=1).tolist(),
           "kernels": {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]}
                       for k, v in prof.items() if v[1]},
           "lazy": {"ms_per_step": lms, "value": wd.draft_nodes / (lms / 1e3),
                    "rows_streamed_per_step": int(lout["accept_len"].sum().item()) + wd.B,
                    "requests_differing_from_eager": int(
                        (lout["out_tokens"] != out["out_tokens"]).any(dim=1).sum().item())},
           "config": f"large_tree shapes (B={wd.B} N={wd.N} V={wd.V} bf16, T=1), grammar "
                     "token boosted by 20"}
    if check:
        par = oracle_parity(xd, wd, {"eager_sample": ("sample", eager_out),
                                     "lazy_sample": ("sample", snapshot(lout))},
                            os.cpu_count() or 1)
        res["parity"] = par["eager_sample"]
        res["lazy"]["vs_oracle"] = par["lazy_sample"]
    del xd
    return res


def bench_small_tries(dev, stream, args, check=False):
    """The two small trie workloads (greedy: B=4, sampling: B=8; N=32, V=151936, bf16 logits),
    one verify call each; L2 flushed before every call. Their 128 and 256 rows fill less
    than one wave of row CTAs, so each row is streamed by several CTAs."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    res = {}
    for name in ("greedy_trie", "sampling_trie"):
        w = W.WORKLOADS[name]
        x = W.make(w, device=dev, seed=w.seed)
        with G.Handle(w.B, w.N, w.V, dev.index if dev.index is not None else 0) as hs:
            out = G.alloc_outputs(w.B, w.N, dev)
            flush = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

            def call():
                if w.mode == "greedy":
                    G.verify_greedy(hs, x["logits"], x["draft_token"], x["parent"], out=out,
                                    stream=stream)
                else:
                    G.verify_sample(hs, x["logits"], x["draft_token"], x["parent"],
                                    w.temperature, x["uniforms"], out=out, stream=stream)

            ms = _time_calls(call, stream, 50, 5, flush)
            moved = x["logits"].numel() * x["logits"].element_size()
            res[name] = {"ms_per_call": ms, "value": w.B * (w.N - 1) / (ms / 1e3), "unit": UNIT,
                         "logits_bytes": moved, "logit_GBps": moved / (ms / 1e3) / 1e9,
                         "roofline": dict(_hbm(moved, ms), bound="hbm"),
                         "kernels_ms": _kernel_split(hs, call, stream, 20, flush),
                         "config": f"{name}: B={w.B} N={w.N} V={w.V} bf16, T={w.temperature}, "
                                   "L2 flushed before every call"}
            if check:
                res[name]["parity"] = oracle_parity(
                    x, w, {"call": ("greedy" if w.mode == "greedy" else "sample",
                                    snapshot(out))}, os.cpu_count() or 1)["call"]
    return res


def bench_budget(h, x, w, dev, stream, args):
    """f4: the large-tree step (mask + eager sampling verify) followed by the device-side budget
    controller, captured once in a CUDA graph and replayed; the node budget starts at 16 of
    64 and the controller moves it (target acceptance ratio 0.5). Rows beyond a request's
    budget are not read."""
    from speculative_decoding_tree_mask_gb300 import binding as G
    B, N, T = w.B, w.N, w.temperature
    n_active = torch.full((B,), 16, dtype=torch.int32, device=dev)
    state = G.budget_state(0.5, 16, dev)
    prm = G.BudgetParams(0.5, 0.25, 0.05, 4, N, 4)
    mask = dict(anc_mask=torch.empty((B, N), dtype=torch.int64, device=dev),
                depth=torch.empty((B, N), dtype=torch.int32, device=dev),
                status=torch.empty(B, dtype=torch.int32, device=dev))
    out = G.alloc_outputs(B, N, dev)
    side = torch.cuda.Stream(dev)

    def step():
        G.spec_build_tree_mask(h, x["parent"], mask["anc_mask"], mask["depth"], mask["status"],
                               side)
        G.spec_verify_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"],
                             out["accept_len"], out["out_tokens"], out["kv_commit"],
                             out["bonus"], out["status"], stream=side)
        G.spec_budget_update(h, prm, out["accept_len"], out["status"], x["parent"], state,
                             n_active, stream=side)

    G.spec_set_node_budget(h, n_active)
    try:
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
            side.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                step()
        stream.wait_stream(side)
        state.copy_(G.budget_state(0.5, 16, dev))
        n_active.fill_(16)
        torch.cuda.synchronize()
        budgets = []
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        steps = 200
        a.record(stream)
        for i in range(steps):
            graph.replay()
        z.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(z) / steps
        ema, budget, nsteps = G.read_budget_state(state)
    finally:
        G.spec_set_node_budget(h, None)
    return {"ms_per_step": ms, "final_budget": budget, "final_ema": ema, "updates": nsteps,
            "path": "tree mask + spec_verify_sample under a device node budget + "
                    "spec_budget_update, one CUDA graph replayed per step",
            "config": "large tree; budget starts at 16 nodes, target ratio 0.5, alpha 0.25, "
                      "band 0.05, step 4, limits 4..64"}


def bench_leg(args):
    """One auxiliary leg on its own (for profiling runs): prints that leg's JSON."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    legs = {"small_tries": lambda: bench_small_tries(dev, stream, args, not args.skip_parity),
            "dense_chain": lambda: bench_dense_chain(dev, stream, args, not args.skip_parity)}
    if args.leg == "kv_commit":
        res = bench_kv_commit(dev, stream, args)
    else:
        res = legs[args.leg]()
    print(json.dumps({"leg": args.leg, **res}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-extra", action="store_true",
                    help="leave out the KV-commit and dense-chain measurements")
    ap.add_argument("--skip-lazy", action="store_true")
    ap.add_argument("--skip-parity", action="store_true",
                    help="leave out the comparison of every leg's outputs with the oracle")
    ap.add_argument("--leg", choices=["small_tries", "dense_chain", "kv_commit"], default=None,
                    help="run one auxiliary leg alone and print its JSON (profiling runs)")
    ap.add_argument("--requests", type=int, default=0,
                    help="requests per rank (default: the workload's 256); for profiling runs")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.leg:
        bench_leg(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
