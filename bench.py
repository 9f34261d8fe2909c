"""Benchmark of the fused commit step (statistics pass + commit rule) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch of synthetic logits:
the statistics pass (x0, prob, entropy for every row), the workload's commit
rule and the canvas update.  The default workload is one LLaDA-8B-shaped
block step: B=1, L=32 rows of V=126464 bf16 logits, suppress the mask id,
greedy, strict threshold 0.95 on 19 candidates.

Our arm replays the steps from CUDA graphs over rotating logit buffers whose
total exceeds 4x the L2 cache, so every step reads its logits from HBM, and
writes then reads buffers of twice the L2 size before each timed region, so
that the region starts from a clean L2 holding none of its inputs.  The
reference arm (--impl reference) times the CPU oracle on the same workload.
Under torchrun each rank runs its own replica on its own GPU (the path shards
by batch row with no collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dllm_workloads as W  # noqa: E402

METRIC = "token_stats+commit logits GB/s (% of GB300 HBM peak); canvas positions/s"
KERNEL_SOURCES = ("dllm_stats_kernels.cuh", "dllm_stats.cuh", "dllm_rules.cuh", "dllm_device.cuh", "dllm_gumbel.cuh",
                  "dllm_stats_greedy.cu", "dllm_stats_sample.cu", "dllm_stats_margin.cu", "dllm_stats_dispatch.cu",
                  "dllm_lmhead.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default="llada", choices=["llada", "tiny", "dream", "large", "loop", "uniform", "mask", "lmhead"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload only: skip the Dream and large sub-records")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", action="store_true",
                    help="eager steps only (no graph, e2e or CPU leg): the command the ncu captures use")
    ap.add_argument("--ready", action="store_true",
                    help="with --profile: launch the steps with DLLM_FLAG_INPUTS_READY (the launch the "
                         "timed graph uses) instead of as a dependent chain")
    ap.add_argument("--batch-rows", type=int, default=None,
                    help="with --profile: only the first N batch rows of the workload (a capture small "
                         "enough for a full ncu section set)")
    return ap.parse_args()


DEFAULT_STEPS = {"llada": 20_000, "tiny": 20_000, "dream": 500, "large": 100}
DEFAULT_WARMUP = {"llada": 3_000, "tiny": 3_000, "dream": 50, "large": 10}
# The other target configurations, measured in the default run beside the
# headline (each on its own timed region): steps per repeat.
SUB_STEPS = {"dream": 250, "large": 60}
MIN_REPEATS = 5          # timed repeats of the K-step region; the median is reported
MIN_TIMED_S = 0.5        # and at least this much summed timed time, so the clock sampler sees it
MAX_REPEATS = 20_000
GRAPH_ROTATIONS = 20     # longest timed graph, in rotations of the logit buffers


def describe(w) -> str:
    rule = {"threshold": f"threshold tau={w.params.get('tau')} strict={w.params.get('strict')}",
            "topk": "top-k k=transfer_schedule(256, 32)[:, 0] = 8",
            "factor+entropy_bound": "factor f=1.0 + entropy bound gamma=0.1"}[w.rule]
    samp = "greedy" if w.temperature == 0 else f"Gumbel-max t={w.temperature}"
    recipe = ""
    if w.name == "llada":
        recipe = (", rows N(0,1) x a per-row scale log-uniform in [3, 60] (the config's 'scale drawn so the top-1 "
                  "probability spans U(0.05, 0.999)', read without a softmax in the generator: top-1 spans "
                  "about 0.02 to 0.999)")
    return (f"{w.name}: B={w.B} L={w.L} V={w.V} {w.dtype}, suppress={w.suppress_ids}, {samp}, {rule}, "
            f"{int(w.candidates.sum())} candidates{recipe}")


def algorithmic_bytes(w) -> int:
    """Bytes one step must move: logits read, stats written (x0, prob, entropy:
    12 B/row), candidate mask read and commit mask written (1 B/row each), the
    canvas write of a committed row (4 B/row, counted for every row)."""
    per_row = 12 + 1 + 1 + 4
    extra = 0
    if w.rule == "factor+entropy_bound":
        extra = w.T * (4 + 1 + 1)     # the entropy-bound pass re-reads entropy and cand, writes its mask
    return w.logit_bytes() + w.T * per_row + extra


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
def gpu_query_id(props, index):
    """An id nvidia-smi understands for this device (UUID when torch gives one)."""
    u = getattr(props, "uuid", None)
    if u:
        u = str(u)
        return u if u.startswith("GPU-") else "GPU-" + u
    return str(index)


class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(sources=None) -> str:
    """Hash of the kernel sources with comments and blank space removed, so
    that only a change of code (not of its comments) invalidates the
    recorded ncu traffic."""
    import hashlib
    import re

    h = hashlib.sha256()
    for name in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "commit_step_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_kernel(workload: str) -> str:
    """Name of the workload's dominant kernel as the committed ncu launch
    summary lists it."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            e = json.load(f).get(workload)
        if e and e.get("kernel"):
            return e["kernel"] + " (fused statistics + commit rule)"
    except (OSError, ValueError):
        pass
    return "dllm statistics kernel (fused statistics + commit rule)"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None).  An entry that names its own
    sources is checked against those alone."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash(e.get("sources")):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def recorded_inst(workload: str):
    """Warp instructions per launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            e = json.load(f).get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash() and e.get("warp_inst_per_launch"):
            return float(e["warp_inst_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def issue_roofline(inst, ms_per_launch, sms, sm_mhz, alg_bytes, hbm_peak):
    """The issue roof of a kernel bound by instruction issue rather than DRAM:
    every SM has four schedulers that each issue at most one warp instruction
    per cycle, so the peak is SMs x 4 x the SM clock sampled under load."""
    if not inst or not sm_mhz:
        return None
    peak = sms * 4 * sm_mhz * 1e6 / 1e9
    achieved = inst / (ms_per_launch / 1e3) / 1e9
    t_full = inst / (peak * 1e9)   # seconds per launch at one instruction per scheduler per cycle
    return {"bound": "issue", "achieved": round(achieved, 1), "peak": round(peak, 1),
            "unit": "G warp instructions/s", "frac": round(achieved / peak, 4), "inst_per_launch": inst,
            "hbm_frac_at_full_issue": round(alg_bytes / t_full / 1e9 / hbm_peak, 4),
            "peak_derivation": f"{sms} SMs x 4 schedulers x 1 warp instruction per cycle x {sm_mhz:.0f} MHz"}


# --------------------------------------------------------------------------
# multi-rank timing: each rank times its own replica; the job takes the max
# --------------------------------------------------------------------------
def max_over_ranks(ms: float, device, world: int) -> float:
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Bytes every rank processed, over the slowest rank's time."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


# --------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload
# --------------------------------------------------------------------------
def oracle_step(w, logits=None, n_threads=0):
    import oracle

    z = w.logits if logits is None else logits
    x0, p, h = oracle.token_stats(z, dtype=w.dtype, temperature=w.temperature, key=w.key,
                                  suppress_ids=w.suppress_ids, row_ids=w.rows, n_threads=n_threads)
    B = z.shape[0] // w.L
    cand = w.candidates[:B]
    p32 = p.astype(np.float32).reshape(B, w.L)
    if w.rule == "threshold":
        oracle.threshold_transfer(p32, cand, w.params["tau"], w.params["strict"])
    elif w.rule == "topk":
        oracle.topk_transfer(p32, cand, np.full(B, 8, np.int32))
    else:
        oracle.factor_transfer(p32, cand, w.params["factor"])
        oracle.entropy_bound_transfer(h.astype(np.float32).reshape(B, w.L), cand, w.params["gamma"])
    return z.nbytes


def _time_oracle(sub, seconds, n_threads):
    done_bytes, n = 0, 0
    t0 = time.perf_counter()
    while True:
        done_bytes += oracle_step(sub, n_threads=n_threads)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return done_bytes, n, time.perf_counter() - t0


def cpu_baseline(w, seconds: float):
    """The oracle as it stands on this host's cores, on a bounded sample of
    the workload: all cores, and (tiny and llada) one core as well."""
    import oracle

    threads = oracle.default_threads()
    # a bounded sample: whole batch rows of the workload, repeated until `seconds` pass
    sub = w
    if w.name in ("dream", "large"):
        rows = np.arange(w.L)   # one batch row
        sub = W.build(w.name, rows=rows)
    done_bytes, n, dt = _time_oracle(sub, seconds, 0)
    unit_rows = sub.logits.shape[0]
    res = {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{n} passes over {unit_rows} rows of the {w.name} workload "
                     f"({sub.logits.nbytes / 1e6:.1f} MB each), {dt:.1f} s, fp64 oracle threaded over rows"}
    if w.name in ("tiny", "llada"):
        b1, n1, dt1 = _time_oracle(sub, max(2.0, seconds / 2), 1)
        res["single_core"] = {"value": b1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} passes over the same {unit_rows} rows, {dt1:.1f} s, one thread"}
    return res


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
class StepRunner:
    """The device buffers and the fused step of one workload: R rotating copies
    of its logits (more than 4x L2 in total when one copy is smaller), the
    candidate mask, a canvas and the packed outputs."""

    def __init__(self, cs, w, dev, l2):
        import torch

        self.cs, self.w, self.dev = cs, w, dev
        nbytes = w.logit_bytes()
        R = max(1, math.ceil(4 * l2 / nbytes)) if nbytes < 4 * l2 else 1
        self.R = min(R, 256)
        if w.dtype == "bf16":
            self.host = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
        else:
            self.host = torch.from_numpy(w.logits)
        base = self.host.to(dev).view(w.B, w.L, w.V)
        self.bufs = [base] + [base.clone() for _ in range(self.R - 1)]
        self.cand = torch.from_numpy(w.candidates).to(dev)
        self.canvas = torch.zeros((w.B, 128 + w.L), dtype=torch.int32, device=dev)
        # The four per-position outputs live in one device buffer (x0, prob,
        # entropy, commit back to back), so a host reads a step's result with
        # one copy.
        T = w.B * w.L
        self.obuf = torch.empty(13 * T, dtype=torch.uint8, device=dev)
        self.x0 = self.obuf[0:4 * T].view(torch.int32).view(w.B, w.L)
        self.prob = self.obuf[4 * T:8 * T].view(torch.float32).view(w.B, w.L)
        self.ent = self.obuf[8 * T:12 * T].view(torch.float32).view(w.B, w.L)
        self.commit = self.obuf[12 * T:13 * T].view(w.B, w.L)
        self.commit2 = torch.empty((w.B, w.L), dtype=torch.uint8, device=dev)
        self.kq = torch.full((w.B,), 8, dtype=torch.int32, device=dev)
        self.ws = cs.workspace(w.B, w.L, w.V, 1 if w.dtype == "bf16" else 0, dev)
        self.out = (self.x0, self.prob, self.ent, self.commit, None)
        self.launches_per_step = 2 if w.rule == "factor+entropy_bound" else 1

    def step(self, i, ready=False):
        # ready: this step's logits do not come from the kernel before it (the
        # rotating buffers were filled before timing), so it may start loading
        # them while that kernel finishes (DLLM_FLAG_INPUTS_READY).
        cs, w = self.cs, self.w
        lg = self.bufs[i % self.R]
        common = dict(suppress_ids=w.suppress_ids, cand=self.cand, canvas=self.canvas, canvas_offset=128,
                      out=self.out, ws=self.ws, inputs_ready=ready)
        if w.rule == "threshold":
            cs.commit_step(lg, rule=cs.RULE_THRESHOLD, tau=w.params["tau"], strict=w.params["strict"], **common)
        elif w.rule == "topk":
            cs.commit_step(lg, rule=cs.RULE_TOPK, k=self.kq, temperature=w.temperature, key=w.key + i, **common)
        else:
            cs.commit_step(lg, rule=cs.RULE_FACTOR, factor=w.params["factor"], **common)
            cs.entropy_bound_transfer(self.ent, self.cand, w.params["gamma"], commit=self.commit2)


def measure_device(runner, steps, warmup, dev, props, world, sample_clocks=True):
    """Times exactly `steps` fused steps per repeat, as CUDA graphs replayed on
    one stream: independent steps (DLLM_FLAG_INPUTS_READY, the pipelined
    figure) and the same steps as a dependent chain, interleaved repeat by
    repeat, with L2 flushed before each timed region.  At least MIN_REPEATS
    repeats and MIN_TIMED_S of summed pipelined time; medians are reported."""
    import torch

    R = runner.R
    # graphs of whole rotations of the buffers, up to GRAPH_ROTATIONS of them:
    # consecutive steps overlap only within a graph, so each graph boundary
    # pays the pipeline's fill once
    G = R * max(1, min(steps // R, GRAPH_ROTATIONS)) if R > 1 else min(50, steps)
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    flush = torch.empty(l2_bytes * 2, dtype=torch.uint8, device=dev)
    clean = torch.zeros(l2_bytes // 2, dtype=torch.int32, device=dev)   # 2x L2, read only

    def flush_l2():
        # writing twice L2's size evicts everything the last region cached; reading
        # another buffer of that size then writes those dirty lines back, so the
        # region starts from a clean L2 and pays for none of the flush's own traffic
        flush.zero_()
        clean.max()

    def capture(ready, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(n):   # eager warm-up on the capture stream
                runner.step(i, ready)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                runner.step(i, ready)
        return g

    reps, rem = divmod(steps, G)
    g = capture(True, G) if reps else None
    g_dep = capture(False, G) if reps else None
    g_rem = capture(True, rem) if rem else None
    g_dep_rem = capture(False, rem) if rem else None
    pipelined = [g] * reps + ([g_rem] if g_rem else [])
    dependent = [g_dep] * reps + ([g_dep_rem] if g_dep_rem else [])
    # warm-up: every graph that is timed is replayed (uploaded) first, then
    # whole graphs until at least `warmup` untimed steps have run
    warm_steps = 0
    with torch.cuda.stream(stream):
        for gr, n in ((g, G), (g_rem, rem), (g_dep, G), (g_dep_rem, rem)):
            if gr is not None:
                gr.replay()
                warm_steps += n
        while warm_steps < warmup:
            (g or g_rem).replay()
            warm_steps += G if g else rem
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()

    def run(seq):
        for gr in seq:
            gr.replay()

    pip, dep = [], []
    sampler = ClockSampler(gpu_query_id(props, dev.index)) if sample_clocks else None
    if sampler:
        sampler.__enter__()
    try:
        n_block = 1
        while len(pip) < MIN_REPEATS or (sum(pip) < MIN_TIMED_S * 1e3 and len(pip) < MAX_REPEATS):
            block = []
            for _ in range(n_block):   # a block of repeats per host sync
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                with torch.cuda.stream(stream):
                    flush_l2()
                    ev[0].record(stream)
                    run(pipelined)
                    ev[1].record(stream)
                    flush_l2()
                    ev[2].record(stream)
                    run(dependent)
                    ev[3].record(stream)
                block.append(ev)
            block[-1][3].synchronize()
            for ev in block:
                pip.append(ev[0].elapsed_time(ev[1]))
                dep.append(ev[2].elapsed_time(ev[3]))
            # about 20 ms of GPU work per host sync
            n_block = int(min(64, max(1, 20.0 / max(1e-3, pip[-1] + dep[-1] + 0.1))))
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
    torch.cuda.synchronize()
    med = statistics.median(pip)
    ms = max_over_ranks(med, dev, world)
    return {"ms": ms, "ms_per_step": ms / steps, "dep_ms_per_step": statistics.median(dep) / steps,
            "repeats": len(pip), "timed_ms_total": sum(pip), "warmup_steps_run": warm_steps, "graph_steps": G,
            "spread": [min(pip) / steps, max(pip) / steps],
            "clocks": sampler.summary() if sampler else None}


def single_launch_us(runner, n):
    import torch

    lat = []
    for i in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        runner.step(i)
        b.record()
        b.synchronize()
        lat.append(a.elapsed_time(b) * 1e3)
    return statistics.median(lat)


def sub_record(cs, name, dev, props, l2, world):
    """One of the other target configurations on its own timed region."""
    import torch

    w = W.build(name)
    runner = StepRunner(cs, w, dev, l2)
    runner.step(0)
    torch.cuda.synchronize()
    steps = SUB_STEPS[name]
    m = measure_device(runner, steps, DEFAULT_WARMUP[name], dev, props, world)
    alg = algorithmic_bytes(w)
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(alg, steps, world, m["ms"])
    rec = {"workload": describe(w), "value": round(value, 2), "unit": "GB/s", "steps": steps,
           "repeats": m["repeats"], "ms_per_step": m["ms_per_step"],
           "pct_of_hbm_peak": round(100 * value / world / peak, 1),
           "frac": round(value / world / peak, 4), "peak": peak, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
           "dependent_steps": {"ms_per_step": m["dep_ms_per_step"],
                               "value": round(alg / (m["dep_ms_per_step"] / 1e3) / 1e9, 2)},
           "single_launch_us": round(single_launch_us(runner, 5), 2),
           "traffic": recorded_traffic(name), "kernel": recorded_kernel(name), "clocks": m["clocks"],
           "workspace_fault": cs.workspace_fault(runner.ws)}
    clk = (m["clocks"] or {}).get("sm_mhz") or getattr(props, "clock_rate", 0) / 1e3
    roof = issue_roofline(recorded_inst(name), m["ms_per_step"], props.multi_processor_count, clk, alg, peak)
    if roof:
        rec["issue_roofline"] = roof
    del runner
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import commit_step_gb300 as cs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if args.batch_rows is not None:
        if not args.profile:
            raise SystemExit("--batch-rows is for --profile captures only")
        full = W.build(args.workload, rows=np.arange(0))
        nb = max(1, min(args.batch_rows, full.B))
        w = W.build(args.workload, rows=np.arange(nb * full.L))
        w = dataclasses.replace(w, B=nb, rows=None, candidates=w.candidates[:nb])
    else:
        w = W.build(args.workload)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[w.name]
    warmup_req = args.warmup if args.warmup is not None else DEFAULT_WARMUP[w.name]
    warmup = max(3, warmup_req)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    runner = StepRunner(cs, w, dev, l2)
    nbytes = w.logit_bytes()
    R = runner.R

    runner.step(0)
    torch.cuda.synchronize()
    if args.profile:
        for i in range(warmup + steps):
            runner.step(i, args.ready)
        torch.cuda.synchronize()
        return {"profile": w.name, "steps": warmup + steps, "workspace_fault": cs.workspace_fault(runner.ws)}, w

    m = measure_device(runner, steps, warmup, dev, props, world)
    ms = m["ms"]
    ms_per_step = m["ms_per_step"]
    dep_ms_per_step = m["dep_ms_per_step"]
    single_us = single_launch_us(runner, min(200, 10 * R))

    # e2e through the public API with host buffers (copies inside the timed region)
    pinned = runner.host.contiguous().pin_memory().view(w.B, w.L, w.V)
    e2e_steps = max(50, min(2000, steps // 10)) if w.name in ("llada", "tiny") else 50

    # One C call per step (dllm_commit_step_host): the logits' copy to the
    # device, the fused step, and one read of x0/prob/entropy/commit.
    host_step = cs.HostStep(pinned, rule={"threshold": cs.RULE_THRESHOLD, "topk": cs.RULE_TOPK}.get(w.rule, cs.RULE_FACTOR),
                            tau=w.params.get("tau", 0.0), strict=w.params.get("strict", False), k=runner.kq,
                            factor=w.params.get("factor", 0.0), temperature=w.temperature, key=w.key,
                            suppress_ids=w.suppress_ids, cand=runner.cand, canvas=runner.canvas, canvas_offset=128,
                            ws=runner.ws)
    for _ in range(3):
        host_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(e2e_steps):
        host_step()
    b.record()
    b.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dev, world)
    ok = cs.workspace_fault(runner.ws)

    alg = algorithmic_bytes(w)
    value = whole_job_gbs(alg, steps, world, ms)
    peak, peak_kind = measured_peaks()
    lps = runner.launches_per_step
    kernel_ms = ms_per_step
    achieved = alg / (kernel_ms / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warmup_req, "repeats": m["repeats"], "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded generator, dllm_workloads.py)",
        "config": {"workload": describe(w), "global_batch": w.B * world, "seq_len": w.L, "vocab": w.V,
                   "parallelism": f"replicas x{world} (batch rows shard, no collective)",
                   "l2": (f"{R} rotating logit buffers, {R * nbytes / 1e6:.0f} MB total vs L2 {l2 / 1e6:.0f} MB"
                          if R > 1 else f"one {nbytes / 1e6:.0f} MB buffer, larger than L2 {l2 / 1e6:.0f} MB")
                         + "; L2 flushed before each timed repeat (a 2x L2 write, then a 2x L2 read of "
                           "another buffer so that no dirty line of the flush is written back inside the region)",
                   "launch": f"CUDA graphs of up to {m['graph_steps']} independent steps, programmatic dependent "
                             "launch, DLLM_FLAG_INPUTS_READY (logits resident before timing)",
                   "timing": f"median of {m['repeats']} repeats of exactly {steps} steps, interleaved with the "
                             f"dependent chain; {m['timed_ms_total']:.0f} ms timed in total; "
                             f"{m['warmup_steps_run']} untimed warm-up steps (every timed graph replayed first)"},
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "dependent_steps": {"ms_per_step": dep_ms_per_step,
                            "value": round(alg / (dep_ms_per_step / 1e3) / 1e9, 2), "unit": "GB/s",
                            "note": "each step waits for the previous kernel before reading its logits"},
        "spread_ms_per_step": m["spread"],
        "single_launch_us": round(single_us, 2),
        "positions_per_s": round(w.B * w.L * steps * world / (ms / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(w.name),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "kernel": recorded_kernel(w.name)},
        "e2e": {"value": round(alg / (e2e_ms / 1e3) / 1e9 * world, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(nbytes), "d2h_bytes_per_step": int(w.T * 13),
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "path": "dllm_commit_step_host: pinned host logits -> device copy -> fused "
                        "step -> one host copy of x0/prob/entropy/commit"},
        "gpu_launches": steps * lps * m["repeats"],
        "gpu_launches_note": "our kernels in the pipelined timed regions (steps x launches per step x repeats)",
        "clocks": m["clocks"],
        "workspace_fault": ok,
    }
    del runner, host_step, pinned
    torch.cuda.empty_cache()
    if w.name == "llada" and not args.no_extra:
        # the other configurations the target names, each on its own timed region
        res["workloads"] = {name: sub_record(cs, name, dev, props, l2, world) for name in ("dream", "large")}
    return res, w


def run_loop(args, rank, world):
    """The block-decode loop workload: B=4, P=128, gen_len=1024, block_len=32,
    V=126464 bf16, strict threshold 0.95 then editing 0.9, max_post_steps=4;
    a seeded generator emits each step's block rows.  Reports the commit
    steps' GB/s and canvas positions per second (B * gen_len / the summed GPU
    time of the commit steps)."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import commit_step_gb300 as cs
    from commit_step_gb300.decode import decode_with_editing

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    spec = W.loop_spec()
    gen = W.LoopGenerator(spec)
    prompt = torch.from_numpy(gen.prompt).to(dev)
    model = lambda bi, st, c0, n: gen.device_logits(bi, st, c0, n)
    kw = dict(gen_len=spec.gen_len, block_len=spec.block_len, mask_id=spec.mask_id, threshold=spec.tau,
              editing_threshold=spec.tau_edit, max_post_steps=spec.max_post_steps, suppress_ids=[spec.mask_id])
    _, warm_forwards = decode_with_editing(model, prompt, **kw)   # warm-up: one whole decode
    times, trace = [], []
    torch.cuda.synchronize()
    with ClockSampler(gpu_query_id(torch.cuda.get_device_properties(dev), dev.index)) as clk:
        out, forwards = decode_with_editing(model, prompt, step_times=times, trace=trace, **kw)
    total_ms = float(sum(times))
    rows_per_step = spec.B * spec.block_len
    bytes_per_step = rows_per_step * (spec.V * 2 + 18)
    peak, peak_kind = measured_peaks()
    value = bytes_per_step * forwards / (total_ms / 1e3) / 1e9 * world
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": forwards,
        "warmup": warm_forwards,
        "ms_per_step": total_ms / forwards, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded generator, dllm_workloads.py)",
        "config": {"workload": "loop: B=4, P=128, gen_len=1024, block_len=32 (aligned), V=126464 bf16, strict "
                               "threshold 0.95 then edit 0.9, max_post_steps=4",
                   "global_batch": spec.B * world, "seq_len": spec.block_len, "vocab": spec.V,
                   "parallelism": f"replicas x{world}", "l2": "per-step rows are written by the generator just before"
                                                              " the step (L2-warm, as in a real loop)"},
        "positions_per_s": round(spec.B * spec.gen_len * world / (total_ms / 1e3), 1),
        "forwards": forwards, "commits": int(sum(t[2] for t in trace)), "edits": int(sum(t[3] for t in trace)),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "gpu_launches": forwards, "clocks": clk.summary(),
    }


def run_uniform(args, rank, world):
    """The uniform-noise loop workload: B=1, canvas N=256, V=262144 bf16 (a
    DiffusionGemma-sized vocabulary), 48 steps at most, entropy bound 0.1,
    temperatures 0.8 -> 0.4, stop when stable once and mean entropy < 0.005;
    a seeded generator makes each position confident from a random onset
    step in [0, 24].  Reports the GB/s of the per-step GPU work (the fused
    statistics + acceptance launch, noise, re-noising, stopping update) and
    canvas positions per second of that time."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    from commit_step_gb300.decode import decode_uniform

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    spec = W.uniform_spec()
    gen = W.UniformGenerator(spec)
    buf = torch.empty((spec.B * spec.N, spec.V), dtype=torch.bfloat16, device=dev)
    model = lambda st, c: gen.device_logits(st, out=buf)
    kw = dict(batch=spec.B, canvas_len=spec.N, vocab_size=spec.V, key=spec.key, num_steps=spec.num_steps,
              entropy_bound=spec.entropy_bound, t_min=spec.t_min, t_max=spec.t_max,
              stability_threshold=spec.stability_threshold, confidence_threshold=spec.confidence_threshold)
    _, warm_steps = decode_uniform(model, **kw)                 # warm-up: one whole decode
    times = []
    torch.cuda.synchronize()
    with ClockSampler(gpu_query_id(torch.cuda.get_device_properties(dev), dev.index)) as clk:
        out, steps = decode_uniform(model, step_times=times, **kw)
    total_ms = float(sum(times))
    rows = spec.B * spec.N
    bytes_per_step = rows * (spec.V * 2 + 12 + 1 + 4 * 4)    # logits; stats out; accepted; noise/canvas/argmax traffic
    peak, _ = measured_peaks()
    value = bytes_per_step * steps / (total_ms / 1e3) / 1e9 * world
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warm_steps, "ms_per_step": total_ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator, dllm_workloads.py)",
        "config": {"workload": f"uniform: B={spec.B}, canvas {spec.N}, V={spec.V} bf16, <= {spec.num_steps} steps, "
                               f"entropy bound {spec.entropy_bound}, T {spec.t_max} -> {spec.t_min}",
                   "global_batch": spec.B * world, "seq_len": spec.N, "vocab": spec.V,
                   "parallelism": f"replicas x{world}",
                   "l2": "per-step logits (134 MB) are written by the generator just before the step"},
        "positions_per_s": round(rows * steps * world / (total_ms / 1e3), 1),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "gpu_launches": 5 * steps, "clocks": clk.summary(),
    }


def run_mask(args, rank, world):
    """block_causal_mask of an 8192-token window in blocks of 32 (a
    LLaDA2-style window), fp32 additive: 256 MiB of pure writes per call.
    Reports the write GB/s (graph replay of independent calls, CUDA events)."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import commit_step_gb300 as cs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    L, bl = 8192, 32
    steps = args.steps if args.steps is not None else 2000
    warmup = max(3, args.warmup if args.warmup is not None else 10)
    outs = [torch.empty((L, L), dtype=torch.float32, device=dev) for _ in range(2)]
    G = 10
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for i in range(G):
            cs.block_causal_mask(L, bl, out=outs[i % 2], stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):
            cs.block_causal_mask(L, bl, out=outs[i % 2], stream=stream)
    reps = max(1, steps // G)
    with torch.cuda.stream(stream):
        for _ in range(max(1, warmup // G)):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_query_id(torch.cuda.get_device_properties(dev), dev.index)) as clk:
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        e1.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dev, world)
    n = reps * G
    nbytes = L * L * 4
    value = nbytes * n * world / (ms / 1e3) / 1e9
    peak, kind = measured_peaks()
    # the pure-write ceiling beside it: torch's fill of the same two buffers,
    # replayed the same way (a library kernel, timed for reference only)
    gf = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(G):
            outs[i % 2].fill_(0.0)
    torch.cuda.synchronize()
    with torch.cuda.graph(gf, stream=stream):
        for i in range(G):
            outs[i % 2].fill_(0.0)
    with torch.cuda.stream(stream):
        gf.replay()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            gf.replay()
    f1.record(stream)
    f1.synchronize()
    fill_gbs = nbytes * n / (f0.elapsed_time(f1) / 1e3) / 1e9
    return {
        "metric": "block_causal_mask write GB/s", "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": n, "warmup": max(1, warmup // G) * G, "ms_per_step": ms / n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (mask of an 8192-token window)",
        "config": {"workload": f"block_causal_mask L={L} block_len={bl} fp32 additive", "l2": "two 256 MiB outputs, "
                   "alternating (each larger than L2)"},
        "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / world / peak, 4), "traffic": recorded_traffic("mask"),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({kind})"},
        "write_ceiling": {"fill_gbs": round(fill_gbs, 1), "frac_of_fill": round(value / world / fill_gbs, 4),
                          "what": "torch fill_ of the same two 256 MiB buffers in the same graphs, timed after ours"},
        "gpu_launches": n, "clocks": clk.summary(),
    }


def run_lmhead(args, rank, world):
    """The LM head fused with the statistics pass at the LLaDA-8B LM head
    shape: 32 hidden states (one 32-token block) x a 126464 x 4096 bf16
    weight, greedy, suppressing the mask id.  Reports the GB/s of the bytes
    the fused call must read (weight + hidden, the logits never written), the
    tensor-core rate, and the unfused path (cuBLAS logits, then token_stats)
    timed the same way."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import commit_step_gb300 as cs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    T, d, V = 32, 4096, 126464
    h, w, _ = W.lm_head_inputs(0, T, d, V)
    hd = torch.from_numpy(h.view(np.int16)).to(dev).view(torch.bfloat16)
    wd = torch.from_numpy(w.view(np.int16)).to(dev).view(torch.bfloat16)
    del w
    out = (torch.empty(T, dtype=torch.int32, device=dev), torch.empty(T, device=dev), torch.empty(T, device=dev))
    steps = args.steps if args.steps is not None else 400
    warmup = max(3, args.warmup if args.warmup is not None else 10)
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    logits16 = torch.empty((T, V), dtype=torch.bfloat16, device=dev)

    def fused():
        cs.lm_head_stats(hd, wd, suppress_ids=[126336], out=out, stream=stream)

    def unfused():
        torch.matmul(hd, wd.t(), out=logits16)
        cs.token_stats(logits16, suppress_ids=[126336], out=out, stream=stream)

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize()
        G = 20
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(G):
                fn()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, n // G)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / (reps * G), reps * G

    with ClockSampler(gpu_query_id(torch.cuda.get_device_properties(dev), dev.index)) as clk:
        ms, n = timed(fused, steps)
    ms = max_over_ranks(ms, dev, world)
    ms_unfused, _ = timed(unfused, max(20, steps // 4))
    nbytes = V * d * 2 + T * d * 2
    value = nbytes / (ms / 1e3) / 1e9 * world
    peak, kind = measured_peaks()
    flops = 2.0 * T * d * V
    return {
        "metric": "fused LM head + token_stats GB/s (weight read)", "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": n, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator, dllm_workloads.lm_head_inputs)",
        "config": {"workload": f"LM head T={T} d={d} V={V} bf16 (LLaDA-8B head shape), greedy, suppress mask id",
                   "l2": "the 1.04 GB weight is larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / world / peak, 4), "traffic": recorded_traffic("lmhead"),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({kind})", "kernel": recorded_kernel("lmhead")},
        "tensor_tflops": round(flops / (ms / 1e3) / 1e12, 1),
        "unfused": {"ms_per_step": ms_unfused, "path": "torch.matmul (cuBLAS) to bf16 logits, then token_stats",
                    "speedup_of_fused": round(ms_unfused / ms, 3)},
        "gpu_launches": 2 * n, "clocks": clk.summary(),
    }


def run_reference(args, rank, world):
    w = W.build(args.workload)
    steps = args.steps if args.steps is not None else 3
    warmup = args.warmup if args.warmup is not None else 1
    sub = w if w.name in ("llada", "tiny") else W.build(w.name, rows=np.arange(w.L))
    import oracle

    for _ in range(max(0, min(warmup, 3))):
        oracle_step(sub)
    t0 = time.perf_counter()
    done = 0
    n = max(1, steps)
    for _ in range(n):
        done += oracle_step(sub)
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": n, "warmup": warmup, "ms_per_step": dt * 1e3 / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator, dllm_workloads.py)",
        "config": {"workload": describe(w), "global_batch": w.B * world, "seq_len": w.L, "vocab": w.V,
                   "parallelism": f"replicas x{world} (batch rows shard, no collective)",
                   "sample": f"{sub.logits.shape[0]} rows per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": f"{n} steps over {sub.logits.shape[0]} rows of the {w.name} workload"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)))
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.workload in ("loop", "uniform", "mask", "lmhead"):
        res = {"loop": run_loop, "uniform": run_uniform, "mask": run_mask,
               "lmhead": run_lmhead}[args.workload](args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        return 0
    res, w = run_ours(args, rank, world)
    if rank == 0:
        # the oracle baseline is timed at N=1 only (one replica's host cores)
        if world == 1 and not args.no_cpu_baseline and not args.profile:
            res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
