"""Benchmark of batched draft verification on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one verification call over one batch of the workload: two kernels
on one stream, the row-statistics kernel (streams every logit once) and the
walk kernel (one thread-block cluster per sequence: accept tests, residual
or bonus pass, inverse-CDF draw), chained with programmatic dependent launch.
The default workload is the largest one, the three-model PipeSpec cascade
B=128, gamma1=8, gamma2=4, V=128256, bf16, T=1.0 (one 689.5 MB call: the
M_0, M_1 and M_2 logit rows); --workload selects any of
workloads.synth.SPECS (e.g. the 128256-vocabulary sampling chain
sampling_chain_b64_g5_v128256_bf16_a60).  Inputs are synthetic and seeded.

Timing: W warm-up steps, then a loaded soak of about one second (clocks are
sampled over it and the timed region), then exactly K steps between CUDA
events on the launching stream, with a barrier and a device synchronize on
both sides; the max over ranks is reported.  Consecutive steps rotate over
enough distinct copies of the input batch (more than 3x the L2 size in
total) that every step reads its logits from HBM.  The steps are replayed
from a CUDA graph that holds one call per input copy.

Printed on rank 0: one JSON line with the metric (verified draft tokens/s),
logits GB/s, the HBM roofline of the verification call (algorithmic bytes
over the call's average duration in the timed region: both kernels, so a
lower bound for the statistics kernel alone), the end-to-end number through
the public call with host buffers, and the CPU oracle timed on a bounded
sample.

--impl reference times the CPU oracle itself (the slow, plainly written
reference) on the same workload and prints the same JSON line with
"impl": "reference".
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "cascade_b128_g8_g4_v128256_bf16"
METRIC = "verified draft tokens/sec and logits GB/s vs GB300 HBM peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["draft_verification_gb300/csrc/verify.cu", "draft_verification_gb300/csrc/stats.cuh",
                  "draft_verification_gb300/csrc/walk.cuh", "draft_verification_gb300/csrc/common.cuh"]
# the kernels of one call (statistics, then walk); greedy calls use the
# greedy walk kernels
KERNELS = {"chain": ["stats_kernel", "chain_walk_kernel"], "tree": ["stats_kernel", "tree_kernel"],
           "cascade": ["stats_kernel", "cascade_walk_kernel"], "compact": ["compact_kernel"],
           "pipeline": ["stats_kernel", "pipeline_walk_kernel"],
           "clasp": ["clasp_init_kernel", "clasp_step_kernel", "clasp_backtrack_kernel"]}
COMPACT_METRIC = "cache rows compacted/sec and GB/s moved vs GB300 HBM peak (1 GPU)"
COMPACT_SOURCES = ["draft_verification_gb300/csrc/compact.cu"]
ASYNC_SOURCES = KERNEL_SOURCES + ["draft_verification_gb300/csrc/pipeline_async.cu"]
CLASP_METRIC = "CLaSp layer selections/sec and weight GB/s vs GB300 HBM and bf16 tensor peaks (1 GPU)"
CLASP_SOURCES = ["draft_verification_gb300/csrc/clasp.cu"]
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="plain eager loop for an ncu capture: warm-up + steps calls, one input copy")
    ap.add_argument("--consulted-only", action="store_true",
                    help="sampling chains: read each position's rows only while no earlier position was rejected")
    return ap.parse_args()


# --------------------------------------------------------------------------
# workload bookkeeping (sizes only)
# --------------------------------------------------------------------------

def draft_tokens_per_call(w) -> int:
    s = w["spec"]
    if w["kind"] == "chain":
        return s.B * s.gamma
    if w["kind"] == "tree":
        return s.B * (w["parent"].shape[1] - 1)
    if w["kind"] == "pipeline":
        return s.B * s.windows[0]
    return s.B * (s.gamma1 + s.gamma2)


def chain_groups(B: int, rows: int, V: int, elt: int, min_seqs: int = 16) -> int:
    """Batch groups of one chain (or tree) call, as the library plans them:
    at most 4, each with at least 40 MB of logits and 16 sequences (4 trees)."""
    return max(1, min(4, B // min_seqs, int(B * rows * V * elt / 40e6)))


def launches_per_call(w) -> int:
    """Kernels of the library launched by one verification call: statistics
    and walk per batch group for chains and trees, statistics and walk for
    the other kinds, one walk kernel in consulted-only mode."""
    s = w["spec"]
    if CONSULTED and (w["kind"] == "tree" or (w["kind"] == "chain" and not s.greedy)):
        return 1  # the consulted-only walk computes its own statistics
    elt = 2 if s.dtype == "bf16" else 4
    if w["kind"] == "chain":
        rows = s.gamma + 1 if s.greedy else 2 * s.gamma + 1
        return 2 * chain_groups(s.B, rows, s.V, elt)
    if w["kind"] == "tree":
        n = int(w["parent"].shape[1])
        return 2 * chain_groups(s.B, n if s.greedy else 2 * n, s.V, elt, min_seqs=4)
    return 2


def compute_dtype(logit_dtype: str) -> str:
    """Arithmetic of the verification path: float32 throughout, on logits
    stored as bfloat16 or float32."""
    return "bf16 in, f32 accumulate" if logit_dtype == "bf16" else "f32"


def workload_config(w) -> dict:
    s = w["spec"]
    cfg = {"workload": s.name, "kind": w["kind"], "batch": s.B, "vocab": s.V,
           "logit_dtype": s.dtype, "mode": "greedy" if s.greedy else "sampling",
           "temperature": s.temperature}
    if w["kind"] == "chain":
        cfg["gamma"] = s.gamma
        cfg["alpha_target"] = s.alpha_target
    elif w["kind"] == "tree":
        cfg["nodes"] = int(w["parent"].shape[1])
        cfg["max_depth"] = w["max_depth"]
        cfg["alpha_target"] = s.alpha_target
    elif w["kind"] == "pipeline":
        cfg.update(models=s.k, windows=list(s.windows), final_bonus=s.final_bonus)
    else:
        cfg.update(gamma1=s.gamma1, gamma2=s.gamma2, alpha01_target=s.alpha01_target,
                   alpha12_target=s.alpha12_target)
    return cfg


# --------------------------------------------------------------------------
# replicas: one process per GPU, each verifying its own batch (no exchange)
# --------------------------------------------------------------------------

def replica_seed(seed: int, rank: int) -> int:
    """Each replica draws its own seeded batch."""
    return seed + rank


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest replica's time (every rank gets it)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_call: float, world: int, ms_per_call: float) -> float:
    """Units all replicas processed per second, timed by the slowest one."""
    return units_per_call * world / (ms_per_call * 1e-3)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            mp = json.load(fh)
        for k in ("hbm_gbs", "hbm_GBps", "hbm"):
            if k in mp:
                return float(mp[k]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"


def measured_tensor_peak(sustained: bool):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as fh:
            mp = json.load(fh)
        if key in mp:
            return float(mp[key]), f"measured (MEASURED_PEAKS.json {key})"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16, no MEASURED_PEAKS.json)"


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES if sources is None else sources:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, sources=None):
    """DRAM bytes of one call (all its kernels, caches flushed) from the
    committed ncu launch-list summary, if it was taken on the current kernel
    source; else None."""
    path = os.path.join(ROOT, "profiles", f"launches_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as fh:
        for line in fh:
            if line.startswith("- ") and " = " in line:
                k, v = line[2:].split(" = ", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_hash") != kernel_source_hash(sources):
        return None
    try:
        return int(float(fields["dram_bytes_per_call"]))
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch
        self.proc = None
        props = torch.cuda.get_device_properties(device)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            self.gpu = "GPU-" + str(uuid)
        else:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.gpu = vis.split(",")[device.index] if vis else str(device.index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# --------------------------------------------------------------------------

def oracle_rate(w, budget_s: float):
    """Verified draft tokens/s of the CPU oracle on whole calls of the
    workload, repeated until about `budget_s` seconds of CPU work."""
    from oracle import verify as V  # the reference is only used on this leg
    s = w["spec"]
    sample_B = s.B
    done = 0
    t0 = time.perf_counter()
    calls = 0
    while True:
        if w["kind"] == "chain":
            V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"],
                           s.temperature, s.greedy, s.dtype, V=s.V)
        elif w["kind"] == "tree":
            V.verify_tree(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"],
                          w["prefix_len"], s.temperature, s.greedy, w["max_depth"], s.dtype, V=s.V)
        elif w["kind"] == "pipeline":
            from oracle import pipeline as Pp
            Pp.verify_pipeline(w["models"], w["tokens"], w["us"], w["vs"], s.temperature, s.greedy,
                               s.final_bonus, s.dtype, V=s.V, base=w["base"])
        else:
            V.verify_cascade(w["l0"], w["l1"], w["l2"], w["tokens"], w["u1"], w["v1"], w["u2"],
                             w["v2"], w["base0"], w["base1"], s.temperature, s.greedy, s.dtype, V=s.V)
        calls += 1
        done += draft_tokens_per_call(w)
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el, f"{calls} whole calls of {sample_B} sequences ({el:.1f} s, float64 NumPy)", el


def subset(w, nseq):
    """The first nseq sequences of a workload (for a bounded CPU sample)."""
    import dataclasses
    out = dict(w)
    out["spec"] = dataclasses.replace(w["spec"], B=nseq)
    for k, v in w.items():
        if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == w["spec"].B:
            out[k] = v[:nseq]
        elif isinstance(v, list):
            out[k] = [x[:nseq] for x in v]
    if w["kind"] == "pipeline":
        out["base"] = w["base"][:, :nseq]
    return out


def bounded_sample(w, budget_s):
    """Shrink the batch so one oracle call takes at most about budget_s / 3."""
    from oracle import verify as V  # noqa: F401
    probe = subset(w, 1)
    t0 = time.perf_counter()
    oracle_rate(probe, 0.0)
    per_seq = time.perf_counter() - t0
    nseq = max(1, min(w["spec"].B, int(budget_s / 3 / max(per_seq, 1e-6))))
    return subset(w, nseq), nseq


def run_reference(args, w):
    sample, nseq = bounded_sample(w, args.cpu_seconds)
    rate, desc, el = oracle_rate(sample, args.cpu_seconds)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * draft_tokens_per_call(w) / rate,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {nseq} of {w['spec'].B} sequences; " + desc},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def device_inputs(w, dev):
    import torch
    s = w["spec"]

    def logits(a):
        if s.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    out = {}
    if w["kind"] == "pipeline":
        out["models"] = [logits(m) for m in w["models"]]
        out["us"] = [torch.from_numpy(u).to(dev) for u in w["us"]]
        out["vs"] = [torch.from_numpy(v).to(dev) for v in w["vs"]]
    for k, v in w.items():
        if not isinstance(v, np.ndarray):
            continue
        if k in ("target", "draft", "l0", "l1", "l2"):
            out[k] = logits(v)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    return out


CONSULTED = False  # set from --consulted-only


def make_plan(w, t, workspace=None):
    import draft_verification_gb300 as dv
    s = w["spec"]
    if w["kind"] == "chain":
        return dv.ChainPlan(t["target"], t["draft"], t["tokens"], t["u"], t["v"], t["prefix_len"],
                            greedy=s.greedy, temperature=s.temperature, workspace=workspace,
                            consulted_only=CONSULTED and not s.greedy)
    if w["kind"] == "tree":
        return dv.TreePlan(t["parent"], t["tokens"], t["target"], t["draft"], t["u"], t["v"],
                           t["prefix_len"], max_depth=w["max_depth"], greedy=s.greedy,
                           temperature=s.temperature, workspace=workspace, consulted_only=CONSULTED)
    if w["kind"] == "pipeline":
        models = [None if (s.greedy and i == 0) else m[:, :, :s.V] for i, m in enumerate(t["models"])]
        return dv.PipelinePlan(models, t["tokens"], s.windows, t["us"], t["vs"], t["base"], greedy=s.greedy,
                               temperature=s.temperature, final_bonus=s.final_bonus, V=s.V,
                               workspace=workspace)
    return dv.CascadePlan(t["l0"], t["l1"], t["l2"], t["tokens"], t["u1"], t["v1"], t["u2"], t["v2"],
                          t["base0"], t["base1"], greedy=s.greedy, temperature=s.temperature,
                          workspace=workspace)


def run_ours(args, w, rank, world, dist):
    import torch
    import draft_verification_gb300 as dv
    from workloads.synth import logit_bytes

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dv.build_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    bytes_per_call = logit_bytes(w)
    n_sets = max(2, math.ceil(3 * l2 / bytes_per_call) + 1)
    n_sets = min(n_sets, max(2, int(0.5 * props.total_memory // max(bytes_per_call, 1))))

    base = device_inputs(w, dev)
    def clone(v):
        return [x.clone() for x in v] if isinstance(v, list) else v.clone()

    sets = [base] + [{k: clone(v) for k, v in base.items()} for _ in range(n_sets - 1)]
    ws = torch.empty(max(16, int(plan_workspace(w))), dtype=torch.uint8, device=dev)
    plans = [make_plan(w, t, ws) for t in sets]
    stream = torch.cuda.Stream(dev)

    def one_pass(s):
        for p in plans:
            p.run(s)

    # warm-up (eager), then capture one call per input copy into a graph
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            plans[i % n_sets].run(stream)
    stream.synchronize()
    launch = "cuda_graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            one_pass(stream)
        stream.synchronize()
    except Exception as exc:  # graph capture unavailable: time eager launches
        launch = f"eager ({type(exc).__name__})"
        graph = None

    def run_steps(k):
        full, rest = divmod(k, n_sets)
        for _ in range(full):
            if graph is not None:
                graph.replay()
            else:
                one_pass(stream)
        for i in range(rest):
            plans[i].run(stream)

    clocks = ClockSampler(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:  # loaded soak so the clocks settle
            run_steps(n_sets * 20)
            stream.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
    clock_info = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, dev)

    # the roofline's unit is one verification call; its average duration is
    # the timed region's (CUDA events around K back-to-back calls replayed
    # from the graph), which includes no host enqueue time
    kernel_ms = ms

    # end to end through the public call, host buffers in and out
    e2e = e2e_rate(args, w, dev, stream)

    tokens = draft_tokens_per_call(w)
    value = whole_job_rate(tokens, world, ms)
    logits_gbs = bytes_per_call / (ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    kernel_gbs = bytes_per_call / (kernel_ms * 1e-3) / 1e9
    check = plans[0].run(stream)
    stream.synchronize()
    s = w["spec"]
    accepted = None
    if w["kind"] == "chain":
        accepted = float((check["accept_len"].float() + 1).mean().item())
    roof_bytes, roof_unit = bytes_per_call, "one verification call"
    if w["kind"] == "chain" and CONSULTED and not s.greedy:
        # the rows the rule consults: 2 (a + 1) after a rejection at a, 2 gamma + 1 otherwise
        a = check["accept_len"].cpu().numpy().astype(np.int64)
        rows = np.where(a < s.gamma, 2 * (a + 1), 2 * s.gamma + 1)
        roof_bytes = int(rows.sum()) * s.V * (2 if s.dtype == "bf16" else 4)
        roof_unit = "one verification call (consulted rows only)"
        kernel_gbs = roof_bytes / (kernel_ms * 1e-3) / 1e9
    if w["kind"] == "tree" and CONSULTED:
        # the rows the walk reads: at every node it stands at, the target row,
        # and (sampling) the draft row when the node has children
        nodes = check["path_nodes"].cpu().numpy()
        has_kids = np.zeros(w["parent"].shape, bool)
        for b in range(s.B):
            has_kids[b, np.unique(w["parent"][b, 1:])] = True
        rows = 0
        for b in range(s.B):
            for n in nodes[b]:
                if n >= 0:
                    rows += 1 + (0 if s.greedy else int(has_kids[b, n]))
        roof_bytes = rows * s.V * (2 if s.dtype == "bf16" else 4)
        roof_unit = "one verification call (consulted rows only)"
        kernel_gbs = roof_bytes / (kernel_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": compute_dtype(s.dtype), "data": "synthetic (seeded; shapes of the pages' model families)",
        "config": dict(workload_config(w), parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                       consulted_only=bool(CONSULTED and (w["kind"] == "tree" or
                                                           (w["kind"] == "chain" and not s.greedy))),
                       l2_policy=f"rotating {n_sets} input copies ({n_sets * bytes_per_call / 2**20:.0f} MB "
                                 f"> 3 x L2 {l2 / 2**20:.0f} MB)", launch=launch),
        "logits_gbs": logits_gbs,
        "logits_frac_of_peak": logits_gbs / peak,
        "accepted_tokens_per_s": None if accepted is None else accepted * s.B * world / (ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": "+".join(KERNELS[w["kind"]]), "unit_of_work": roof_unit,
                     "achieved": kernel_gbs,
                     "peak": peak, "unit": "GB/s", "frac": kernel_gbs / peak, "peak_source": peak_src,
                     "kernel_ms": kernel_ms, "algorithmic_bytes": roof_bytes,
                     "traffic": None if CONSULTED else profiled_traffic(s.name),
                     "traffic_note": "DRAM read + write bytes of one call from the committed ncu capture, "
                                     "caches flushed before each launch (an upper bound for re-reads)"},
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_call(w),
        "clocks": clock_info,
    }
    return line


def plan_workspace(w):
    import draft_verification_gb300 as dv
    s = w["spec"]
    if w["kind"] == "chain":
        return dv.workspace_bytes("chain", s.B, s.gamma, s.V)
    if w["kind"] == "tree":
        return dv.workspace_bytes("tree", s.B, int(w["parent"].shape[1]), s.V)
    if w["kind"] == "pipeline":
        import ctypes
        from draft_verification_gb300 import _lib
        win = (ctypes.c_int * (_lib.SPEC_MAX_MODELS - 1))(*s.windows)
        return int(_lib.lib().spec_pipeline_workspace_size(s.B, s.k, win, int(s.final_bonus), s.V))
    return dv.workspace_bytes("cascade", s.B, s.gamma1, s.gamma2, s.V)


def e2e_rate(args, w, dev, stream):
    """Same metric through the public verify_* call with pinned host tensors:
    each step copies the step's inputs to the device and reads the results
    back (both inside the timed region)."""
    import torch
    import draft_verification_gb300 as dv
    s = w["spec"]
    if w["kind"] == "pipeline":
        return pipeline_e2e(args, w, dev, stream)
    host = {}
    for k, v in w.items():
        if isinstance(v, np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(v))
            if k in ("target", "draft", "l0", "l1", "l2") and s.dtype == "bf16":
                t = t.view(torch.int16).view(torch.bfloat16)
            host[k] = t.pin_memory()
    h2d = sum(t.numel() * t.element_size() for k, t in host.items()
              if not (s.greedy and k in ("draft", "l0", "u", "v", "u1", "v1", "u2", "v2")))

    def call():
        with torch.cuda.stream(stream):
            if w["kind"] == "chain":
                o = dv.verify_chain(host["target"], None if s.greedy else host["draft"], host["tokens"],
                                    host["u"], host["v"], host["prefix_len"], greedy=s.greedy,
                                    temperature=s.temperature, device=dev, stream=stream,
                                    consulted_only=CONSULTED and not s.greedy)
            elif w["kind"] == "tree":
                o = dv.verify_tree(host["parent"], host["tokens"], host["target"], host["draft"],
                                   host["u"], host["v"], host["prefix_len"], max_depth=w["max_depth"],
                                   greedy=s.greedy, temperature=s.temperature, device=dev, stream=stream,
                                   consulted_only=CONSULTED)
            else:
                o = dv.verify_cascade(host["l0"], host["l1"], host["l2"], host["tokens"], host["u1"],
                                      host["v1"], host["u2"], host["v2"], host["base0"], host["base1"],
                                      greedy=s.greedy, temperature=s.temperature, device=dev,
                                      stream=stream)
        return o

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    d2h = 0
    for _ in range(n):
        o = call()
        stream.synchronize()
        d2h = sum(v.numel() * v.element_size() for v in o.values())
    el = time.perf_counter() - t0
    return {"value": draft_tokens_per_call(w) / (el / n), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": 1000.0 * el / n, "steps": n}


# --------------------------------------------------------------------------
# cache compaction after a tree verification (a workload of its own)
# --------------------------------------------------------------------------

def compact_rows(w) -> int:
    """Cache rows one compaction call writes (the root and the kept nodes of
    every sequence the verifier did not flag)."""
    ok = w["path_nodes"][:, 0] >= 0
    return int(np.sum(np.where(ok, w["path_len"] + 1, 0)))


def compact_bytes(w) -> int:
    """Algorithmic bytes of one call: every written row read once and written once."""
    return 2 * compact_rows(w) * w["spec"].row_bytes


def compact_oracle_rate(w, budget_s: float):
    from oracle import compact as K  # the reference is only used on this leg
    t0 = time.perf_counter()
    calls = 0
    while True:
        K.compact_tree_path(w["tree_rows"], w["cache"], w["path_nodes"], w["path_len"], w["prefix_len"])
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return compact_rows(w) * calls / el, f"{calls} whole calls ({el:.1f} s, NumPy row copies)"


def compact_config(w) -> dict:
    s = w["spec"]
    return {"workload": s.name, "kind": "compact", "batch": s.B, "tree_nodes": int(len(w["parent"])),
            "max_depth": s.max_depth, "row_bytes": s.row_bytes, "cache_rows": int(w["cache"].shape[1]),
            "rows_per_call": compact_rows(w)}


def run_compact(args, w):
    import torch
    import draft_verification_gb300 as dv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dv.build_library()
    s = w["spec"]
    W = s.row_bytes
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    moved = compact_bytes(w)
    set_bytes = w["tree_rows"].nbytes + w["cache"].nbytes
    n_sets = max(2, math.ceil(3 * l2 / max(moved, 1)) + 1)
    n_sets = min(n_sets, max(2, int(0.5 * props.total_memory // max(set_bytes, 1))))
    tree0 = torch.from_numpy(w["tree_rows"]).to(dev)
    cache0 = torch.from_numpy(w["cache"]).to(dev)
    paths = {k: torch.from_numpy(np.ascontiguousarray(w[k])).to(dev) for k in ("path_nodes", "path_len", "prefix_len")}
    sets = [(tree0, cache0)] + [(tree0.clone(), cache0.clone()) for _ in range(n_sets - 1)]
    stream = torch.cuda.Stream(dev)

    def call(i):
        t, c = sets[i]
        dv.compact_tree_path(t[:, :, :W], c[:, :, :W], paths["path_nodes"], paths["path_len"],
                             paths["prefix_len"], stream=stream)

    def one_pass():
        for i in range(n_sets):
            call(i)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            call(i % n_sets)
    stream.synchronize()
    launch = "cuda_graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            one_pass()
        stream.synchronize()
    except Exception as exc:
        launch = f"eager ({type(exc).__name__})"
        graph = None

    def run_steps(k):
        full, rest = divmod(k, n_sets)
        for _ in range(full):
            if graph is not None:
                graph.replay()
            else:
                one_pass()
        for i in range(rest):
            call(i)

    clocks = ClockSampler(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            run_steps(n_sets * 20)
            stream.synchronize()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps

    # end to end through the public call: host tree rows, cache and paths
    # in, the cache back out, every step
    host = {k: torch.from_numpy(np.ascontiguousarray(w[k])).pin_memory()
            for k in ("tree_rows", "cache", "path_nodes", "path_len", "prefix_len")}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host["cache"].numel()
    out = torch.empty_like(host["cache"]).pin_memory()

    def e2e_call():
        with torch.cuda.stream(stream):
            d = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
            dv.compact_tree_path(d["tree_rows"][:, :, :W], d["cache"][:, :, :W], d["path_nodes"], d["path_len"],
                                 d["prefix_len"], stream=stream)
            out.copy_(d["cache"], non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_call()
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(n):
        e2e_call()
    el = time.perf_counter() - t0

    rows = compact_rows(w)
    peak, peak_src = measured_peak()
    gbs = moved / (ms * 1e-3) / 1e9
    return {
        "metric": COMPACT_METRIC, "value": rows / (ms * 1e-3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random bytes; root paths drawn on the 64-node tree)",
        "config": dict(compact_config(w), parallelism="1 GPU", launch=launch,
                       l2_policy=f"rotating {n_sets} copies of tree rows and cache "
                                 f"({n_sets * moved / 2**20:.0f} MB moved per rotation > 3 x L2 {l2 / 2**20:.0f} MB)"),
        "roofline": {"bound": "hbm", "kernel": "compact_kernel", "unit_of_work": "one compaction call",
                     "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src,
                     "kernel_ms": ms, "algorithmic_bytes": moved,
                     "traffic": profiled_traffic(s.name, COMPACT_SOURCES)},
        "e2e": {"value": rows / (el / n), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": 1000.0 * el / n, "steps": n},
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }


def compact_main(args, w, rank):
    if args.impl == "reference":
        if rank == 0:
            rate, desc = compact_oracle_rate(w, args.cpu_seconds)
            print(json.dumps({
                "impl": "reference", "metric": COMPACT_METRIC, "value": rate, "unit": "rows/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * compact_rows(w) / rate, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "u8", "data": "synthetic", "config": compact_config(w),
                "cpu_baseline": {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": desc},
                "e2e": {"value": rate, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
        return
    if args.profile:
        import torch
        import draft_verification_gb300 as dv
        dev = torch.device("cuda", 0)
        dv.build_library()
        W = w["spec"].row_bytes
        tree = torch.from_numpy(w["tree_rows"]).to(dev)
        cache = torch.from_numpy(w["cache"]).to(dev)
        p = {k: torch.from_numpy(np.ascontiguousarray(w[k])).to(dev) for k in ("path_nodes", "path_len", "prefix_len")}
        for _ in range(args.warmup + args.steps):
            dv.compact_tree_path(tree[:, :, :W], cache[:, :, :W], p["path_nodes"], p["path_len"], p["prefix_len"])
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": w["spec"].name, "calls": args.warmup + args.steps}))
        return
    if rank != 0:
        return  # one GPU: the other ranks of a replica launch have nothing to add
    line = run_compact(args, w)
    if not args.no_cpu_baseline:
        rate, desc = compact_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# CLaSp layer selection (a workload of its own)
# --------------------------------------------------------------------------

def clasp_columns(spec) -> int:
    """GEMM columns of one call: two bfloat16 terms of every state that may
    keep its layer and can still reach (L, M), summed over the layers."""
    L, M = spec.L, spec.M
    n = 0
    for i in range(1, L + 1):
        lo, last_keep = max(0, M - (L - i)), min(i - 1, M)
        n += max(0, last_keep - lo + 1)
    return 2 * spec.B * n


def clasp_bytes(spec) -> int:
    """Algorithmic HBM bytes of one call: every weight read once, the hidden
    states read once (the DP's states and products stay in L2)."""
    return spec.L * spec.d * spec.d * 2 + spec.B * (spec.L + 1) * spec.d * 4


def clasp_flops(spec) -> int:
    return 2 * spec.d * spec.d * clasp_columns(spec)


def clasp_oracle_rate(w, budget_s: float):
    """Selections/s of the oracle on whole sequences until the budget is
    spent; cores = process CPU time over wall time (NumPy's BLAS may use
    several threads for the matrix-vector products)."""
    from oracle import clasp as K  # the reference is only used on this leg
    from workloads import synth
    s = w["spec"]
    Wv = synth.clasp_weight_values(w)
    t0, c0 = time.perf_counter(), time.process_time()
    n = 0
    while True:
        K.clasp_dp(w["hidden"][n % s.B].astype(np.float64), Wv, s.M)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    cores = (time.process_time() - c0) / el
    return n / el, f"{n} whole sequences ({el:.1f} s; NumPy float64, BLAS matrix-vector products)", round(cores, 1)


def clasp_config(w) -> dict:
    s = w["spec"]
    return {"workload": s.name, "kind": "clasp", "batch": s.B, "layers": s.L, "width": s.d, "skips": s.M,
            "layer": "x + W x, W bf16 ~ N(0, %.2f^2/d)" % s.scale, "gemm_columns_per_call": clasp_columns(s)}


def run_clasp(args, w):
    import torch
    import draft_verification_gb300 as dv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dv.build_library()
    s = w["spec"]
    hidden = torch.from_numpy(w["hidden"]).to(dev)
    weights = torch.from_numpy(w["weights"].view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.Stream(dev)
    plan = dv.ClaspPlan(hidden, weights, s.M)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            plan.run(stream)
    stream.synchronize()
    launch = "cuda_graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            plan.run(stream)
        stream.synchronize()
    except Exception as exc:
        launch = f"eager ({type(exc).__name__})"
        graph = None

    def run_steps(k):
        for _ in range(k):
            if graph is not None:
                graph.replay()
            else:
                plan.run(stream)

    clocks = ClockSampler(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            run_steps(50)
            stream.synchronize()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps

    # end to end through the public call: the hidden states from pinned host
    # memory every step, the skip masks and scores back; the weights are the
    # model's parameters and stay resident
    host_h = torch.from_numpy(w["hidden"]).pin_memory()
    h2d = host_h.numel() * 4

    def e2e_call():
        with torch.cuda.stream(stream):
            o = dv.clasp_layer_select(host_h, weights, s.M, device=dev, stream=stream)
        stream.synchronize()
        return o

    for _ in range(2):
        e2e_call()
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(n):
        o = e2e_call()
    el = time.perf_counter() - t0
    d2h = sum(v.numel() * v.element_size() for v in o.values())

    hbm_peak, hbm_src = measured_peak()
    tc_peak, tc_src = measured_tensor_peak(sustained=False)
    gbs = clasp_bytes(s) / (ms * 1e-3) / 1e9
    tfs = clasp_flops(s) / (ms * 1e-3) / 1e12
    hbm_frac, tc_frac = gbs / hbm_peak, tfs / tc_peak
    # the roofline bound is the resource the call would saturate first
    t_hbm = clasp_bytes(s) / (hbm_peak * 1e9)
    t_tc = clasp_flops(s) / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": hbm_frac,
                "peak_source": hbm_src, "algorithmic_bytes": clasp_bytes(s)}
    else:
        roof = {"bound": "tensor", "achieved": tfs, "peak": tc_peak, "unit": "TFLOP/s", "frac": tc_frac,
                "peak_source": tc_src, "algorithmic_flops": clasp_flops(s)}
    roof.update({"kernel": "whole call: per layer one cuBLAS bf16 GEMM + clasp_step_kernel",
                 "unit_of_work": "one layer-selection call", "kernel_ms": ms,
                 "other": {"hbm_GBps": gbs, "hbm_frac": hbm_frac, "tensor_TFLOPs": tfs, "tensor_frac": tc_frac},
                 "traffic": profiled_traffic(s.name, CLASP_SOURCES)})
    return {
        "metric": CLASP_METRIC, "value": s.B / (ms * 1e-3), "unit": "selections/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x2 split, f32 accumulate",
        "data": "synthetic (seeded bf16 residual layers; hidden states of the full stack plus noise)",
        "config": dict(clasp_config(w), parallelism="1 GPU", launch=launch,
                       l2_policy=f"weights {clasp_bytes(s) / 2**20:.0f} MB per call > L2: every call streams them"),
        "roofline": roof,
        "e2e": {"value": s.B / (el / n), "unit": "selections/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": 1000.0 * el / n, "steps": n,
                "note": "hidden states host to device each step; weights resident"},
        "gpu_launches": args.steps * (s.L + 2),
        "clocks": clock_info,
    }


def clasp_main(args, w, rank):
    s = w["spec"]
    if args.impl == "reference":
        if rank == 0:
            rate, desc, cores = clasp_oracle_rate(w, args.cpu_seconds)
            print(json.dumps({
                "impl": "reference", "metric": CLASP_METRIC, "value": rate, "unit": "selections/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * s.B / rate, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": clasp_config(w),
                "cpu_baseline": {"value": rate, "unit": "selections/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": rate, "unit": "selections/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
        return
    if args.profile:
        import torch
        import draft_verification_gb300 as dv
        dev = torch.device("cuda", 0)
        dv.build_library()
        hidden = torch.from_numpy(w["hidden"]).to(dev)
        weights = torch.from_numpy(w["weights"].view(np.int16)).to(dev).view(torch.bfloat16)
        plan = dv.ClaspPlan(hidden, weights, s.M)
        for _ in range(args.warmup + args.steps):
            plan.run()
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": s.name, "calls": args.warmup + args.steps}))
        return
    if rank != 0:
        return  # one GPU: the other ranks of a replica launch have nothing to add
    line = run_clasp(args, w)
    if not args.no_cpu_baseline:
        rate, desc, cores = clasp_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "selections/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# PipeSpec stages at independent buffer offsets (asynchronous snapshot)
# --------------------------------------------------------------------------

def async_rows(spec) -> int:
    """Logit rows of one call per sequence: each stage's M_s rows (window + 1)
    and, sampling, its M_{s-1} rows (window)."""
    return sum(w + 1 + (0 if spec.greedy else w) for w in spec.windows)


def async_bytes(spec) -> int:
    return spec.B * async_rows(spec) * spec.V * (2 if spec.dtype == "bf16" else 4)


def async_tokens(spec) -> int:
    return spec.B * sum(spec.windows)


def async_launches_per_call(spec) -> int:
    """One chain verification per stage (statistics and walk per batch
    group), then the combine kernel."""
    elt = 2 if spec.dtype == "bf16" else 4
    return 1 + sum(2 * chain_groups(spec.B, w + 1 if spec.greedy else 2 * w + 1, spec.V, elt)
                   for w in spec.windows)


def async_config(w) -> dict:
    s = w["spec"]
    return {"workload": s.name, "kind": "pipeline_async", "batch": s.B, "models": s.k, "windows": list(s.windows),
            "vocab": s.V, "dtype": s.dtype, "temperature": s.temperature, "final_bonus": s.final_bonus,
            "greedy": s.greedy, "logit_bytes_per_call": async_bytes(s)}


def async_oracle_rate(w, budget_s: float):
    from oracle import pipeline_async as A  # the reference is only used on this leg
    s = w["spec"]
    t0 = time.perf_counter()
    n = 0
    while True:
        b = n % s.B
        sub = lambda xs: [x[b:b + 1] for x in xs]
        A.verify_pipeline_async(sub(w["targets"]), None if s.greedy else sub(w["drafts"]), sub(w["tokens"]),
                                sub(w["us"]), sub(w["vs"]), w["length"][:, b:b + 1], s.temperature, s.greedy,
                                s.final_bonus, s.dtype, V=s.V)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return n * sum(s.windows) / el, f"{n} whole sequences ({el:.1f} s, float64 NumPy)"


def run_pipeline_async(args, w):
    import torch
    import draft_verification_gb300 as dv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dv.build_library()
    s = w["spec"]
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    nbytes = async_bytes(s)
    n_sets = max(2, math.ceil(3 * l2 / nbytes) + 1)

    def logits(a):
        t = torch.from_numpy(a).to(dev)
        return (t.view(torch.bfloat16) if s.dtype == "bf16" else t)[:, :, :s.V]

    small = dict(tokens=[torch.from_numpy(t).to(dev) for t in w["tokens"]],
                 length=torch.from_numpy(w["length"]).to(dev),
                 us=[torch.from_numpy(u).to(dev) for u in w["us"]], vs=[torch.from_numpy(v).to(dev) for v in w["vs"]])
    base_t = [logits(x.view(np.int16) if s.dtype == "bf16" else x) for x in w["targets"]]
    base_d = [logits(x.view(np.int16) if s.dtype == "bf16" else x) for x in w["drafts"]]
    sets = [(base_t, base_d)] + [([t.clone() for t in base_t], [d.clone() for d in base_d]) for _ in range(n_sets - 1)]
    plans = [dv.PipelineAsyncPlan(t, None if s.greedy else d, small["tokens"], small["length"],
                                  None if s.greedy else small["us"], None if s.greedy else small["vs"],
                                  greedy=s.greedy, temperature=s.temperature, final_bonus=s.final_bonus)
             for t, d in sets]
    stream = torch.cuda.Stream(dev)

    def one_pass():
        for p in plans:
            p.run(stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            plans[i % n_sets].run(stream)
    stream.synchronize()
    launch = "cuda_graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            one_pass()
        stream.synchronize()
    except Exception as exc:
        launch = f"eager ({type(exc).__name__})"
        graph = None

    def run_steps(k):
        full, rest = divmod(k, n_sets)
        for _ in range(full):
            if graph is not None:
                graph.replay()
            else:
                one_pass()
        for i in range(rest):
            plans[i].run(stream)

    clocks = ClockSampler(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            run_steps(n_sets * 10)
            stream.synchronize()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps

    # end to end through the public call: host logits, tokens, uniforms and
    # lengths in, the outputs back, every step
    def pin(a, is_logits=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if is_logits and s.dtype == "bf16":
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory()

    host_t = [pin(x[:, :, :s.V], True) for x in w["targets"]]
    host_d = None if s.greedy else [pin(x[:, :, :s.V], True) for x in w["drafts"]]
    host_tok = [pin(t) for t in w["tokens"]]
    host_len = pin(w["length"])
    host_u = None if s.greedy else [pin(u) for u in w["us"]]
    host_v = None if s.greedy else [pin(v) for v in w["vs"]]
    h2d = sum(t.numel() * t.element_size() for t in host_t + (host_d or []) + host_tok + (host_u or []) +
              (host_v or [])) + host_len.numel() * 4

    def e2e_call():
        with torch.cuda.stream(stream):
            o = dv.verify_pipeline_async(host_t, host_d, host_tok, host_len, host_u, host_v, greedy=s.greedy,
                                         temperature=s.temperature, final_bonus=s.final_bonus, V=s.V, device=dev,
                                         stream=stream)
        stream.synchronize()
        return o

    for _ in range(2):
        e2e_call()
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(n):
        o = e2e_call()
    el = time.perf_counter() - t0
    d2h = sum(v.numel() * v.element_size() for v in o.values())

    peak, peak_src = measured_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": async_tokens(s) / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": compute_dtype(s.dtype),
        "data": "synthetic (seeded logits; windows drawn from the drafter's softmax)",
        "config": dict(async_config(w), parallelism="1 GPU", launch=launch,
                       l2_policy=f"rotating {n_sets} copies of the logits "
                                 f"({n_sets * nbytes / 2**20:.0f} MB > 3 x L2 {l2 / 2**20:.0f} MB)"),
        "roofline": {"bound": "hbm", "kernel": "whole call: per stage stats_kernel + chain_walk_kernel, then "
                                               "pipeline_async_combine_kernel",
                     "unit_of_work": "one asynchronous snapshot", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": peak_src, "kernel_ms": ms, "algorithmic_bytes": nbytes,
                     "traffic": profiled_traffic(s.name, ASYNC_SOURCES)},
        "e2e": {"value": async_tokens(s) / (el / n), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": 1000.0 * el / n, "steps": n},
        "gpu_launches": args.steps * async_launches_per_call(s),
        "clocks": clock_info,
    }


def pipeline_async_main(args, w, rank):
    s = w["spec"]
    if args.impl == "reference":
        if rank == 0:
            rate, desc = async_oracle_rate(w, args.cpu_seconds)
            print(json.dumps({
                "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * async_tokens(s) / rate,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": async_config(w),
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
        return
    if args.profile:
        import torch
        import draft_verification_gb300 as dv
        dev = torch.device("cuda", 0)
        dv.build_library()

        def logits(a):
            t = torch.from_numpy(a.view(np.int16) if s.dtype == "bf16" else a).to(dev)
            return (t.view(torch.bfloat16) if s.dtype == "bf16" else t)[:, :, :s.V]

        d = lambda xs: [torch.from_numpy(x).to(dev) for x in xs]
        plan = dv.PipelineAsyncPlan([logits(x) for x in w["targets"]],
                                    None if s.greedy else [logits(x) for x in w["drafts"]], d(w["tokens"]),
                                    torch.from_numpy(w["length"]).to(dev), None if s.greedy else d(w["us"]),
                                    None if s.greedy else d(w["vs"]), greedy=s.greedy, temperature=s.temperature,
                                    final_bonus=s.final_bonus)
        for _ in range(args.warmup + args.steps):
            plan.run()
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": s.name, "calls": args.warmup + args.steps}))
        return
    if rank != 0:
        return  # one GPU: the other ranks of a replica launch have nothing to add
    line = run_pipeline_async(args, w)
    if not args.no_cpu_baseline:
        rate, desc = async_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


def pipeline_e2e(args, w, dev, stream):
    """e2e_rate for the k-model pipeline (lists of per-model inputs)."""
    import torch
    import draft_verification_gb300 as dv
    s = w["spec"]

    def pin(a, logits=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if logits and s.dtype == "bf16":
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory()

    models = [None if (s.greedy and i == 0) else pin(m[:, :, :s.V], True) for i, m in enumerate(w["models"])]
    us = None if s.greedy else [pin(u) for u in w["us"]]
    vs = None if s.greedy else [pin(v) for v in w["vs"]]
    tokens, base = pin(w["tokens"]), pin(w["base"])
    h2d = sum(m.numel() * m.element_size() for m in models if m is not None) + tokens.numel() * 4 + base.numel() * 4
    if not s.greedy:
        h2d += sum(u.numel() * 4 for u in us) + sum(v.numel() * 4 for v in vs)

    def call():
        with torch.cuda.stream(stream):
            return dv.verify_pipeline(models, tokens, s.windows, us, vs, base, greedy=s.greedy,
                                      temperature=s.temperature, final_bonus=s.final_bonus, V=s.V, device=dev,
                                      stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    d2h = 0
    for _ in range(n):
        o = call()
        stream.synchronize()
        d2h = sum(v.numel() * v.element_size() for v in o.values())
    el = time.perf_counter() - t0
    return {"value": draft_tokens_per_call(w) / (el / n), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": 1000.0 * el / n, "steps": n}


def run_profile(args, w):
    """W + K eager calls on one input copy, nothing else (an ncu target)."""
    import torch
    import draft_verification_gb300 as dv
    dev = torch.device("cuda", 0)
    dv.build_library()
    plan = make_plan(w, device_inputs(w, dev))
    for _ in range(args.warmup + args.steps):
        plan.run()
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": w["spec"].name, "calls": args.warmup + args.steps}))


# --------------------------------------------------------------------------
# LM head folded into the verification (spec_verify_chain_lm_head)
# --------------------------------------------------------------------------
LM_HEAD_SOURCES = ["draft_verification_gb300/csrc/lm_head.cu", "draft_verification_gb300/csrc/tc.cuh"] + \
    KERNEL_SOURCES


def lm_head_flops(spec) -> int:
    """2 * rows * d * V per head: the products the head kernels compute."""
    rows_t = spec.B * (spec.gamma + 1)
    rows_d = 0 if spec.greedy else spec.B * spec.gamma
    return 2 * spec.V * (rows_t * spec.d_target + rows_d * spec.d_draft)


def lm_head_bytes(spec) -> int:
    """Algorithmic HBM bytes: each head's weights once and the hidden states."""
    heads = spec.V * spec.d_target * 2 + (0 if spec.greedy or spec.gamma == 0 else spec.V * spec.d_draft * 2)
    hidden = spec.B * ((spec.gamma + 1) * spec.d_target + (0 if spec.greedy else spec.gamma * spec.d_draft)) * 2
    return heads + hidden


def lm_head_config(w) -> dict:
    s = w["spec"]
    return {"workload": s.name, "kind": "lm_head", "batch": s.B, "gamma": s.gamma, "vocab": s.V,
            "d_target": s.d_target, "d_draft": s.d_draft, "shared_head": s.d_target == s.d_draft,
            "mode": "greedy" if s.greedy else "sampling", "temperature": s.temperature,
            "alpha_target": s.alpha_target}


def lm_head_device(w, dev):
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    wt = bf(w["w_target"])
    wd = wt if w["w_draft"] is w["w_target"] else bf(w["w_draft"])
    return dict(h_target=bf(w["h_target"]), h_draft=bf(w["h_draft"]), w_target=wt, w_draft=wd,
                tokens=torch.from_numpy(w["tokens"]).to(dev), u=torch.from_numpy(w["u"]).to(dev),
                v=torch.from_numpy(w["v"]).to(dev), prefix_len=torch.from_numpy(w["prefix_len"]).to(dev))


def lm_head_plan(w, t):
    import draft_verification_gb300 as dv
    s = w["spec"]
    return dv.LmHeadChainPlan(t["h_target"], t["h_draft"], t["w_target"], t["w_draft"], t["tokens"], t["u"],
                              t["v"], t["prefix_len"], greedy=s.greedy, temperature=s.temperature)


def lm_head_oracle_rate(w, budget_s: float):
    """Verified draft tokens/s of the oracle on whole sequences (exact
    float64 products, then the chain rule) until the budget is spent."""
    from oracle import lm_head as LH  # the reference is only used on this leg
    s = w["spec"]
    wt = LH.bf16_values(w["w_target"])
    wd = wt if w["w_draft"] is w["w_target"] else LH.bf16_values(w["w_draft"])
    t0, c0 = time.perf_counter(), time.process_time()
    n = 0
    while True:
        b = n % s.B
        LH.verify_chain_from_hidden(LH.bf16_values(w["h_target"][b:b + 1]), LH.bf16_values(w["h_draft"][b:b + 1]),
                                    wt, wd, w["tokens"][b:b + 1], w["u"][b:b + 1], w["v"][b:b + 1],
                                    w["prefix_len"][b:b + 1], s.temperature, s.greedy)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    cores = (time.process_time() - c0) / el
    return n * s.gamma / el, (f"{n} whole sequences ({el:.1f} s; NumPy float64 products and chain rule)",
                              round(cores, 1))


def run_lm_head(args, w):
    import torch
    import draft_verification_gb300 as dv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dv.build_library()
    s = w["spec"]
    t = lm_head_device(w, dev)
    plan = lm_head_plan(w, t)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            plan.run(stream)
    stream.synchronize()
    launch = "cuda_graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            plan.run(stream)
        stream.synchronize()
    except Exception as exc:
        launch = f"eager ({type(exc).__name__})"
        graph = None

    def run_steps(k):
        for _ in range(k):
            if graph is not None:
                graph.replay()
            else:
                plan.run(stream)

    clocks = ClockSampler(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            run_steps(20)
            stream.synchronize()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps

    # end to end: the hidden states from pinned host memory every step, the
    # outputs back; the heads are model parameters and stay resident
    host = {k: torch.from_numpy(np.ascontiguousarray(w[k]).view(np.int16)).pin_memory()
            for k in ("h_target", "h_draft")}
    host.update({k: torch.from_numpy(w[k]).pin_memory() for k in ("tokens", "u", "v", "prefix_len")})
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    dev_in = {k: torch.empty_like(x, device=dev) for k, x in host.items()}
    e2e_plan = dv.LmHeadChainPlan(dev_in["h_target"].view(torch.bfloat16), dev_in["h_draft"].view(torch.bfloat16),
                                  t["w_target"], t["w_draft"], dev_in["tokens"], dev_in["u"], dev_in["v"],
                                  dev_in["prefix_len"], greedy=s.greedy, temperature=s.temperature,
                                  workspace=plan.workspace)
    outs_host = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in e2e_plan.out.items()}
    d2h = sum(x.numel() * x.element_size() for x in outs_host.values())

    def e2e_call():
        with torch.cuda.stream(stream):
            for k in host:
                dev_in[k].copy_(host[k], non_blocking=True)
            e2e_plan.run(stream)
            for k, x in e2e_plan.out.items():
                outs_host[k].copy_(x, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_call()
    n = max(3, args.e2e_steps)
    t0 = time.perf_counter()
    for _ in range(n):
        e2e_call()
    el = time.perf_counter() - t0

    hbm_peak, hbm_src = measured_peak()
    tc_peak, tc_src = measured_tensor_peak(sustained=True)
    flops, nbytes = lm_head_flops(s), lm_head_bytes(s)
    tfs = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    if flops / (tc_peak * 1e12) >= nbytes / (hbm_peak * 1e9):
        roof = {"bound": "tensor", "achieved": tfs, "peak": tc_peak, "unit": "TFLOP/s", "frac": tfs / tc_peak,
                "peak_source": tc_src, "algorithmic_flops": flops}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                "peak_source": hbm_src, "algorithmic_bytes": nbytes}
    launches = 2 if (s.greedy or s.gamma == 0) else 3
    roof.update({"kernel": "whole call: one head kernel per head (lm_head_pair_kernel on CTA pairs or lm_head_kernel, as the library picks) + chain walk", "unit_of_work": "one call",
                 "kernel_ms": ms,
                 "other": {"tensor_TFLOPs": tfs, "tensor_frac": tfs / tc_peak, "weights_GBps": gbs,
                           "hbm_frac": gbs / hbm_peak},
                 "traffic": profiled_traffic(s.name, LM_HEAD_SOURCES)})
    tokens = s.B * s.gamma
    return {
        "metric": METRIC, "value": tokens / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, f32 accumulate (tcgen05)",
        "data": "synthetic (seeded bf16 hidden states and LM heads)",
        "config": dict(lm_head_config(w), parallelism="1 GPU", launch=launch,
                       l2_policy=f"heads {nbytes / 2**20:.0f} MB per call > L2: every call streams them"),
        "roofline": roof,
        "e2e": {"value": tokens / (el / n), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": 1000.0 * el / n, "steps": n,
                "note": "hidden states, tokens and uniforms host to device each step; heads resident"},
        "gpu_launches": args.steps * launches,
        "clocks": clock_info,
    }


def lm_head_main(args, w, rank):
    s = w["spec"]
    if args.impl == "reference":
        if rank == 0:
            rate, (desc, cores) = lm_head_oracle_rate(w, args.cpu_seconds)
            print(json.dumps({
                "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * s.B * s.gamma / rate, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": lm_head_config(w),
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
        return
    if args.profile:
        import torch
        import draft_verification_gb300 as dv
        dev = torch.device("cuda", 0)
        dv.build_library()
        plan = lm_head_plan(w, lm_head_device(w, dev))
        for _ in range(args.warmup + args.steps):
            plan.run()
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": s.name, "calls": args.warmup + args.steps}))
        return
    if rank != 0:
        return
    line = run_lm_head(args, w)
    if not args.no_cpu_baseline:
        rate, (desc, cores) = lm_head_oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)


def main():
    global CONSULTED
    args = parse()
    CONSULTED = args.consulted_only
    from workloads import synth
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.workload in synth.COMPACT_SPECS:
        compact_main(args, synth.make(synth.COMPACT_SPECS[args.workload], seed=replica_seed(args.seed, rank)), rank)
        return
    if args.workload in synth.PIPELINE_ASYNC_SPECS:
        pipeline_async_main(args, synth.make(synth.PIPELINE_ASYNC_SPECS[args.workload],
                                             seed=replica_seed(args.seed, rank)), rank)
        return
    if args.workload in synth.CLASP_SPECS:
        clasp_main(args, synth.make(synth.CLASP_SPECS[args.workload], seed=replica_seed(args.seed, rank)), rank)
        return
    if args.workload in synth.LM_HEAD_SPECS:
        lm_head_main(args, synth.make(synth.LM_HEAD_SPECS[args.workload], seed=replica_seed(args.seed, rank)), rank)
        return
    specs = dict(synth.SPECS, **synth.PIPELINE_SPECS)
    if args.workload not in specs:
        raise SystemExit(f"unknown workload {args.workload}; choose from "
                         f"{sorted(specs) + sorted(synth.COMPACT_SPECS) + sorted(synth.CLASP_SPECS) + sorted(synth.PIPELINE_ASYNC_SPECS) + sorted(synth.LM_HEAD_SPECS)}")
    w = synth.make(specs[args.workload], seed=replica_seed(args.seed, rank))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    if args.profile:
        run_profile(args, w)
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_ours(args, w, rank, world, dist)
    if rank == 0 and not args.no_cpu_baseline:
        sample, nseq = bounded_sample(w, args.cpu_seconds)
        rate, desc, _ = oracle_rate(sample, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {nseq} of {w['spec'].B} sequences; " + desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
