"""Benchmark of the sparse-attention hot path on GB300.

Headline: the sparse-prefill workload (B=2, S1=2048, S2=16384, N1=64, N2=8,
Dk=192, Dv=128 with value = key prefix, topK=2048, fp16, BSND, causal), the
largest top-K configuration.  One step = one call of the top-K entry point
over the whole workload, inputs resident in HBM.  The same JSON line carries a
`workloads` object with one record per other workload (GQA decode, MLA decode
and MTP, the operator page's call example, block-sparse plain / causal /
per-element mask, variable block-sparse), each with its own step time,
roofline, end-to-end figure and CPU-oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--sub all|none|a,b,...]

The K timed steps of a workload are captured once into a CUDA graph (the
public entry point called K times on one stream) and replayed, timed with
CUDA events on that stream: the device time of K back-to-back calls, without
the Python-side cost of each call.  `e2e` times the same entry point called
eagerly from Python with the step's inputs copied in from pinned host memory
and its outputs read back every step.

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the headline workload.  Under torchrun every rank runs
an independent replica of the workload (weak scaling, no collective on the
data path); timing is the max over ranks.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "sparse-attn effective TFLOP/s & gathered-KV GB/s, fraction of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEADLINE = "sparse_prefill"
SUB_WORKLOADS = ("gqa_decode", "mla_decode", "mla_mtp", "call_example", "bsr", "bsr_causal",
                 "bsr_mask", "bsr_fp8", "varbsr")
ALL_WORKLOADS = sorted(synth.SFA_WORKLOADS) + sorted(synth.BSR_WORKLOADS) + \
    sorted(synth.VARBSR_WORKLOADS)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=ALL_WORKLOADS)
    ap.add_argument("--sub", default="auto",
                    help="other workloads recorded under `workloads`: all, none or a comma "
                         "list (auto = all with the default headline, none otherwise)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the gather-only probe of the top-K workloads")
    ap.add_argument("--eager", action="store_true",
                    help="time eager calls instead of a captured CUDA graph")
    ap.add_argument("--replicas", type=int, default=0,
                    help="input replicas rotated over the steps (0 = enough to exceed L2 4x; "
                         "1 keeps a profiling capture small)")
    return ap.parse_args(argv)


def sub_workloads(args):
    if args.sub == "auto":
        return list(SUB_WORKLOADS) if args.workload == HEADLINE else []
    if args.sub == "none":
        return []
    if args.sub == "all":
        return [w for w in SUB_WORKLOADS if w != args.workload]
    names = [w for w in args.sub.split(",") if w]
    bad = [w for w in names if w not in ALL_WORKLOADS]
    if bad:
        raise SystemExit(f"unknown workloads: {bad}")
    return [w for w in names if w != args.workload]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device):
    """The largest of every rank's value (the slowest rank's step time):
    an all-reduce MAX over the default process group (no-op for one rank)."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms, world):
    """Units processed by all ranks together per second, each rank running an
    independent replica of the workload and the step time being the max over
    ranks (weak scaling)."""
    return world * units_per_rank / (ms * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------------------------
# clocks sampling during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def merge_clocks(parts):
    parts = [c for c in parts if c]
    if not parts:
        return None
    sm = [c["sm_mhz"] for c in parts if c.get("sm_mhz") is not None]
    smax = [c["sm_max_mhz"] for c in parts if c.get("sm_max_mhz") is not None]
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted({r for c in parts for r in c["reasons"]}),
            "samples": sum(c["samples"] for c in parts)}


# ---------------------------------------------------------------------------
# figures from a committed ncu summary (only while the kernel sources it was
# taken on are unchanged)

def kernel_source_sha(files):
    """sha256 over the named kernel sources (file name + bytes, in order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_serving_sfa_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def committed_profile(workload):
    """Per-launch figures of the workload's main kernel from its committed ncu
    summary (profiles/<workload>_ncu.md): {"dram": bytes, "lts": bytes or
    None}, or None when the summary is missing or its kernel sources have
    changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{workload}_ncu.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    src = re.search(r"^sources:\s*(.+)$", text, re.M)
    sha = re.search(r"^source_sha256:\s*([0-9a-f]+)", text, re.M)
    val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not src or not sha or not val:
        return None
    try:
        if sha.group(1) != kernel_source_sha(src.group(1).split()):
            return None
    except OSError:
        return None
    lts = re.search(r"^lts_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    return {"dram": float(val.group(1)), "lts": float(lts.group(1)) if lts else None}


def committed_traffic(workload):
    prof = committed_profile(workload)
    return None if prof is None else prof["dram"]


# main kernel of each workload (what the roofline object describes)
MAIN_KERNEL = {
    "tiny": "generic top-K kernel",
    "gqa_decode": "sfa_decode_kernel (one launch per call; split index lists merged in-kernel)",
    "sparse_prefill": "sfa_decode_kernel (one launch per call; whole index lists per CTA)",
    "mla_decode": "sfa_mla_kernel (one launch per call: the two ranges of every index list run as "
                  "one 4-CTA cluster and merge in distributed shared memory)",
    "mla_mtp": "sfa_mla_kernel + sfa_mla_combine (two launches per call; time is the call's)",
    "call_example": "sfa_decode_kernel (one launch per call; whole index lists per CTA)",
    "bsr": "bsr_tc_wide_kernel (one launch per bsr_run)",
    "bsr_causal": "bsr_tc_wide_kernel, causal mode (one launch per bsr_run)",
    "bsr_mask": "bsr_tc_kernel, per-element mask (one launch per bsr_run)",
    "bsr_fp8": "bsr_tc_wide_kernel, E4M3 instantiation (one launch per bsr_run_scaled)",
    "varbsr": "bsr_tc_wide_kernel, variable mode (one launch per varbsr_run)",
}


# ---------------------------------------------------------------------------
# timing

def device_time(step, steps, eager, world):
    """Device time of `steps` back-to-back calls of step(i) on the current
    stream: captured once into a CUDA graph and replayed (or, with `eager` or
    when capture fails, called from Python), CUDA events on that stream,
    barrier + synchronize on both sides.  Returns (ms per step, kernels
    launched in the timed region, how the steps were launched)."""
    import sparse_attention_serving_sfa_gb300 as sfa
    stream = torch.cuda.current_stream()
    graph, mode, per_graph = None, "eager", 0
    if not eager:
        try:
            graph = torch.cuda.CUDAGraph()
            l0 = sfa.sfa_kernel_launches()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                for i in range(steps):
                    step(i)
            per_graph = sfa.sfa_kernel_launches() - l0
            graph.replay()           # one untimed replay
            torch.cuda.synchronize()
            mode = f"CUDA graph of the {steps} calls, replayed once"
        except Exception as e:  # noqa: BLE001 - fall back to eager calls
            graph = None
            mode = f"eager (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    l0 = sfa.sfa_kernel_launches()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(steps):
            step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = per_graph if graph is not None else sfa.sfa_kernel_launches() - l0
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps, world, "cuda")
    return ms, int(launches), mode


E2E_SCHEDULE = ("every step copies its inputs in from pinned host memory and its outputs back; "
                "two device buffer sets, copies on two copy streams overlapping the neighbouring "
                "steps' calls")


def e2e_time(h2d, compute, d2h, n, warm, world, eager=False):
    """Event-timed end-to-end steps through the public API, run as a serving
    loop runs them: two sets of device buffers; step i's inputs copy in from
    pinned host memory on a copy stream while step i - 1 computes, its call
    runs once they have landed, and its outputs copy back to pinned host
    memory on a second copy stream while step i + 1 computes.  The timed
    region holds every step's copies in and out and ends when the last
    step's outputs are on the host.  h2d(i, b), compute(i, b) and d2h(i, b)
    issue step i's work on buffer set b on the current stream.  As for the
    device time, the n steps are captured once into a CUDA graph (copies,
    calls and the streams' event edges) and replayed, unless `eager` or the
    capture fails.  Returns (ms per step, how the steps were launched)."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of set b landed
    done = [torch.cuda.Event() for _ in range(2)]    # the call on set b finished
    back = [torch.cuda.Event() for _ in range(2)]    # outputs of set b on the host

    def run(m):
        cs = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cs)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        with torch.cuda.stream(s_in):
            h2d(0, 0)
            ready[0].record(s_in)
        for i in range(m):
            b = i & 1
            if i + 1 < m:
                if i >= 1:
                    s_in.wait_event(done[b ^ 1])      # step i - 1 has read set b ^ 1
                with torch.cuda.stream(s_in):
                    h2d(i + 1, b ^ 1)
                    ready[b ^ 1].record(s_in)
            cs.wait_event(ready[b])
            if i >= 2:
                cs.wait_event(back[b])                # step i - 2's outputs are out
            compute(i, b)
            done[b].record(cs)
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                d2h(i, b)
                back[b].record(s_out)
        for b in range(min(m, 2)):
            cs.wait_event(back[b])

    stream = torch.cuda.current_stream()
    run(warm)
    torch.cuda.synchronize()
    graph, mode = None, "eager"
    if not eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                run(n)
            graph.replay()           # one untimed replay
            torch.cuda.synchronize()
            mode = f"CUDA graph of the {n} steps (copies and calls), replayed once"
        except Exception as e:  # noqa: BLE001 - fall back to eager steps
            graph = None
            mode = f"eager (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        run(n)
    ev1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(ev0.elapsed_time(ev1) / n, world, "cuda"), mode


def nbytes(t):
    return t.numel() * t.element_size()


# ---------------------------------------------------------------------------
# top-K workloads

def sfa_config(case, world):
    return {"workload": case.name, "B": case.B, "S1": case.S1, "S2": case.S2, "N1": case.N1,
            "N2": case.N2, "Dk": case.Dk, "Dv": case.Dv, "topK": case.topK,
            "layout": case.layout, "causal": case.causal,
            "value_is_key_prefix": case.value_is_key_prefix, "index": case.index_kind,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def roofline_terms(work, peaks):
    """Time bounds of the survey's roofline: gathered bytes at the measured
    HBM copy peak and useful FLOPs at the measured bf16 burst tensor peak."""
    t_hbm = work["gathered_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    return t_hbm, t_tc


def run_sfa(name, args, world, rank, cpu_target_s):
    import sparse_attention_serving_sfa_gb300 as sfa
    case = synth.SFA_WORKLOADS[name]
    host = synth.make_sfa_inputs(case)
    counts = synth.sfa_counts(case, host["idx"])
    prefix = case.value_is_key_prefix
    # Rotating replicas: consecutive steps read different copies whose
    # gathered bytes together exceed L2 several times, so every step gathers
    # from HBM (no flush needed between steps).
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    reps = args.replicas if args.replicas > 0 else max(1, -(-4 * l2 // counts["gathered_bytes"]) + 1)
    reps = min(reps, 12)
    replicas = []
    for _ in range(reps):
        d = {"q": host["q"].cuda(), "k": host["k"].cuda(), "idx": host["idx"].cuda()}
        d["v"] = d["k"] if prefix else host["v"].cuda()
        replicas.append(d)
    if case.layout == "BSND":
        out_shape, lse_shape = (case.B, case.S1, case.N1, case.Dv), (case.B, case.S1, case.N1)
    else:
        out_shape, lse_shape = (case.B, case.N1, case.S1, case.Dv), (case.B, case.N1, case.S1)
    tdt = replicas[0]["q"].dtype
    out = torch.empty(out_shape, dtype=tdt, device="cuda")
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")
    ws_bytes = sfa.sfa_workspace_size(case.B, case.S1, case.N1, case.N2, case.Dk, case.Dv,
                                      case.topK)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

    def call(d, q=None, idx=None, o=None, l=None, ready=False):
        sfa.sfa_run_ex(d["q"] if q is None else q, d["k"], d["v"], d["idx"] if idx is None else idx,
                       case.B, case.S1, case.S2, case.N1, case.N2, case.Dk, case.Dv, case.topK,
                       case.scale, case.layout, case.causal, case.dtype,
                       out if o is None else o, lse if l is None else l,
                       torch.cuda.current_stream(), workspace=ws, value_is_key_prefix=prefix,
                       inputs_ready=ready)

    for i in range(max(args.warmup, 3) + reps):
        call(replicas[i % reps])
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.2)
    ms, launches, mode = device_time(lambda i: call(replicas[i % reps]), args.steps, args.eager,
                                     world)
    clocks = sampler.stop()

    # the same calls with sfa_options.inputs_ready (the inputs of every call
    # exist before the previous call starts, as they do here): the
    # small-group and MLA kernels then gather while the previous call finishes
    ready = None
    if MAIN_KERNEL.get(name, "").startswith(("sfa_decode_kernel", "sfa_mla_kernel")):
        r_ms, _, r_mode = device_time(lambda i: call(replicas[i % reps], ready=True), args.steps,
                                      args.eager, world)
        ready = {"what": "sfa_options.inputs_ready = 1: a call waits for the previous one only "
                         "before its first write", "us_per_call": r_ms * 1e3,
                 "value": whole_job_rate(counts["gathered_bytes"], r_ms, world) / 1e9, "unit": "GB/s",
                 "launch": r_mode}

    probe = None
    if not args.no_probe:
        probe = gather_probe(case, replicas, reps, args, world, counts, ms)

    e2e = None
    if not args.no_e2e:
        # the KV cache stays resident (as in serving); q and the indices come
        # in from pinned host memory, out and lse go back, every step
        hq, hidx = host["q"].pin_memory(), host["idx"].pin_memory()
        hout = torch.empty(out_shape, dtype=tdt).pin_memory()
        hlse = torch.empty(lse_shape, dtype=torch.float32).pin_memory()
        sets = [{"q": torch.empty_like(replicas[0]["q"]), "idx": torch.empty_like(replicas[0]["idx"]),
                 "out": torch.empty_like(out), "lse": torch.empty_like(lse)} for _ in range(2)]

        def h2d(i, b):
            sets[b]["q"].copy_(hq, non_blocking=True)
            sets[b]["idx"].copy_(hidx, non_blocking=True)

        def compute(i, b):
            t = sets[b]
            call(replicas[i % reps], q=t["q"], idx=t["idx"], o=t["out"], l=t["lse"])

        def d2h(i, b):
            hout.copy_(sets[b]["out"], non_blocking=True)
            hlse.copy_(sets[b]["lse"], non_blocking=True)

        n_e2e = max(min(args.steps, 50), 5)
        e_ms, e_mode = e2e_time(h2d, compute, d2h, n_e2e, min(reps, 3), world, args.eager)
        e2e = {"value": whole_job_rate(counts["gathered_bytes"], e_ms, world) / 1e9,
               "unit": "GB/s", "ms_per_step": e_ms, "steps": n_e2e, "schedule": E2E_SCHEDULE,
               "launch": e_mode,
               "h2d_bytes_per_step": nbytes(hq) + nbytes(hidx),
               "d2h_bytes_per_step": nbytes(hout) + nbytes(hlse)}

    peaks, peak_src = load_peaks()
    gbs = counts["gathered_bytes"] / (ms * 1e-3) / 1e9
    tflops = counts["flops"] / (ms * 1e-3) / 1e12
    t_hbm, t_tc = roofline_terms(counts, peaks)
    prof = committed_profile(name)
    roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": None if prof is None else prof["dram"],
                "peak_source": f"{peak_src} hbm_gbs (copy, read+write bytes)",
                "algorithmic": "gathered K/V bytes of the selected slots per launch",
                "kernel": MAIN_KERNEL.get(name, "sfa_run_ex call") + "; CUDA events on its stream"}
    if prof is not None and prof.get("lts") is not None:
        roofline["l2_traffic"] = prof["lts"]
    cfg = sfa_config(case, world)
    rot = reps * counts["gathered_bytes"]
    cfg["l2"] = (f"not flushed: {reps} rotating input replica(s), {rot >> 20} MiB gathered per "
                 f"rotation {'>' if rot > l2 else '<='} L2 {l2 >> 20} MiB"
                 + ("" if rot > l2 else " (profiling run: not a valid timing)"))
    cfg["launch"] = mode
    rec = {"workload": name, "value": whole_job_rate(counts["gathered_bytes"], ms, world) / 1e9,
           "unit": "GB/s", "ms_per_step": ms, "us_per_call": ms * 1e3, "dtype": case.dtype,
           "config": cfg, "gathered_gbs": world * gbs, "tflops": world * tflops,
           "tensor_frac": tflops / peaks["bf16_tflops"],
           "roofline_time_frac": max(t_hbm, t_tc) / (ms * 1e-3),
           "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
           "gather_probe": probe, "with_inputs_ready": ready,
           "work": {"flops": counts["flops"], "gathered_bytes": counts["gathered_bytes"],
                    "unmasked_slots": counts["unmasked_slots"]}}
    if rank == 0 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = sfa_cpu_baseline(case, host, counts, cpu_target_s)
    del replicas, out, lse, ws
    torch.cuda.empty_cache()
    return rec


def gather_probe(case, replicas, reps, args, world, counts, kernel_ms):
    """The call's K/V row gather alone (sfa_gather_probe: no arithmetic),
    timed like the call on the same replicas: the gather ceiling of the
    workload.  When no two index lists share a KV head's rows (S1 = 1), the
    same byte count read as rows 0 .. topK - 1 of every list (sequential
    rows) is timed too."""
    import sparse_attention_serving_sfa_gb300 as sfa
    peaks, _ = load_peaks()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.empty(2 * sms * 4 + 64, dtype=torch.uint8, device="cuda")

    def timed(idx_of, tma=False):
        def step(i):
            d = replicas[i % reps]
            if tma:
                sfa.sfa_gather_probe_tma(d["k"], d["v"], idx_of(d), case.B, case.S1, case.S2,
                                         case.N2, case.Dk, case.Dv, case.topK, case.layout,
                                         torch.cuda.current_stream())
            else:
                sfa.sfa_gather_probe(d["k"], d["v"], idx_of(d), case.B, case.S1, case.S2, case.N2,
                                     case.Dk, case.Dv, case.topK, case.layout, sink,
                                     torch.cuda.current_stream())
        for i in range(max(args.warmup, 3)):
            step(i)
        torch.cuda.synchronize()
        ms, _, _ = device_time(step, args.steps, args.eager, world)
        gbs = counts["gathered_bytes"] / (ms * 1e-3) / 1e9
        return {"ms_per_step": ms, "gbs": gbs, "frac_of_copy_peak": gbs / peaks["hbm_gbs"]}

    out = {"what": "sfa_gather_probe: the same K/V rows read with coalesced 16-byte loads, no "
                   "arithmetic",
           "random_rows": timed(lambda d: d["idx"])}
    # the same rows by TMA row gathers (tile::gather4), one CTA per SM
    out["random_rows_tma_gather4"] = timed(lambda d: d["idx"], tma=True)
    # the kernel's gather rate as a fraction of the probe's (1.0 = the
    # attention kernel is as fast as reading its rows alone)
    out["kernel_frac_of_probe_rate"] = out["random_rows"]["ms_per_step"] / kernel_ms
    if case.S1 == 1:
        seq = torch.arange(case.topK, dtype=torch.int32, device="cuda").expand(
            replicas[0]["idx"].shape).contiguous()
        out["sequential_rows"] = timed(lambda d: seq)
    return out


def sfa_cpu_baseline(case, host, counts, target_s=10.0):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (whole calls while they fit in ~target_s, else sampled rows
    scaled to a whole call)."""
    import oracle
    rows_total = case.B * case.N1 * case.S1
    t0 = time.perf_counter()
    probe = np.array([[0, 0, 0]])
    oracle.sfa_rows(host["q"], host["k"], host["v"], host["idx"], case.scale, probe, case.layout,
                    case.causal)
    per_row = max(time.perf_counter() - t0, 1e-6)
    est_full = per_row * rows_total / max(oracle.threads(), 1)
    if est_full < target_s / 2:
        reps = 0
        t0 = time.perf_counter()
        while True:
            oracle.sfa(host["q"], host["k"], host["v"], host["idx"], case.scale, case.layout,
                       case.causal)
            reps += 1
            if time.perf_counter() - t0 > target_s / 2 or reps >= 20:
                break
        sec = (time.perf_counter() - t0) / reps
        sample = f"{reps} whole calls ({rows_total} output rows each)"
    else:
        n = max(int(target_s / per_row * max(oracle.threads(), 1) / 2), 16)
        n = min(n, rows_total)
        rng = np.random.default_rng(0)
        flat = rng.choice(rows_total, size=n, replace=False)
        rows = np.stack([flat // (case.N1 * case.S1), (flat // case.S1) % case.N1,
                         flat % case.S1], axis=1)
        t0 = time.perf_counter()
        oracle.sfa_rows(host["q"], host["k"], host["v"], host["idx"], case.scale, rows,
                        case.layout, case.causal)
        sec = (time.perf_counter() - t0) * rows_total / n
        sample = f"{n} of {rows_total} output rows, time scaled to a whole call"
    return {"value": counts["gathered_bytes"] / sec / 1e9, "unit": "GB/s",
            "cores": oracle.threads(), "kind": "oracle", "sample": sample,
            "seconds_per_call": sec}


# ---------------------------------------------------------------------------
# block-sparse workloads

def run_bsr(name, args, world, rank, cpu_target_s):
    """Block-sparse workloads (tensor-bound): one step = one bsr_run (or
    varbsr_run) over the whole 16384 x 16384 pattern (plan built once,
    outside the timed region)."""
    import sparse_attention_serving_sfa_gb300 as sfa
    variable = name in synth.VARBSR_WORKLOADS
    if variable:
        case = synth.VARBSR_WORKLOADS[name]
        x = synth.make_varbsr_inputs(case)
        counts = synth.varbsr_counts(case, x["block_mask_map"], x["block_row_sz"],
                                     x["block_col_sz"])
        plan = sfa.varbsr_plan(x["block_mask_map"], x["block_row_sz"], x["block_col_sz"],
                               case.Hq, case.Hkv, case.d, causal=case.causal,
                               sm_scale=case.sm_scale, dtype=case.dtype)
        run = sfa.varbsr_run
        lse_shape = (case.Hq, case.M)
        shape_cfg = {"layout": "HND", "MB": case.MB, "NB": case.NB,
                     "block_sizes": "per kv head, uniform random cut points (mean "
                                    f"{case.M // case.MB} x {case.N // case.NB})",
                     "key_tiles": int(plan.int_ws.cpu().view(torch.int32)[case.Hkv * case.MB])}
    else:
        case = synth.BSR_WORKLOADS[name]
        x = synth.make_bsr_inputs(case)
        counts = synth.bsr_counts(case, x["indptr"], x["indices"], x["mask"])
        plan = sfa.bsr_plan(x["indptr"], x["indices"], case.M, case.N, case.R, case.C, case.Hq,
                            case.Hkv, case.d, sm_scale=case.sm_scale, dtype=case.dtype,
                            causal=case.causal, mask=x["mask"])
        run = sfa.bsr_run
        lse_shape = (case.M, case.Hq)
        shape_cfg = {"layout": "NHD", "R": case.R, "C": case.C, "nnz_blocks": counts["nnz"],
                     "element_mask_keep": case.mask_keep or None}
        if case.fp8:
            # q / k / v in E4M3 with per-head scales, fp16 out
            sfa.bsr_plan_set_data_types(plan, case.fp8, case.fp8, case.dtype)
            scales = [x[n].cuda() for n in ("scale_q", "scale_k", "scale_v")]

            def run(pl, q_, k_, v_, out_, lse_, stream_):
                sfa.bsr_run_scaled(pl, q_, k_, v_, *scales, out=out_, lse=lse_, stream=stream_)
            shape_cfg["fp8"] = {"q_k_v": case.fp8, "out": case.dtype,
                                "scales": "per head, max |x| / 448"}
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    out_dtype = {"f16": torch.float16, "bf16": torch.bfloat16}[case.dtype]
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")

    def call(qq, o=None, l=None):
        run(plan, qq, k, v, out if o is None else o, lse if l is None else l,
            torch.cuda.current_stream())

    for _ in range(max(args.warmup, 3)):
        call(q)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.2)
    ms, launches, mode = device_time(lambda i: call(q), args.steps, args.eager, world)
    clocks = sampler.stop()

    e2e = None
    if not args.no_e2e:
        # K/V resident (the KV cache); q in from pinned host memory, out and
        # lse back, every step
        hq = x["q"].pin_memory()
        hout = torch.empty(hq.shape, dtype=out_dtype).pin_memory()
        hlse = torch.empty(lse_shape, dtype=torch.float32).pin_memory()
        sets = [{"q": torch.empty_like(q), "out": torch.empty_like(out), "lse": torch.empty_like(lse)}
                for _ in range(2)]

        def h2d(i, b):
            sets[b]["q"].copy_(hq, non_blocking=True)

        def compute(i, b):
            call(sets[b]["q"], o=sets[b]["out"], l=sets[b]["lse"])

        def d2h(i, b):
            hout.copy_(sets[b]["out"], non_blocking=True)
            hlse.copy_(sets[b]["lse"], non_blocking=True)

        n_e2e = max(min(args.steps, 20), 5)
        e_ms, e_mode = e2e_time(h2d, compute, d2h, n_e2e, 2, world, args.eager)
        e2e = {"value": whole_job_rate(counts["flops"], e_ms, world) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e_ms, "steps": n_e2e, "schedule": E2E_SCHEDULE, "launch": e_mode,
               "h2d_bytes_per_step": nbytes(hq),
               "d2h_bytes_per_step": nbytes(hout) + nbytes(hlse)}

    peaks, peak_src = load_peaks()
    tflops = counts["flops"] / (ms * 1e-3) / 1e12
    prof = committed_profile(name)
    fp8 = getattr(case, "fp8", "")
    # a contraction's own dtype: 8-bit MMAs run at twice the 16-bit rate
    # (nominal 4.5 vs 2.25 PFLOP/s dense)
    peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    peak_src_txt = (f"{peak_src} bf16_tflops x 2 (nominal fp8 / bf16 dense ratio 4.5 / 2.25); "
                    "burst: the kernel is timed alone" if fp8 else
                    f"{peak_src} bf16_tflops (burst: the kernel is timed alone; the fp16 dense "
                    "rate is the bf16 rate)")
    cfg = {"workload": case.name, "M": case.M, "N": case.N, **shape_cfg, "Hq": case.Hq,
           "Hkv": case.Hkv, "d": case.d, "p": case.p, "causal": case.causal,
           "l2": "q, out (268 MiB) stream through; K/V (67 MiB) L2-resident by design",
           "launch": mode,
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    rec = {"workload": name, "value": whole_job_rate(counts["flops"], ms, world) / 1e12,
           "unit": "TFLOP/s", "ms_per_step": ms, "us_per_call": ms * 1e3,
           "dtype": fp8 or case.dtype, "config": cfg, "tflops": world * tflops,
           "tensor_frac": tflops / peak,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak,
                        "unit": "TFLOP/s", "frac": tflops / peak,
                        "traffic": None if prof is None else prof["dram"],
                        "peak_source": peak_src_txt,
                        "algorithmic": "useful FLOPs (4 * d per allowed row, column, qo head)",
                        "kernel": MAIN_KERNEL[name] + "; CUDA events on its stream"},
           "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
           "work": {"flops": counts["flops"], "allowed_elements": counts["allowed"]}}
    if rank == 0 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = bsr_cpu_baseline(case, x, counts, variable, cpu_target_s)
    del q, k, v, out, lse, plan
    torch.cuda.empty_cache()
    return rec


def bsr_cpu_baseline(case, x, counts, variable, target_s):
    """The oracle on sampled query rows (all heads of each row), time scaled
    to the whole pattern."""
    import oracle
    rng = np.random.default_rng(0)

    def run_rows(qrows):
        # every qo head of each query row
        heads = np.arange(case.Hq, dtype=np.int64)
        if variable:
            flat = (heads[None, :] * case.M + qrows[:, None]).reshape(-1)
            oracle.varbsr_rows(x["q"], x["k"], x["v"], x["block_mask_map"], x["block_row_sz"],
                               x["block_col_sz"], case.sm_scale, flat, causal=case.causal)
        else:
            pairs = np.stack([np.repeat(qrows, case.Hq), np.tile(heads, len(qrows))], axis=1)
            if getattr(case, "fp8", ""):
                oracle.bsr_scaled(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M,
                                  case.N, case.R, case.C, case.sm_scale,
                                  scale_q=x["scale_q"].numpy(), scale_k=x["scale_k"].numpy(),
                                  scale_v=x["scale_v"].numpy(), rows=pairs, causal=case.causal)
            else:
                oracle.bsr_rows(x["q"], x["k"], x["v"], x["indptr"], x["indices"], case.M,
                                case.N, case.R, case.C, case.sm_scale, pairs, mask=x["mask"],
                                causal=case.causal)

    t0 = time.perf_counter()
    run_rows(np.array([case.M // 2], dtype=np.int64))
    per_row = max(time.perf_counter() - t0, 1e-6)
    n = int(min(max(target_s / per_row * max(oracle.threads(), 1) / 2, 16), case.M))
    rows = np.sort(rng.choice(case.M, size=n, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    run_rows(rows)
    sec = (time.perf_counter() - t0) * case.M / n
    return {"value": counts["flops"] / sec / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "kind": "oracle", "sample": f"{n} of {case.M} query rows (all heads), time scaled "
                                        "to the whole pattern", "seconds_per_call": sec}


def run_workload(name, args, world, rank, cpu_target_s):
    if name in synth.SFA_WORKLOADS:
        return run_sfa(name, args, world, rank, cpu_target_s)
    return run_bsr(name, args, world, rank, cpu_target_s)


def run_ours(args, rank, world, local):
    import sparse_attention_serving_sfa_gb300 as sfa
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    sfa.build()
    sfa.load()
    # one non-default stream for every call, copy and event (a CUDA graph
    # cannot be captured on the legacy default stream)
    torch.cuda.set_stream(torch.cuda.Stream())
    head = run_workload(args.workload, args, world, rank, cpu_target_s=12.0)
    subs = {}
    for name in sub_workloads(args):
        subs[name] = run_workload(name, args, world, rank, cpu_target_s=4.0)
    res = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": head["dtype"], "data": "synthetic (seeded generator, shapes of the workload)",
           "config": head["config"]}
    for key in ("us_per_call", "gathered_gbs", "tflops", "tensor_frac", "roofline_time_frac",
                "roofline", "e2e", "gpu_launches", "cpu_baseline", "gather_probe",
                "with_inputs_ready", "work"):
        if key in head:
            res[key] = head[key]
    res["gpu_launches"] = head["gpu_launches"]
    res["clocks"] = merge_clocks([head.get("clocks")] + [r.get("clocks") for r in subs.values()])
    if subs:
        for r in subs.values():
            r.pop("clocks", None)
        res["workloads"] = subs
    if world > 1:
        torch.distributed.destroy_process_group()
    return res


def run_reference(args, rank, world):
    """The CPU oracle as it stands on the headline workload's config: each
    step is one bounded sample of the workload."""
    import oracle
    oracle.build()
    name = args.workload
    if name in synth.SFA_WORKLOADS:
        case = synth.SFA_WORKLOADS[name]
        host = synth.make_sfa_inputs(case)
        counts = synth.sfa_counts(case, host["idx"])

        def sample(t):
            return sfa_cpu_baseline(case, host, counts, target_s=t)
        unit, units, cfg = "GB/s", counts["gathered_bytes"] / 1e9, sfa_config(case, world)
    else:
        variable = name in synth.VARBSR_WORKLOADS
        case = (synth.VARBSR_WORKLOADS if variable else synth.BSR_WORKLOADS)[name]
        x = synth.make_varbsr_inputs(case) if variable else synth.make_bsr_inputs(case)
        counts = (synth.varbsr_counts(case, x["block_mask_map"], x["block_row_sz"],
                                      x["block_col_sz"]) if variable
                  else synth.bsr_counts(case, x["indptr"], x["indices"], x["mask"]))

        def sample(t):
            return bsr_cpu_baseline(case, x, counts, variable, t)
        unit, units, cfg = "TFLOP/s", counts["flops"] / 1e12, {"workload": name}
    cb = sample(4.0)
    for _ in range(max(args.warmup, 0)):
        sample(1.0)
    n_steps = max(min(args.steps, 5), 1)
    secs = [sample(3.0)["seconds_per_call"] for _ in range(n_steps)]
    sec = float(np.mean(secs))
    val = units / sec
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": world,
            "steps": n_steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator, shapes of the workload)",
            "config": cfg,
            "cpu_baseline": {"value": val, "unit": unit, "cores": oracle.threads(),
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def reference_runs_on(rank):
    """The reference arm (the CPU oracle) runs on rank 0 only; other ranks
    exit without work."""
    return rank == 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if not reference_runs_on(rank):
            return 0
        print(json.dumps(run_reference(args, rank, world)))
        return 0
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res))
    return 0


if __name__ == "__main__":
    sys.exit(main())
