"""Benchmark of the sparse-attention hot path on GB300.

One step = one call of the top-K sparse flash attention entry point over the
GQA-decode workload (B=16, S1=1, S2=8192, N1=32, N2=8, Dk=Dv=128, topK=1024,
bf16, BNSD, causal), inputs resident in HBM.  Steps run back to back over
rotating replicas of the inputs whose gathered bytes exceed L2 several times,
so every step gathers from HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload.  Under torchrun every rank runs an
independent replica of the workload (weak scaling, no collective on the data
path); timing is the max over ranks.
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
UNIT = "GB/s"   # gathered-KV bytes per second (the decode workload is HBM-bound)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_decode",
                    choices=sorted(synth.SFA_WORKLOADS) + sorted(synth.BSR_WORKLOADS)
                    + sorted(synth.VARBSR_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--replicas", type=int, default=0,
                    help="input replicas rotated over the steps (0 = enough to exceed L2 4x; "
                         "1 keeps a profiling capture small)")
    return ap.parse_args()


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


def dtype_name(case):
    return {"f16": "f16", "bf16": "bf16"}[case.dtype]


def config_of(case, world):
    return {"workload": case.name, "B": case.B, "S1": case.S1, "S2": case.S2, "N1": case.N1,
            "N2": case.N2, "Dk": case.Dk, "Dv": case.Dv, "topK": case.topK,
            "layout": case.layout, "causal": case.causal,
            "value_is_key_prefix": case.value_is_key_prefix, "index": case.index_kind,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


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


# ---------------------------------------------------------------------------
# traffic figure from a committed ncu summary (only while the kernel source
# it was taken on is unchanged)

def kernel_source_sha(files):
    """sha256 over the named kernel sources (file name + bytes, in order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_serving_sfa_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def committed_traffic(workload):
    """DRAM bytes per launch of the workload's main kernel from its committed
    ncu summary (profiles/<workload>_ncu.md), or None when the summary is
    missing or its kernel sources have changed since it was taken."""
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
    return float(val.group(1))


# main kernel of each top-K workload (what the roofline object describes)
MAIN_KERNEL = {
    "tiny": "generic top-K kernel",
    "gqa_decode": "sfa_decode_kernel (one launch per sfa_run_ex call; split index lists merged in-kernel)",
    "sparse_prefill": "sfa_decode_kernel (one launch per sfa_run_ex call; split index lists merged in-kernel)",
    "mla_decode": "sfa_mla_kernel + sfa_mla_combine (two launches per sfa_run_ex call; time is the call's)",
    "mla_mtp": "sfa_mla_kernel + sfa_mla_combine (two launches per sfa_run_ex call; time is the call's)",
    "call_example": "sfa_decode_kernel (one launch per sfa_run_ex call; whole index lists per CTA)",
}


# ---------------------------------------------------------------------------

def run_bsr(args, rank, world, local):
    """Block-sparse workloads (tensor-bound): one step = one bsr_run (or
    varbsr_run) over the whole 16384 x 16384 pattern (plan built once, outside
    the timed region)."""
    import sparse_attention_serving_sfa_gb300 as sfa

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    sfa.build()
    sfa.load()
    variable = args.workload in synth.VARBSR_WORKLOADS
    if variable:
        case = synth.VARBSR_WORKLOADS[args.workload]
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
        kernel = "bsr_tc_wide_kernel, variable mode (one launch per varbsr_run)"
    else:
        case = synth.BSR_WORKLOADS[args.workload]
        x = synth.make_bsr_inputs(case)
        counts = synth.bsr_counts(case, x["indptr"], x["indices"], x["mask"])
        plan = sfa.bsr_plan(x["indptr"], x["indices"], case.M, case.N, case.R, case.C, case.Hq,
                            case.Hkv, case.d, sm_scale=case.sm_scale, dtype=case.dtype,
                            causal=case.causal, mask=x["mask"])
        run = sfa.bsr_run
        lse_shape = (case.M, case.Hq)
        shape_cfg = {"layout": "NHD", "R": case.R, "C": case.C, "nnz_blocks": counts["nnz"],
                     "element_mask_keep": case.mask_keep or None}
        kernel = ("bsr_tc_kernel, per-element mask (one launch per bsr_run)" if case.mask_keep > 0
                  else "bsr_tc_wide_kernel (one launch per bsr_run)")
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    out = torch.empty_like(q)
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        run(plan, q, k, v, out, lse, stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = sfa.sfa_kernel_launches()
    ev0.record(stream)
    for _ in range(args.steps):
        run(plan, q, k, v, out, lse, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = sfa.sfa_kernel_launches() - launches0
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, "cuda")
    peaks, peak_src = load_peaks()
    tflops = counts["flops"] / (ms * 1e-3) / 1e12
    res = {"metric": METRIC, "value": whole_job_rate(counts["flops"], ms, world) / 1e12,
           "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": case.dtype, "data": "synthetic (seeded generator, shapes of the workload)",
           "config": {"workload": case.name, "M": case.M, "N": case.N, **shape_cfg,
                      "Hq": case.Hq, "Hkv": case.Hkv, "d": case.d, "p": case.p,
                      "causal": case.causal,
                      "l2": "q, out (268 MiB) stream through; K/V (67 MiB) L2-resident by design",
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
           "roofline": {"bound": "tensor", "achieved": tflops,
                        "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                        "frac": tflops / peaks["bf16_tflops_sustained"],
                        "traffic": committed_traffic(case.name),
                        "peak_source": f"{peak_src} bf16_tflops_sustained (fp16 dense rate is the same)",
                        "kernel": kernel},
           "gpu_launches": launches, "clocks": clocks,
           "work": {"flops": counts["flops"], "allowed_elements": counts["allowed"]}}
    if world > 1:
        torch.distributed.destroy_process_group()
    return res


def run_ours(args, rank, world, local):
    import sparse_attention_serving_sfa_gb300 as sfa

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    sfa.build()
    sfa.load()
    case = synth.SFA_WORKLOADS[args.workload]
    host = synth.make_sfa_inputs(case)
    counts = synth.sfa_counts(case, host["idx"])
    prefix = case.value_is_key_prefix
    # Rotating replicas of the inputs: consecutive steps read different
    # copies, and the replicas' gathered bytes together exceed L2 several
    # times, so every step gathers from HBM (no flush needed between steps).
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    reps = args.replicas if args.replicas > 0 else max(2, -(-4 * l2 // counts["gathered_bytes"]) + 1)
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
    stream = torch.cuda.current_stream()
    ws_bytes = sfa.sfa_workspace_size(case.B, case.S1, case.N1, case.N2, case.Dk, case.Dv,
                                      case.topK)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

    def step(d, q=None, idx=None):
        sfa.sfa_run_ex(d["q"] if q is None else q, d["k"], d["v"], d["idx"] if idx is None else idx,
                       case.B, case.S1, case.S2, case.N1, case.N2, case.Dk, case.Dv, case.topK,
                       case.scale, case.layout, case.causal, case.dtype, out, lse, stream,
                       workspace=ws, value_is_key_prefix=prefix)

    for i in range(max(args.warmup, 3) + reps):
        step(replicas[i % reps])
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = sfa.sfa_kernel_launches()
    wall0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.steps):
        step(replicas[i % reps])
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = sfa.sfa_kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, "cuda")

    # end to end through the same entry point with host buffers: every step
    # copies its q and indices from pinned host memory and reads the output
    # and lse back (the KV cache stays resident, as it does in serving)
    e2e = None
    if not args.no_e2e:
        hq = host["q"].pin_memory()
        hidx = host["idx"].pin_memory()
        hout = torch.empty(out_shape, dtype=tdt).pin_memory()
        hlse = torch.empty(lse_shape, dtype=torch.float32).pin_memory()
        dq = torch.empty_like(replicas[0]["q"])
        didx = torch.empty_like(replicas[0]["idx"])
        n_e2e = max(args.steps // 4, 20)

        def e2e_step(i):
            dq.copy_(hq, non_blocking=True)
            didx.copy_(hidx, non_blocking=True)
            step(replicas[i % reps], q=dq, idx=didx)
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        for i in range(reps):
            e2e_step(i)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(ev0.elapsed_time(ev1) / n_e2e, world, "cuda")
        h2d = hq.numel() * hq.element_size() + hidx.numel() * 4
        d2h = hout.numel() * hout.element_size() + hlse.numel() * 4
        e2e = {"value": whole_job_rate(counts["gathered_bytes"], e_ms, world) / 1e9, "unit": UNIT,
               "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks, peak_src = load_peaks()
    gbs = counts["gathered_bytes"] / (ms * 1e-3) / 1e9
    tflops = counts["flops"] / (ms * 1e-3) / 1e12
    roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": committed_traffic(args.workload),
                "peak_source": f"{peak_src} hbm_gbs (copy, read+write bytes)",
                "kernel": MAIN_KERNEL.get(args.workload, "sfa_run_ex call") + "; CUDA events on its stream"}
    t_roof = max(counts["gathered_bytes"] / (peaks["hbm_gbs"] * 1e9),
                 counts["flops"] / (peaks["bf16_tflops"] * 1e12))
    cfg = config_of(case, world)
    rot = reps * counts["gathered_bytes"]
    cfg["l2"] = (f"not flushed: {reps} rotating input replicas, {rot >> 20} MiB gathered per "
                 f"rotation {'>' if rot > l2 else '<='} L2 {l2 >> 20} MiB"
                 + ("" if rot > l2 else " (profiling run: not a valid timing)"))
    res = {"metric": METRIC, "value": whole_job_rate(counts["gathered_bytes"], ms, world) / 1e9,
           "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": dtype_name(case), "data": "synthetic (seeded generator, shapes of the workload)",
           "config": cfg,
           "tflops": world * tflops, "us_per_call": ms * 1e3,
           "tensor_frac": tflops / peaks["bf16_tflops"],
           "roofline_time_frac": t_roof / (ms * 1e-3),
           "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
           "clocks": clocks, "wall_s_timed_loop": wall,
           "work": {"flops": counts["flops"], "gathered_bytes": counts["gathered_bytes"],
                    "unmasked_slots": counts["unmasked_slots"]}}
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(case, host, counts)
    if world > 1:
        torch.distributed.destroy_process_group()
    return res


def cpu_baseline(case, host, counts, target_s=10.0):
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
    return {"value": counts["gathered_bytes"] / sec / 1e9, "unit": UNIT,
            "cores": oracle.threads(), "kind": "oracle", "sample": sample,
            "seconds_per_call": sec}


def run_reference(args, rank, world):
    import oracle
    case = synth.SFA_WORKLOADS[args.workload]
    host = synth.make_sfa_inputs(case)
    counts = synth.sfa_counts(case, host["idx"])
    oracle.build()
    cb = cpu_baseline(case, host, counts, target_s=4.0)
    # steps: each step is one bounded sample of the workload
    secs = []
    for _ in range(max(args.warmup, 0)):
        cpu_baseline(case, host, counts, target_s=1.0)
    n_steps = min(args.steps, 5)
    for _ in range(n_steps):
        secs.append(cpu_baseline(case, host, counts, target_s=2.0)["seconds_per_call"])
    sec = float(np.mean(secs))
    val = counts["gathered_bytes"] / sec / 1e9
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": n_steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded generator, shapes of the workload)",
            "config": config_of(case, world),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.threads(),
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
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
    if args.workload in synth.BSR_WORKLOADS or args.workload in synth.VARBSR_WORKLOADS:
        res = run_bsr(args, rank, world, local)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res))
    return 0


if __name__ == "__main__":
    sys.exit(main())
