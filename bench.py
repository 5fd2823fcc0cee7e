"""Benchmark of the NVFP4 block-scaled grouped GEMM on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--sf-path fused]
                    [--impl ours|reference] [--all-configs]

One step = one nvfp4_ggemm_run call over the whole grouped problem (scale
permutation, tile scheduling, loads, block-scaled MMAs, fp16 epilogue), with
inputs resident in HBM. Every timed call starts with its inputs out of L2:
by default the bench cycles through copies of the inputs that together hold
at least three times the L2 (`--l2 rotate`); `--l2 flush` writes a 256 MB
buffer before every call instead. Both are timed and reported; each call is
timed with CUDA events on its stream.
Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on
the host cores instead (bounded samples of the same workload).

N > 1 (torchrun): every rank runs its own replica of the workload (the
operation needs no exchange); the reported time is the maximum over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_fp4_grouped_gb300 import synth  # noqa: E402

METRIC = "µs/call, FP4 TFLOPS and GB/s as fraction of roofline, NVFP4 grouped GEMM"
UNIT = "µs/call"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_PER_BF16 = 13.5 / 2.25  # nominal dense ratio
# Nominal GB300 figures (HBM3e ~8 TB/s, dense FP4 13.5 PFLOP/s): a second
# roofline fraction beside the one against the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_FP4_TFLOPS = 13500.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["block_scaled_fp4_grouped_gb300/csrc/ggemm_kernels.cu",
                  "block_scaled_fp4_grouped_gb300/csrc/ptx.cuh",
                  "block_scaled_fp4_grouped_gb300/csrc/ggemm_internal.h"]


def code_tokens(text: str) -> str:
    """C/C++ source with comments removed and whitespace collapsed, so that a
    comment edit does not change the hash of the code the counters were
    taken on (string literals in these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def traffic_for(config: str, sf_path: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{config}/{sf_path}")
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129 << 20
ROTATE_FACTOR = 3       # rotated input sets hold at least 3x the L2
ROTATE_MAX_SETS = 64
SLEEP_CYCLES = 200_000  # ~100 us at 2 GHz: longer than the host's enqueue of one call


def time_config(name: str, sf_path: str, steps: int, warmup: int, seed: int = 0, torch=None, flush=None,
                want_e2e: bool = False, tuning=None, l2: str = "rotate"):
    """Device timing of one config. Returns a dict of measurements.

    Two ways to start every timed call with its inputs out of L2:
    "rotate" keeps R copies of the inputs and outputs (R * their size >= 3x
    the L2, each copy with its own plan, so no table upload happens inside
    the timed region) and cycles through them, so a call's inputs were last
    read R - 1 calls ago with at least twice the L2 of other data read since;
    "flush" writes a 256 MB buffer before every call, which leaves L2 full of
    dirty lines that the call's reads must first write back. Both are
    timed; `l2` picks the one reported as the headline (problems too small
    for R <= 64 copies to cover 3x the L2 always use "flush")."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    prob = synth.make_problem(name, seed=seed)
    K, N = prob.K, prob.N
    kw = dict(sf_layout="raw", sf_path="fused")
    if sf_path == "relayout":
        kw = dict(sf_layout="raw", sf_path="relayout")
    elif sf_path == "relayout-cached":
        kw = dict(sf_layout="raw", sf_path="relayout", cache_b_scales=True)
    elif sf_path == "atom":
        kw = dict(sf_layout="atom", sf_path="fused")
    kw.update(tuning or {})
    set_bytes = synth.algorithmic_bytes(prob.M, N, K)
    n_sets = -(-ROTATE_FACTOR * L2_BYTES // set_bytes)
    rotate_ok = n_sets <= ROTATE_MAX_SETS
    if not rotate_ok:
        l2 = "flush"
    n_sets = max(2, n_sets) if rotate_ok else 1

    def make_set():
        dev = lambda arrs: [torch.from_numpy(a).cuda() for a in arrs]
        A, B, SFA, SFB = dev(prob.A), dev(prob.B), dev(prob.SFA), dev(prob.SFB)
        if sf_path == "atom":
            SFA = [_atom(torch, nb, s, m, K) for s, m in zip(SFA, prob.M)]
            SFB = [_atom(torch, nb, s, N, K) for s in SFB]
        C = [torch.empty((m, N), dtype=torch.float16, device="cuda") for m in prob.M]
        gg = nb.GroupedGemm(prob.M, N, K, **kw)
        if kw.get("cache_b_scales"):
            gg.prepare_b_scales(SFB)
            SFB_run = [None] * len(SFB)
        else:
            SFB_run = SFB
        return gg, gg.bind(A, B, SFA, SFB_run, C)

    sets = [make_set() for _ in range(n_sets)]
    info = sets[0][0].info()
    stream = torch.cuda.current_stream()

    def check():
        for gg, _ in sets:
            st, detail = gg.sync_status()
            if st != nb.NVFP4_OK:
                raise RuntimeError(f"{name}: device status {nb.nvfp4_status_string(st)} ({detail:#x})")

    def before_call(mode):
        # Something for the GPU to do while the host enqueues the call, so
        # that the start event is not followed by host launch latency: the
        # flush itself, or (rotation) a short device-side sleep that touches
        # no memory.
        if mode == "flush":
            flush.zero_()
        else:
            torch.cuda._sleep(SLEEP_CYCLES)

    def timed(mode):
        # warm-up: every set at least once (uploads its table), then W calls
        for i in range(max(warmup, len(sets) if mode == "rotate" else 1)):
            _, call = sets[i % len(sets)] if mode == "rotate" else sets[0]
            before_call(mode)
            call()
        check()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            _, call = sets[i % len(sets)] if mode == "rotate" else sets[0]
            before_call(mode)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        check()
        return [a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends)], wall

    modes = {m: timed(m) for m in (["rotate", "flush"] if rotate_ok else ["flush"])}
    us, wall = modes[l2]
    out = {
        "prob": prob, "info": info, "us": us, "wall_s": wall, "l2": l2, "n_sets": n_sets,
        "us_mean": statistics.fmean(us), "us_median": statistics.median(us),
        "us_min": min(us), "us_p90": sorted(us)[int(0.9 * (len(us) - 1))],
        "by_l2": {m: {"us_mean": statistics.fmean(v[0]), "us_median": statistics.median(v[0]),
                      "us_min": min(v[0])} for m, v in modes.items()},
        "bytes": set_bytes, "flops": synth.algorithmic_flops(prob.M, N, K),
        "launches_per_call": info.kernels_per_run,
    }
    if want_e2e:
        out["e2e"] = time_e2e(prob, kw, steps, warmup, torch, nb)
    for gg, _ in sets:
        gg.close()
    return out


def l2_text(r):
    if r["l2"] == "rotate":
        return (f"inputs larger than L2: {r['n_sets']} copies of the inputs and outputs "
                f"({r['n_sets']} x {r['bytes'] / 1e6:.1f} MB), cycled call by call, no flush write")
    return "flushed before every timed call (256 MB write)"


def _atom(torch, nb, sf, rows, K):
    out = torch.zeros(nb.nvfp4_sf_atom_bytes(rows, K), dtype=torch.uint8, device="cuda")
    assert nb.nvfp4_sf_relayout(sf, out, rows, K) == nb.NVFP4_OK
    return out


def time_e2e(prob, kw, steps, warmup, torch, nb):
    """Same metric through nvfp4_ggemm_run_host: pinned host inputs copied in,
    C copied back, every step."""
    kw = {k: v for k, v in kw.items() if k != "cache_b_scales"}
    if kw.get("sf_layout") == "atom":
        kw = dict(sf_layout="raw", sf_path="fused")
    pin = lambda arrs: [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in arrs]
    A, B, SFA, SFB = pin(prob.A), pin(prob.B), pin(prob.SFA), pin(prob.SFB)
    C = [torch.empty((m, prob.N), dtype=torch.float16).pin_memory() for m in prob.M]
    h2d = sum(t.numel() * t.element_size() for t in A + B + SFA + SFB)
    d2h = sum(t.numel() * t.element_size() for t in C)
    n = max(3, min(steps, 50))
    with nb.GroupedGemm(prob.M, prob.N, prob.K, **kw) as gg:
        call = gg.bind_host(A, B, SFA, SFB, C)
        for _ in range(max(1, min(warmup, 3))):
            call()
        times = []
        for _ in range(n):
            t0 = time.perf_counter()
            call()
            times.append((time.perf_counter() - t0) * 1e6)
    return {"value": statistics.fmean(times), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "median": statistics.median(times)}


def oracle_sample_time(prob, budget_s: float):
    """Time the oracle (as it stands) on a bounded sample of `prob`: whole
    groups while they fit the budget, else a row subset of the largest
    group. Returns (µs per full call extrapolated by flops, threads, sample
    text)."""
    import oracle as oracle_pkg
    O = oracle_pkg.get()
    threads = os.cpu_count() or 1
    total_flops = synth.algorithmic_flops(prob.M, prob.N, prob.K)
    g0 = int(np.argmax(prob.M))
    # size the sample from 4 rows per thread of the largest group (after a warm-up call)
    probe = max(1, min(prob.M[g0], 4 * threads))
    O.group_gemm(prob.A[g0][:4], prob.B[g0], prob.SFA[g0][:4], prob.SFB[g0], prob.K, nthreads=threads)
    t0 = time.perf_counter()
    O.group_gemm(prob.A[g0][:probe], prob.B[g0], prob.SFA[g0][:probe], prob.SFB[g0], prob.K, nthreads=threads)
    per_row = max((time.perf_counter() - t0) / probe, 1e-7)
    groups, est = [], 0.0
    for g, m in enumerate(prob.M):
        if m > 0 and est + m * per_row <= budget_s:
            groups.append(g)
            est += m * per_row
    if groups:
        t0 = time.perf_counter()
        for g in groups:
            O.group_gemm(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K, nthreads=threads)
        dt = time.perf_counter() - t0
        rows = sum(prob.M[g] for g in groups)
        sample_flops = 2 * rows * prob.N * prob.K
        what = (f"{len(groups)} of {sum(1 for m in prob.M if m > 0)} groups ({rows} of {sum(prob.M)} rows) "
                f"x N={prob.N} x K={prob.K} ({dt:.2f} s)")
    else:
        take = int(max(8, min(prob.M[g0], budget_s / per_row)))
        t0 = time.perf_counter()
        O.group_gemm(prob.A[g0][:take], prob.B[g0], prob.SFA[g0][:take], prob.SFB[g0], prob.K, nthreads=threads)
        dt = time.perf_counter() - t0
        sample_flops = 2 * take * prob.N * prob.K
        what = f"group {g0}: {take} of {prob.M[g0]} rows x N={prob.N} x K={prob.K} ({dt:.2f} s)"
    us_full = dt * 1e6 * total_flops / sample_flops
    if sample_flops < total_flops:
        what += ", scaled by flops"
    return us_full, threads, what


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    prob = synth.make_problem(args.config, seed=0)
    per_step = []
    cores = os.cpu_count() or 1
    sample = ""
    budget = max(0.5, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        us, cores, sample = oracle_sample_time(prob, budget)
        if i >= args.warmup:
            per_step.append(us)
    value = statistics.fmean(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.config, prob),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(name, prob):
    spec = synth.CONFIGS.get(name)
    desc = name
    if spec is not None:
        if spec.m_fixed:
            mdesc = f"M={list(spec.m_fixed)}"
        else:
            mdesc = f"M_g multiples of {spec.m_step} in [{spec.m_lo},{spec.m_hi}]"
        desc = f"{name}: g={spec.G} N={spec.N} K={spec.K} {mdesc}, seed 0"
    return {"workload": desc, "M": list(prob.M), "N": prob.N, "K": prob.K,
            "values": "E2M1 codes uniform over 16; E4M3 scales 2^e(1+u), e in [-4,2]",
            "scales": "raw row-major [rows, K/16] E4M3 per call"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c4")
    ap.add_argument("--sf-path", default="fused", choices=["fused", "relayout", "relayout-cached", "atom"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--all-configs", action="store_true", help="also time every config (extra key)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--tile-n", type=int, default=0, help="widest output tile (0 = library default)")
    ap.add_argument("--b-stages", type=int, default=0)
    ap.add_argument("--a-stages", type=int, default=0)
    ap.add_argument("--l2", default="rotate", choices=["rotate", "flush"],
                    help="how every timed call starts with its inputs out of L2 (both are timed)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        # no collective on this arm: rank 0 times the oracle, the others exit
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()

    import torch
    from block_scaled_fp4_grouped_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    barrier(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    hbm, bf16, peak_src = measured_peaks()
    fp4_peak_tflops = bf16 * FP4_PER_BF16

    barrier(world)
    with ClockSampler(local) as clocks:
        tuning = dict(tile_n=args.tile_n, b_stages=args.b_stages, a_stages=args.a_stages)
        r = time_config(args.config, args.sf_path, args.steps, args.warmup, torch=torch, flush=flush,
                        want_e2e=not args.no_e2e, tuning=tuning, l2=args.l2)
    barrier(world)
    us = max_over_ranks(world, r["us_mean"], device)
    prob = r["prob"]
    bytes_, flops = r["bytes"], r["flops"]
    achieved_gbs = bytes_ / (r["us_mean"] * 1e-6) / 1e9
    tflops = flops / (r["us_mean"] * 1e-6) / 1e12
    t_roof_us = max(flops / (fp4_peak_tflops * 1e12), bytes_ / (hbm * 1e9)) * 1e6
    t_roof_nominal_us = max(flops / (NOMINAL_FP4_TFLOPS * 1e12), bytes_ / (NOMINAL_HBM_GBS * 1e9)) * 1e6
    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": dict(workload_config(args.config, prob), sf_path=args.sf_path,
                       l2=l2_text(r),
                       max_tile_n=r["info"].tile_n, grid=r["info"].grid, chunks=r["info"].chunks,
                       b_stages=r["info"].b_stages, a_stages=r["info"].a_stages,
                       parallelism=f"replicas x{world}"),
        "us_median": r["us_median"], "us_min": r["us_min"], "us_p90": r["us_p90"],
        "us_by_l2_protocol": {m: {k: round(v, 2) for k, v in d.items()} for m, d in r["by_l2"].items()},
        "tflops_fp4": tflops, "gbs": achieved_gbs,
        "roofline_fraction": t_roof_us / r["us_mean"],
        "roofline_time_us": t_roof_us,
        "roofline_fraction_nominal": t_roof_nominal_us / r["us_mean"],
        "roofline_time_us_nominal": t_roof_nominal_us,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm, "traffic": traffic_for(args.config, args.sf_path),
                     "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": bytes_,
                     "kernel": "ggemm_kernel" if args.sf_path != "relayout" else "ggemm_kernel + sf_relayout_kernel"},
        "gpu_launches": r["launches_per_call"] * args.steps,
        "clocks": clocks.summary(),
        "timed_wall_s": r["wall_s"],
    }
    if "e2e" in r:
        e2e = r["e2e"]
        line["e2e"] = {"value": e2e["value"], "unit": UNIT, "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                       "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}
    if args.all_configs and rank == 0:
        per = {}
        for name in ["c0", "c1", "c2", "c3", "c4", "c1_page", "c2_page", "c3_page", "c4_page"]:
            for path in ["fused", "relayout", "relayout-cached"]:
                q = time_config(name, path, max(20, args.steps // 2), args.warmup, torch=torch, flush=flush,
                                tuning=tuning if path == args.sf_path else None, l2=args.l2)
                t_roof = max(q["flops"] / (fp4_peak_tflops * 1e12), q["bytes"] / (hbm * 1e9)) * 1e6
                t_nom = max(q["flops"] / (NOMINAL_FP4_TFLOPS * 1e12), q["bytes"] / (NOMINAL_HBM_GBS * 1e9)) * 1e6
                per[f"{name}/{path}"] = {"us_mean": round(q["us_mean"], 2), "us_median": round(q["us_median"], 2),
                                         "us_min": round(q["us_min"], 2),
                                         "gbs": round(q["bytes"] / (q["us_mean"] * 1e-6) / 1e9, 1),
                                         "tflops": round(q["flops"] / (q["us_mean"] * 1e-6) / 1e12, 1),
                                         "roofline_fraction": round(t_roof / q["us_mean"], 3),
                                         "roofline_fraction_nominal": round(t_nom / q["us_mean"], 3),
                                         "chunks": q["info"].chunks, "grid": q["info"].grid, "l2": q["l2"],
                                         "us_mean_flush": round(q["by_l2"]["flush"]["us_mean"], 2)}
        line["per_config"] = per
    if rank == 0 and not args.no_cpu_baseline:
        us_cpu, cores, sample = oracle_sample_time(prob, budget_s=10.0)
        line["cpu_baseline"] = {"value": us_cpu, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
