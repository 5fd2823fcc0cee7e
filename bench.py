"""Benchmark of the NVFP4 block-scaled grouped GEMM on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--sf-path fused]
                    [--impl ours|reference] [--all-configs] [--serial-launch]

One step = one nvfp4_ggemm_run call over the whole grouped problem (scale
permutation, tile scheduling, loads, block-scaled MMAs, fp16 epilogue), with
inputs resident in HBM. The headline times K steps back to back between one
pair of CUDA events on the launching stream, the calls using in turn copies
of the inputs that together hold at least three times the L2 (so every call
starts with its inputs out of L2); a device-side sleep ahead of the start
event covers the host's enqueue. Also reported, labelled: one call between
its own events (isolated), one call after a 256 MB flush write, back-to-back
calls on one copy (warm L2), the host's cost per call, the same call on host
buffers (e2e), every config c0-c4, and the CPU oracle's time.
Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on
the host cores instead (the whole problem every step).

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
SM_GHZ_FOR_SLEEP = 2.2  # cycles per ns used to size device sleeps (>= the top SM clock)
MAX_STREAM_SLEEP_NS = 400e6


def _flavour(sf_path: str):
    kw = dict(sf_layout="raw", sf_path="fused")
    if sf_path == "relayout":
        kw = dict(sf_layout="raw", sf_path="relayout")
    elif sf_path == "relayout-cached":
        kw = dict(sf_layout="raw", sf_path="relayout", cache_b_scales=True)
    elif sf_path == "fused-cached":
        kw = dict(sf_layout="raw", sf_path="fused", cache_b_scales=True)
    elif sf_path == "atom":
        kw = dict(sf_layout="atom", sf_path="fused")
    return kw


def time_config(name: str, sf_path: str, steps: int, warmup: int, seed: int = 0, torch=None, flush=None,
                want_e2e: bool = False, tuning=None, host_calls: int = 50, prob=None):
    """Device timing of one config. Returns a dict of measurements.

    Every timed call starts with its inputs out of L2 (except the labelled
    warm-L2 protocol): R copies of the inputs and outputs (R * their size >=
    3x the L2, each copy with its own plan, so no table upload happens inside
    a timed region) are used in turn, so a call's inputs were last read R - 1
    calls earlier with at least twice the L2 of other data read since.
    Protocols, all timed with CUDA events on the launching stream:

    * "stream" (the headline): `steps` calls back to back between one pair
      of events, cycling through the copies; a device-side sleep ahead of the
      start event covers the host's enqueue of all of them, so the timed
      region holds GPU work only. Per call = elapsed / steps.
    * "isolated": one call between its own events, a short device sleep
      before each (the host has enqueued the call before its start event
      runs), cycling through the copies.
    * "flush": one call between its own events after a 256 MB write, on one
      copy (it leaves L2 full of dirty lines the call's reads write back).
    * "warm": `steps` calls back to back on one copy, nothing flushed
      (warm L2 as far as the copy fits in it).
    * "stream_b_static": as "stream", with plans that declare B and SFB
      static (the b_static option: no kernel before a call writes them, as
      for model weights), so each call streams B while the previous one
      finishes. Reported beside the headline, not as it.
    * "stream_inputs_static": as "stream", with plans that declare all four
      inputs static (b_static = 2: every load may start while the previous
      call finishes; only the C stores wait for it). Reported beside the
      headline, not as it.
    Problems too small for 64 copies to cover 3x the L2 (c0) run "flush"
    and "warm" only, and report "flush" as the headline.
    Host cost: the enqueue time of one call (the C call from Python, plan
    cached) and the wall time of one call followed by a stream
    synchronisation."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    if prob is None:
        prob = synth.make_problem(name, seed=seed)
    K, N = prob.K, prob.N
    kw = _flavour(sf_path)
    kw.update(tuning or {})
    set_bytes = synth.algorithmic_bytes(prob.M, N, K)
    n_sets = -(-ROTATE_FACTOR * L2_BYTES // set_bytes)
    rotate_ok = n_sets <= ROTATE_MAX_SETS
    n_sets = max(2, n_sets) if rotate_ok else 1

    def make_set():
        dev = lambda arrs: [torch.from_numpy(a).cuda() for a in arrs]
        A, B, SFA, SFB = dev(prob.A), dev(prob.B), dev(prob.SFA), dev(prob.SFB)
        if sf_path == "atom":
            SFA = [_atom(torch, nb, s, m, K) for s, m in zip(SFA, prob.M)]
            SFB = [_atom(torch, nb, s, N, K) for s in SFB]
        C = [torch.empty((m, N), dtype=torch.float16, device="cuda") for m in prob.M]
        gg = nb.GroupedGemm(prob.M, N, K, **kw)
        gs = nb.GroupedGemm(prob.M, N, K, **dict(kw, b_static=1))
        gi = nb.GroupedGemm(prob.M, N, K, **dict(kw, b_static=2))
        if kw.get("cache_b_scales"):
            for plan in (gg, gs, gi):
                plan.prepare_b_scales(SFB)
            SFB_run = [None] * len(SFB)
        else:
            SFB_run = SFB
        return (gg, gg.bind(A, B, SFA, SFB_run, C), gs, gs.bind(A, B, SFA, SFB_run, C),
                gi, gi.bind(A, B, SFA, SFB_run, C))

    sets = [make_set() for _ in range(n_sets)]
    info = sets[0][0].info()
    stream = torch.cuda.current_stream()

    def check():
        for gg, _, gs, _, gi, _ in sets:
            for plan in (gg, gs, gi):
                st, detail = plan.sync_status()
                if st != nb.NVFP4_OK:
                    raise RuntimeError(f"{name}: device status {nb.nvfp4_status_string(st)} ({detail:#x})")

    # warm-up: every copy at least once (uploads its table), then W calls;
    # the enqueue time of a call is taken here too
    enq = []
    for i in range(max(warmup, len(sets))):
        _, call, _, call_s, _, call_i = sets[i % len(sets)]
        torch.cuda._sleep(SLEEP_CYCLES)
        t0 = time.perf_counter()
        call()
        enq.append(time.perf_counter() - t0)
        call_s()
        call_i()
    torch.cuda.synchronize()
    check()
    enqueue_s = statistics.median(enq[len(sets):] or enq)

    def stream_block(order, which=1):
        """Calls sets[order[i]] back to back between one event pair (which: 1
        the default plans, 3 the plans that declare B static, 5 those that
        declare every input static). Returns (µs per call, whether the
        device waited for the host)."""
        sleep_ns = 50e3 + 3.0 * enqueue_s * 1e9 * len(order)
        for _attempt in range(4):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            torch.cuda._sleep(int(min(sleep_ns, MAX_STREAM_SLEEP_NS) * SM_GHZ_FOR_SLEEP))
            start.record(stream)
            for j in order:
                sets[j][which]()
            end.record(stream)
            late = start.query()  # the timed region had begun before the last call was enqueued
            torch.cuda.synchronize()
            if not late or sleep_ns >= MAX_STREAM_SLEEP_NS:
                return start.elapsed_time(end) * 1e3 / len(order), late
            sleep_ns *= 4
        return start.elapsed_time(end) * 1e3 / len(order), late

    def per_call(mode):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            call = sets[i % len(sets)][1] if mode == "isolated" else sets[0][1]
            if mode == "flush":
                flush.zero_()
            else:
                torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends)]

    out = {"prob": prob, "info": info, "n_sets": n_sets, "rotate": rotate_ok,
           "bytes": set_bytes, "flops": synth.algorithmic_flops(prob.M, N, K),
           "launches_per_call": info.kernels_per_run}
    by = {}
    t_wall0 = time.perf_counter()
    if rotate_ok:
        us, late = stream_block([i % len(sets) for i in range(steps)])
        by["stream"] = {"us_mean": us, "host_bound": bool(late)}
        us, late = stream_block([i % len(sets) for i in range(steps)], which=3)
        by["stream_b_static"] = {"us_mean": us, "host_bound": bool(late)}
        us, late = stream_block([i % len(sets) for i in range(steps)], which=5)
        by["stream_inputs_static"] = {"us_mean": us, "host_bound": bool(late)}
        v = per_call("isolated")
        by["isolated"] = {"us_mean": statistics.fmean(v), "us_median": statistics.median(v), "us_min": min(v),
                          "us_p90": sorted(v)[int(0.9 * (len(v) - 1))]}
    v = per_call("flush")
    by["flush"] = {"us_mean": statistics.fmean(v), "us_median": statistics.median(v), "us_min": min(v),
                   "us_p90": sorted(v)[int(0.9 * (len(v) - 1))]}
    us, late = stream_block([0] * steps)
    by["warm"] = {"us_mean": us, "host_bound": bool(late)}
    out["timed_wall_s"] = time.perf_counter() - t_wall0
    check()
    out["headline"] = "stream" if rotate_ok else "flush"
    out["us_mean"] = by[out["headline"]]["us_mean"]
    out["by"] = by
    # host cost per call with the plan cached
    call = sets[0][1]
    torch.cuda.synchronize()
    walls = []
    for _ in range(host_calls):
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        walls.append(time.perf_counter() - t0)
    out["host"] = {"enqueue_us": enqueue_s * 1e6, "call_and_sync_us": statistics.median(walls) * 1e6}
    if want_e2e:
        out["e2e"] = time_e2e(prob, kw, steps, warmup, torch, nb)
    for gg, _, gs, _, gi, _ in sets:
        gg.close()
        gs.close()
        gi.close()
    return out


def l2_text(r):
    if r["rotate"]:
        return (f"inputs larger than L2: {r['n_sets']} copies of the inputs and outputs "
                f"({r['n_sets']} x {r['bytes'] / 1e6:.1f} MB) used in turn, no flush write")
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


def oracle_time(prob, nthreads: int = 0, groups=None):
    """Wall time (s) of the oracle, as it stands, on `prob` (every group, or
    the listed ones) with `nthreads` host threads (0 = all cores). Returns
    (seconds, threads used)."""
    import oracle as oracle_pkg
    O = oracle_pkg.get()
    threads = nthreads or (os.cpu_count() or 1)
    t0 = time.perf_counter()
    for g in (range(prob.G) if groups is None else groups):
        if prob.M[g] > 0:
            O.group_gemm(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K, nthreads=threads)
    return time.perf_counter() - t0, threads


REFERENCE_BUDGET_S = 150.0  # wall time the reference arm's measured steps may take


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only): every timed step is
    the whole problem of the workload; the warm-up steps run its smallest
    group (they only load the oracle and warm the caches). Steps stop early
    when the next one would take the measured steps past REFERENCE_BUDGET_S
    (the line says how many were measured); a step is never a sample."""
    if rank != 0:
        return
    prob = headline_problem(args)
    g_small = int(np.argmin([m if m > 0 else 1 << 30 for m in prob.M]))
    for _ in range(args.warmup):
        oracle_time(prob, groups=[g_small])
    per_step, cores = [], os.cpu_count() or 1
    t_all = time.perf_counter()
    for _ in range(args.steps):
        if per_step and time.perf_counter() - t_all + statistics.fmean(per_step) * 1e-6 > REFERENCE_BUDGET_S:
            break
        sec, cores = oracle_time(prob)
        per_step.append(sec * 1e6)
    wall = time.perf_counter() - t_all
    value = statistics.fmean(per_step)
    measured = len(per_step)
    sample = (f"the whole {args.config} problem every step ({len(prob.M)} groups, {sum(prob.M)} rows x "
              f"N={prob.N} x K={prob.K}), {measured} steps in {wall:.1f} s; warm-up steps: group {g_small} only")
    if measured < args.steps:
        sample += (f"; {measured} of the {args.steps} steps asked were measured, the next would have taken the "
                   f"run past {REFERENCE_BUDGET_S:.0f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.config, prob),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "steps_measured": measured,
        "timed_wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def headline_problem(args):
    """The timed workload: the config's problem, or with --k its M list and N
    at another K (values drawn afresh, seed 0)."""
    prob = synth.make_problem(args.config, seed=0)
    if args.k:
        prob = synth.make_problem("custom", seed=0, M=list(prob.M), N=prob.N, K=args.k)
    return prob


def workload_config(name, prob):
    spec = synth.CONFIGS.get(name)
    desc = name
    if spec is not None:
        if spec.m_fixed:
            mdesc = f"M={list(spec.m_fixed)}"
        else:
            mdesc = f"M_g multiples of {spec.m_step} in [{spec.m_lo},{spec.m_hi}]"
        desc = f"{name}: g={spec.G} N={spec.N} K={spec.K} {mdesc}, seed 0"
        if prob.K != spec.K:
            desc = f"{name}'s M list and N (g={spec.G} N={spec.N}) at K={prob.K}, seed 0"
    return {"workload": desc, "M": list(prob.M), "N": prob.N, "K": prob.K,
            "values": "E2M1 codes uniform over 16; E4M3 scales 2^e(1+u), e in [-4,2]",
            "scales": "raw row-major [rows, K/16] E4M3 per call"}


PER_CONFIGS = ["c0", "c1", "c2", "c3", "c4"]
PAGE_CONFIGS = ["c1_page", "c2_page", "c3_page", "c4_page"]


def roofline_time_us(flops, bytes_, fp4_tflops, hbm_gbs):
    return max(flops / (fp4_tflops * 1e12), bytes_ / (hbm_gbs * 1e9)) * 1e6


def config_summary(q, fp4_peak_tflops, hbm):
    """Per-config figures of one time_config result."""
    us = q["us_mean"]
    t_roof = roofline_time_us(q["flops"], q["bytes"], fp4_peak_tflops, hbm)
    t_nom = roofline_time_us(q["flops"], q["bytes"], NOMINAL_FP4_TFLOPS, NOMINAL_HBM_GBS)
    by = {m: {k: (round(v, 2) if isinstance(v, float) else v) for k, v in d.items()} for m, d in q["by"].items()}
    return {"us": round(us, 2), "protocol": q["headline"], "us_by_protocol": by,
            "gbs": round(q["bytes"] / (us * 1e-6) / 1e9, 1), "tflops": round(q["flops"] / (us * 1e-6) / 1e12, 1),
            "roofline_fraction": round(t_roof / us, 3), "roofline_time_us": round(t_roof, 2),
            "roofline_fraction_nominal": round(t_nom / us, 3),
            "algorithmic_bytes": q["bytes"], "flops": q["flops"],
            "host_us": {k: round(v, 2) for k, v in q["host"].items()},
            "grid": q["info"].grid, "chunks": q["info"].chunks, "M": list(q["prob"].M),
            "row_units": q["info"].row_units, "split_acc": q["info"].split_acc}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="c4")
    ap.add_argument("--k", type=int, default=0,
                    help="time the config's M list and N at another K (a multiple of 64; 0 = the config's K)")
    ap.add_argument("--sf-path", default="fused", choices=["fused", "fused-cached", "relayout", "relayout-cached", "atom"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--all-configs", action="store_true",
                    help="also time the pages' M lists and the re-layout paths (extra key)")
    ap.add_argument("--no-per-config", action="store_true", help="skip the c0-c4 table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--tile-n", type=int, default=0, help="widest output tile (0 = library default)")
    ap.add_argument("--b-stages", type=int, default=0)
    ap.add_argument("--a-stages", type=int, default=0)
    ap.add_argument("--serial-launch", action="store_true",
                    help="plain kernel launches (no overlap of a call's set-up with the previous call)")
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
    tuning = dict(tile_n=args.tile_n, b_stages=args.b_stages, a_stages=args.a_stages,
                  serial_launch=args.serial_launch)

    barrier(world)
    with ClockSampler(local) as clocks:
        r = time_config(args.config, args.sf_path, args.steps, args.warmup, torch=torch, flush=flush,
                        want_e2e=not args.no_e2e, tuning=tuning, prob=headline_problem(args))
    barrier(world)
    us = max_over_ranks(world, r["us_mean"], device)
    prob = r["prob"]
    bytes_, flops = r["bytes"], r["flops"]
    achieved_gbs = bytes_ / (us * 1e-6) / 1e9
    tflops = flops / (us * 1e-6) / 1e12
    t_roof_us = roofline_time_us(flops, bytes_, fp4_peak_tflops, hbm)
    t_roof_nominal_us = roofline_time_us(flops, bytes_, NOMINAL_FP4_TFLOPS, NOMINAL_HBM_GBS)
    iso = r["by"].get("isolated", r["by"]["flush"])
    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": dict(workload_config(args.config, prob), sf_path=args.sf_path,
                       l2=l2_text(r),
                       timing=("K calls back to back between one event pair (a device sleep ahead of the "
                               "start event covers the host's enqueue); value = elapsed / K"
                               if r["headline"] == "stream" else "one call between its own events"),
                       launch="plain" if args.serial_launch else "set-up overlaps the previous call",
                       max_tile_n=r["info"].tile_n, grid=r["info"].grid, chunks=r["info"].chunks,
                       b_stages=r["info"].b_stages, a_stages=r["info"].a_stages,
                       parallelism=f"replicas x{world}"),
        "us_isolated_call": {k: round(v, 2) for k, v in iso.items()},
        "us_b_static": (round(r["by"]["stream_b_static"]["us_mean"], 2) if "stream_b_static" in r["by"] else None),
        "b_static_note": ("the same back-to-back calls with the b_static option (the caller declares B and "
                          "SFB unwritten by the previous kernel, as for inference weights): each call streams "
                          "B while the previous call's last CTAs finish; A, SFA and C still wait"),
        "us_inputs_static": (round(r["by"]["stream_inputs_static"]["us_mean"], 2)
                             if "stream_inputs_static" in r["by"] else None),
        "inputs_static_note": ("the same back-to-back calls with b_static = 2 (the caller declares all four "
                               "inputs unwritten by the previous kernel): every load may start while the previous "
                               "call finishes, only the C stores wait"),
        "us_by_protocol": {m: {k: (round(v, 2) if isinstance(v, float) else v) for k, v in d.items()}
                           for m, d in r["by"].items()},
        "host_us_per_call": {k: round(v, 2) for k, v in r["host"].items()},
        "tflops_fp4": tflops, "gbs": achieved_gbs,
        "roofline_fraction": t_roof_us / us,
        "roofline_time_us": t_roof_us,
        "roofline_fraction_nominal": t_roof_nominal_us / us,
        "roofline_time_us_nominal": t_roof_nominal_us,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm,
                     "traffic": traffic_for(args.config, args.sf_path) if not args.k else None,
                     "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": bytes_,
                     "kernel": ("ggemm_kernel + sf_relayout_kernel" if args.sf_path.startswith("relayout")
                                    else "ggemm_kernel")},
        "gpu_launches": r["launches_per_call"] * args.steps,
        "clocks": clocks.summary(),
        "timed_wall_s": r["timed_wall_s"],
    }
    if "e2e" in r:
        e2e = r["e2e"]
        line["e2e"] = {"value": e2e["value"], "unit": UNIT, "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                       "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}
    if rank == 0 and not args.no_per_config:
        per = {}
        names = PER_CONFIGS + (PAGE_CONFIGS if args.all_configs else [])
        paths = ["fused"] + (["relayout", "relayout-cached"] if args.all_configs else [])
        with ClockSampler(local) as clocks_pc:
            for name in names:
                for path in paths:
                    if name == args.config and path == args.sf_path and not args.k:
                        q = r
                    else:
                        q = time_config(name, path, args.steps, args.warmup, torch=torch, flush=flush,
                                        tuning=tuning)
                    per[name if path == "fused" else f"{name}/{path}"] = config_summary(q, fp4_peak_tflops, hbm)
        line["per_config"] = per
        line["per_config_clocks"] = clocks_pc.summary()
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle as it stands, whole problems, all host cores; and c2 on one thread
        by_cfg = {}
        for name in PER_CONFIGS:
            p = prob if name == args.config and not args.k else synth.make_problem(name, seed=0)
            sec, cores = oracle_time(p)
            by_cfg[name] = {"s": round(sec, 3), "threads": cores}
        p2 = synth.make_problem("c2", seed=0)
        sec1, _ = oracle_time(p2, nthreads=1)
        by_cfg["c2_1thread"] = {"s": round(sec1, 3), "threads": 1}
        if args.k:
            sec, cores = oracle_time(prob)
            by_cfg[f"{args.config}_k{args.k}"] = {"s": round(sec, 3), "threads": cores}
        key = f"{args.config}_k{args.k}" if args.k else args.config
        line["cpu_baseline"] = {"value": by_cfg[key]["s"] * 1e6, "unit": UNIT,
                                "cores": by_cfg[key]["threads"], "kind": "oracle",
                                "sample": f"the whole {args.config} problem once (all {len(prob.M)} groups, "
                                          f"{sum(prob.M)} rows, K={prob.K}), not scaled"}
        line["cpu_baseline_by_config"] = by_cfg
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
