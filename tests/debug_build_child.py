"""Run by tests/test_gpu_debug_build.py in a child process whose
NVFP4_GGEMM_LIB names the device-check build (libnvfp4_ggemm_debug.so), so
that every call below goes through the kernel compiled with -DNVFP4_DEBUG.
Prints one JSON object: the library path it loaded, the worst
|gpu - ref| / tolerance of each problem, and for each check site the status
and error word of a call that forces that check to fail, followed by the
status of a good call on the same context."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from block_scaled_fp4_grouped_gb300 import binding as nb, synth  # noqa: E402
from gpu_util import run_gpu, to_device  # noqa: E402


def worst_ratio(got, ref):
    worst = 0.0
    for g, r in zip(got, ref):
        if g.size == 0:
            continue
        d = np.abs(g.astype(np.float64) - r.astype(np.float64)) / (1e-2 + 1e-2 * np.abs(r.astype(np.float64)))
        if not np.isfinite(d).all():
            return float("inf")
        worst = max(worst, float(d.max()))
    return worst


def main():
    import torch
    out = {"lib": nb.LIB_PATH, "parity": {}, "checks": {}}
    O = oracle.get()
    problems = [
        ("c0", synth.make_problem("c0", seed=0), {}),
        ("pairs_ragged", synth.make_problem("custom", seed=71, M=[1, 130, 257, 0, 64], N=328, K=768),
         {"row_units": 2}),
        ("single_rows_split", synth.make_problem("custom", seed=76, M=[1, 130, 257, 0, 64], N=328, K=832),
         {"row_units": 1}),
        ("k_mod_64_lanes", synth.make_problem("custom", seed=72, M=[100, 200], N=256, K=448), {}),
        ("k_mod_128_lanes_classes", synth.make_problem("custom", seed=77, M=[130, 7], N=264, K=640), {}),
        ("k_mod_64_relayout", synth.make_problem("custom", seed=72, M=[100, 200], N=256, K=448),
         {"sf_path": "relayout"}),
        ("atom_layout", synth.make_problem("custom", seed=73, M=[96, 300], N=512, K=1024), {"sf_layout": "atom"}),
        ("tile_128", synth.make_problem("custom", seed=74, M=[129, 64], N=384, K=512), {"tile_n": 128}),
    ]
    for name, prob, kw in problems:
        got = run_gpu(prob, **kw)
        ref, _ = O.grouped(prob)
        out["parity"][name] = worst_ratio(got, ref)
    # raw scale rows loaded by TMA (K % 256 == 0) or copied by the scale
    # producer's lanes; the kernels for single row tiles (split accumulators)
    # and for pairs
    for kind, K in (("tma", 1024), ("lanes", 1152)):
        prob = synth.make_problem("custom", seed=75, M=[200, 64], N=512, K=K)
        ref, _ = O.grouped(prob)
        for units in (1, 2):
            for site in range(0x21, 0x27):
                A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
                C = [torch.zeros((m, prob.N), dtype=torch.float16, device="cuda") for m in prob.M]
                with nb.GroupedGemm(prob.M, prob.N, prob.K, debug_check_fail=site, wait_timeout_ns=100_000_000,
                                    row_units=units) as gg:
                    info = gg.info()
                    gg.run(A, B, SFA, SFB, C)
                    st, word = gg.sync_status()
                got = run_gpu(prob, row_units=units)
                out["checks"][f"{kind}/{units}/{hex(site)}"] = {"status": st, "word": word,
                                                                 "after": worst_ratio(got, ref),
                                                                 "units": int(info.row_units),
                                                                 "split": int(info.split_acc)}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
