"""Helpers for the GPU tests: move a synth.Problem to the device, run it
through the C ABI, and compare against the oracle within the stated
tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref| (inf equal to same-sign inf)."""
from __future__ import annotations

from typing import List, Optional

import numpy as np

ATOL = 1e-2
RTOL = 1e-2


def torch_mod():
    import torch
    return torch


def to_device(arrs, device="cuda"):
    torch = torch_mod()
    return [torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in arrs]


def atom_copy(sf_dev, rows: int, K: int):
    """Atom-layout copy of a raw device scale tensor, made by the library's
    re-layout kernel (itself checked bit-exactly against the oracle)."""
    torch = torch_mod()
    from block_scaled_fp4_grouped_gb300 import binding as nb
    out = torch.zeros(max(1, nb.nvfp4_sf_atom_bytes(rows, K)), dtype=torch.uint8, device=sf_dev.device)
    if rows > 0:
        st = nb.nvfp4_sf_relayout(sf_dev, out, rows, K)
        assert st == nb.NVFP4_OK, nb.nvfp4_status_string(st)
    return out


def run_gpu(prob, sf_layout="raw", sf_path="fused", tile_n=0, cache_b_scales=False, sentinel=None,
            max_ctas=0, use_host=False, b_stages=0, a_stages=0, row_units=0):
    """Returns the list of C_g as numpy float16 arrays."""
    torch = torch_mod()
    from block_scaled_fp4_grouped_gb300 import binding as nb
    K, N = prob.K, prob.N
    if use_host:
        A = [np.ascontiguousarray(a) for a in prob.A]
        B = [np.ascontiguousarray(b) for b in prob.B]
        SFA = [np.ascontiguousarray(s) for s in prob.SFA]
        SFB = [np.ascontiguousarray(s) for s in prob.SFB]
        C = [np.zeros((m, N), np.float16) for m in prob.M]
        with nb.GroupedGemm(prob.M, N, K, sf_layout=sf_layout, sf_path=sf_path, tile_n=tile_n,
                            max_ctas=max_ctas) as gg:
            gg.run_host(A, B, SFA, SFB, C)
            st, detail = gg.sync_status()
            assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(detail))
        return C
    A = to_device(prob.A)
    B = to_device(prob.B)
    SFA = to_device(prob.SFA)
    SFB = to_device(prob.SFB)
    if sf_layout == "atom":
        SFA = [atom_copy(s, m, K) for s, m in zip(SFA, prob.M)]
        SFB = [atom_copy(s, N, K) for s in SFB]
    fill = float("nan") if sentinel is None else sentinel
    C = [torch.full((m, N), fill, dtype=torch.float16, device="cuda") for m in prob.M]
    with nb.GroupedGemm(prob.M, N, K, sf_layout=sf_layout, sf_path=sf_path, tile_n=tile_n,
                        cache_b_scales=cache_b_scales, max_ctas=max_ctas, b_stages=b_stages,
                        a_stages=a_stages, row_units=row_units) as gg:
        if cache_b_scales:
            gg.prepare_b_scales(SFB)
            gg.run(A, B, SFA, [None] * len(SFB), C)
        else:
            gg.run(A, B, SFA, SFB, C)
        st, detail = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(detail))
    torch.cuda.synchronize()
    return [c.cpu().numpy() for c in C]


def close_mask(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):
        ok = np.abs(g - r) <= ATOL + RTOL * np.abs(r)
    return ok | both_inf


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    ok = close_mask(gpu, ref)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} elements outside |d| <= {ATOL} + {RTOL}|ref|; "
                             f"first at {i}: gpu {gpu[i]} ref {ref[i]}")


def assert_bit_exact(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    g = np.asarray(gpu, np.float16)
    r = np.asarray(ref, np.float16)
    same = (g == r) | (np.isnan(g) & np.isnan(r))  # +0 == -0
    if not same.all():
        bad = np.argwhere(~same)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {same.size} elements differ; first at {i}: "
                             f"gpu {g[i]} ref {r[i]}")


def sample_indices(M: int, N: int, count: int, rng: np.random.Generator):
    """Random entries plus the corners and tile edges of an M x N output."""
    rows = list(rng.integers(0, M, count))
    cols = list(rng.integers(0, N, count))
    for m in {0, M - 1, min(M - 1, 127), min(M - 1, 128)}:
        for n in {0, N - 1, min(N - 1, 63), min(N - 1, 64), min(N - 1, 127), min(N - 1, 128)}:
            rows.append(m)
            cols.append(n)
    return np.asarray(rows, np.int32), np.asarray(cols, np.int32)
