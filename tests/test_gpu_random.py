"""Seeded random grouped problems on the GPU against the oracle: per-group
M_g, N_g and K_g drawn across tile and chunk boundaries (empty groups, one
row, partial row tiles and pairs; N_g % 32 != 0; K_g % 256 != 0), random
scale layout and path, random widest tile and grid cap. Every output is
checked for being written; the oracle computes sampled entries, compared
within |gpu - ref| <= 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, atom_copy, sample_indices, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def O():
    return oracle.get()


def _draw(rng, k256):
    G = int(rng.integers(1, 13))
    M = [int(rng.choice([0, 1, rng.integers(1, 129), rng.integers(129, 700)])) for _ in range(G)]
    N = [8 * int(rng.integers(1, 300)) for _ in range(G)]
    # every third case keeps all K_g % 256 == 0 (raw scale rows loaded by the TMA)
    K = [int(256 * rng.integers(1, 12) if k256 else rng.choice([256 * rng.integers(1, 12), 64 * rng.integers(1, 48)]))
         for _ in range(G)]
    layout = "raw" if k256 else str(rng.choice(["raw", "atom"]))
    path = "fused" if k256 else (str(rng.choice(["fused", "relayout"])) if layout == "raw" else "fused")
    tile_n = int(rng.choice([0, 256, 192, 160, 128, 64]))
    max_ctas = int(rng.choice([0, 0, 1, 7, 64]))
    return M, N, K, layout, path, tile_n, max_ctas


@pytest.mark.parametrize("case", range(15))
def test_random_grouped_problem(O, case):
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    rng = np.random.default_rng(2000 + case)
    M, N, K, layout, path, tile_n, max_ctas = _draw(rng, case % 3 == 0)
    parts = [synth.make_problem("custom", seed=2100 + 37 * case + g, M=[m], N=n, K=k)
             for g, (m, n, k) in enumerate(zip(M, N, K))]
    A = to_device([p.A[0] for p in parts])
    B = to_device([p.B[0] for p in parts])
    SFA = to_device([p.SFA[0] for p in parts])
    SFB = to_device([p.SFB[0] for p in parts])
    if layout == "atom":
        SFA = [atom_copy(s, m, k) for s, m, k in zip(SFA, M, K)]
        SFB = [atom_copy(s, n, k) for s, n, k in zip(SFB, N, K)]
    C = [torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda") for m, n in zip(M, N)]
    what = f"case {case}: G={len(M)} M={M} N={N} K={K} {layout}/{path} tile_n={tile_n} max_ctas={max_ctas}"
    with nb.GroupedGemm(M, N, K, sf_layout=layout, sf_path=path, tile_n=tile_n, max_ctas=max_ctas) as gg:
        gg.run(A, B, SFA, SFB, C)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (what, nb.nvfp4_status_string(st), hex(word))
    torch.cuda.synchronize()
    for g, p in enumerate(parts):
        if M[g] == 0:
            continue
        got = C[g].cpu().numpy()
        assert not np.isnan(got).any(), f"{what}: group {g} has unwritten elements"
        rows, cols = sample_indices(M[g], N[g], 300, rng)
        ref16, _ = O.group_entries(p.A[0], p.B[0], p.SFA[0], p.SFB[0], K[g], rows, cols)
        assert_close(got[rows, cols], ref16, f"{what}: group {g}")
