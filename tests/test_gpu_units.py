"""Units of work of one 128-row tile, and split accumulators, on the GPU
against the oracle.

A plan's units of work are pairs of 128-row tiles (sharing every B stage)
or single row tiles (option row_units, or the plan's own choice). When every
CTA walks one tile of single row tiles, a tile of at most 192 columns adds
its even and odd 64-k slices into the two accumulator halves and the
epilogue sums them in fp32. These tests force each unit count on ragged and
workload shapes and compare with the oracle within |gpu - ref| <= 1e-2 +
1e-2 |ref|; the exact cases (power-of-two scales of small span, so every
partial sum is exact in fp32) must match bit for bit whichever accumulator
takes a slice; K of one 64-k slice leaves the odd accumulator unused."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def O():
    return oracle.get()


def _plan_units(prob, **options):
    from block_scaled_fp4_grouped_gb300 import binding as nb
    with nb.GroupedGemm(prob.M, prob.N, prob.K, **options) as gg:
        info = gg.info()
        return int(info.row_units), int(info.split_acc)


RAGGED = dict(M=[1, 127, 129, 0, 200, 384, 64], N=328, K=768)


@pytest.mark.parametrize("row_units", [1, 2])
@pytest.mark.parametrize("tile_n", [0, 192, 96, 32])
def test_forced_units_ragged(O, row_units, tile_n):
    prob = synth.make_problem("custom", seed=31, **RAGGED)
    units, split = _plan_units(prob, row_units=row_units, tile_n=tile_n)
    assert units == row_units
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, tile_n=tile_n, row_units=row_units)
    for g in range(prob.G):
        assert_close(got[g], ref[g], f"row_units {row_units} tile_n {tile_n} group {g} (split {split})")


@pytest.mark.parametrize("cfg", ["c1", "c2", "c1_page", "c2_page"])
@pytest.mark.parametrize("row_units", [0, 1, 2])
def test_two_group_workloads_every_element(O, cfg, row_units):
    """The 2-group workloads at seed 0 with each unit count (0: the plan's
    choice, single row tiles with split accumulators), every element."""
    prob = synth.make_problem(cfg, seed=0)
    units, split = _plan_units(prob, row_units=row_units)
    assert units == (1 if row_units in (0, 1) else 2)
    if row_units == 0:
        assert split == 1
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, row_units=row_units)
    for g in range(prob.G):
        assert not np.isnan(got[g]).any(), f"{cfg} group {g}: an element was never written"
        assert_close(got[g], ref[g], f"{cfg} row_units {row_units} group {g}")


@pytest.mark.parametrize("K", [64, 128, 192, 256, 320, 704, 1088])
def test_split_accumulators_exact_bit_for_bit(O, K):
    """Single row tiles, one tile per CTA, power-of-two scales of span 4:
    every fp32 partial sum is exact, so the two accumulators' sum is too and
    the GPU equals the oracle bit for bit, for K of one to many slices
    (K = 64: the odd accumulator is never written nor read)."""
    prob = synth.make_problem("custom", seed=40 + K, M=[140, 1, 300, 0, 64], N=392, K=K)
    rng = np.random.default_rng(40 + K)
    for g in range(prob.G):
        prob.SFA[g] = (((rng.integers(-2, 2, prob.SFA[g].shape) + 7) << 3)).astype(np.uint8)
        prob.SFB[g] = (((rng.integers(-2, 2, prob.SFB[g].shape) + 7) << 3)).astype(np.uint8)
    units, split = _plan_units(prob, row_units=1)
    assert (units, split) == (1, 1)
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, row_units=1)
    for g in range(prob.G):
        assert np.array_equal(got[g].view(np.uint16), ref[g].view(np.uint16)), f"K={K} group {g}"


def test_single_row_units_with_several_tiles_per_cta(O):
    """More single-row-tile chunks than one tile per CTA (a small grid): no
    split; tiles double-buffer their accumulators as usual."""
    prob = synth.make_problem("custom", seed=50, M=[400, 256, 77], N=1000, K=512)
    units, split = _plan_units(prob, row_units=1, max_ctas=7)
    assert (units, split) == (1, 0)
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, row_units=1, max_ctas=7)
    for g in range(prob.G):
        assert_close(got[g], ref[g], f"group {g}")


@pytest.mark.parametrize("layout,path", [("raw", "fused"), ("raw", "relayout"), ("atom", "fused")])
def test_split_accumulators_on_the_other_scale_paths(O, layout, path):
    prob = synth.make_problem("custom", seed=60, M=[448, 320], N=3072, K=1088)
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, sf_layout=layout, sf_path=path, row_units=1)
    for g in range(prob.G):
        assert_close(got[g], ref[g], f"{layout}/{path} group {g}")
