"""The work split (nvfp4_ggemm_schedule), checked on the host.

Every group's pairs of 128-row tiles own ceil(N/32) consecutive chunks of 32
columns; CTA c takes chunks [cta_begin[c], cta_begin[c+1]). These tests
check the split against properties fixed by that definition: the ranges
partition the chunks; when there are no more pairs than CTAs, each range
lies in one pair and the most tiles any CTA needs (a tile is at most 192
columns for two row tiles, tile_n for one) is the fewest with which the
pairs fit the grid or fewer (a CTA that takes two or more tiles of a pair
with two row tiles takes one chunk fewer per tile, when a tile holds more
than two chunks); otherwise the ranges are equal to within one chunk."""
import random

import pytest

from block_scaled_fp4_grouped_gb300 import binding as nb
from block_scaled_fp4_grouped_gb300 import build as nbuild


@pytest.fixture(scope="module", autouse=True)
def built():
    nbuild.build()


def pairs_of(M):
    """(chunk offset, row tiles in the pair) of every pair, in chunk order."""
    out = []
    for m in M:
        tiles = -(-m // 128)
        for t in range(0, tiles, 2):
            out.append(min(2, tiles - t))
    return out


def caps(tile_n):
    tile_n = tile_n or 256
    kernel = 128 if tile_n <= 128 else 256
    single = tile_n // 32
    pair = min(single, (192 if kernel >= 192 else kernel) // 32)
    return single, pair


def per_cta(cap, rows, passes):
    """Chunks a CTA takes from one pair when it walks at most `passes` tiles:
    tiles of two row tiles are one chunk narrower once there are two or more."""
    return passes * (cap - 1 if rows == 2 and passes > 1 and cap > 2 else cap)


def ctas_needed(M, N, tile_n, passes):
    """CTAs needed when each takes at most `passes` tiles inside one pair."""
    single, pair = caps(tile_n)
    n = -(-N // 32)
    return sum(-(-n // per_cta(pair if rows == 2 else single, rows, passes)) for rows in pairs_of(M))


def check(M, N, tile_n, max_ctas):
    st, cb = nb.nvfp4_ggemm_schedule(M, N, tile_n, max_ctas)
    assert st == nb.NVFP4_OK
    n = -(-N // 32)
    segs = pairs_of(M)
    total = len(segs) * n
    grid = len(cb) - 1
    if total == 0:
        assert grid == 0
        return cb
    assert 1 <= grid <= max_ctas
    assert cb[0] == 0 and cb[-1] == total
    assert all(b > a for a, b in zip(cb, cb[1:])), "every CTA gets at least one chunk"
    single, pair = caps(tile_n)
    if len(segs) <= max_ctas:
        fewest = next(P for P in range(1, 10 ** 6) if ctas_needed(M, N, tile_n, P) <= max_ctas)
        most = 0
        for a, b in zip(cb, cb[1:]):
            s = a // n
            assert (b - 1) // n == s, f"range [{a},{b}) crosses a pair boundary"
            cap = pair if segs[s] == 2 else single
            most = max(most, -(-(b - a) // cap))
        # narrower pair tiles may leave a CTA fewer tiles than passes, never more
        assert most <= fewest, (most, fewest)
    else:
        sizes = [b - a for a, b in zip(cb, cb[1:])]
        assert grid == min(total, max_ctas)
        assert max(sizes) - min(sizes) <= 1
    return cb


def test_page_shape_gets_one_tile_per_cta():
    # four-group-pairs-and-singles shape of the largest timed workload
    M = [80, 176, 128, 72, 64, 248, 96, 160]
    cb = check(M, 4096, 0, 152)
    assert len(cb) - 1 == 152
    widths = [b - a for a, b in zip(cb, cb[1:])]
    assert max(widths) == 8  # 128 chunks over 17 CTAs per one-tile group


def test_skinny_wide_shape_takes_two_passes_per_cta():
    M = [40, 76, 168, 72, 164, 148, 196, 160]
    cb = check(M, 7168, 0, 152)
    assert len(cb) - 1 == 152
    widths = [b - a for a, b in zip(cb, cb[1:])]
    assert max(widths) <= 12  # two tiles of at most 6 chunks in the two-row-tile pairs


def test_more_pairs_than_ctas_uses_equal_ranges():
    M = [256] * 40
    cb = check(M, 1024, 0, 16)
    assert len(cb) - 1 == 16


@pytest.mark.parametrize("tile_n", [0, 256, 224, 192, 128, 96, 32])
def test_random_shapes(tile_n):
    rng = random.Random(1234 + tile_n)
    for _ in range(200):
        G = rng.randint(1, 12)
        M = [rng.choice([0, rng.randint(1, 700)]) for _ in range(G)]
        N = 8 * rng.randint(1, 1200)
        max_ctas = rng.choice([1, 3, 37, 148, 152, 192])
        check(M, N, tile_n, max_ctas)


def test_empty_problem_has_no_ctas():
    st, cb = nb.nvfp4_ggemm_schedule([0, 0], 256, 0, 152)
    assert st == nb.NVFP4_OK and cb == [0]


@pytest.mark.parametrize("kw", [dict(tile_n=80), dict(tile_n=288), dict(max_ctas=0), dict(max_ctas=193),
                                dict(N=12), dict(M=[-1])])
def test_bad_arguments(kw):
    args = dict(M=[64], N=256, tile_n=0, max_ctas=152)
    args.update(kw)
    st, _ = nb.nvfp4_ggemm_schedule(args["M"], args["N"], args["tile_n"], args["max_ctas"])
    assert st in (nb.NVFP4_ERR_INVALID_ARG, nb.NVFP4_ERR_UNSUPPORTED_SHAPE)


def _check_shapes(M, N, K, tile_n, max_ctas):
    """Per-group N_g and K_g: the ranges partition the chunks (pairs of group g
    own ceil(N_g/32) chunks each); with no more pairs than CTAs every range
    lies in one pair and the most k-stages any CTA needs (tiles x ceil(K_g/256)) is
    the smallest budget with which the pairs fit the grid."""
    st, cb = nb.nvfp4_ggemm_schedule(M, N, tile_n, max_ctas, K=K)
    assert st == nb.NVFP4_OK
    single, pair = caps(tile_n)
    segs = []  # (first chunk, chunks, cap, k tiles)
    base = 0
    for m, n, k in zip(M, N, K):
        tiles = -(-m // 128)
        for t in range(0, tiles, 2):
            c = -(-n // 32)
            segs.append((base, c, pair if tiles - t >= 2 else single, -(-k // 256), min(2, tiles - t)))
            base += c
    total = base
    grid = len(cb) - 1
    if total == 0:
        assert grid == 0
        return
    assert cb[0] == 0 and cb[-1] == total and all(b > a for a, b in zip(cb, cb[1:]))
    if len(segs) > max_ctas:
        return
    def seg_of(x):
        return next(i for i, s in enumerate(segs) if s[0] <= x < s[0] + s[1])
    def need(budget):
        return sum(-(-c // per_cta(cap, rows, max(1, budget // kt))) for _, c, cap, kt, rows in segs)
    fewest = next(B for B in range(1, 10 ** 7) if need(B) <= max_ctas)
    for a, b in zip(cb, cb[1:]):
        i = seg_of(a)
        assert seg_of(b - 1) == i, f"range [{a},{b}) crosses a pair boundary"
        _, c, cap, kt, _ = segs[i]
        stages = -(-(b - a) // cap) * kt
        # within the smallest fitting budget, or one pass where a pass alone exceeds it
        assert stages <= max(fewest, kt), (stages, fewest, kt)


@pytest.mark.parametrize("tile_n", [0, 192, 128])
def test_random_per_group_shapes(tile_n):
    rng = random.Random(77 + tile_n)
    for _ in range(150):
        G = rng.randint(1, 10)
        M = [rng.choice([0, rng.randint(1, 600)]) for _ in range(G)]
        N = [8 * rng.randint(1, 700) for _ in range(G)]
        K = [rng.choice([256 * rng.randint(1, 24), 64 * rng.randint(1, 96)]) for _ in range(G)]
        _check_shapes(M, N, K, tile_n, rng.choice([1, 7, 64, 152]))


def test_per_group_bad_shapes():
    for N, K in (([256, 12], [256, 256]), ([256, 256], [256, 300])):
        st, _ = nb.nvfp4_ggemm_schedule([64, 64], N, 0, 152, K=K)
        assert st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE


# ------------------------------------------------- units of one row tile

def check_single(M, N, tile_n, max_ctas):
    """row_units = 1: every group's ceil(M_g/128) row tiles own ceil(N/32)
    chunks each; the same properties as for pairs, with every segment one
    row tile wide (tiles of at most tile_n). Returns (cta_begin, split)."""
    st, cb, units, split = nb.nvfp4_ggemm_schedule_units(M, N, tile_n, max_ctas, 256, 1)
    assert st == nb.NVFP4_OK and units == 1
    n = -(-N // 32)
    segs = sum(-(-m // 128) for m in M)
    total = segs * n
    grid = len(cb) - 1
    if total == 0:
        assert grid == 0
        return cb, split
    assert 1 <= grid <= max_ctas
    assert cb[0] == 0 and cb[-1] == total
    assert all(b > a for a, b in zip(cb, cb[1:]))
    single, _ = caps(tile_n)
    tiles = [-(-(b - a) // single) for a, b in zip(cb, cb[1:])]
    if segs <= max_ctas:
        fewest = next(P for P in range(1, 10 ** 6) if segs * -(-n // (P * single)) <= max_ctas)
        for a, b in zip(cb, cb[1:]):
            assert (b - 1) // n == a // n, f"range [{a},{b}) crosses a row tile boundary"
        assert max(tiles) <= fewest
        # split accumulators exactly when every CTA walks one tile
        assert split == (1 if max(tiles) == 1 else 0)
    return cb, split


@pytest.mark.parametrize("tile_n", [0, 256, 192, 128, 64])
def test_single_row_units_random_shapes(tile_n):
    rng = random.Random(4321 + tile_n)
    for _ in range(150):
        G = rng.randint(1, 10)
        M = [rng.choice([0, rng.randint(1, 700)]) for _ in range(G)]
        N = 8 * rng.randint(1, 1200)
        check_single(M, N, tile_n, rng.choice([1, 5, 37, 152, 192]))


def test_pairs_through_the_units_entry_match_the_pair_schedule():
    rng = random.Random(99)
    for _ in range(100):
        M = [rng.randint(0, 700) for _ in range(rng.randint(1, 8))]
        N = 8 * rng.randint(1, 900)
        st, cb, units, split = nb.nvfp4_ggemm_schedule_units(M, N, 0, 152, 256, 2)
        assert st == nb.NVFP4_OK and units == 2 and split == 0
        assert cb == nb.nvfp4_ggemm_schedule(M, N, 0, 152)[1]


@pytest.mark.parametrize("cfg,want", [("c0", 2), ("c1", 1), ("c2", 1), ("c3", 2), ("c4", 2),
                                      ("c1_page", 1), ("c2_page", 1), ("c3_page", 2), ("c4_page", 2)])
def test_automatic_units_on_the_workloads(cfg, want):
    """Pairs stay unless their tiles would be at most four chunks wide while
    one-row-tile units give every CTA a single tile: the two 2-group
    workloads (tall groups, narrow N) take single row tiles with split
    accumulators; the 8-group ones and the small case keep pairs."""
    import numpy as np
    from block_scaled_fp4_grouped_gb300 import synth
    if cfg.endswith("_page"):
        d = synth.PAGE_SHAPES[cfg]
        M, N, K = d["M"], d["N"], d["K"]
    else:
        spec = synth.CONFIGS[cfg]
        M, N, K = synth.draw_m_list(spec, np.random.default_rng(0)), spec.N, spec.K
    st, cb, units, split = nb.nvfp4_ggemm_schedule_units(M, N, 0, 152, K, 0)
    assert st == nb.NVFP4_OK and units == want
    assert split == (1 if want == 1 else 0)
    if want == 1:
        assert cb == nb.nvfp4_ggemm_schedule_units(M, N, 0, 152, K, 1)[1]
    else:
        assert cb == nb.nvfp4_ggemm_schedule(M, N, 0, 152, K)[1]


def test_automatic_units_rule_on_random_shapes():
    """Whenever the choice is single row tiles, every CTA walks one tile and
    the pair split's two-row-tile tiles would be at most four chunks wide."""
    rng = random.Random(7)
    for _ in range(200):
        M = [rng.randint(0, 600) for _ in range(rng.randint(1, 6))]
        N = 8 * rng.randint(1, 700)
        st, cb, units, split = nb.nvfp4_ggemm_schedule_units(M, N, 0, 152, 256, 0)
        assert st == nb.NVFP4_OK and units in (1, 2)
        if units == 1:
            assert split == 1
            assert max(b - a for a, b in zip(cb, cb[1:])) <= 8
            n = -(-N // 32)
            _, cb2 = nb.nvfp4_ggemm_schedule(M, N, 0, 152)
            segs = pairs_of(M)
            widest = 0
            for a, b in zip(cb2, cb2[1:]):
                if segs[a // n] == 2:
                    cap = 6
                    pt = -(-(b - a) // cap)
                    widest = max(widest, -(-(b - a) // pt))
            assert 0 < widest <= 4


@pytest.mark.parametrize("row_units", [-1, 3])
def test_units_entry_rejects_bad_unit_counts(row_units):
    st, cb, units, split = nb.nvfp4_ggemm_schedule_units([64], 256, 0, 152, 256, row_units)
    assert st == nb.NVFP4_ERR_INVALID_ARG


def test_units_entry_random_per_group_shapes():
    """Per-group N_g and K_g, every unit count: the ranges partition the
    chunks of the units the call reports (ceil(M_g/128/units) units of
    ceil(N_g/32) chunks per group), and split accumulators only come with
    single row tiles."""
    rng = random.Random(2024)
    for _ in range(150):
        G = rng.randint(1, 9)
        M = [rng.choice([0, rng.randint(1, 900)]) for _ in range(G)]
        N = [8 * rng.randint(1, 600) for _ in range(G)]
        K = [64 * rng.randint(1, 120) for _ in range(G)]
        row_units = rng.choice([0, 1, 2])
        max_ctas = rng.choice([1, 9, 64, 152, 192])
        st, cb, units, split = nb.nvfp4_ggemm_schedule_units(M, N, rng.choice([0, 128, 256]), max_ctas, K,
                                                             row_units)
        assert st == nb.NVFP4_OK
        assert units in (1, 2) and (row_units == 0 or units == row_units)
        assert split in (0, 1) and (units == 1 or split == 0)
        total = sum(-(-(-(-m // 128)) // units) * -(-n // 32) for m, n in zip(M, N))
        if total == 0:
            assert cb == [0]
            continue
        assert cb[0] == 0 and cb[-1] == total and 1 <= len(cb) - 1 <= max_ctas
        assert all(b > a for a, b in zip(cb, cb[1:]))
