"""Per-group N_g and K_g (nvfp4_ggemm_plan_shapes) on the GPU against the oracle.

Group g computes C_g[M_g, N_g] from A_g[M_g, K_g] and B_g[N_g, K_g] with their
own scales; the oracle computes each group on its own (it is a per-group
definition), so the comparison is element by element within the stated
tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|. The shapes mix N_g that are and
are not multiples of 32 and 256, K_g of one to many 256-k stages, groups of
one and two 128-row tiles, an empty group and a partial last row tile."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, atom_copy, to_device

pytestmark = pytest.mark.gpu

SHAPES = [  # (M_g, N_g, K_g)
    (200, 328, 768),
    (64, 4096, 256),
    (0, 512, 512),
    (130, 72, 2048),
    (256, 1000, 1536),
    (17, 8, 256),
    (384, 2056, 1024),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def O():
    return oracle.get()


def _groups(seed):
    parts = [synth.make_problem("custom", seed=seed + g, M=[m], N=n, K=k) for g, (m, n, k) in enumerate(SHAPES)]
    return parts


def _run(parts, sf_layout="raw", sf_path="fused", use_host=False, cache_b_scales=False):
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    M = [p.M[0] for p in parts]
    N = [p.N for p in parts]
    K = [p.K for p in parts]
    if use_host:
        A = [np.ascontiguousarray(p.A[0]) for p in parts]
        B = [np.ascontiguousarray(p.B[0]) for p in parts]
        SFA = [np.ascontiguousarray(p.SFA[0]) for p in parts]
        SFB = [np.ascontiguousarray(p.SFB[0]) for p in parts]
        C = [np.zeros((m, n), np.float16) for m, n in zip(M, N)]
        with nb.GroupedGemm(M, N, K) as gg:
            gg.run_host(A, B, SFA, SFB, C)
            st, word = gg.sync_status()
            assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
        return C
    A = to_device([p.A[0] for p in parts])
    B = to_device([p.B[0] for p in parts])
    SFA = to_device([p.SFA[0] for p in parts])
    SFB = to_device([p.SFB[0] for p in parts])
    if sf_layout == "atom":
        SFA = [atom_copy(s, m, k) for s, m, k in zip(SFA, M, K)]
        SFB = [atom_copy(s, n, k) for s, n, k in zip(SFB, N, K)]
    C = [torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda") for m, n in zip(M, N)]
    with nb.GroupedGemm(M, N, K, sf_layout=sf_layout, sf_path=sf_path, cache_b_scales=cache_b_scales) as gg:
        if cache_b_scales:
            gg.prepare_b_scales(SFB)
            gg.run(A, B, SFA, [None] * len(SFB), C)
        else:
            gg.run(A, B, SFA, SFB, C)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    torch.cuda.synchronize()
    return [c.cpu().numpy() for c in C]


@pytest.mark.parametrize("layout,path,cached", [("raw", "fused", False), ("raw", "relayout", False),
                                                ("raw", "relayout", True), ("atom", "fused", False)])
def test_per_group_shapes_match_the_oracle(O, layout, path, cached):
    parts = _groups(seed=500)
    got = _run(parts, sf_layout=layout, sf_path=path, cache_b_scales=cached)
    for g, p in enumerate(parts):
        assert got[g].shape == (p.M[0], p.N)
        if p.M[0] == 0:
            continue
        ref, _, _ = O.group_gemm(p.A[0], p.B[0], p.SFA[0], p.SFB[0], p.K)
        assert not np.isnan(got[g]).any(), f"group {g}: an element was never written"
        assert_close(got[g], ref, f"group {g} (M={p.M[0]}, N={p.N}, K={p.K})")


def test_per_group_shapes_through_host_buffers(O):
    parts = _groups(seed=600)
    got = _run(parts, use_host=True)
    for g, p in enumerate(parts):
        if p.M[0] == 0:
            continue
        ref, _, _ = O.group_gemm(p.A[0], p.B[0], p.SFA[0], p.SFB[0], p.K)
        assert_close(got[g], ref, f"group {g}")


def test_uniform_call_equals_per_group_call_bitwise():
    prob = synth.make_problem("custom", seed=700, M=[150, 0, 300], N=384, K=1024)
    parts = []
    for g, m in enumerate(prob.M):
        q = synth.Problem("part", prob.N, prob.K, [m], seed=700)
        q.A, q.B, q.SFA, q.SFB = [prob.A[g]], [prob.B[g]], [prob.SFA[g]], [prob.SFB[g]]
        parts.append(q)
    per_group = _run(parts)
    from gpu_util import run_gpu
    uniform = run_gpu(prob)
    for g in range(prob.G):
        assert np.array_equal(per_group[g].view(np.uint16), uniform[g].view(np.uint16))


def test_strided_c_writes_only_its_columns():
    """nvfp4_ggemm_run_strided: each C_g is a column slice of a wider fp16
    matrix (row stride ldc_g > N_g). The slice must equal the dense result
    bit for bit, and the columns around it must keep their sentinel."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    from gpu_util import run_gpu
    prob = synth.make_problem("custom", seed=800, M=[150, 0, 300, 40], N=328, K=1024)
    dense = run_gpu(prob)
    A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
    pads = [(16, 40), (8, 8), (0, 24), (64, 0)]  # columns before / after each slice
    wide = [torch.full((m, lo + prob.N + hi), -7.0, dtype=torch.float16, device="cuda")
            for m, (lo, hi) in zip(prob.M, pads)]
    C = [w[:, lo:lo + prob.N] for w, (lo, _) in zip(wide, pads)]
    ldc = [w.shape[1] for w in wide]
    with nb.GroupedGemm(prob.M, prob.N, prob.K) as gg:
        gg.run_strided(A, B, SFA, SFB, C, ldc)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
        with pytest.raises(nb.Nvfp4Error):
            gg.run_strided(A, B, SFA, SFB, C, [prob.N - 8] + ldc[1:])  # stride below N
    torch.cuda.synchronize()
    for g, (m, (lo, hi)) in enumerate(zip(prob.M, pads)):
        w = wide[g].cpu().numpy()
        assert np.array_equal(w[:, lo:lo + prob.N].view(np.uint16), dense[g].view(np.uint16))
        assert (w[:, :lo] == -7.0).all() and (w[:, lo + prob.N:] == -7.0).all()


def test_bound_call_equals_run_bitwise():
    """GroupedGemm.bind: pointer arrays built once, then repeated calls. Two
    bound buffer sets on one plan (one dense, one strided) must each equal
    the plain call bit for bit, called in alternation."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    from gpu_util import run_gpu
    prob = synth.make_problem("custom", seed=900, M=[96, 260, 0, 33], N=264, K=768)
    dense = run_gpu(prob)
    A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
    C1 = [torch.full((m, prob.N), 3.0, dtype=torch.float16, device="cuda") for m in prob.M]
    wide = [torch.full((m, prob.N + 24), -5.0, dtype=torch.float16, device="cuda") for m in prob.M]
    C2 = [w[:, 8:8 + prob.N] for w in wide]
    with nb.GroupedGemm(prob.M, prob.N, prob.K) as gg:
        call1 = gg.bind(A, B, SFA, SFB, C1)
        call2 = gg.bind(A, B, SFA, SFB, C2, ldc=[prob.N + 24] * prob.G)
        for _ in range(3):
            call1()
            call2()
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    torch.cuda.synchronize()
    for g in range(prob.G):
        assert np.array_equal(C1[g].cpu().numpy().view(np.uint16), dense[g].view(np.uint16))
        w = wide[g].cpu().numpy()
        assert np.array_equal(w[:, 8:8 + prob.N].view(np.uint16), dense[g].view(np.uint16))
        assert (w[:, :8] == -5.0).all() and (w[:, 8 + prob.N:] == -5.0).all()


SHAPES_K64 = [  # (M_g, N_g, K_g): most K_g are not multiples of 256
    (200, 328, 320),
    (64, 256, 64),
    (130, 72, 832),
    (0, 512, 192),
    (257, 1000, 1088),
    (17, 8, 128),
    (96, 520, 256),
    (33, 4096, 448),
    (3, 64, 320),
    (1, 40, 64),
    (6, 96, 1216),
]


@pytest.mark.parametrize("layout,path,cached", [("raw", "fused", False), ("raw", "fused", True),
                                                ("raw", "relayout", True), ("atom", "fused", False)])
def test_k_multiple_of_64_matches_the_oracle(O, layout, path, cached):
    """K_g % 64 == 0 with a partial last 256-k tile: A and B past K_g come
    from the TMA's zero fill, the last tile issues only its live 64-k MMA
    slices and loads only its live scale atoms. Raw scale rows are not
    16-byte TMA rows here: on the FUSED path the scale producer's lanes copy
    them (one kernel), on the RELAYOUT path the re-layout kernel runs first;
    the plan says which."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    parts = [synth.make_problem("custom", seed=1000 + g, M=[m], N=n, K=k)
             for g, (m, n, k) in enumerate(SHAPES_K64)]
    with nb.GroupedGemm([p.M[0] for p in parts], [p.N for p in parts], [p.K for p in parts],
                        sf_layout=layout, sf_path=path) as gg:
        info = gg.info()
        assert info.sf_path == (nb.NVFP4_SF_RELAYOUT if path == "relayout" else nb.NVFP4_SF_FUSED)
        assert info.kernels_per_run == (2 if path == "relayout" else 1)
    got = _run(parts, sf_layout=layout, sf_path=path, cache_b_scales=cached)
    for g, p in enumerate(parts):
        assert got[g].shape == (p.M[0], p.N)
        if p.M[0] == 0:
            continue
        ref, _, _ = O.group_gemm(p.A[0], p.B[0], p.SFA[0], p.SFB[0], p.K)
        assert not np.isnan(got[g]).any(), f"group {g}: an element was never written"
        assert_close(got[g], ref, f"group {g} (M={p.M[0]}, N={p.N}, K={p.K})")


@pytest.mark.parametrize("layout,path,cached,K", [("raw", "fused", False, 7104), ("raw", "fused", False, 7040),
                                                  ("raw", "fused", True, 7104), ("raw", "fused", True, 7040),
                                                  ("raw", "relayout", False, 7104), ("raw", "relayout", True, 7104),
                                                  ("atom", "fused", False, 7104)])
def test_k7104_on_the_largest_m_list_sampled(O, layout, path, cached, K):
    """The K % 64 workload that is timed: the 8-group N = 4096 M list at
    K = 7104 (27 whole 256-k tiles and a last tile of three 64-k slices),
    through each path a caller can take (raw scale rows copied by the scale
    producer's lanes, raw scales re-laid out every call,
    with the B scales cached by the plan, and atom-layout scales read by
    3-D tensor-map boxes whose atoms past K are zero-filled); sampled
    entries and the output's tile edges against the oracle. K = 7040 (rows
    of 440 bytes) takes the FUSED path's 16- and 8-byte row classes."""
    from gpu_util import run_gpu, sample_indices
    M = synth.make_problem("c4", seed=0).M
    prob = synth.make_problem("custom", seed=1200, M=M, N=4096, K=K)
    got = run_gpu(prob, sf_layout=layout, sf_path=path, cache_b_scales=cached)
    rng = np.random.default_rng(1200)
    for g in range(prob.G):
        rows, cols = sample_indices(prob.M[g], prob.N, 400, rng)
        ref16, _ = O.group_entries(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K, rows, cols)
        assert_close(got[g][rows, cols], ref16, f"K={K} {layout}/{path} group {g}")
        assert not np.isnan(got[g]).any(), f"group {g}: an element was never written"


@pytest.mark.parametrize("K,cached", [(7104, False), (7040, False), (7104, True)])
def test_k_multiple_of_64_fused_largest_m_list_every_element(O, K, cached):
    """The FUSED path with lane-copied raw scale rows on the largest M list
    at K = 7104 (4-byte pieces) and K = 7040 (16- and 8-byte row classes):
    every element against the oracle, which does the whole problem in
    seconds on the host cores. With cache_b_scales the B scales are copied
    once into rows padded to 16 bytes and loaded by TMA."""
    from gpu_util import run_gpu
    M = synth.make_problem("c4", seed=0).M
    prob = synth.make_problem("custom", seed=1400, M=M, N=4096, K=K)
    got = run_gpu(prob, cache_b_scales=cached)
    ref, _ = O.grouped(prob)
    for g in range(prob.G):
        assert not np.isnan(got[g]).any(), f"group {g}: an element was never written"
        assert_close(got[g], ref[g], f"K={K} group {g}")


@pytest.mark.parametrize("K", [1216, 1152], ids=["rows_4mod8", "rows_8mod16"])
@pytest.mark.parametrize("opts", [dict(tile_n=128), dict(tile_n=64), dict(b_stages=4, a_stages=2),
                                  dict(row_units=1), dict(max_ctas=7)],
                         ids=["tile128", "tile64", "stages4x2", "single_rows", "grid7"])
def test_k_multiple_of_64_fused_with_other_options(O, opts, K):
    """A raw-scale FUSED plan with K % 256 != 0 runs the kernels whose scale
    producer copies the raw rows: the widest-tile kernel with its default
    ring depths, whatever tile width or depths the options ask for (the tile
    width still caps the tiles). Scale rows of 76 bytes go in 4-byte
    pieces, rows of 72 bytes in 16- and 8-byte pieces by row class. Every
    option must still give the oracle's result, and the plan must say which
    kernel configuration it runs."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    from gpu_util import run_gpu
    prob = synth.make_problem("custom", seed=1300, M=[300, 64, 129, 17], N=520, K=K)
    with nb.GroupedGemm(prob.M, prob.N, prob.K, **opts) as gg:
        info = gg.info()
        assert (info.sf_path, info.kernels_per_run) == (nb.NVFP4_SF_FUSED, 1)
        assert (info.b_stages, info.a_stages) == (3, 3)
        assert info.tile_n == opts.get("tile_n", 256)
    ref, _ = O.grouped(prob)
    got = run_gpu(prob, **opts)
    for g in range(prob.G):
        assert not np.isnan(got[g]).any(), f"group {g}: an element was never written"
        assert_close(got[g], ref[g], f"{opts} group {g}")


def test_k_multiple_of_64_uniform_and_exact(O):
    """One K for every group (nvfp4_ggemm_plan), K = 704 = 2 x 256 + 192,
    with power-of-two scales of span 4 so that every fp32 partial sum is
    exact: the GPU must equal the oracle bit for bit."""
    from gpu_util import run_gpu
    prob = synth.make_problem("custom", seed=1100, M=[140, 64, 0, 300], N=392, K=704)
    rng = np.random.default_rng(1100)
    for g in range(prob.G):
        # E4M3 codes of 2^e, e in [-2, 1]: (e + 7) << 3
        prob.SFA[g] = (((rng.integers(-2, 2, prob.SFA[g].shape) + 7) << 3)).astype(np.uint8)
        prob.SFB[g] = (((rng.integers(-2, 2, prob.SFB[g].shape) + 7) << 3)).astype(np.uint8)
    ref, _ = O.grouped(prob)
    got = run_gpu(prob)
    for g in range(prob.G):
        assert np.array_equal(got[g].view(np.uint16), ref[g].view(np.uint16)), f"group {g}"


@pytest.mark.parametrize("path,cached", [("fused", False), ("fused", True), ("relayout", False)])
def test_k_multiple_of_64_mixed_with_256_bit_exact(O, path, cached):
    """One plan whose groups mix K_g % 256 == 0 and K_g % 256 != 0 (on the
    FUSED path the scale producer loads the first kind by TMA and copies the
    second with its lanes, K_g % 128 == 0 in 8-byte pieces and the rest in
    4-byte ones; on the RELAYOUT path all are re-laid out), M_g % 4 != 0 and
    M_g < 4, with power-of-two scales of span 4 so that every fp32 partial
    sum is exact: the GPU must equal the oracle bit for bit, every row of
    every group."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    shapes = [(141, 392, 704), (3, 64, 320), (66, 256, 512), (299, 128, 1088), (7, 520, 64), (130, 200, 1024)]
    parts = [synth.make_problem("custom", seed=1200 + g, M=[m], N=n, K=k) for g, (m, n, k) in enumerate(shapes)]
    rng = np.random.default_rng(1200)
    for p in parts:
        p.SFA[0] = (((rng.integers(-2, 2, p.SFA[0].shape) + 7) << 3)).astype(np.uint8)
        p.SFB[0] = (((rng.integers(-2, 2, p.SFB[0].shape) + 7) << 3)).astype(np.uint8)
    with nb.GroupedGemm([p.M[0] for p in parts], [p.N for p in parts], [p.K for p in parts], sf_path=path) as gg:
        want = (nb.NVFP4_SF_RELAYOUT, 2) if path == "relayout" else (nb.NVFP4_SF_FUSED, 1)
        assert (gg.info().sf_path, gg.info().kernels_per_run) == want
    got = _run(parts, sf_path=path, cache_b_scales=cached)
    for g, p in enumerate(parts):
        ref, _, _ = O.group_gemm(p.A[0], p.B[0], p.SFA[0], p.SFB[0], p.K)
        assert np.array_equal(got[g].view(np.uint16), ref.view(np.uint16)), f"group {g} {shapes[g]}"


@pytest.mark.parametrize("layout", ["raw", "atom"])
def test_batched_groups_match_the_oracle(O, layout):
    """nvfp4_ggemm_plan_batched / run_batched: every group is `batch`
    independent problems laid out [batch][rows][cols], one pointer per group
    and a byte stride per operand. C's batches are padded apart; the padding
    must keep its sentinel. K_g % 256 != 0 in one group (its raw scale rows
    copied by the scale producer's lanes)."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    shapes = [(100, 256, 512), (0, 128, 256), (200, 520, 320), (33, 64, 1024)]
    L = 3
    probs = [[synth.make_problem("custom", seed=1200 + 10 * g + b, M=[m], N=n, K=k) for b in range(L)]
             for g, (m, n, k) in enumerate(shapes)]
    dev = lambda arrs: torch.from_numpy(np.ascontiguousarray(np.stack(arrs))).cuda()
    A = [dev([q.A[0] for q in ps]) for ps in probs]
    B = [dev([q.B[0] for q in ps]) for ps in probs]
    SFA = [dev([q.SFA[0] for q in ps]) for ps in probs]
    SFB = [dev([q.SFB[0] for q in ps]) for ps in probs]
    if layout == "atom":
        SFA = [torch.stack([atom_copy(s[b], m, k) for b in range(L)]) for s, (m, n, k) in zip(SFA, shapes)]
        SFB = [torch.stack([atom_copy(s[b], n, k) for b in range(L)]) for s, (m, n, k) in zip(SFB, shapes)]
    pad = 64  # fp16 elements between C batches
    Cbuf = [torch.full((L * (m * n + pad) + 8,), -3.0, dtype=torch.float16, device="cuda") for m, n, k in shapes]
    strides = []
    for g, (m, n, k) in enumerate(shapes):
        strides += [A[g][0].numel(), B[g][0].numel(), SFA[g][0].numel(), SFB[g][0].numel(), 2 * (m * n + pad)]
    with nb.GroupedGemm([m for m, _, _ in shapes], [n for _, n, _ in shapes], [k for _, _, k in shapes],
                        batch=L, sf_layout=layout) as gg:
        gg.run_batched(A, B, SFA, SFB, Cbuf, strides)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
        with pytest.raises(nb.Nvfp4Error):
            gg.run_batched(A, B, SFA, SFB, Cbuf, [s + 8 if i == 4 else s for i, s in enumerate(strides)])
    torch.cuda.synchronize()
    for g, (m, n, k) in enumerate(shapes):
        buf = Cbuf[g].cpu().numpy()
        for b in range(L):
            off = b * (m * n + pad)
            if m:
                q = probs[g][b]
                ref, _, _ = O.group_gemm(q.A[0], q.B[0], q.SFA[0], q.SFB[0], k)
                assert_close(buf[off:off + m * n].reshape(m, n), ref, f"group {g} batch {b}")
            assert (buf[off + m * n:off + m * n + pad] == -3.0).all(), f"group {g} batch {b}: padding written"


def test_bound_host_call_equals_run_host_bitwise():
    """GroupedGemm.bind_host: nvfp4_ggemm_run_host on host buffers marshalled
    once, called twice, equals the device-buffer call bit for bit."""
    from block_scaled_fp4_grouped_gb300 import binding as nb
    from gpu_util import run_gpu
    prob = synth.make_problem("custom", seed=950, M=[200, 0, 64], N=320, K=512)
    dense = run_gpu(prob)
    A = [np.ascontiguousarray(a) for a in prob.A]
    B = [np.ascontiguousarray(b) for b in prob.B]
    SFA = [np.ascontiguousarray(a) for a in prob.SFA]
    SFB = [np.ascontiguousarray(b) for b in prob.SFB]
    C = [np.full((m, prob.N), np.nan, np.float16) for m in prob.M]
    with nb.GroupedGemm(prob.M, prob.N, prob.K) as gg:
        call = gg.bind_host(A, B, SFA, SFB, C)
        call()
        call()
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    for g in range(prob.G):
        assert np.array_equal(C[g].view(np.uint16), dense[g].view(np.uint16))


def test_run_host_pinned_buffers_through_the_sms_bitwise():
    """run_host on pinned host tensors: one launch moves every input over the
    host link into the plan's buffers and one moves C back (SM loads and
    stores of host memory the GPU can address). Equal, bit for bit, to the
    device-buffer call; unaligned host views fall back to one copy per
    buffer and must give the same result."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    parts = [synth.make_problem("custom", seed=960 + g, M=[m], N=n, K=k)
             for g, (m, n, k) in enumerate([(200, 328, 768), (0, 512, 512), (64, 4096, 256), (17, 8, 320)])]
    M = [p.M[0] for p in parts]
    N = [p.N for p in parts]
    K = [p.K for p in parts]
    pin = lambda arrs: [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in arrs]
    A, B = pin([p.A[0] for p in parts]), pin([p.B[0] for p in parts])
    SFA, SFB = pin([p.SFA[0] for p in parts]), pin([p.SFB[0] for p in parts])
    dense = _run(parts)  # the same plan shapes on device buffers
    C = [torch.full((m, n), float("nan"), dtype=torch.float16).pin_memory() for m, n in zip(M, N)]
    with nb.GroupedGemm(M, N, K) as gg:
        call = gg.bind_host(A, B, SFA, SFB, C)
        call()
        call()
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
        for g in range(len(M)):
            assert np.array_equal(C[g].numpy().view(np.uint16), dense[g].view(np.uint16)), f"group {g}"
        # the same problem from host views that start 8 bytes in: one copy per buffer
        big = [torch.zeros(a.numel() + 16, dtype=torch.uint8).pin_memory() for a in A]
        A2 = []
        for b, a in zip(big, A):
            b[8:8 + a.numel()] = a.reshape(-1)
            A2.append(b[8:8 + a.numel()].view(a.shape))
        C2 = [torch.full((m, n), float("nan"), dtype=torch.float16).pin_memory() for m, n in zip(M, N)]
        gg.run_host(A2, B, SFA, SFB, C2)
        for g in range(len(M)):
            assert np.array_equal(C2[g].numpy().view(np.uint16), dense[g].view(np.uint16)), f"unaligned, group {g}"
