"""The allocation-free entry point, nvfp4_ggemm_run_noalloc.

Some callers cannot call cudaMalloc: code that runs under a fixed device
memory budget or hands all device memory to its own allocator, code inside a
region where an allocation would synchronise the device, plugins that must
not grow their host process's device footprint. This entry point serves
them: it keeps its tensor maps and error word in a static device array
instead of a plan. Here it is called through the C ABI two times in a row
on different problems, and each result is compared with the CPU oracle and
with the plan-based nvfp4_ggemm_run, within the tolerance the other GPU
tests use; two calls with K % 256 != 0 are checked against the oracle; a
call of the size of the largest workload (8 groups, K = 7168) is checked on
sampled entries; the device's free memory must not change
over several calls; and a call made while the stream is being captured into
a graph must be refused without enqueuing anything. This file is collected
last so that a run stopping at the first failure has already run every
other test."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, run_gpu, sample_indices, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


def _inputs(prob):
    import torch
    A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
    C = [torch.full((m, prob.N), float("nan"), dtype=torch.float16, device="cuda") for m in prob.M]
    return A, B, SFA, SFB, C


def _run_noalloc(prob, bufs=None):
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    A, B, SFA, SFB, C = bufs if bufs is not None else _inputs(prob)
    st, word = nb.nvfp4_ggemm_run_noalloc(prob.M, prob.N, prob.K, A, B, SFA, SFB, C, wait=True)
    assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    assert word == 0
    torch.cuda.synchronize()
    return [c.cpu().numpy() for c in C]


def test_noalloc_matches_oracle_and_plan_entry_on_two_calls_in_a_row():
    first = synth.make_problem("custom", seed=31, M=[1, 127, 129, 0, 200, 384, 64], N=328, K=768)
    second = synth.make_problem("c1", seed=32)
    got1 = _run_noalloc(first)
    got2 = _run_noalloc(second)
    O = oracle.get()
    for prob, got in ((first, got1), (second, got2)):
        want = run_gpu(prob)
        ref, _ = O.grouped(prob)
        for g in range(prob.G):
            assert got[g].shape == want[g].shape
            assert not np.isnan(got[g]).any(), "an output element was never written"
            assert_close(got[g], ref[g], f"{prob.name} group {g} against the oracle")
            assert_close(got[g], want[g], f"{prob.name} group {g} against nvfp4_ggemm_run")


@pytest.mark.parametrize("K", [704, 1152])
def test_noalloc_k_multiple_of_64_against_oracle(K):
    """K % 256 != 0: scale rows of 44 bytes (copied in 4-byte pieces) and of
    72 bytes (8-byte pieces), every element against the oracle."""
    prob = synth.make_problem("custom", seed=33, M=[130, 1, 0, 256, 77], N=200, K=K)
    got = _run_noalloc(prob)
    ref, _ = oracle.get().grouped(prob)
    for g in range(prob.G):
        assert not np.isnan(got[g]).any(), "an output element was never written"
        assert_close(got[g], ref[g], f"K={K} group {g}")


def test_noalloc_largest_workload_sampled_against_oracle():
    prob = synth.make_problem("c4", seed=0)
    got = _run_noalloc(prob)
    O = oracle.get()
    rng = np.random.default_rng(5)
    for g in range(prob.G):
        assert not np.isnan(got[g]).any(), "an output element was never written"
        rows, cols = sample_indices(prob.M[g], prob.N, 300, rng)
        want, _ = O.group_entries(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K, rows, cols)
        assert_close(got[g][rows, cols], want, f"c4 group {g}")


def test_noalloc_leaves_device_free_memory_unchanged():
    import torch
    probs = [synth.make_problem("custom", seed=50 + i, M=m, N=256, K=512)
             for i, m in enumerate(([64], [128, 0, 31], [300, 7, 64, 1]))]
    bufs = [_inputs(p) for p in probs]
    _run_noalloc(probs[0], bufs[0])  # first call on the device: its one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for p, b in zip(probs, bufs):
            _run_noalloc(p, b)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"


def test_noalloc_refuses_a_stream_being_captured():
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    prob = synth.make_problem("custom", seed=60, M=[64], N=256, K=256)
    A, B, SFA, SFB, C = _inputs(prob)
    _run_noalloc(prob, (A, B, SFA, SFB, C))
    x = torch.zeros(16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    statuses = []
    with torch.cuda.graph(graph):
        x.add_(1.0)
        statuses.append(nb.nvfp4_ggemm_run_noalloc(prob.M, prob.N, prob.K, A, B, SFA, SFB, C)[0])
    assert statuses == [nb.NVFP4_ERR_INVALID_ARG]
    graph.replay()
    torch.cuda.synchronize()
    assert float(x[0]) == 1.0
    # the entry point still works once the capture has ended
    _run_noalloc(prob, (A, B, SFA, SFB, C))


def test_noalloc_rejects_more_groups_than_its_array_holds():
    from block_scaled_fp4_grouped_gb300 import binding as nb
    G = 65
    st, _ = nb.nvfp4_ggemm_run_noalloc([64] * G, 256, 256, [0] * G, [0] * G, [0] * G, [0] * G, [0] * G)
    assert st == nb.NVFP4_ERR_INVALID_ARG or st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
    st, _ = nb.nvfp4_ggemm_run_noalloc([64] * G, 256, 256, [16] * G, [16] * G, [16] * G, [16] * G, [16] * G)
    assert st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
