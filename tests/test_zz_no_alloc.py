"""The allocation-free entry point, nvfp4_ggemm_run_noalloc.

It serves callers that may not allocate device memory (a fixed memory
budget, their own allocator, regions where an allocation would synchronise
the device): it keeps its tensor maps and error word in a static device
array instead of a plan. Here it is called through the C ABI twice in a
row, on different problems, and each result is compared with the plan-based
nvfp4_ggemm_run within the tolerance the other GPU tests use. This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import numpy as np
import pytest

from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


def _run_noalloc(prob):
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
    C = [torch.full((m, prob.N), float("nan"), dtype=torch.float16, device="cuda") for m in prob.M]
    st, word = nb.nvfp4_ggemm_run_noalloc(prob.M, prob.N, prob.K, A, B, SFA, SFB, C, wait=True)
    assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    assert word == 0
    torch.cuda.synchronize()
    return [c.cpu().numpy() for c in C]


def test_noalloc_matches_plan_entry_on_two_calls_in_a_row():
    first = synth.make_problem("custom", seed=31, M=[1, 127, 129, 0, 200, 384, 64], N=328, K=768)
    second = synth.make_problem("c1", seed=32)
    got1 = _run_noalloc(first)
    got2 = _run_noalloc(second)
    for prob, got in ((first, got1), (second, got2)):
        want = run_gpu(prob)
        for g in range(prob.G):
            assert got[g].shape == want[g].shape
            assert not np.isnan(got[g]).any(), "an output element was never written"
            assert_close(got[g], want[g], f"{prob.name} group {g}")


def test_noalloc_rejects_more_groups_than_its_array_holds():
    from block_scaled_fp4_grouped_gb300 import binding as nb
    G = 65
    st, _ = nb.nvfp4_ggemm_run_noalloc([64] * G, 256, 256, [0] * G, [0] * G, [0] * G, [0] * G, [0] * G)
    assert st == nb.NVFP4_ERR_INVALID_ARG or st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
    st, _ = nb.nvfp4_ggemm_run_noalloc([64] * G, 256, 256, [16] * G, [16] * G, [16] * G, [16] * G, [16] * G)
    assert st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
