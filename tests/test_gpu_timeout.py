"""Failure detection on the GPU without a GPU fault.

Every pipeline wait in the kernel is bounded by the plan's wait_timeout_ns.
The test-only option debug_skip_load makes the B producer of CTA 0 leave
one stage load unissued, so the MMA thread's wait for that stage (and then
the other waits of that CTA) run out: the kernel records (status, wait
site, block) in the device error word, every role leaves its loop, drains
its own asynchronous work, releases TMEM and returns. The host reads the
status with nvfp4_ggemm_sync_status, and the context stays usable: a plain
run afterwards matches the oracle."""
import numpy as np
import pytest

import oracle
from block_scaled_fp4_grouped_gb300 import synth
from gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_scaled_fp4_grouped_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def O():
    return oracle.get()


def _inputs(prob):
    import torch
    A, B, SFA, SFB = to_device(prob.A), to_device(prob.B), to_device(prob.SFA), to_device(prob.SFB)
    C = [torch.full((m, prob.N), float("nan"), dtype=torch.float16, device="cuda") for m in prob.M]
    return A, B, SFA, SFB, C


@pytest.mark.parametrize("row_units", [1, 2])
@pytest.mark.parametrize("skip", [1, 3])
def test_a_wait_that_runs_out_is_reported_and_the_context_survives(O, skip, row_units):
    """Both kernel families: single row tiles with split accumulators (the
    plan's own choice for this shape) and pairs of row tiles."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    prob = synth.make_problem("custom", seed=41, M=[200, 64, 0, 130], N=512, K=1024)
    A, B, SFA, SFB, C = _inputs(prob)
    with nb.GroupedGemm(prob.M, prob.N, prob.K, debug_skip_load=skip, wait_timeout_ns=20_000_000,
                        row_units=row_units) as gg:
        assert gg.info().row_units == row_units
        gg.run(A, B, SFA, SFB, C)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_ERR_TIMEOUT, (nb.nvfp4_status_string(st), hex(word))
        assert word & 0xFF == nb.NVFP4_ERR_TIMEOUT
        assert (word >> 8) & 0xFF in range(1, 14), hex(word)  # a documented wait site
        assert word >> 16 == 0, "only CTA 0 had a load left out"
        st, word = gg.sync_status()
        assert (st, word) == (nb.NVFP4_OK, 0), "the error word is cleared once read"
    torch.cuda.synchronize()
    # the same problem through a plain plan
    A, B, SFA, SFB, C = _inputs(prob)
    with nb.GroupedGemm(prob.M, prob.N, prob.K, row_units=row_units) as gg:
        gg.run(A, B, SFA, SFB, C)
        st, word = gg.sync_status()
        assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
    for g in range(prob.G):
        got = C[g].cpu().numpy()
        ref, _, _ = O.group_gemm(prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], prob.K)
        assert not np.isnan(got).any()
        assert_close(got, ref, f"group {g} after the timed-out run")
