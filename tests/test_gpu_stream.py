"""Back-to-back calls on one stream, through the C ABI.

A GEMM launched right after another kernel of its stream starts its set-up
while that kernel finishes (programmatic dependent launch) and must not load
an operand before that kernel has completed. Here the second GEMM reads, as
its A operand, the bytes the first GEMM writes to C (any byte is a valid
pair of E2M1 codes), so a load issued too early would see the previous
contents of that buffer. Both plans' tables are uploaded by a first round
of calls; the checked round changes the first GEMM's inputs with a torch
kernel and then enqueues both GEMMs with nothing between them, so both
launches overlap their predecessor. The expected values are the oracle's on
the bytes read back after the stream has drained. A second test does the same
for raw scales whose rows are not 16-byte units (K % 256 != 0), copied by the
GEMM's scale producer on the FUSED path and by the re-layout kernel ahead of
the GEMM on the RELAYOUT path: either must read scales a kernel wrote just
before it only after that kernel has completed."""
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


def _new_inputs(prob, seed):
    other = synth.make_problem("custom", seed=seed, M=prob.M, N=prob.N, K=prob.K)
    return other


@pytest.mark.parametrize("serial,b_static", [(False, False), (True, False), (False, True)],
                         ids=["overlapped", "plain", "overlapped_b_static"])
def test_second_gemm_reads_what_the_first_wrote(serial, b_static):
    """b_static (B and SFB never written by the previous kernel) lets a GEMM
    stream B before the previous kernel completes; A, which the previous
    kernel writes here, must still be read only after it."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    # first GEMM: one group, 256 x 4096 x 7168 (a few microseconds of work)
    p1 = synth.make_problem("custom", seed=41, M=[256], N=4096, K=7168)
    A1, B1, SFA1, SFB1 = to_device(p1.A), to_device(p1.B), to_device(p1.SFA), to_device(p1.SFB)
    C1 = [torch.zeros((256, 4096), dtype=torch.float16, device="cuda")]
    # second GEMM: A2 is the first 256 x 4096 bytes of C1 (K2 = 8192)
    p2 = synth.make_problem("custom", seed=42, M=[256], N=512, K=8192)
    A2 = [C1[0].view(torch.uint8).reshape(-1)[: 256 * 4096].view(256, 4096)]
    B2, SFA2, SFB2 = to_device(p2.B), to_device(p2.SFA), to_device(p2.SFB)
    C2 = [torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")]
    g1 = nb.GroupedGemm(p1.M, p1.N, p1.K, serial_launch=serial, b_static=b_static)
    g2 = nb.GroupedGemm(p2.M, p2.N, p2.K, serial_launch=serial, b_static=b_static)
    try:
        call1 = g1.bind(A1, B1, SFA1, SFB1, C1)
        call2 = g2.bind(A2, B2, SFA2, SFB2, C2)
        call1()
        call2()
        torch.cuda.synchronize()
        for rnd in range(3):
            q = _new_inputs(p1, 100 + rnd)
            a_new = torch.from_numpy(q.A[0]).cuda()
            sfa_new = torch.from_numpy(q.SFA[0]).cuda()
            torch.cuda.synchronize()
            # torch kernels write the first GEMM's new A and SFA, then both
            # GEMMs follow with nothing between them
            torch.bitwise_xor(a_new, 0, out=A1[0])
            torch.bitwise_xor(sfa_new, 0, out=SFA1[0])
            call1()
            call2()
            for gg in (g1, g2):
                st, word = gg.sync_status()
                assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
            c1 = C1[0].cpu().numpy()
            a2 = A2[0].cpu().numpy()
            c2 = C2[0].cpu().numpy()
            O = oracle.get()
            # the first GEMM used the new inputs (sampled entries)
            rng = np.random.default_rng(rnd)
            rows = rng.integers(0, 256, 300).astype(np.int32)
            cols = rng.integers(0, 4096, 300).astype(np.int32)
            want1, _ = O.group_entries(q.A[0], p1.B[0], q.SFA[0], p1.SFB[0], p1.K, rows, cols)
            assert_close(c1[rows, cols], want1, f"round {rnd}: first GEMM")
            # the second GEMM read the first GEMM's output of this round
            want2, _, _ = O.group_gemm(a2, p2.B[0], p2.SFA[0], p2.SFB[0], p2.K)
            assert not np.isnan(c2).any()
            assert_close(c2, want2, f"round {rnd}: second GEMM on the first GEMM's output")
    finally:
        g1.close()
        g2.close()


@pytest.mark.parametrize("path,cached", [("fused", False), ("fused", True), ("relayout", False), ("relayout", True)],
                         ids=["fused_lanes", "fused_lanes_cached_b_scales", "relayout", "relayout_cached_b_scales"])
def test_relayout_reads_scales_the_previous_kernel_wrote(path, cached):
    """K % 256 != 0: on the FUSED path the GEMM's scale producer copies the
    raw scale rows with its lanes; on the RELAYOUT path the re-layout kernel
    runs ahead of the GEMM. Each kernel is launched to overlap its
    predecessor. Here a torch kernel writes the
    second GEMM's A scales (from the first GEMM's output, masked to finite
    E4M3 codes) right before the call, so a scale copy that read its
    input before that kernel completed would see the previous contents."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    p1 = synth.make_problem("custom", seed=43, M=[256], N=4096, K=7168)
    A1, B1, SFA1, SFB1 = to_device(p1.A), to_device(p1.B), to_device(p1.SFA), to_device(p1.SFB)
    C1 = [torch.zeros((256, 4096), dtype=torch.float16, device="cuda")]
    K2 = 8128  # K % 256 == 192: raw scale rows of 508 bytes
    p2 = synth.make_problem("custom", seed=44, M=[256], N=512, K=K2)
    c1_bytes = C1[0].view(torch.uint8).reshape(-1)
    A2 = [c1_bytes[: 256 * K2 // 2].view(256, K2 // 2)]
    src_sfa = c1_bytes[1 << 20: (1 << 20) + 256 * K2 // 16].view(256, K2 // 16)
    SFA2 = [torch.zeros((256, K2 // 16), dtype=torch.uint8, device="cuda")]
    B2, SFB2 = to_device(p2.B), to_device(p2.SFB)
    C2 = [torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")]
    g1 = nb.GroupedGemm(p1.M, p1.N, p1.K)
    g2 = nb.GroupedGemm(p2.M, p2.N, K2, sf_path=path, cache_b_scales=cached)
    try:
        if path == "relayout":
            assert g2.info().sf_path == nb.NVFP4_SF_RELAYOUT and g2.info().kernels_per_run == 2
        else:
            assert g2.info().sf_path == nb.NVFP4_SF_FUSED and g2.info().kernels_per_run == 1
        if cached:
            g2.prepare_b_scales(SFB2)
        call1 = g1.bind(A1, B1, SFA1, SFB1, C1)
        call2 = g2.bind(A2, B2, SFA2, SFB2, C2)
        call1()
        call2()
        torch.cuda.synchronize()
        for rnd in range(3):
            q = _new_inputs(p1, 200 + rnd)
            a_new = torch.from_numpy(q.A[0]).cuda()
            torch.cuda.synchronize()
            torch.bitwise_xor(a_new, 0, out=A1[0])
            call1()
            # finite scale codes (sign 0, exponent <= 5) from the first GEMM's output
            torch.bitwise_and(src_sfa, 0x2F, out=SFA2[0])
            call2()
            for gg in (g1, g2):
                st, word = gg.sync_status()
                assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
            a2 = A2[0].cpu().numpy()
            sfa2 = SFA2[0].cpu().numpy()
            c2 = C2[0].cpu().numpy()
            want2, _, _ = oracle.get().group_gemm(a2, p2.B[0], sfa2, p2.SFB[0], K2)
            assert not np.isnan(c2).any()
            assert_close(c2, want2, f"round {rnd}: re-layout of scales the previous kernel wrote")
    finally:
        g1.close()
        g2.close()


def test_all_inputs_static_still_orders_the_c_stores():
    """b_static = 2: the caller declares that the kernel before the GEMM
    writes none of its inputs, so every load may start during that kernel's
    last CTAs, but the C stores must still wait for it. Here the kernel
    before the second GEMM (the first GEMM) reads, as its A operand, the
    buffer the second GEMM writes as C; a store issued too early would change
    what the first GEMM read. The second GEMM's inputs are written once, long
    before, so the declaration holds."""
    import torch
    from block_scaled_fp4_grouped_gb300 import binding as nb
    p2 = synth.make_problem("custom", seed=45, M=[256], N=4096, K=7168)
    A2, B2, SFA2, SFB2 = to_device(p2.A), to_device(p2.B), to_device(p2.SFA), to_device(p2.SFB)
    C2 = [torch.zeros((256, 4096), dtype=torch.float16, device="cuda")]
    # the first GEMM reads the first 256 x 4096 bytes of C2 as its A (K1 = 8192)
    p1 = synth.make_problem("custom", seed=46, M=[256], N=512, K=8192)
    A1 = [C2[0].view(torch.uint8).reshape(-1)[: 256 * 4096].view(256, 4096)]
    B1, SFA1, SFB1 = to_device(p1.B), to_device(p1.SFA), to_device(p1.SFB)
    C1 = [torch.full((256, 512), float("nan"), dtype=torch.float16, device="cuda")]
    g1 = nb.GroupedGemm(p1.M, p1.N, p1.K)
    g2 = nb.GroupedGemm(p2.M, p2.N, p2.K, b_static=2)
    O = oracle.get()
    try:
        call1 = g1.bind(A1, B1, SFA1, SFB1, C1)
        call2 = g2.bind(A2, B2, SFA2, SFB2, C2)
        call2()
        call1()
        torch.cuda.synchronize()
        want2, _, _ = O.group_gemm(p2.A[0], p2.B[0], p2.SFA[0], p2.SFB[0], p2.K)
        for rnd in range(3):
            # C2 is zeroed so that its next write changes the bytes the first GEMM reads
            C2[0].zero_()
            a1_before = A1[0].cpu().numpy().copy()
            call1()  # reads C2's bytes (zeros)
            call2()  # overwrites C2; its loads may start early, its stores may not
            for gg in (g1, g2):
                st, word = gg.sync_status()
                assert st == nb.NVFP4_OK, (nb.nvfp4_status_string(st), hex(word))
            want1, _, _ = O.group_gemm(a1_before, p1.B[0], p1.SFA[0], p1.SFB[0], p1.K)
            assert_close(C1[0].cpu().numpy(), want1, f"round {rnd}: the first GEMM read C2 before it was written")
            assert_close(C2[0].cpu().numpy(), want2, f"round {rnd}: the second GEMM with every input static")
    finally:
        g1.close()
        g2.close()
