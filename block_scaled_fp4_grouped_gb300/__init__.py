"""NVFP4 block-scaled grouped GEMM for GB300 (sm_103a).

The compute lives in the C-ABI library `libnvfp4_ggemm.so` (CUDA kernels
with inline PTX, host plan/run logic in C++); `binding` marshals arguments
to it. `synth` draws the seeded synthetic workloads.
"""
