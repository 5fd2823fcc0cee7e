// Host <-> device copies for nvfp4_ggemm_run_host through the SMs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

// Copies between host memory the GPU can address (pinned, mapped) and
// device memory, all in one launch: the SMs move every job's bytes over the
// host link (as fast as the copy engine there), without a copy engine's
// per-copy set-up. src and dst of a job are 16-byte aligned.
constexpr int kMaxIoJobs = 96;
struct IoJob {
    const uint8_t *src;
    uint8_t *dst;
    uint64_t bytes;
};
struct IoCopyParams {
    IoJob jobs[kMaxIoJobs];
    int32_t njobs;
};
cudaError_t io_copy_launch(const IoCopyParams &p, int sm_count, cudaStream_t stream);

}  // namespace nvfp4
