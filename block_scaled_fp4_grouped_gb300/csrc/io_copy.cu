// Host <-> device copies for nvfp4_ggemm_run_host: the SMs load host memory
// the GPU can address (pinned, mapped) and store it to device memory, or the
// reverse, for every job of a call in one launch.
#include "io_copy.h"

namespace nvfp4 {
namespace {

// Every block takes part in every job: 16-byte units by grid stride, the
// job's last bytes (fewer than 16) by its first threads.
__global__ void __launch_bounds__(256) io_copy_kernel(const __grid_constant__ IoCopyParams p)
{
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    for (int j = 0; j < p.njobs; ++j) {
        const IoJob job = p.jobs[j];
        const uint64_t n16 = job.bytes / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(job.src);
        uint4 *d = reinterpret_cast<uint4 *>(job.dst);
        uint64_t i = tid;
        for (; i + 3 * nthreads < n16; i += 4 * nthreads) {
            const uint4 a = s[i], b = s[i + nthreads], c = s[i + 2 * nthreads], e = s[i + 3 * nthreads];
            d[i] = a;
            d[i + nthreads] = b;
            d[i + 2 * nthreads] = c;
            d[i + 3 * nthreads] = e;
        }
        for (; i < n16; i += nthreads) d[i] = s[i];
        const uint64_t tail = job.bytes - 16 * n16;
        if (tid < tail) job.dst[16 * n16 + tid] = job.src[16 * n16 + tid];
    }
}

}  // namespace

cudaError_t io_copy_launch(const IoCopyParams &p, int sm_count, cudaStream_t stream)
{
    if (p.njobs <= 0) return cudaSuccess;
    io_copy_kernel<<<sm_count * 4, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
