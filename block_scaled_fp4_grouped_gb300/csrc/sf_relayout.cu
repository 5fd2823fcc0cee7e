// Scale re-layout: raw row-major E4M3 block scales [rows][K/16] into the
// tensor cores' atom layout, K/64 atoms of 512 bytes per 128-row block (the
// 128 x 4 scale-factor atom of the block-scaled MMA: byte 16 i + 4 j + c of
// an atom holds row i + 32 j, k-block c). The RELAYOUT path runs it before
// the GEMM; nvfp4_sf_relayout runs it alone.
#include <cstdint>

#include "ggemm_internal.h"

namespace nvfp4 {
namespace {

// One block of 4 warps per item = (matrix, 128-row block, 16 words of each
// row: 16 atoms). Each warp first finds the item's job with a 32-way search
// of the job table (one load per lane per level: one level for up to 32
// jobs). The warps read the block's rows into shared memory, each warp 32
// rows, half a warp per row with lane w taking 32-bit word w % 16 (64
// contiguous bytes of a row per half warp); every thread issues its 16 loads
// before it writes any, so an item costs one trip to memory. Then warp a
// writes atoms a, a + 4, a + 8 and a + 12: lane i gathers the words of rows
// i, i + 32, i + 64 and i + 96 and stores them as the atom's 16 bytes at
// 16 i, so every atom is one 512-byte coalesced store. Rows past `rows` are
// written as zero; words past K/64 (a last item narrower than 16 atoms) are
// not written.
__global__ void __launch_bounds__(kRelayoutThreads) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    constexpr int kWarps = kRelayoutThreads / 32;
    constexpr int kRowsPerWarp = kTileM / kWarps;
    __shared__ uint32_t tile[kTileM][kRelayoutWords + 1];  // + 1: conflict-free column reads
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
        RelayoutJob job;
        if (p.jobs == nullptr) {
            job = p.single;
        } else {
            // the last job whose item_begin <= item (jobs[lo] always qualifies)
            int lo = 0, n = p.njobs;
            while (n > 1) {
                const int step = (n + 31) / 32;
                const int idx = lo + lane * step;
                const bool ok = lane * step < n && p.jobs[idx].item_begin <= item;
                const int k = 31 - __clz(__ballot_sync(0xFFFFFFFFu, ok));
                lo += k * step;
                n = min(step, n - k * step);
            }
            job = p.jobs[lo];
        }
        const int words = job.K / 64;  // 32-bit words (atoms) per row; K is a multiple of 64
        const int per_block = (words + kRelayoutWords - 1) / kRelayoutWords;
        const int l = item - job.item_begin;
        const int rb = l / per_block;
        const int w0 = (l % per_block) * kRelayoutWords;
        const int nw = min(kRelayoutWords, words - w0);
        const size_t row_bytes = (size_t)(job.K / 16);
        const int col = lane & 15;
        const int r0 = warp * kRowsPerWarp + (lane >> 4);
        uint32_t v[kRowsPerWarp / 2];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp / 2; ++i) {
            const int row = rb * kTileM + r0 + 2 * i;
            v[i] = 0;
            if (row < job.rows && col < nw)
                v[i] = __ldg(reinterpret_cast<const uint32_t *>(job.src + (size_t)row * row_bytes) + w0 + col);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp / 2; ++i) tile[r0 + 2 * i][col] = v[i];
        __syncthreads();
        for (int a = warp; a < nw; a += kWarps)
            *reinterpret_cast<uint4 *>(job.dst + ((size_t)rb * words + w0 + a) * kSfAtomBytes + 16 * lane) =
                make_uint4(tile[lane][a], tile[lane + 32][a], tile[lane + 64][a], tile[lane + 96][a]);
        __syncthreads();
    }
}

// One warp per row of one job: the row's K/16 raw bytes as 4-byte words,
// then zero words up to sf_padded_row_bytes(K). The job is found by a
// 32-way search of the job table as above.
__global__ void __launch_bounds__(256) sf_pad_kernel(const __grid_constant__ RelayoutParams p)
{
    const int lane = threadIdx.x & 31;
    const int warps = (int)(blockDim.x >> 5);
    for (int item = blockIdx.x * warps + (int)(threadIdx.x >> 5); item < p.total_items; item += gridDim.x * warps) {
        int lo = 0, n = p.njobs;
        while (n > 1) {
            const int step = (n + 31) / 32;
            const int idx = lo + lane * step;
            const bool ok = lane * step < n && p.jobs[idx].item_begin <= item;
            const int k = 31 - __clz(__ballot_sync(0xFFFFFFFFu, ok));
            lo += k * step;
            n = min(step, n - k * step);
        }
        const RelayoutJob job = p.jobs[lo];
        const int r = item - job.item_begin;
        const int in_words = job.K / 64;  // K/16 bytes, a multiple of 4
        const int out_words = sf_padded_row_bytes(job.K) / 4;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(job.src + (size_t)r * (size_t)(job.K / 16));
        uint32_t *dst = reinterpret_cast<uint32_t *>(job.dst + (size_t)r * (size_t)sf_padded_row_bytes(job.K));
        for (int w = lane; w < out_words; w += 32) dst[w] = w < in_words ? __ldg(src + w) : 0u;
    }
}

}  // namespace

cudaError_t sf_pad_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream)
{
    if (p.total_items <= 0 || p.jobs == nullptr) return cudaSuccess;
    const int warps = 8;
    int blocks = (p.total_items + warps - 1) / warps;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    sf_pad_kernel<<<blocks, warps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t relayout_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream)
{
    if (p.total_items <= 0) return cudaSuccess;
    const int cap = sm_count * 16;  // 9 KB of shared memory and 128 threads a block: 16 fit an SM
    const int blocks = p.total_items < cap ? p.total_items : cap;
    sf_relayout_kernel<<<blocks, kRelayoutThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
