// A grouped-GEMM entry point that allocates nothing, for callers that may
// not call cudaMalloc: code running under a fixed memory budget or a custom
// device allocator, code inside a region where allocation would
// synchronise the device, plugins that must not grow the process's device
// footprint. The work it needs beyond the caller's inputs and outputs (the
// per-group tensor maps the kernel reads and the device error word) lives in
// one file-scope device array that every GPU loading the library holds
// until the process exits. It runs the same persistent GEMM kernel as
// nvfp4_ggemm_run on the raw-scale FUSED path with its default tiles.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "ggemm_internal.h"
#include "nvfp4_ggemm.h"

namespace nvfp4 {
namespace {

constexpr int kNoAllocMaxGroups = 64;
constexpr size_t kTableBytes = sizeof(GroupDesc) * kNoAllocMaxGroups;          // 104 KB
constexpr size_t kPrefixOffset = kTableBytes;                                   // int32[G+1]
constexpr size_t kErrOffset = kPrefixOffset + 512;                              // uint32 error word
constexpr size_t kScratchBytes = kErrOffset + 256;
static_assert(sizeof(int32_t) * (kNoAllocMaxGroups + 1) <= 512, "prefix area");
static_assert(kScratchBytes <= 112 * 1024, "the array stays within 112 KB");

// The scratch: problem table, chunk prefix sums, error word (the CTA start
// records travel in the kernel parameters). In host code this
// name is only a host-side stand-in; the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
uint8_t *g_scratch_addr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

bool aligned16_p(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The default raw-scale kernels: pairs of row tiles and single row tiles,
// each without and with the lane copies of raw scale rows (K % 256 != 0).
int noalloc_variant(int unit, bool lanes) { return ggemm_variant_index(kMaxTileN, 0, 0, true, unit, lanes); }

// First call on a device (that device current): look up the scratch array's
// device address, raise the shared-memory limit of the four kernels, fetch
// the tensor-map encoder.
nvfp4_status_t setup_device(int dev)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev]) return NVFP4_OK;
    if (!tensor_map_encoder()) return NVFP4_ERR_CUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NVFP4_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    for (int unit = 1; unit <= 2; ++unit)
        for (int lanes = 0; lanes < 2; ++lanes)
            if (ggemm_configure(noalloc_variant(unit, lanes != 0)) != cudaSuccess) return NVFP4_ERR_CUDA;
    g_sm_count[dev] = sms;
    g_scratch_addr[dev] = static_cast<uint8_t *>(ptr);
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" NVFP4_API nvfp4_status_t nvfp4_ggemm_run_noalloc(int num_groups, const int32_t *M, int32_t N, int32_t K,
                                                             const void *const *A, const void *const *B,
                                                             const void *const *SFA, const void *const *SFB,
                                                             void *const *C, void *stream, uint32_t *status_out)
{
    if (status_out) *status_out = 0;
    // --- arguments (nothing is enqueued before these pass)
    if (num_groups < 1 || !M || !A || !B || !SFA || !SFB || !C) return NVFP4_ERR_INVALID_ARG;
    if (num_groups > kNoAllocMaxGroups) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (N < 8 || N > (1 << 20) || N % 8 != 0 || K < 64 || K > (1 << 18) || K % 64 != 0)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    for (int g = 0; g < num_groups; ++g) {
        if (M[g] < 0 || M[g] > (1 << 20)) return NVFP4_ERR_INVALID_ARG;
        if (M[g] == 0) continue;
        if (!A[g] || !B[g] || !SFA[g] || !SFB[g] || !C[g]) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16_p(A[g]) || !aligned16_p(B[g]) || !aligned16_p(SFA[g]) || !aligned16_p(SFB[g]) ||
            !aligned16_p(C[g]))
            return NVFP4_ERR_ALIGNMENT;
    }
    const bool lanes = K % 256 != 0;  // scale rows the TMA cannot load: the scale producer copies them
    const int variant2 = noalloc_variant(2, lanes);
    const int variant1 = noalloc_variant(1, lanes);
    if (variant2 < 0 || variant1 < 0 || noalloc_variant(2, !lanes) < 0 || noalloc_variant(1, !lanes) < 0)
        return NVFP4_ERR_CUDA;

    // --- a call made while `stream` is being captured into a graph is refused
    //     before anything is enqueued: the copy below reads a host buffer
    //     that later calls rewrite
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    if (capture != cudaStreamCaptureStatusNone) return NVFP4_ERR_INVALID_ARG;

    // --- device and one-time set-up
    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    }
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return NVFP4_ERR_UNSUPPORTED_DEVICE;
    nvfp4_status_t st = setup_device(dev);
    if (st != NVFP4_OK) {
        cudaGetLastError();
        return st;
    }
    uint8_t *scratch = g_scratch_addr[dev];

    // --- schedule and tensor maps, built in a host buffer of this thread
    alignas(128) static thread_local uint8_t table[kTableBytes + 512];
    std::memset(table, 0, sizeof(table));
    auto *groups = reinterpret_cast<GroupDesc *>(table);
    auto *prefix = reinterpret_cast<int32_t *>(table + kPrefixOffset);
    const int n_chunks = ceil_div_i(N, kChunkN);
    GroupShape shapes[kNoAllocMaxGroups];
    long most = 0;
    for (int g = 0; g < num_groups; ++g) {
        shapes[g] = group_shape(M[g], N, K);
        most += (long)shapes[g].m_tiles * n_chunks;
    }
    if (most > 0x7FFFFFFF) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    // the same units of work a plan with default options would use
    const int cap_single = kMaxTileN / kChunkN;
    const int cap_pair = pair_cap_chunks(kMaxTileN);
    const int max_ctas = std::min(g_sm_count[dev], kMaxCtas);
    const UnitChoice uc = choose_units(shapes, num_groups, cap_single, cap_pair, max_ctas, 0);
    long total = 0;
    for (int g = 0; g < num_groups; ++g) {
        GroupDesc &d = groups[g];
        d.M = M[g];
        d.m_tiles = ceil_div_i(M[g], kTileM);
        d.m_units = ceil_div_i(d.m_tiles, uc.unit);
        d.chunk_begin = (int32_t)total;
        prefix[g] = (int32_t)total;
        total += (long)d.m_units * n_chunks;
        if (M[g] == 0) continue;
        if (!fill_group_desc(d, M[g], N, K, A[g], B[g], SFA[g], SFB[g], C[g], true, uc.unit))
            return NVFP4_ERR_CUDA;
        d.chunk_begin = prefix[g];
    }
    prefix[num_groups] = (int32_t)total;
    if (total == 0) return NVFP4_OK;
    int32_t cta_begin[kMaxCtas + 1];
    int32_t counts[kMaxCtas];
    const int grid = schedule_ctas(shapes, num_groups, uc.unit, cap_single, cap_pair, max_ctas, cta_begin, counts);
    if (grid < 1) return NVFP4_OK;
    CtaRange ranges[kMaxCtas];
    fill_cta_ranges(ranges, cta_begin, grid, prefix, shapes, num_groups, uc.unit, cap_single, cap_pair);

    // --- upload (pageable source: the copy call returns once the bytes are
    //     staged, so the buffer may be rewritten by the next call), clear the
    //     error word, launch
    const size_t used = sizeof(GroupDesc) * (size_t)num_groups;
    if (cudaMemcpyAsync(scratch, table, used, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(scratch + kPrefixOffset, prefix, sizeof(int32_t) * (size_t)(num_groups + 1),
                        cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemsetAsync(scratch + kErrOffset, 0, sizeof(uint32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    GemmParams gp{};
    for (int g = 0; g < std::min(num_groups, kParamGroups); ++g) gp.pmaps[g] = groups[g].maps;
    gp.groups = reinterpret_cast<const GroupDesc *>(scratch);
    gp.chunk_prefix = reinterpret_cast<const int32_t *>(scratch + kPrefixOffset);
    pack_cta_starts(gp.cta, ranges, grid, (int)total, shapes);
    order_ctas(gp.order, ranges, grid, prefix, shapes, uc.unit, cap_single, cap_pair);
    gp.err = reinterpret_cast<uint32_t *>(scratch + kErrOffset);
    gp.timeout_ns = 2000000000ull;
    gp.G = num_groups;
    gp.cap_single = cap_single;
    gp.cap_pair = cap_pair;
    gp.debug_skip_load = 0;
    gp.split_acc = uc.split ? 1 : 0;
    if (ggemm_launch(uc.unit == 1 ? variant1 : variant2, gp, grid, s, false) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }

    // --- optional: wait and report the device error word
    if (status_out) {
        uint32_t word = 0;
        if (cudaStreamSynchronize(s) != cudaSuccess ||
            cudaMemcpy(&word, scratch + kErrOffset, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
        *status_out = word;
        if (word != 0) return (word & 0xFFu) == NVFP4_ERR_TIMEOUT ? NVFP4_ERR_TIMEOUT : NVFP4_ERR_DEVICE_FAULT;
    }
    return NVFP4_OK;
}
