// Shared between the host plan code and the kernels: the device problem
// table, kernel parameters and launch entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kTileM = 128;  // rows of one MMA (cta_group::1, M = 128)
constexpr int kTileK = 256;  // k per pipeline stage: one 128-byte swizzle row of E2M1
constexpr int kMmaK = 64;    // k per tcgen05.mma of kind::mxf4nvf4
constexpr int kSfAtomBytes = 512;  // scales of 128 rows x 64 k

// Wait sites recorded in the error word (bits 8-15).
enum WaitSite : uint32_t {
    kSiteEmpty = 1,      // producer waiting for a free stage
    kSiteFull = 2,       // MMA (or scale permuter) waiting for loaded data
    kSiteSfReady = 3,    // MMA waiting for permuted scales
    kSiteAccEmpty = 4,   // MMA waiting for the epilogue to free TMEM
    kSiteAccFull = 5,    // epilogue waiting for the accumulator
    kSiteMmaDrain = 6,   // MMA thread waiting for its own tcgen05 work at exit
    kSiteLoadDrain = 7,  // producer waiting for its own loads at exit
};

// One entry of the device-resident problem table. Tensor maps must be
// 64-byte aligned (CUtensorMap itself is declared 128-byte aligned); every map describes one group's buffer exactly, so the
// TMA zero-fills rows past M_g / N on loads and drops them on stores.
struct alignas(128) GroupDesc {
    CUtensorMap tmA;    // A_g as bytes [M_g][K/2]; box 128 B x 128 rows; 128-byte swizzle
    CUtensorMap tmB;    // B_g as bytes [N][K/2];   box 128 B x BN rows;  128-byte swizzle
    CUtensorMap tmC;    // C_g fp16 [M_g][N];       box 64 x 32;          128-byte swizzle
    CUtensorMap tmSFA;  // raw SFA_g bytes [M_g][K/16]; box 16 B x 128 rows (fused path)
    CUtensorMap tmSFB;  // raw SFB_g bytes [N][K/16];   box 16 B x BN rows  (fused path)
    const uint8_t *sfa_atoms;  // atom-layout SFA_g (atom path)
    const uint8_t *sfb_atoms;  // atom-layout SFB_g (atom path)
    int32_t M;
    int32_t m_tiles;   // ceil(M / 128)
    int32_t m_groups;  // ceil(m_tiles / tiles per unit)
    int32_t unit_begin;
    int32_t pad[8];
};
static_assert(sizeof(GroupDesc) % 128 == 0, "GroupDesc must keep tensor maps 64-byte aligned");

struct GemmParams {
    const GroupDesc *groups;      // [G]
    const int32_t *unit_prefix;   // [G+1]: first work unit of each group
    uint32_t *err;                // device error word
    uint64_t timeout_ns;
    int32_t G, N, K;
    int32_t k_tiles;              // K / 256
    int32_t total_units;
    int32_t debug_skip_load;      // test-only fault injection (0 = off)
};

// One matrix for the scale re-layout kernel.
struct RelayoutJob {
    const uint8_t *src;  // raw [rows][K/16]
    uint8_t *dst;        // atoms
    int32_t rows;
    int32_t item_begin;  // prefix over jobs of ceil(rows/128) * (K/256)
};

struct RelayoutParams {
    const RelayoutJob *jobs;  // device array, or nullptr to use `single`
    RelayoutJob single;
    int32_t njobs;
    int32_t K;
    int32_t total_items;
};

// GEMM kernel variants (tile width, row tiles per unit, stages, scale path).
struct GemmVariant {
    int tile_n;
    int m_tiles;
    int stages;
    bool sf_raw;
};

// Returns the variant index for (tile_n, sf_raw), or -1.
int ggemm_variant_index(int tile_n, bool sf_raw);
GemmVariant ggemm_variant(int index);
int ggemm_smem_bytes(int index);
int ggemm_threads();
cudaError_t ggemm_configure(int index);  // raises the dynamic shared-memory limit (per device)
cudaError_t ggemm_launch(int index, const GemmParams &p, int grid, cudaStream_t stream);

cudaError_t relayout_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream);

}  // namespace nvfp4
