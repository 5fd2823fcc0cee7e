// Shared between the host code and the kernels: the device problem table,
// kernel parameters and launch entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kTileM = 128;        // rows of one MMA (cta_group::1, M = 128)
constexpr int kTileK = 256;        // k per pipeline stage: one 128-byte swizzle row of E2M1
constexpr int kMmaK = 64;          // k per tcgen05.mma of kind::mxf4nvf4
constexpr int kSfAtomBytes = 512;  // scales of 128 rows x 64 k in the atom layout
constexpr int kChunkN = 32;        // scheduling grain along N (columns)
constexpr int kMaxTileN = 256;     // widest output tile any kernel variant supports
constexpr int kMaxCtas = 192;      // largest persistent grid (the CTA start records travel in the kernel parameters)
constexpr int kRowTilesPerUnit = 2;  // 128-row tiles of A that share every B stage
constexpr int kNumRowBoxes = 4;    // B / SFB box heights 32, 64, 128, 256 rows (32 << i)
constexpr int kSfKTiles = 2;       // k tiles (of 256) per raw-scale TMA box: 32 bytes of each scale row

// Operands a GEMM launch may load before the previous kernel of its stream
// has completed (GemmParams::early), because the caller declared that
// kernel does not write them; all others, and the C stores, wait for it.
constexpr int32_t kEarlyB = 1, kEarlySfb = 2, kEarlyA = 4, kEarlySfa = 8;

// Wait sites recorded in the error word (bits 8-15).
enum WaitSite : uint32_t {
    kSiteBEmpty = 1,     // B producer waiting for a free stage
    kSiteBFull = 2,      // MMA waiting for a B stage
    kSiteAEmpty = 3,     // A producer waiting for a free stage
    kSiteAFull = 4,      // MMA waiting for an A stage
    kSiteSfFree = 5,     // scale writers waiting for a scale buffer in TMEM
    kSiteSfReady = 6,    // MMA waiting for the scales of a stage
    kSiteAccEmpty = 7,   // MMA waiting for the epilogue to free the accumulator
    kSiteAccFull = 8,    // epilogue waiting for the accumulator
    kSiteMmaDrain = 9,   // MMA thread waiting for its own tcgen05 work at exit
    kSiteLoadDrain = 10, // a producer waiting for its own loads at exit
    kSiteSEmpty = 11,    // scale producer waiting for a free scale stage
    kSiteSFull = 12,     // scale writers waiting for a scale stage
    kSiteTileCheck = 13, // a tile larger than the CTA's ring slots (never expected)
    // device checks of the debug build (-DNVFP4_DEBUG), each guarding one
    // kind of operation; a failed check skips the operation
    kSiteCheckLoadB = 0x21,  // B stage load: shared-memory range, 1024-byte alignment, 16-byte x
    kSiteCheckLoadA = 0x22,  // A stage load: the same
    kSiteCheckLoadSf = 0x23, // scale stage loads: range inside the stage, source alignment
    kSiteCheckMma = 0x24,    // a stage's MMAs: accumulator and scale columns in TMEM, operand ranges
    kSiteCheckSfSt = 0x25,   // scale writers: TMEM scale-buffer columns
    kSiteCheckEpi = 0x26,    // epilogue: accumulator columns read, C row alignment of wide stores
};

// Timeline build (compiled with -DNVFP4_TRACE only; the library built for
// use has none of it): the kernel stores %globaltimer at the points below,
// one row of kTraceSlots per CTA, into the buffer GemmParams::trace names.
constexpr int kTraceSlots = 64;
enum TraceSlot : int {
    kTrStart = 0,        // CTA entry
    kTrPrologue = 1,     // after the prologue barrier (TMEM address known)
    kTrDepWait = 2,      // A producer: released by the previous kernel of the stream
    kTrBFirst = 3,       // B producer: first load issued
    kTrAFirst = 4,       // A producer: first load issued
    kTrSFirst = 5,       // scale producer: first load issued
    kTrMmaFirstData = 6, // MMA thread: first B stage landed
    kTrMmaFirstCommit = 7,
    kTrBLast = 8,        // B producer: last load issued
    kTrEnd = 9,          // CTA exit (after the final barrier)
    kTrTiles = 10,       // number of tiles the MMA thread walked
    kTrStages = 11,      // number of k stages the MMA thread issued
    kTrSfFirst = 12,     // scale writers: first TMEM scale buffer written
    kTrSmId = 13,        // the SM the CTA ran on (a value, not a time)
    kTrBarInit = 14,     // thread 0: barriers initialised
    kTrTmemAlloc = 15,   // warp 1: TMEM allocated
    kTrWalked = 57,      // the last producer lane at its first tile
    kTrTileMmaEnd = 16,  // + tile (< 8): last commit of the tile's MMAs
    kTrTileEpiStart = 24,// + tile: epilogue warp 2 saw the accumulator full
    kTrTileEpiEnd = 32,  // + tile: epilogue warp 2 released the accumulator
    kTrTileFirstData = 40, // + tile: MMA thread saw the tile's first B stage land
    kTrTileEpiEndAll = 48, // + tile: the last epilogue warp released the accumulator
};

// One entry of the device-resident problem table. Every tensor map
// describes one group's buffer exactly, so the TMA zero-fills rows past
// M_g / N_g (no memory traffic). A stage of a tile loads each operand with
// as few boxes as its row count allows: the tile's one or two 128-row tiles
// of A (and SFA) in one box of 128 or 256 rows, its 32c columns of B (and
// SFB) in the boxes of 256, 128, 64 and 32 rows that sum to 32c (at most
// three). Each TMA instruction costs issue time in the SM's copy unit, so
// few large boxes keep a CTA's stages at the memory's pace.
struct alignas(128) GroupMaps {
    CUtensorMap tmA[2];    // A_g bytes [M_g][K_g/2];  boxes 128 B x 128 / 256 rows; 128-byte swizzle
    CUtensorMap tmB[kNumRowBoxes];    // B_g bytes [N_g][K_g/2]; boxes 128 B x (32 << i) rows; 128-byte swizzle
    // raw scales: SFA_g [M_g][K_g/16], boxes 32 B x 128 / 256 rows; SFB_g
    // [N_g][K_g/16], boxes 32 B x (32 << i) rows. Atom layout: the atoms of one
    // k tile (4 x 512 B) of i + 1 consecutive 128-row blocks.
    CUtensorMap tmSFA[2];
    CUtensorMap tmSFB[kNumRowBoxes];
};
constexpr int kNumMaps = 2 + kNumRowBoxes + 2 + kNumRowBoxes;
static_assert(sizeof(GroupMaps) == kNumMaps * sizeof(CUtensorMap), "the maps are consecutive");

struct alignas(128) GroupDesc {
    GroupMaps maps;
    uint16_t *C;               // C_g fp16 [M_g][ldc], columns [0, N_g) written
    int32_t M;
    int32_t m_tiles;      // ceil(M / 128)
    int32_t m_units;      // ceil(m_tiles / row tiles per unit): passes over B
    int32_t chunk_begin;  // first scheduling chunk of this group (prefix sum)
    int32_t b_keep;       // 1: B is read by more than one unit of row tiles (keep it in L2)
    int32_t N;            // N_g
    int32_t k_tiles;      // ceil(K_g / 256)
    int32_t n_chunks;     // ceil(N_g / 32)
    int32_t ldc;          // row stride of C_g in elements (>= N_g, a multiple of 8)
    int32_t k_last;       // 64-k slices in the last k tile (1..4; 4 when K_g % 256 == 0)
    // raw scales whose rows (K_g/16 bytes) are not whole 16-byte units
    // (K_g % 256 != 0): no scale tensor maps; the scale producer's lanes copy
    // the rows from these pointers. sf_row_bytes = K_g/16 then, else 0.
    int32_t sf_row_bytes;
    int32_t sfb_tma;          // 1: SFB is a copy with rows padded to 16 bytes, loaded by TMA (tmSFB)
    const uint8_t *sfa_rows;  // SFA_g [M_g][K_g/16]
    const uint8_t *sfb_rows;  // SFB_g [N_g][K_g/16] (unused when sfb_tma)
};
static_assert(sizeof(GroupDesc) % 128 == 0, "GroupDesc must keep tensor maps 64-byte aligned");

// CTA c's chunk range and the group it starts in (host side).
struct alignas(32) CtaRange {
    int32_t begin, end;   // chunks [begin, end)
    int32_t g;            // group holding chunk `begin`
    int32_t g_base;       // chunk_prefix[g]
    int32_t g_tiles;      // m_tiles of group g
    int32_t max_chunks;   // widest tile the CTA will walk (sizes its B ring slots)
    int32_t max_rows;     // most row tiles in one of its tiles (sizes its A ring slots)
    int32_t g_rows;       // M of group g
};
static_assert(sizeof(CtaRange) == 32, "one sector per CTA");

// Per-group shape for the host scheduling helpers.
struct GroupShape {
    int32_t m_tiles;   // ceil(M_g / 128)
    int32_t n_chunks;  // ceil(N_g / 32)
    int32_t k_tiles;   // ceil(K_g / 256)
    int32_t M;
    int32_t k_last;    // 64-k slices in the last k tile (1..4)
};

// k tiles of 256 and 64-k slices in the last one, for K a multiple of 64.
inline int k_tiles_of(int K) { return (K + 255) / 256; }
inline int k_last_of(int K) { return (K / 64 - 1) % 4 + 1; }
inline GroupShape group_shape(int M, int N, int K)
{
    return GroupShape{(M + 127) / 128, (N + 31) / 32, k_tiles_of(K), M, k_last_of(K)};
}

// What a CTA needs to start, packed into 16 bytes of the kernel parameters
// so that no role reads memory before its first load. CTA c's range ends
// where CTA c + 1's begins (a sentinel follows the last CTA).
struct CtaStart {
    int32_t begin;    // first chunk
    int32_t g_base;   // chunk_prefix[g]
    uint32_t rows;    // group g: M (bits 0-20) | ceil(K / 256) (bits 21-31)
    uint32_t packed;  // g (bits 0-9) | widest tile in chunks - 1 (10-12) | most row tiles - 1 (13) |
                      // group g's 64-k slices in its last k tile - 1 (14-15) | group g's ceil(N / 32) (16-31)
};
static_assert(sizeof(CtaStart) == 16, "packed start record");

// The one packing of CtaStart's fields, used by the host and the kernel.
#if defined(__CUDACC__)
#define NVFP4_HD __host__ __device__ __forceinline__
#else
#define NVFP4_HD inline
#endif
NVFP4_HD uint32_t cta_pack_rows(int M, int k_tiles) { return (uint32_t)(M & 0x1FFFFF) | ((uint32_t)(k_tiles & 0x7FF) << 21); }
// max_chunks 1..8, max_rows 1..2, k_last 1..4 (a CTA with no tile packs 1s)
NVFP4_HD uint32_t cta_pack(int g, int max_chunks, int max_rows, int k_last, int n_chunks)
{
    return (uint32_t)(g & 0x3FF) | ((uint32_t)((max_chunks - 1) & 0x7) << 10) |
           ((uint32_t)((max_rows - 1) & 0x1) << 13) | ((uint32_t)((k_last - 1) & 0x3) << 14) |
           ((uint32_t)(n_chunks & 0xFFFF) << 16);
}
NVFP4_HD int cta_rows_m(uint32_t rows) { return (int)(rows & 0x1FFFFFu); }
NVFP4_HD int cta_rows_ktiles(uint32_t rows) { return (int)(rows >> 21); }
NVFP4_HD int cta_group(uint32_t packed) { return (int)(packed & 0x3FFu); }
NVFP4_HD int cta_max_chunks(uint32_t packed) { return (int)((packed >> 10) & 0x7u) + 1; }
NVFP4_HD int cta_max_rows(uint32_t packed) { return (int)((packed >> 13) & 0x1u) + 1; }
NVFP4_HD int cta_k_last(uint32_t packed) { return (int)((packed >> 14) & 0x3u) + 1; }
NVFP4_HD int cta_n_chunks(uint32_t packed) { return (int)(packed >> 16); }

// Work decomposition: a plan's units of work are pairs of 128-row tiles
// (unit 2; the last unit of a group with an odd tile count has one) or
// single row tiles (unit 1). Group g owns m_units_g * ceil(N_g/32) chunks (32
// columns of one unit), numbered after the chunks of groups 0..g-1
// (chunk_prefix), unit by unit; a unit is a "segment" of ceil(N_g/32) chunks.
// CTA c takes the chunk range [cta_begin[c], cta_begin[c+1]) and walks it as
// tiles inside one segment of up to cap_pair chunks (segments with two row
// tiles, whose accumulators share TMEM) or cap_single chunks (one row tile).
// The tensor maps of the first kParamGroups groups also travel in the
// kernel parameters: a map in parameter space needs no proxy fence before
// the TMA reads it (a map in global memory, written by a host copy, needs an
// acquire fence, a memory round trip that takes microseconds while the
// other SMs stream at full bandwidth).
constexpr int kParamGroups = 8;

struct GemmParams {
    GroupMaps pmaps[kParamGroups];  // maps of groups 0 .. min(G, kParamGroups) - 1
    const GroupDesc *groups;       // [G]
    const int32_t *chunk_prefix;   // [G+1]
    CtaStart cta[kMaxCtas + 1];    // [grid + 1]
    uint8_t order[kMaxCtas];       // block b walks range order[b] (a permutation of 0 .. grid - 1)
    uint32_t *err;                 // device error word
    uint64_t timeout_ns;
    int32_t G;
    int32_t cap_single;            // chunks per tile, one row tile (1..MAXN/32)
    int32_t cap_pair;              // chunks per tile, two row tiles
    int32_t debug_skip_load;       // test-only fault injection (0 = off)
    int32_t early;                 // kEarly* bits: operands loaded before the previous kernel completes
    int32_t debug_check_fail;      // debug build, test only: the check site forced to fail (0 = none)
    int32_t split_acc;             // kernels for single row tiles: 1 = a tile of at most half the
                                   // accumulator columns adds its even and odd 64-k slices into the
                                   // two halves, which the epilogue sums (two MMA chains, not one)
#ifdef NVFP4_TRACE
    unsigned long long *trace;     // [grid][kTraceSlots] timeline of this launch, or null
#endif
};

// Fills ranges[0..grid) from cta_begin[0..grid] and the group layout, walking
// each range exactly as the kernel does to bound its tiles; pack_cta_starts
// turns them into the kernel's start records (grid + 1 entries).
void fill_cta_ranges(CtaRange *ranges, const int32_t *cta_begin, int grid, const int32_t *chunk_prefix,
                     const GroupShape *shapes, int G, int unit, int cap_single, int cap_pair);
// Raw scale rows of K/16 bytes padded to a multiple of 16 bytes (a TMA row).
__host__ __device__ inline int sf_padded_row_bytes(int K) { return ((K / 16 + 15) / 16) * 16; }

void pack_cta_starts(CtaStart *out, const CtaRange *ranges, int grid, int total_chunks, const GroupShape *shapes);

// Which block walks which range: the ranges sorted by an estimate of their
// work, heaviest first. Blocks are placed on SMs in index order as the
// previous kernel's CTAs leave them, so the lowest indices start first and
// the heaviest ranges get the most time. The estimate counts the bytes a
// range moves through HBM (its B strip with SFB, its C) and, for each tile of
// two row tiles that another tile of the CTA follows, four times that tile's
// C: such a tile fills both accumulator halves, so the next tile's MMAs wait
// for its whole epilogue (timed on the GPU: the heaviest-first order matches
// or beats every input group order tried, by up to 1.2 us on the skinny
// 8-group shape).
void order_ctas(uint8_t *order, const CtaRange *ranges, int grid, const int32_t *chunk_prefix, const GroupShape *shapes,
                int unit, int cap_single, int cap_pair);

// The scale re-layout kernel's unit of work: 128 rows of a matrix by 16
// 32-bit words of each row (16 atoms, 1024 k).
constexpr int kRelayoutWords = 16;
constexpr int kRelayoutThreads = 128;
inline int relayout_items_of(int rows, int K) { return ((rows + 127) / 128) * ((K / 64 + kRelayoutWords - 1) / kRelayoutWords); }

// One matrix for the scale re-layout kernel.
struct RelayoutJob {
    const uint8_t *src;  // raw [rows][K/16]
    uint8_t *dst;        // atoms
    int32_t rows;
    int32_t K;           // a multiple of 64
    int32_t item_begin;  // prefix over jobs of relayout_items_of(rows, K)
    int32_t pad;
};

struct RelayoutParams {
    const RelayoutJob *jobs;  // device array, or nullptr to use `single`
    RelayoutJob single;
    int32_t njobs;
    int32_t total_items;
};

// GEMM kernel variants: widest tile, B ring depth, A ring depth, scale path,
// 128-row tiles per unit of work (each configuration is built for 2 and 1),
// and whether the scale producer's lanes copy raw scale rows the TMA cannot
// load (built for the default raw-scale configuration only).
struct GemmVariant {
    int max_n;
    int b_stages;
    int a_stages;
    bool sf_raw;
    int unit;
    bool lanes;
};

// Returns the variant index, or -1. b_stages / a_stages 0 pick the default
// depths for (max_n, sf_raw, unit, lanes).
int ggemm_variant_index(int max_n, int b_stages, int a_stages, bool sf_raw, int unit, bool lanes = false);
GemmVariant ggemm_variant(int index);
int ggemm_smem_bytes(int index);
int ggemm_threads();
cudaError_t ggemm_configure(int index);  // raises the dynamic shared-memory limit (per device)
// overlap_prev: launch with programmatic stream serialisation, so that the
// kernel's set-up overlaps the end of the previous kernel on the stream (the
// kernel waits for that kernel to complete before its first operand load).
cudaError_t ggemm_launch(int index, const GemmParams &p, int grid, cudaStream_t stream, bool overlap_prev);

cudaError_t relayout_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream);
// Copies raw scale rows into padded rows (the pad zero) for the jobs of p
// (item_begin: the prefix of rows over the jobs; dst rows of
// sf_padded_row_bytes(K) bytes).
cudaError_t sf_pad_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream);

// Host helpers shared by the plan path and the allocation-free entry point.

// Widest tile, in chunks, of a unit with two row tiles for a kernel whose
// widest tile is max_n columns (their accumulators share TMEM).
int pair_cap_chunks(int max_n);

// Splits the chunks of all segments (units of `unit` row tiles, group by
// group) into per-CTA ranges, written to cta_begin[0..grid], and returns grid
// (<= max_ctas <= kMaxCtas). With no more segments than max_ctas, every range
// lies inside one segment: the split takes the smallest per-CTA budget of
// k-stages (passes over K_g times ceil(K_g / 256)) that fits max_ctas CTAs, and
// spare CTAs then shorten the longest ranges; otherwise the chunks are split
// into equal contiguous ranges. counts is scratch for kMaxCtas ints.
int schedule_ctas(const GroupShape *shapes, int G, int unit, int cap_single, int cap_pair, int max_ctas,
                  int32_t *cta_begin, int32_t *counts);

// Row tiles per unit of work, and whether one-row-tile tiles split their
// accumulator, for a plan over these shapes. forced 2: pairs; forced 1:
// single row tiles; 0: pairs, unless their tiles would be at most four
// chunks wide (narrow tiles: the stage's MMA chains, not the bytes, set the
// pace) while single row tiles give every CTA one tile in no more k-stages
// than pairs do. split: single row tiles and every CTA walks one tile; the
// kernel then adds the even and odd 64-k slices of each such tile of at most
// half the accumulator columns into the two halves (one MMA waits for the
// previous one into the same accumulator, so two chains per stage take
// about half as long).
struct UnitChoice {
    int unit;
    bool split;
};
UnitChoice choose_units(const GroupShape *shapes, int G, int cap_single, int cap_pair, int max_ctas, int forced);
using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                       const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                       CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();  // nullptr when the driver has none

// Fills one table entry (tensor maps, pointers, counts) for group g with
// M_g > 0. sf_raw: encode the raw-scale maps; else the atom-layout maps.
// sfb_padded (raw scales): SFB is a copy whose rows are padded to
// sf_padded_row_bytes(K), loaded by TMA whatever K is.
bool fill_group_desc(GroupDesc &d, int M, int N, int K, const void *A, const void *B, const void *SFA,
                     const void *SFB, void *C, bool sf_raw, int unit, bool sfb_padded = false);

}  // namespace nvfp4
