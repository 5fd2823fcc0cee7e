// Device code: the persistent warp-specialised NVFP4 grouped GEMM, for
// sm_103a (the scale re-layout kernel is in sf_relayout.cu).
//
// GEMM structure (one CTA per SM, persistent, 16 warps):
//   warp 0      B producer: per 256-k stage, TMA loads of the tile's B rows
//               (128-byte swizzle) into the B ring. B is the operand streamed
//               from HBM; a slot holds nothing else, so it is refilled as
//               soon as its MMAs have read it.
//   warp 6      A producer: the tile's one or two 128-row A tiles (one box
//               each; rows past M_g are the TMA's zero fill) into the A
//               ring; A is small and re-read from L2.
//   warp 7      scale producer: the stage's A and B scales into a ring of NS
//               small stages, running ahead of the operands.
//   warps 8-11  scale writers: each gathers a scale stage from shared memory
//               into the TMEM layout the block-scaled MMA reads (32 lanes x
//               4 columns per 128 rows, the same in every lane quarter), then
//               waits for one of two TMEM scale buffers and writes its
//               quarter with tcgen05.st. Raw row-major and atom-layout
//               scales are both handled here, off the tensor pipe and ahead
//               of the MMAs.
//   warp 1      allocates TMEM; one lane issues kind::mxf4nvf4 block16 MMAs
//               (M = 128 per row tile, N = tile width up to MAXN) into fp32
//               accumulators, then commits one stage-completion barrier that
//               frees the stage's A and B slots and its TMEM scale buffer.
//               The accumulator columns are two halves: a one-row-tile tile
//               of at most 192 columns takes one, alternating, so its MMAs
//               overlap the previous tile's epilogue.
//   warps 2-5,  epilogue: tcgen05.ld of the accumulators (lane quarter
//   12-15       warp % 4; the two warps of a quarter split the 32-column
//               blocks), RN to fp16, 32- or 16-byte stores of each row
//               straight to C.
// The producer lanes walk to their first tile before the prologue barrier.
// Work: group g owns m_units_g x ceil(N_g/32) chunks (32 columns of one unit
// of work: a pair of 128-row tiles, or one row tile when the plan chooses
// single row tiles); the chunks of all groups are numbered through prefix
// sums, and the host gives every CTA a contiguous chunk range (its start
// record travels in the kernel parameters). A CTA walks its range as tiles
// inside one unit: up to 192 columns when the unit has two row tiles (their
// accumulators share TMEM) and up to MAXN when it has one. Both row tiles of
// a pair share every B stage, so each B strip is read from HBM once, by one
// SM. With single row tiles (the UNIT = 1 instances) and one tile per CTA
// (split_acc), a tile of at most 192 columns adds its even and odd 64-k
// slices into the two accumulator halves, and the epilogue sums them: an
// MMA waits for the previous one into the same accumulator, so two chains
// halve that wait. The host keeps every range inside one unit when it can
// and picks the smallest per-CTA budget of k-stages that fits the grid, so a
// CTA streams its B strip in as few passes over K as possible. Block b walks range
// order[b]: the host hands the ranges out heaviest first, as blocks with low
// indices reach their SMs first.
//
// Every mbarrier wait is bounded by the plan's timeout: on expiry the waiter
// records (status, site, block) in the error word, raises a CTA-wide abort
// flag and leaves its loop; all warps then drain their own asynchronous
// work, TMEM is released and the kernel returns normally.
#include <cstddef>

#include <cuda_fp16.h>

#include "ggemm_internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

using namespace ptx;

constexpr int kWarpBProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;    // epilogue warps 2-5: even 32-column blocks
constexpr int kWarpEpi1 = 12;   // epilogue warps 12-15: odd 32-column blocks
constexpr int kNumEpiWarps = 8;
constexpr int kWarpAProducer = 6;
constexpr int kWarpSProducer = 7;
constexpr int kWarpSf0 = 8;
constexpr int kNumSfWarps = 4;
constexpr int kThreads = 16 * 32;

constexpr int kATileBytes = kTileM * (kTileK / 2);  // 16384: 128 rows x 128 B
constexpr int kSfTileBytes = 4 * kSfAtomBytes;       // 2048: scales of 128 rows x 256 k
constexpr int kBRowBoxBytes = 32 * (kTileK / 2);     // 4096: one 32-row B box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kStatusTimeout = 6;  // NVFP4_ERR_TIMEOUT
constexpr uint32_t kStatusFault = 7;    // NVFP4_ERR_DEVICE_FAULT
constexpr int kSfCols = 32 + 32;        // TMEM scale columns per stage: SFA 2 tiles x 4 x 4, SFB 4 x 8

constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

// Stage-completion ring: the MMA thread commits one barrier per stage, done[s %
// kDoneRing], and every ring the MMAs read (A, B, TMEM scale buffers) takes
// its "slot free" signal from it: the slot that stage s reuses in a ring of
// depth D was last read by stage s - D. A ring is at most kDoneRing deep, so
// a producer waiting for stage s - D can never see that barrier two phases on.
// The A and B rings are fixed byte regions; each CTA cuts them into as many
// slots (up to kDoneRing) as its widest tile allows, so narrow tiles keep
// more stages in flight.
constexpr int kDoneRing = 16;

// Timeline stamps (the -DNVFP4_TRACE build only; nothing otherwise).
#ifdef NVFP4_TRACE
__device__ __forceinline__ void trace_at(const GemmParams &p, int slot)
{
    if (p.trace) p.trace[(size_t)blockIdx.x * kTraceSlots + slot] = globaltimer_ns();
}
__device__ __forceinline__ void trace_val(const GemmParams &p, int slot, unsigned long long v)
{
    if (p.trace) p.trace[(size_t)blockIdx.x * kTraceSlots + slot] = v;
}
__device__ __forceinline__ void trace_max(const GemmParams &p, int slot)
{
    if (p.trace) atomicMax(p.trace + (size_t)blockIdx.x * kTraceSlots + slot, (unsigned long long)globaltimer_ns());
}
#define NVFP4_TRACE_AT(slot) trace_at(p, (slot))
#define NVFP4_TRACE_VAL(slot, v) trace_val(p, (slot), (v))
#define NVFP4_TRACE_MAX(slot) trace_max(p, (slot))
#else
#define NVFP4_TRACE_AT(slot) ((void)0)
#define NVFP4_TRACE_VAL(slot, v) ((void)0)
#define NVFP4_TRACE_MAX(slot) ((void)0)
#endif

// Device checks of the debug build (-DNVFP4_DEBUG): NVFP4_CHECK(cond, site)
// is a Roles member call that, when cond is false (or the test-only option
// names the site), records (device fault, site) in the error word, raises the
// CTA's abort flag and returns false, and the caller skips the operation it
// guards; NVFP4_CHECK_WARP is the same for a whole warp, true only if it
// holds on every lane. In the release build both are the constant true and
// cost nothing.
#ifdef NVFP4_DEBUG
#define NVFP4_CHECK(cond, site) check((cond), (site))
#define NVFP4_CHECK_WARP(cond, site) __all_sync(0xffffffffu, check((cond), (site)))
#else
#define NVFP4_CHECK(cond, site) true
#define NVFP4_CHECK_WARP(cond, site) true
#endif

template <int MAXN, int NB, int NA, int NS, bool RAW>
struct Cfg {
    static_assert(MAXN % 32 == 0 && MAXN >= 32 && MAXN <= kMaxTileN, "tile width");
    // widest tile of a unit with two row tiles: both accumulators share TMEM
    static constexpr int kPairN = MAXN >= 192 ? 192 : MAXN;
    static constexpr int kBStage = MAXN * (kTileK / 2);
    static constexpr int kAStage = kRowTilesPerUnit * kATileBytes;
    // scale stage: raw scales cover kKS k tiles (rows of 16 * kKS bytes): SFA
    // (128 rows per row tile) then SFB (MAXN rows); atom-layout scales cover
    // one k tile: SFA (2 KB per row tile) then up to three 128-row atom
    // groups covering the tile's columns
    static constexpr int kKS = RAW ? kSfKTiles : 1;
    static constexpr int kSfRow = 16 * kKS;
    static constexpr int kSfaTile = RAW ? kTileM * kSfRow : kSfTileBytes;
    static constexpr int kSfaBytes = kRowTilesPerUnit * kSfaTile;
    static constexpr int kSfbRegion = RAW ? MAXN * kSfRow : 3 * kSfTileBytes;
    static constexpr int kSStage = align1k(kSfaBytes + kSfbRegion);
    static constexpr int kOffARing = 0;
    static constexpr int kOffBRing = NA * kAStage;
    static constexpr int kOffSRing = kOffBRing + NB * kBStage;
    // accumulator columns: two halves of kPairN, one per row tile of a pair
    static constexpr int kAccCols = kRowTilesPerUnit * kPairN;
    static_assert(MAXN <= kAccCols, "a one-row-tile unit fits the accumulator columns");
    static constexpr int kSfBase = kAccCols;
    static constexpr int kNT0 = ((int)kTmemCols - kSfBase) / kSfCols;
    static constexpr int kNT = kNT0 > 6 ? 6 : kNT0;  // TMEM scale buffers
    static constexpr int kOffBars = kOffSRing + NS * kSStage;
    static constexpr int kBRing = NB * kBStage;  // bytes
    static constexpr int kARing = NA * kAStage;
    static constexpr int kNumBars = kDoneRing + kDoneRing + 2 * NS + kNT + kDoneRing + 2 + 2 + 1;
    static constexpr int kOffTmemSlot = kOffBars + 8 * kNumBars;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1024
    static_assert(kNT >= 2, "at least two TMEM scale buffers");
    static_assert(NB >= 2 && NA >= 2 && kNT <= kDoneRing, "ring depths");
    static_assert(kSfBase + kNT * kSfCols <= (int)kTmemCols, "TMEM budget");
    static_assert(kBStage % 1024 == 0 && kAStage % 1024 == 0, "stages keep 1024-byte swizzle alignment");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct Unit {
    int g;
    int mt0;     // first 128-row tile of the unit
    int mtu;     // row tiles in the unit (1 or 2)
    int n0;      // first column
    int ncols;   // tile width: a multiple of 32
    bool keep;   // the group has more units of row tiles, which read B again
    int M;       // rows of the group
    int N;       // columns of the group
    int k_tiles; // ceil(K of the group / 256)
    int k_last;  // 64-k slices in the last k tile (1..4)
};

// Walks this CTA's contiguous range of chunks as tiles, for units of UNIT
// 128-row tiles (the plan's row tiles per unit, 1 or 2).
template <int UNIT>
struct Walker {
    static_assert(UNIT == 1 || UNIT == 2, "row tiles per unit");
    int pos, end;
    // the part of the range inside the current unit (plen chunks from ch0)
    // is cut into pt tiles of equal width (to within one chunk); pi = next tile
    int plen = 0, pt = 0, pi = 0;
    int g, g_base, g_tiles, g_rows, g_chunks, g_ktiles, g_klast, g_cols = -1, mt0 = 0, mtu = 0, ch0 = 0;

    __device__ __forceinline__ explicit Walker(const GemmParams &p)
    {
        const int c = p.order[blockIdx.x];  // the range this block walks
        const CtaStart &r = p.cta[c];
        pos = r.begin;
        end = p.cta[c + 1].begin;
        g = cta_group(r.packed);
        g_base = r.g_base;
        g_rows = cta_rows_m(r.rows);
        g_ktiles = cta_rows_ktiles(r.rows);
        g_chunks = cta_n_chunks(r.packed);
        g_klast = cta_k_last(r.packed);
        g_tiles = (g_rows + kTileM - 1) / kTileM;
    }

    __device__ __forceinline__ bool next(const GemmParams &p, Unit &t)
    {
        if (pi == pt) {
            if (pos >= end) return false;
            // groups past the one holding `pos` (only ranges that span groups get here)
            while (pos >= g_base + (UNIT == 1 ? g_tiles : (g_tiles + 1) >> 1) * g_chunks) {
                ++g;
                const GroupDesc &gd = p.groups[g];
                g_base = __ldg(p.chunk_prefix + g);
                g_rows = gd.M;
                g_tiles = gd.m_tiles;
                g_chunks = gd.n_chunks;
                g_ktiles = gd.k_tiles;
                g_klast = gd.k_last;
                g_cols = gd.N;
            }
            const int local = pos - g_base;
            const int mp = local / g_chunks;
            ch0 = local - mp * g_chunks;
            mt0 = mp * UNIT;
            mtu = min(UNIT, g_tiles - mt0);
            plen = min(g_chunks - ch0, end - pos);
            const int cap = mtu == 2 ? p.cap_pair : p.cap_single;
            pt = (plen + cap - 1) / cap;
            pi = 0;
            pos += plen;
        }
        const int c0 = (int)((long long)plen * pi / pt);
        const int c1 = (int)((long long)plen * (pi + 1) / pt);
        ++pi;
        t.g = g;
        t.mt0 = mt0;
        t.mtu = mtu;
        t.n0 = (ch0 + c0) * kChunkN;
        t.ncols = (c1 - c0) * kChunkN;
        t.keep = g_tiles > UNIT;
        t.M = g_rows;
        t.k_tiles = g_ktiles;
        t.k_last = g_klast;
        // N itself is only in the table; a bound that never cuts a live column
        // (the chunks cover N) serves until a role reads it
        t.N = g_cols >= 0 ? g_cols : g_chunks * kChunkN;
        return true;
    }
};

__device__ __forceinline__ void record_error(uint32_t *err, uint32_t status, uint32_t site)
{
    const uint32_t word = status | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16);
    atomicCAS(err, 0u, word);
}

// Slow path of wait_phase, kept out of line so that the common case (the
// phase has already completed) costs one try_wait and no call.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             const GemmParams &p, uint32_t site)
{
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_error(p.err, kStatusTimeout, site);
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait for phase `parity` of `bar`. False when another warp aborted
// or the timeout expired (then this thread records the error and aborts).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const GemmParams &p, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, p, site);
}

// The same bounded wait written inline, for a call site that holds many live
// registers (a call to the out-of-line slow path would spill them).
__device__ __forceinline__ bool wait_phase_inline(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                  const GemmParams &p, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_error(p.err, kStatusTimeout, site);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Bounded wait that ignores the abort flag: used at exit for a thread's own
// asynchronous work, which always completes unless it was never issued.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, const GemmParams &p, uint32_t site)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_error(p.err, kStatusTimeout, site);
            return false;
        }
    }
    return true;
}

// Warp-uniform bounded wait: every lane waits (each acquires the barrier),
// and the warp proceeds only if all lanes saw the phase complete.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                const GemmParams &p, uint32_t site)
{
    const bool ok = wait_phase(bar, parity, abort_flag, p, site);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits)
{
    const __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Orders every later use of v after the preceding tcgen05.wait::ld (the
// registers of a tcgen05.ld are written asynchronously).
__device__ __forceinline__ void pin_registers(uint32_t (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[i]));
}

// RN to fp16 and stores of 32 accumulator columns of one C row, starting at
// column col0 (a multiple of 32); columns >= N are not written. wide: the row
// is 32-byte aligned and N % 16 == 0, so two 32-byte stores cover the block;
// otherwise four 16-byte stores (N % 8 == 0). The stores carry an L2
// evict-first policy: C is written once and never read here, so its lines
// should be the first to leave L2 rather than lines other work still holds.
__device__ __forceinline__ void store_row_block(uint16_t *crow, int col0, int N, const uint32_t (&v)[32], bool wide,
                                                uint64_t pol)
{
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = pack_half2(v[2 * i], v[2 * i + 1]);
    if (wide) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (col0 + 16 * j < N)
                asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(
                                 crow + col0 + 16 * j),
                             "r"(h[8 * j + 0]), "r"(h[8 * j + 1]), "r"(h[8 * j + 2]), "r"(h[8 * j + 3]),
                             "r"(h[8 * j + 4]), "r"(h[8 * j + 5]), "r"(h[8 * j + 6]), "r"(h[8 * j + 7]), "l"(pol)
                             : "memory");
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (col0 + 8 * j < N)
                asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(crow + col0 + 8 * j),
                             "r"(h[4 * j + 0]), "r"(h[4 * j + 1]), "r"(h[4 * j + 2]), "r"(h[4 * j + 3]), "l"(pol)
                             : "memory");
    }
}

// The accumulator columns as two halves of kPairN columns, each with its own
// full / empty barrier pair. A tile with one row tile at most kPairN columns
// wide takes one half, the halves alternating, so that its MMAs run while
// the epilogue drains the previous tile from the other half; any other tile
// (two row tiles, or wider) takes both. The MMA thread and the epilogue walk
// the same tiles and so make the same choices.
struct AccTrack {
    uint32_t parity = 0;  // bit h: phase parity of half h's barriers
    int next = 0;         // the half a one-half tile takes
    __device__ __forceinline__ uint32_t par(int h) const { return (parity >> h) & 1u; }
    __device__ __forceinline__ void advance(int h0, bool both)
    {
        if (both) {
            parity ^= 3u;
            next = 0;
        } else {
            parity ^= 1u << h0;
            next = h0 ^ 1;
        }
    }
};

// A ring of mbarrier-guarded stages: position (stage, phase) advanced in step.
struct RingPos {
    int stage = 0;
    uint32_t phase = 0;
    template <int N>
    __device__ __forceinline__ void advance()
    {
        if (++stage == N) {
            stage = 0;
            phase ^= 1u;
        }
    }
    __device__ __forceinline__ void advance(int n)
    {
        if (++stage == n) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// First and count of the 128-row scale blocks that cover columns [n0, n0+ncols) of N.
__device__ __forceinline__ void sfb_blocks(int n0, int ncols, int N, int &b0, int &nblk)
{
    b0 = n0 / 128;
    const int last = min(n0 + ncols, N) - 1;
    nblk = last / 128 - b0 + 1;
}

// Rows [row0, row0 + 32 * chunks) of an operand (chunks 1..8) in the fewest
// boxes: 256, 128, 64 and 32 rows from maps[3], maps[2], maps[1], maps[0]
// (those whose bit is set in `chunks`), placed one after another from dst,
// `row_bytes` of shared memory per row.
__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap *maps, int32_t x, int32_t row0, int chunks,
                                         uint32_t row_bytes, uint32_t bar, uint64_t policy)
{
#pragma unroll
    for (int i = kNumRowBoxes - 1; i >= 0; --i) {
        if (chunks & (1 << i)) {
            tma_load_2d(dst, maps + i, x, row0, bar, policy);
            dst += (uint32_t)(kChunkN << i) * row_bytes;
            row0 += kChunkN << i;
        }
    }
}

// The tensor maps of group g: in the kernel parameters for the first
// kParamGroups groups, else in the problem table.
__device__ __forceinline__ const GroupMaps *maps_of(const GemmParams &p, int g)
{
    return g < kParamGroups ? &p.pmaps[g] : &p.groups[g].maps;
}

// The maps a producer thread has prepared, for one group at a time: on a
// map's first use the thread prefetches it, after an acquire fence when the
// map is in the problem table (written to global memory by a host copy, so
// the tensormap proxy must be ordered after that write; a memory round trip
// that can take microseconds while the other SMs stream). Parameter-space
// maps need no fence. For its first tile a producer does this before it
// waits for the previous kernel of the stream.
struct MapUse {
    int g = -1;
    uint32_t done = 0;  // bit i: map i of group g prepared
    __device__ __forceinline__ const CUtensorMap *use(const GroupMaps *gm, int group, const CUtensorMap *m)
    {
        if (group != g) {
            g = group;
            done = 0;
        }
        const uint32_t bit = 1u << (uint32_t)(m - &gm->tmA[0]);
        if (!(done & bit)) {
            if (group >= kParamGroups) fence_tensormap_acquire(m);
            prefetch_tensormap(m);
            done |= bit;
        }
        return m;
    }
    // the boxes of tma_rows for `chunks` rows of 32
    __device__ __forceinline__ void use_rows(const GroupMaps *gm, int group, const CUtensorMap *maps, int chunks)
    {
#pragma unroll
        for (int i = 0; i < kNumRowBoxes; ++i)
            if (chunks & (1 << i)) use(gm, group, maps + i);
    }
};

template <int MAXN, int NB, int NA, int NS, bool RAW, int UNIT, bool LANES>
struct Roles {
    using C = Cfg<MAXN, NB, NA, NS, RAW>;
    using Walker = nvfp4::Walker<UNIT>;
    static constexpr int NT = C::kNT;

    uint8_t *smem;
    uint32_t sbase;
    volatile int *abort_flag;
    const GemmParams &p;
    int max_chunks, max_rows;  // bound on this CTA's tiles
    int nb, na;                // slots of the B and A rings for this CTA
    uint32_t b_slot, a_slot;   // their sizes in bytes

    __device__ Roles(uint8_t *s, const GemmParams &params)
        : smem(s), sbase(smem_addr(s)), abort_flag(reinterpret_cast<volatile int *>(s + C::kOffAbort)), p(params)
    {
        size_rings();
    }

    // Size the ring slots from this CTA's widest tile and most row tiles.
    __device__ void size_rings()
    {
        const uint32_t packed = p.cta[p.order[blockIdx.x]].packed;
        max_chunks = min(max(cta_max_chunks(packed), 1), MAXN / kChunkN);
        max_rows = min(max(cta_max_rows(packed), 1), kRowTilesPerUnit);
        b_slot = (uint32_t)max_chunks * kBRowBoxBytes;
        a_slot = (uint32_t)max_rows * kATileBytes;
        nb = min(kDoneRing, C::kBRing / (int)b_slot);
        na = min(kDoneRing, C::kARing / (int)a_slot);
    }

    // A tile wider or taller than the slots this CTA cut its rings into
    // (the host bounds both; this only guards the shared-memory writes).
    __device__ __forceinline__ bool tile_fits(const Unit &t) const
    {
        if (t.ncols <= max_chunks * kChunkN && t.mtu <= max_rows) return true;
        record_error(p.err, kStatusFault, kSiteTileCheck);
        *abort_flag = 1;
        return false;
    }

    // A tile that adds its even and odd 64-k slices into the two accumulator
    // halves (the plan's split_acc: one row tile, at most half the columns)
    __device__ __forceinline__ bool split_tile(const Unit &t) const
    {
        if constexpr (UNIT == 2) return false;  // pairs: never (the code below compiles away)
        return p.split_acc != 0 && t.ncols <= C::kPairN;
    }

#ifdef NVFP4_DEBUG
    __device__ __forceinline__ bool check(bool cond, uint32_t site) const
    {
        if (cond && p.debug_check_fail != (int)site) return true;
        record_error(p.err, kStatusFault, site);
        *abort_flag = 1;
        return false;
    }
#endif
    // `bytes` of shared memory from dst lie inside [sbase + lo, sbase + hi)
    // and dst is 1024-byte aligned (the 128-byte swizzle's atom)
    __device__ __forceinline__ bool smem_in(uint32_t dst, uint32_t bytes, int lo, int hi) const
    {
        return dst >= sbase + (uint32_t)lo && dst + bytes <= sbase + (uint32_t)hi && (dst & 1023u) == 0;
    }

    static constexpr int kBarDone = 2 * kDoneRing + 2 * NS + NT;
    __device__ __forceinline__ uint32_t bar(int i) const { return sbase + C::kOffBars + 8 * i; }
    __device__ __forceinline__ uint32_t b_full(int s) const { return bar(s); }
    __device__ __forceinline__ uint32_t a_full(int s) const { return bar(kDoneRing + s); }
    __device__ __forceinline__ uint32_t s_full(int s) const { return bar(2 * kDoneRing + s); }
    __device__ __forceinline__ uint32_t s_empty(int s) const { return bar(2 * kDoneRing + NS + s); }
    __device__ __forceinline__ uint32_t sf_ready(int b) const { return bar(2 * kDoneRing + 2 * NS + b); }
    __device__ __forceinline__ uint32_t done(int d) const { return bar(kBarDone + d); }
    __device__ __forceinline__ uint32_t acc_full(int a) const { return bar(kBarDone + kDoneRing + a); }
    __device__ __forceinline__ uint32_t acc_empty(int a) const { return bar(kBarDone + kDoneRing + 2 + a); }
    __device__ __forceinline__ uint32_t drain() const { return bar(kBarDone + kDoneRing + 4); }
    // Wait until the MMAs of stage j (< 0: none) have completed.
    __device__ __forceinline__ bool wait_done(int j, uint32_t site) const
    {
        if (j < 0) return true;
        return wait_phase(done(j % kDoneRing), (uint32_t)(j / kDoneRing) & 1u, abort_flag, p, site);
    }
    __device__ __forceinline__ uint32_t b_stage(int s) const { return sbase + C::kOffBRing + (uint32_t)s * b_slot; }
    __device__ __forceinline__ uint32_t a_stage(int s) const { return sbase + C::kOffARing + (uint32_t)s * a_slot; }
    __device__ __forceinline__ uint32_t s_stage(int s) const { return sbase + C::kOffSRing + s * C::kSStage; }

    __device__ void init_barriers()
    {
        for (int s = 0; s < kDoneRing; ++s) {
            mbar_init(b_full(s), 1);
            mbar_init(a_full(s), 1);
        }
        for (int d = 0; d < kDoneRing; ++d) mbar_init(done(d), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(s_full(s), LANES ? 32 : 1);  // 32: a warp-wide scale producer
            mbar_init(s_empty(s), kNumSfWarps);
        }
        for (int b = 0; b < NT; ++b) mbar_init(sf_ready(b), kNumSfWarps);
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), kNumEpiWarps);
        }
        mbar_init(drain(), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }

    // ------------------------------------------------------------- B producer
    __device__ void b_producer(Walker wk, Unit t, bool have)
    {
        const uint64_t pol_stream = policy_evict_first();  // read by one row tile only
        const uint64_t pol_keep = policy_evict_normal();    // read again by the group's other row tiles
        RingPos r;
        uint32_t issued_mask = 0, issued_parity = 0;
        MapUse maps;
        int loads = 0, seq = 0;
        if (have) maps.use_rows(maps_of(p, t.g), t.g, maps_of(p, t.g)->tmB, t.ncols / kChunkN);
        bool ok = true;
        for (bool more = have; ok && more; more = wk.next(p, t)) {
            if (!tile_fits(t)) {
                ok = false;
                break;
            }
            const GroupMaps *gm = maps_of(p, t.g);
            maps.use_rows(gm, t.g, gm->tmB, t.ncols / kChunkN);
            const uint64_t pol = t.keep ? pol_keep : pol_stream;
            const int chunks = t.ncols / kChunkN;
            const uint32_t bytes = (uint32_t)t.ncols * (kTileK / 2);
            for (int kt = 0; kt < t.k_tiles; ++kt) {
                if (!wait_done(seq - nb, kSiteBEmpty)) {
                    ok = false;
                    break;
                }
                ++seq;
                ++loads;
                const bool skip =
                    (p.debug_skip_load > 0 && blockIdx.x == 0 && loads == p.debug_skip_load) ||
                    !NVFP4_CHECK(smem_in(b_stage(r.stage), bytes, C::kOffBRing, C::kOffBRing + C::kBRing) &&
                                     chunks >= 1 && chunks <= MAXN / kChunkN && t.n0 >= 0 &&
                                     ((kt * (kTileK / 2)) & 15) == 0,
                                 kSiteCheckLoadB);
                if (!skip) {
                    const uint32_t fb = b_full(r.stage);
                    mbar_arrive_expect_tx(fb, bytes);
                    // B may be written by the previous kernel, unless the caller says otherwise
                    if (loads == 1 && !(p.early & kEarlyB)) griddep_wait();
                    tma_rows(b_stage(r.stage), gm->tmB, kt * (kTileK / 2), t.n0, chunks, kTileK / 2, fb, pol);
                    issued_mask |= 1u << r.stage;
                    issued_parity = (issued_parity & ~(1u << r.stage)) | (r.phase << r.stage);
                    if (loads == 1) NVFP4_TRACE_AT(kTrBFirst);
                    NVFP4_TRACE_AT(kTrBLast);
                } else {
                    issued_mask &= ~(1u << r.stage);  // nothing in flight for this stage
                }
                r.advance(nb);
            }
        }
        for (int s = 0; s < nb; ++s)
            if ((issued_mask >> s) & 1u) wait_drain(b_full(s), (issued_parity >> s) & 1u, p, kSiteLoadDrain);
    }

    // ------------------------------------------------------------- A producer
    __device__ void a_producer(Walker wk, Unit t, bool have)
    {
        const uint64_t pol = policy_evict_last();  // A tiles are re-read by every column tile
        RingPos r;
        uint32_t issued_mask = 0, issued_parity = 0;
        MapUse maps;
        int seq = 0;
        bool first = true;
        bool ok = true;
        for (bool more = have; ok && more; more = wk.next(p, t)) {
            if (!tile_fits(t)) {
                ok = false;
                break;
            }
            const GroupMaps *gm = maps_of(p, t.g);
            // the unit's one or two 128-row tiles in one box; rows past M_g
            // are the TMA's zero fill, and their accumulator rows are never stored
            const CUtensorMap *map = maps.use(gm, t.g, &gm->tmA[t.mtu - 1]);
            for (int kt = 0; kt < t.k_tiles; ++kt) {
                if (!wait_done(seq - na, kSiteAEmpty)) {
                    ok = false;
                    break;
                }
                ++seq;
                if (!NVFP4_CHECK(smem_in(a_stage(r.stage), (uint32_t)t.mtu * kATileBytes, C::kOffARing,
                                         C::kOffARing + C::kARing) &&
                                     t.mtu >= 1 && t.mtu <= kRowTilesPerUnit && t.mt0 >= 0,
                                 kSiteCheckLoadA)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = a_full(r.stage);
                mbar_arrive_expect_tx(fb, (uint32_t)t.mtu * kATileBytes);
                if (first) {
                    // A may be written by the previous kernel, unless the caller says otherwise
                    if (!(p.early & kEarlyA)) griddep_wait();
                    NVFP4_TRACE_AT(kTrDepWait);
                }
                tma_load_2d(a_stage(r.stage), map, kt * (kTileK / 2), t.mt0 * kTileM, fb, pol);
                if (first) {
                    first = false;
                    NVFP4_TRACE_AT(kTrAFirst);
                }
                issued_mask |= 1u << r.stage;
                issued_parity = (issued_parity & ~(1u << r.stage)) | (r.phase << r.stage);
                r.advance(na);
            }
        }
        for (int s = 0; s < na; ++s)
            if ((issued_mask >> s) & 1u) wait_drain(a_full(s), (issued_parity >> s) & 1u, p, kSiteLoadDrain);
    }

    // --------------------------------------------------------- scale producer
    __device__ void s_producer(Walker wk, Unit t, bool have)
    {
        const uint64_t pol = policy_evict_normal();
        RingPos r;
        uint32_t issued_mask = 0, issued_parity = 0;
        MapUse maps;
        bool first = true;
        bool ok = true;

        for (bool more = have; ok && more; more = wk.next(p, t)) {
            const GroupMaps *gm = maps_of(p, t.g);
            const int chunks = t.ncols / kChunkN;
            int b0 = 0, nblk = 0;
            sfb_blocks(t.n0, t.ncols, t.N, b0, nblk);
            maps.use(gm, t.g, &gm->tmSFA[t.mtu - 1]);
            if (RAW) maps.use_rows(gm, t.g, gm->tmSFB, chunks);
            else if (nblk >= 1 && nblk <= 3) maps.use(gm, t.g, &gm->tmSFB[nblk - 1]);
            const int s_tiles = (t.k_tiles + C::kKS - 1) / C::kKS;  // scale stages of this tile
            for (int ks = 0; ks < s_tiles; ++ks) {
                // atom layout: whole boxes of four atoms per 128-row block, the
                // atoms past K_g of a partial last k tile filled with zeros
                const uint32_t bytes = RAW ? (uint32_t)(t.mtu * kTileM + t.ncols) * C::kSfRow
                                           : (uint32_t)(t.mtu + nblk) * kSfTileBytes;
                if (!wait_phase(s_empty(r.stage), r.phase ^ 1u, abort_flag, p, kSiteSEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = s_full(r.stage);
                const uint32_t st = s_stage(r.stage);
                if (!NVFP4_CHECK(st >= sbase + C::kOffSRing && st + C::kSStage <= sbase + C::kOffSRing + NS * C::kSStage &&
                                     (RAW ? (uint32_t)t.mtu * kTileM * C::kSfRow <= (uint32_t)C::kSfaBytes &&
                                                (uint32_t)t.ncols * C::kSfRow <= (uint32_t)C::kSfbRegion &&
                                                ((ks * C::kSfRow) & 15) == 0
                                          : nblk >= 1 && nblk <= 3 && nblk * kSfTileBytes <= C::kSfbRegion),
                                 kSiteCheckLoadSf)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fb, bytes);
                // the scales may be written by the previous kernel: on the first
                // stage, part 0 loads those the caller declared it does not write,
                // then part 1 waits for it and loads the rest
                const bool sfa_early = !first || (p.early & kEarlySfa);
                const bool sfb_early = !first || (p.early & kEarlySfb);
                for (int part = 0; part < 2; ++part) {
                    const bool sfa_now = part == 0 ? sfa_early : !sfa_early;
                    const bool sfb_now = part == 0 ? sfb_early : !sfb_early;
                    if (part == 1 && !(sfa_early && sfb_early)) griddep_wait();
                    if (RAW) {
                        // scale bytes [16 * kt0, 16 * (kt0 + kKS)) of each row: k tiles kt0 .. kt0 + kKS - 1;
                        // the unit's row tiles in one box, the tile's columns in the fewest boxes
                        const int x = ks * C::kSfRow;
                        if (sfa_now) tma_load_2d(st, &gm->tmSFA[t.mtu - 1], x, t.mt0 * kTileM, fb, pol);
                        if (sfb_now) tma_rows(st + C::kSfaBytes, gm->tmSFB, x, t.n0, chunks, C::kSfRow, fb, pol);
                    } else {
                        // the four atoms of k tile ks for the unit's row tiles
                        // and for the 128-row blocks under the tile's columns,
                        // one box each: 2 KB per 128-row block, block after block
                        if (sfa_now) tma_load_3d(st, &gm->tmSFA[t.mtu - 1], 0, ks * 4, t.mt0, fb, pol);
                        if (sfb_now) tma_load_3d(st + C::kSfaBytes, &gm->tmSFB[nblk - 1], 0, ks * 4, b0, fb, pol);
                    }
                }
                if (first) {
                    first = false;
                    NVFP4_TRACE_AT(kTrSFirst);
                }
                issued_mask |= 1u << r.stage;
                issued_parity = (issued_parity & ~(1u << r.stage)) | (r.phase << r.stage);
                r.advance<NS>();
            }
        }
        for (int s = 0; s < NS; ++s)
            if ((issued_mask >> s) & 1u) wait_drain(s_full(s), (issued_parity >> s) & 1u, p, kSiteLoadDrain);
    }

    // Bytes [x, x + kSfRow) of rows r_first, r_first + period, ... (< rows)
    // of raw scale rows of row_bytes bytes each, counted from row row0 of
    // src, into consecutive kSfRow-byte rows of shared memory at dst (the
    // layout a TMA box gives), by the warp's 32 lanes in cp.async pieces of
    // PIECE bytes: a lane keeps one piece position of the row and steps
    // through the rows. Pieces past a row's end (64-k slices past K_g,
    // which are never issued) are not copied; every piece copied lies
    // inside its row.
    template <int PIECE>
    __device__ __forceinline__ void copy_sf_pieces(uint32_t dst, const uint8_t *src, int row0, int r_first,
                                                   int period, int rows, int row_bytes, int x, int lane)
    {
        constexpr int P = C::kSfRow / PIECE;  // pieces per row
        constexpr int R = 32 / P;             // rows per pass of the warp
        const int c = lane % P;
        const int off = x + PIECE * c;
        if (off + PIECE > row_bytes) return;
        int r = r_first + period * (lane / P);
        if (r >= rows) return;
        const int step = period * R;
        const uint8_t *sp = src + (size_t)(row0 + r) * row_bytes + off;
        uint32_t dp = dst + (uint32_t)(r * C::kSfRow + PIECE * c);
        const size_t s_step = (size_t)step * row_bytes;
#pragma unroll 4
        for (; r < rows; r += step) {
            if (PIECE == 16) cp_async_16(dp, sp);
            else if (PIECE == 8) cp_async_8(dp, sp);
            else cp_async_4(dp, sp);
            sp += s_step;
            dp += step * C::kSfRow;
        }
    }

    // Bytes [x, x + kSfRow) of `rows` raw scale rows (row0 on) of a row
    // length with row_bytes % 8 == 0 into the stage at dst, rows inside the
    // matrix only. Row starts (src 16-byte aligned) alternate between 16-byte
    // and 8-byte alignment, and each of the two classes of rows takes the
    // widest piece its start allows; a row's last window (past its end) goes
    // in 4-byte pieces.
    __device__ __forceinline__ void copy_sf_rows(uint32_t dst, const uint8_t *src, int row0, int rows, int row_bytes,
                                                 int x, int lane)
    {
        if (x + C::kSfRow <= row_bytes) {
            const int r16 = row0 & 1;  // the first row r with (row0 + r) even: 16-byte aligned
            copy_sf_pieces<16>(dst, src, row0, r16, 2, rows, row_bytes, x, lane);
            copy_sf_pieces<8>(dst, src, row0, r16 ^ 1, 2, rows, row_bytes, x, lane);
        } else {
            copy_sf_pieces<4>(dst, src, row0, 0, 1, rows, row_bytes, x, lane);
        }
    }

    // The scale producer of the raw-scale kernels built for groups whose raw
    // scale rows are not whole 16-byte units (LANES): the whole warp runs this
    // loop and the stage barriers count 32 arrivals. For such a group's tiles
    // every lane copies its share of the stage's rows with cp.async and arms
    // an arrive that fires once its copies have landed; for the other groups
    // lane 0 loads by TMA as s_producer does and arrives with the byte count,
    // and the other lanes arrive at once. (Kernels of their own, so that the
    // kernels every other plan runs carry none of this code.)
    __device__ void s_producer_lanes(Walker wk, Unit t, bool have, int lane)
    {
        static_assert(RAW && LANES, "raw-scale kernels built with the lane copies only");
        const uint64_t pol = policy_evict_normal();
        RingPos r;
        uint32_t issued_mask = 0, issued_parity = 0;
        MapUse maps;
        bool first = true;
        bool ok = true;

        for (bool more = have; ok && more; more = wk.next(p, t)) {
            const GroupMaps *gm = maps_of(p, t.g);
            const int chunks = t.ncols / kChunkN;
            // raw rows the lanes copy (read once per tile): this group's row
            // bytes, else 0 (TMA)
            const GroupDesc *gd = &p.groups[t.g];
            const int row_bytes = gd->sf_row_bytes;
            const uint8_t *sfa_rows = gd->sfa_rows;
            const uint8_t *sfb_rows = gd->sfb_rows;
            // SFB a copy with rows padded to 16 bytes: loaded by TMA even here
            const bool sfb_tma = row_bytes != 0 && gd->sfb_tma != 0;
            const int a_rows = min(t.mtu * kTileM, t.M - t.mt0 * kTileM);  // rows inside the matrices
            const int b_rows = min(t.ncols, t.N - t.n0);
            if (lane == 0 && (row_bytes == 0 || sfb_tma)) {
                if (row_bytes == 0) maps.use(gm, t.g, &gm->tmSFA[t.mtu - 1]);
                maps.use_rows(gm, t.g, gm->tmSFB, chunks);
            }
            const int s_tiles = (t.k_tiles + C::kKS - 1) / C::kKS;  // scale stages of this tile
            for (int ks = 0; ks < s_tiles; ++ks) {
                if (!warp_wait_phase(s_empty(r.stage), r.phase ^ 1u, abort_flag, p, kSiteSEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = s_full(r.stage);
                const uint32_t st = s_stage(r.stage);
                if (!NVFP4_CHECK(st >= sbase + C::kOffSRing && st + C::kSStage <= sbase + C::kOffSRing + NS * C::kSStage &&
                                     (uint32_t)t.mtu * kTileM * C::kSfRow <= (uint32_t)C::kSfaBytes &&
                                     (uint32_t)t.ncols * C::kSfRow <= (uint32_t)C::kSfbRegion &&
                                     ((ks * C::kSfRow) & 15) == 0 &&
                                     (row_bytes == 0 || (row_bytes % 4 == 0 &&
                                                         ((reinterpret_cast<uintptr_t>(sfa_rows) |
                                                           reinterpret_cast<uintptr_t>(sfb_tma ? nullptr : sfb_rows)) &
                                                          15u) == 0)),
                                 kSiteCheckLoadSf)) {
                    ok = false;
                    break;
                }
                // the scales may be written by the previous kernel: on the first
                // stage, part 0 loads those the caller declared it does not write,
                // then part 1 waits for it and loads the rest
                const bool sfa_early = !first || (p.early & kEarlySfa);
                const bool sfb_early = !first || (p.early & kEarlySfb);
                const int x = ks * C::kSfRow;  // scale bytes [x, x + kSfRow) of each row
                // Rows whose length is 4 mod 8 bytes go in 4-byte pieces (16- and
                // 8-byte pieces for the rows that allow them were slower there);
                // rows of 8-byte multiples in 16- and 8-byte pieces, from a
                // single copy of that code (four inlined copies were slower)
                // An SFB loaded by TMA adds its bytes to the stage barrier (lane 0,
                // before its own arrive below, so the phase cannot complete first).
                if (sfb_tma && lane == 0) mbar_expect_tx(fb, (uint32_t)t.ncols * C::kSfRow);
                if (row_bytes % 8 != 0) {
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1 && !(sfa_early && sfb_early)) griddep_wait();
                        if (part == 0 ? sfa_early : !sfa_early)
                            copy_sf_pieces<4>(st, sfa_rows, t.mt0 * kTileM, 0, 1, a_rows, row_bytes, x, lane);
                        if (part == 0 ? sfb_early : !sfb_early) {
                            if (!sfb_tma)
                                copy_sf_pieces<4>(st + C::kSfaBytes, sfb_rows, t.n0, 0, 1, b_rows, row_bytes, x, lane);
                            else if (lane == 0)
                                tma_rows(st + C::kSfaBytes, gm->tmSFB, x, t.n0, chunks, C::kSfRow, fb, pol);
                        }
                    }
                    cp_async_mbar_arrive_noinc(fb);
                } else if (row_bytes != 0) {
                    // (part, operand) = (i / 2, i % 2): SFA then SFB, those loaded
                    // early first
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        const bool sfb = (i & 1) != 0;
                        const bool early = sfb ? sfb_early : sfa_early;
                        if (i == 2 && !(sfa_early && sfb_early)) griddep_wait();
                        if (!(i < 2 ? early : !early)) continue;
                        if (sfb && sfb_tma) {
                            if (lane == 0) tma_rows(st + C::kSfaBytes, gm->tmSFB, x, t.n0, chunks, C::kSfRow, fb, pol);
                        } else {
                            copy_sf_rows(sfb ? st + C::kSfaBytes : st, sfb ? sfb_rows : sfa_rows,
                                         sfb ? t.n0 : t.mt0 * kTileM, sfb ? b_rows : a_rows, row_bytes, x, lane);
                        }
                    }
                    cp_async_mbar_arrive_noinc(fb);
                } else if (lane == 0) {
                    mbar_arrive_expect_tx(fb, (uint32_t)(t.mtu * kTileM + t.ncols) * C::kSfRow);
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1 && !(sfa_early && sfb_early)) griddep_wait();
                        if (part == 0 ? sfa_early : !sfa_early)
                            tma_load_2d(st, &gm->tmSFA[t.mtu - 1], x, t.mt0 * kTileM, fb, pol);
                        if (part == 0 ? sfb_early : !sfb_early)
                            tma_rows(st + C::kSfaBytes, gm->tmSFB, x, t.n0, chunks, C::kSfRow, fb, pol);
                    }
                } else {
                    mbar_arrive(fb);
                }
                if (first) {
                    first = false;
                    if (lane == 0) NVFP4_TRACE_AT(kTrSFirst);
                }
                issued_mask |= 1u << r.stage;
                issued_parity = (issued_parity & ~(1u << r.stage)) | (r.phase << r.stage);
                r.advance<NS>();
            }
        }
        for (int s = 0; s < NS; ++s)
            if ((issued_mask >> s) & 1u) wait_drain(s_full(s), (issued_parity >> s) & 1u, p, kSiteLoadDrain);
        cp_async_wait_all();  // this thread's copies, whatever became of the stages
    }

    // ------------------------------------------------------------ scale writers
    // TMEM scale layout for one stage (scale buffer b at column S = base + 64b):
    //   SFA, row tile mt, 64-k slice kk: columns S + 16mt + 4kk + c (c = 0..3),
    //   lane i holds the four 16-k scales of the tile's row 32c + i;
    //   SFB, 64-k slice kk: columns S + 32 + 8kk + c (c = 0..7), lane i holds
    //   those of tile column 32c + i.
    // Every lane quarter holds the same values; warp q writes quarter q.
    __device__ void sf_writer(uint32_t tmem, int warp, int lane)
    {
        const int q = warp & 3;
        RingPos rs, rt;
        int seq = 0;
        bool ok = true;
        Walker wk(p);
        Unit t;
        while (ok && wk.next(p, t)) {
            int b0 = 0, nblk = 0;
            sfb_blocks(t.n0, t.ncols, t.N, b0, nblk);
            const int s0 = (t.n0 % 128) / 32;
            for (int kt = 0; kt < t.k_tiles; ++kt) {
                const int sub = kt % C::kKS;  // k tile within the scale stage
                // gather from shared memory first, then wait for the TMEM scale
                // buffer (the MMAs that read it two stages ago) only to write it
                if (sub == 0 && !warp_wait_phase(s_full(rs.stage), rs.phase, abort_flag, p, kSiteSFull)) {
                    ok = false;
                    break;
                }
                ++seq;
                const uint8_t *sa = smem + C::kOffSRing + rs.stage * C::kSStage;
                const uint8_t *sb = sa + C::kSfaBytes;
                uint32_t va[32], vb[32];
                if (RAW) {
                    // raw rows: row r's scales at r * kSfRow, this k tile's 16 bytes
                    // at 16 * sub; word kk = the 64-k slice kk. Rows past M_g hold
                    // stale bytes; their accumulator rows are never stored.
                    const uint8_t *ra = sa + 16 * sub;
                    const uint8_t *rb = sb + 16 * sub;
#pragma unroll
                    for (int mt = 0; mt < kRowTilesPerUnit; ++mt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 w = (mt < t.mtu) ? *reinterpret_cast<const uint4 *>(
                                                               ra + mt * C::kSfaTile + C::kSfRow * (32 * c + lane))
                                                         : make_uint4(0u, 0u, 0u, 0u);
                            va[16 * mt + 0 + c] = w.x;
                            va[16 * mt + 4 + c] = w.y;
                            va[16 * mt + 8 + c] = w.z;
                            va[16 * mt + 12 + c] = w.w;
                        }
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        // rows past the widest tile lie outside this stage's scale region
                        const uint4 w = (32 * c < MAXN)
                                            ? *reinterpret_cast<const uint4 *>(rb + C::kSfRow * (32 * c + lane))
                                            : make_uint4(0u, 0u, 0u, 0u);
                        vb[0 + c] = w.x;
                        vb[8 + c] = w.y;
                        vb[16 + c] = w.z;
                        vb[24 + c] = w.w;
                    }
                } else {
                    // atom groups: atom kk row i holds rows i, i+32, i+64, i+96 (words 0..3)
#pragma unroll
                    for (int mt = 0; mt < kRowTilesPerUnit; ++mt)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint4 w = (mt < t.mtu) ? *reinterpret_cast<const uint4 *>(
                                                               sa + mt * kSfTileBytes + kk * kSfAtomBytes + 16 * lane)
                                                         : make_uint4(0u, 0u, 0u, 0u);
                            va[16 * mt + 4 * kk + 0] = w.x;
                            va[16 * mt + 4 * kk + 1] = w.y;
                            va[16 * mt + 4 * kk + 2] = w.z;
                            va[16 * mt + 4 * kk + 3] = w.w;
                        }
                    // tile column 32c + i is row n0 + 32c + i: atom group (s0 + c) / 4,
                    // word (s0 + c) % 4 of that group's row i
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int idx = s0 + c;
                        const bool in = (idx >> 2) < nblk;
                        const uint8_t *src = sb + (idx >> 2) * kSfTileBytes + 16 * lane + 4 * (idx & 3);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            vb[8 * kk + c] = in ? *reinterpret_cast<const uint32_t *>(src + kk * kSfAtomBytes) : 0u;
                    }
                }
                const int jd = seq - 1 - NT;  // the stage whose MMAs last read this TMEM scale buffer
                if (jd >= 0 && !__all_sync(0xffffffffu, wait_phase_inline(done(jd % kDoneRing),
                                                                           (uint32_t)(jd / kDoneRing) & 1u,
                                                                           abort_flag, p, kSiteSfFree))) {
                    ok = false;
                    break;
                }
                const uint32_t col = (uint32_t)(C::kSfBase + rt.stage * kSfCols);
                if (!NVFP4_CHECK_WARP(col >= (uint32_t)C::kSfBase && col + kSfCols <= kTmemCols, kSiteCheckSfSt)) {
                    ok = false;
                    break;
                }
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + col;
                tmem_st_32x32b_x32(taddr, va);
                tmem_st_32x32b_x32(taddr + 32, vb);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                const bool stage_done = (sub == C::kKS - 1) || (kt == t.k_tiles - 1);
                if (seq == 1 && lane == 0 && q == 0) NVFP4_TRACE_AT(kTrSfFirst);
                if (lane == 0) {
                    if (stage_done) mbar_arrive(s_empty(rs.stage));
                    mbar_arrive(sf_ready(rt.stage));
                }
                if (stage_done) rs.advance<NS>();
                rt.advance<NT>();
            }
        }
        tmem_st_wait();
    }

    // ------------------------------------------------------------- MMA issuer
    __device__ void mma_issuer(uint32_t tmem)
    {
        RingPos ra, rb, rt;
        AccTrack acc;
        int seq = 0, tile = 0;
        bool ok = true;
        Walker wk(p);
        Unit t;
        while (ok && wk.next(p, t)) {
            const bool split = split_tile(t);
            const bool both = t.mtu > 1 || t.ncols > C::kPairN || split;
            const int h0 = both ? 0 : acc.next;
            if (!wait_phase(acc_empty(h0), acc.par(h0) ^ 1u, abort_flag, p, kSiteAccEmpty) ||
                (both && !wait_phase(acc_empty(1), acc.par(1) ^ 1u, abort_flag, p, kSiteAccEmpty)))
                break;
            tc_fence_after_sync();
            const uint32_t d = tmem + (uint32_t)(h0 * C::kPairN);
            const uint32_t idesc = idesc_mxf4nvf4_m128((uint32_t)t.ncols);
            for (int kt = 0; kt < t.k_tiles; ++kt) {
                if (!wait_phase(b_full(rb.stage), rb.phase, abort_flag, p, kSiteBFull) ||
                    !wait_phase(a_full(ra.stage), ra.phase, abort_flag, p, kSiteAFull) ||
                    !wait_phase(sf_ready(rt.stage), rt.phase, abort_flag, p, kSiteSfReady)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (seq == 0) NVFP4_TRACE_AT(kTrMmaFirstData);
                if (kt == 0 && tile < 8) NVFP4_TRACE_AT(kTrTileFirstData + tile);
                const uint32_t sa = a_stage(ra.stage);
                const uint32_t sb = b_stage(rb.stage);
                const uint32_t sf = tmem + (uint32_t)(C::kSfBase + rt.stage * kSfCols);
                // a last k tile of K % 256 != 0 holds fewer live 64-k slices
                const int slices = kt + 1 == t.k_tiles ? t.k_last : 4;
                // (debug build) accumulator and scale columns inside their TMEM
                // regions, operands inside their rings; a failed check skips
                // the stage's MMAs, and the commit below still frees the stage
                const bool issue = NVFP4_CHECK(
                    (split ? C::kPairN : (h0 + t.mtu - 1) * C::kPairN) + t.ncols <= C::kAccCols &&
                        C::kSfBase + rt.stage * kSfCols + kSfCols <= (int)kTmemCols &&
                        smem_in(sa, (uint32_t)t.mtu * kATileBytes, C::kOffARing, C::kOffARing + C::kARing) &&
                        smem_in(sb, (uint32_t)t.ncols * (kTileK / 2), C::kOffBRing, C::kOffBRing + C::kBRing),
                    kSiteCheckMma);
                if (split) {
                    // slice kk into half kk & 1; each half starts from its first slice
#pragma unroll
                    for (int kk = 0; kk < 4 && issue; ++kk)
                        if (kk < slices)
                            tc_mma_nvf4(d + (uint32_t)((kk & 1) * C::kPairN), desc_sw128_kmajor(sa + kk * 32),
                                        desc_sw128_kmajor(sb + kk * 32), idesc, sf + kk * 4, sf + 32 + kk * 8,
                                        (kt | (kk >> 1)) != 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4 && issue; ++kk) {
                        const uint64_t bdesc = desc_sw128_kmajor(sb + kk * 32);
#pragma unroll
                        for (int mt = 0; mt < kRowTilesPerUnit; ++mt)
                            if (mt < t.mtu && kk < slices)
                                tc_mma_nvf4(d + (uint32_t)(mt * C::kPairN),
                                            desc_sw128_kmajor(sa + mt * kATileBytes + kk * 32), bdesc, idesc,
                                            sf + mt * 16 + kk * 4, sf + 32 + kk * 8, (kt | kk) != 0 ? 1u : 0u);
                    }
                }
                // the stages and the scale buffer are free once these MMAs have read them
                tc_commit(done(seq % kDoneRing));
                if (seq == 0) NVFP4_TRACE_AT(kTrMmaFirstCommit);
                ++seq;
                ra.advance(na);
                rb.advance(nb);
                rt.advance<NT>();
            }
            if (!ok) break;
            tc_commit(acc_full(h0));
            if (both) tc_commit(acc_full(1));
            acc.advance(h0, both);
            if (tile < 8) NVFP4_TRACE_AT(kTrTileMmaEnd + tile);
            ++tile;
        }
        NVFP4_TRACE_VAL(kTrTiles, (unsigned long long)tile);
        NVFP4_TRACE_VAL(kTrStages, (unsigned long long)seq);
        // All tcgen05 work issued by this thread completes before TMEM is released.
        tc_commit(drain());
        wait_drain(drain(), 0, p, kSiteMmaDrain);
    }

    // --------------------------------------------------------------- epilogue
    __device__ void epilogue(uint32_t tmem, int warp, int lane)
    {
        const int q = warp & 3;                    // the TMEM lane quarter this warp may read
        const int h = warp >= kWarpEpi1 ? 1 : 0;   // which half of the 32-column blocks
        const uint64_t pol_c = policy_evict_first();
        AccTrack acc;
        Walker wk(p);
        Unit t;
        int tile = 0;
        while (wk.next(p, t)) {
            const GroupDesc *gd = p.groups + t.g;
            // the tile's C fields are read here, before the accumulator wait:
            // the wait is ordered before every later load, so a load written
            // after it would only start once the accumulator is full
            const int N = gd->N;
            const int ldc = gd->ldc;
            uint16_t *const cbase = gd->C;
            const bool split = split_tile(t);
            const bool both = t.mtu > 1 || t.ncols > C::kPairN || split;
            const int h0 = both ? 0 : acc.next;
            // a split tile's odd 64-k slices (none when K_g is one slice)
            const bool odd = split && (t.k_tiles > 1 || t.k_last > 1);
            if (!warp_wait_phase(acc_full(h0), acc.par(h0), abort_flag, p, kSiteAccFull) ||
                (both && !warp_wait_phase(acc_full(1), acc.par(1), abort_flag, p, kSiteAccFull)))
                break;
            tc_fence_after_sync();
            if (warp == kWarpEpi0 && lane == 0 && tile < 8) NVFP4_TRACE_AT(kTrTileEpiStart + tile);
            if (tile == 0) griddep_wait();  // C may be read or written by the previous kernel
            // columns [n0, n0 + 32 * nblk) hold live data; this warp takes blocks
            // h, h + 2, ... with two tcgen05.ld in flight: the next block is read
            // while the current one is converted and stored
            const int nblk = (min(t.ncols, N - t.n0) + 31) / 32;
            const int mine = (nblk - h + 1) / 2;
            const bool wide_st = ((reinterpret_cast<uintptr_t>(cbase) & 31u) == 0) && (N % 16 == 0) && (ldc % 16 == 0);
            bool failed = false;
            uint32_t v0[32], v1[32];
            if (split) {
                // one row tile, its accumulator in the two halves: each block's
                // two partial sums are added in fp32, then stored
                const int row0 = t.mt0 * kTileM + 32 * q;  // warp-uniform
                if (row0 < t.M && mine > 0) {
                    const int row = row0 + lane;
                    const bool live = row < t.M;
                    uint16_t *crow = cbase + (size_t)(live ? row : 0) * (size_t)ldc;
                    if (!NVFP4_CHECK_WARP(C::kPairN + 32 * (h + 2 * (mine - 1) + 1) <= C::kAccCols &&
                                              (!wide_st || !live ||
                                               (reinterpret_cast<uintptr_t>(crow + t.n0 + 32 * h) & 31u) == 0),
                                          kSiteCheckEpi))
                        break;
                    const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * h);
#pragma unroll 1
                    for (int j = 0; j < mine; ++j) {
                        tmem_ld_32x32b_x32(tbase + (uint32_t)(64 * j), v0);
                        if (odd) tmem_ld_32x32b_x32(tbase + (uint32_t)(C::kPairN + 64 * j), v1);
                        tmem_ld_wait();
                        pin_registers(v0);
                        if (odd) {
                            pin_registers(v1);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(v1[i]));
                        }
                        if (live) store_row_block(crow, t.n0 + 32 * (h + 2 * j), N, v0, wide_st, pol_c);
                    }
                }
            } else
#pragma unroll
            for (int mt = 0; mt < kRowTilesPerUnit; ++mt) {
                const int row0 = (t.mt0 + mt) * kTileM + 32 * q;  // warp-uniform
                if (mt >= t.mtu || row0 >= t.M || mine <= 0) continue;
                const int row = row0 + lane;
                const bool live = row < t.M;
                uint16_t *crow = cbase + (size_t)(live ? row : 0) * (size_t)ldc;
                // (debug build) the accumulator columns this warp reads, and the
                // 32-byte alignment of its rows' wide stores
                if (!NVFP4_CHECK_WARP((h0 + mt) * C::kPairN + 32 * (h + 2 * (mine - 1) + 1) <= C::kAccCols &&
                                          (!wide_st || !live ||
                                           (reinterpret_cast<uintptr_t>(crow + t.n0 + 32 * h) & 31u) == 0),
                                      kSiteCheckEpi)) {
                    failed = true;
                    break;
                }
                const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) +
                                       (uint32_t)((h0 + mt) * C::kPairN + 32 * h);
                tmem_ld_32x32b_x32(tbase, v0);
#pragma unroll 1
                for (int j = 0; j < mine; j += 2) {
                    tmem_ld_wait();
                    pin_registers(v0);
                    if (j + 1 < mine) tmem_ld_32x32b_x32(tbase + (uint32_t)(64 * (j + 1)), v1);
                    if (live) store_row_block(crow, t.n0 + 32 * (h + 2 * j), N, v0, wide_st, pol_c);
                    if (j + 1 < mine) {
                        tmem_ld_wait();
                        pin_registers(v1);
                        if (j + 2 < mine) tmem_ld_32x32b_x32(tbase + (uint32_t)(64 * (j + 2)), v0);
                        if (live) store_row_block(crow, t.n0 + 32 * (h + 2 * j + 2), N, v1, wide_st, pol_c);
                    }
                }
            }
            if (failed) break;
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(acc_empty(h0));
                if (both) mbar_arrive(acc_empty(1));
                if (tile < 8) {
                    if (warp == kWarpEpi0) NVFP4_TRACE_AT(kTrTileEpiEnd + tile);
                    NVFP4_TRACE_MAX(kTrTileEpiEndAll + tile);
                }
            }
            acc.advance(h0, both);
            ++tile;
        }
    }
};

template <int MAXN, int NB, int NA, int NS, bool RAW, int UNIT, bool LANES>
__global__ void __launch_bounds__(kThreads, 1) ggemm_kernel(const __grid_constant__ GemmParams p)
{
    using C = Cfg<MAXN, NB, NA, NS, RAW>;
    using Walker = nvfp4::Walker<UNIT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Roles<MAXN, NB, NA, NS, RAW, UNIT, LANES> r(smem, p);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        NVFP4_TRACE_AT(kTrStart);
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        NVFP4_TRACE_VAL(kTrSmId, smid);
    }
    if (threadIdx.x == 0) {
        r.init_barriers();
        NVFP4_TRACE_AT(kTrBarInit);
    }
    if (warp == kWarpMma) {
        tmem_alloc(r.sbase + C::kOffTmemSlot, kTmemCols);
        tmem_relinquish();
        if (lane == 0) NVFP4_TRACE_AT(kTrTmemAlloc);
    }
    // The producers walk to their first tile (a chain of single-thread
    // integer arithmetic of about a microsecond) while the barriers and TMEM
    // are set up; each then continues the walk itself.
    Walker wk0(p);
    Unit t0{};
    bool have0 = false;
    // (every lane of the scale producer's warp when that warp runs as one)
    if ((lane == 0 && (warp == kWarpBProducer || warp == kWarpAProducer || warp == kWarpSProducer)) ||
        (LANES && warp == kWarpSProducer))
    {
        have0 = wk0.next(p, t0);
        NVFP4_TRACE_MAX(kTrWalked);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kOffTmemSlot);
    if (threadIdx.x == 0) NVFP4_TRACE_AT(kTrPrologue);
    // Launched after another kernel of the stream with programmatic
    // serialisation, everything above (barriers, TMEM, the problem table,
    // tensor-map prefetch, the walk to the first tile) overlaps that kernel's
    // last CTAs. The threads that touch global memory the previous kernel
    // may use (the three producers before their first load, the epilogue
    // before its first store) wait for it to complete right there, after
    // preparing that first load: code and parameters a thread touches for
    // the first time cost it memory round trips, which are better spent
    // before the wait than after it. The MMA thread and the scale writers
    // work on shared memory and TMEM only. The next kernel may be scheduled
    // from here on: its CTAs find an SM only as this grid's CTAs exit.
    griddep_launch_dependents();

    if (warp == kWarpBProducer) {
        if (lane == 0) r.b_producer(wk0, t0, have0);
    } else if (warp == kWarpAProducer) {
        if (lane == 0) r.a_producer(wk0, t0, have0);
    } else if (warp == kWarpSProducer) {
        if constexpr (LANES) r.s_producer_lanes(wk0, t0, have0, lane);
        else if (lane == 0) r.s_producer(wk0, t0, have0);
    } else if (warp == kWarpMma) {
        if (lane == 0) r.mma_issuer(tmem);
    } else if ((warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) || warp >= kWarpEpi1) {
        r.epilogue(tmem, warp, lane);
    } else if (warp >= kWarpSf0 && warp < kWarpSf0 + kNumSfWarps) {
        r.sf_writer(tmem, warp, lane);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0) NVFP4_TRACE_AT(kTrEnd);
}


// ------------------------------------------------------------------- variants

using KernelFn = void (*)(GemmParams);

struct VariantEntry {
    GemmVariant v;
    bool is_default;
    KernelFn fn;
    int smem;
};

template <int MAXN, int NB, int NA, int NS, bool RAW, int UNIT, bool LANES = false>
constexpr VariantEntry make_entry(bool is_default)
{
    return VariantEntry{GemmVariant{MAXN, NB, NA, RAW, UNIT, LANES}, is_default,
                        &ggemm_kernel<MAXN, NB, NA, NS, RAW, UNIT, LANES>, Cfg<MAXN, NB, NA, NS, RAW>::kSmemBytes};
}

// (MAXN, B stages, A stages, scale stages, raw scales, row tiles per unit
// [, lane copies of raw scale rows]): each ring configuration for pairs of
// row tiles and for single row tiles
const VariantEntry kVariants[] = {
    make_entry<256, 3, 3, 2, true, 2>(true),  make_entry<256, 3, 3, 3, false, 2>(true),
    make_entry<256, 4, 2, 2, true, 2>(false), make_entry<128, 8, 2, 2, true, 2>(true),
    make_entry<128, 8, 2, 3, false, 2>(true), make_entry<256, 3, 3, 2, true, 1>(true),
    make_entry<256, 3, 3, 3, false, 1>(true), make_entry<256, 4, 2, 2, true, 1>(false),
    make_entry<128, 8, 2, 2, true, 1>(true),  make_entry<128, 8, 2, 3, false, 1>(true),
    make_entry<256, 3, 3, 2, true, 2, true>(true), make_entry<256, 3, 3, 2, true, 1, true>(true),
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

}  // namespace

int ggemm_variant_index(int max_n, int b_stages, int a_stages, bool sf_raw, int unit, bool lanes)
{
    for (int i = 0; i < kNumVariants; ++i) {
        const GemmVariant &v = kVariants[i].v;
        if (v.max_n != max_n || v.sf_raw != sf_raw || v.unit != unit || v.lanes != lanes) continue;
        if (b_stages == 0 && a_stages == 0 && kVariants[i].is_default) return i;
        if (v.b_stages == b_stages && v.a_stages == a_stages) return i;
    }
    return -1;
}

GemmVariant ggemm_variant(int index) { return kVariants[index].v; }

int ggemm_smem_bytes(int index) { return kVariants[index].smem; }

int ggemm_threads() { return kThreads; }

cudaError_t ggemm_configure(int index)
{
    return cudaFuncSetAttribute(kVariants[index].fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kVariants[index].smem);
}

cudaError_t ggemm_launch(int index, const GemmParams &p, int grid, cudaStream_t stream, bool overlap_prev)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = (size_t)kVariants[index].smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap_prev ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kVariants[index].fn, p);
}

}  // namespace nvfp4
