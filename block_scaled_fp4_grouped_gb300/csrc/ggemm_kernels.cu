// Device code: the persistent warp-specialised NVFP4 grouped GEMM and the
// scale re-layout kernel, for sm_103a.
//
// GEMM structure (one CTA per SM, persistent):
//   warp 0      TMA producer: per 256-k stage loads MT A tiles (128 x 128 B),
//               one B tile (BN x 128 B, 128-byte swizzle) and their scales
//               into a ring of NS shared-memory stages on mbarriers.
//   warp 1      allocates TMEM; one lane copies scales to TMEM
//               (tcgen05.cp) and issues kind::mxf4nvf4 block16 MMAs into
//               the accumulator, committing each stage back to the producer.
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, RN to fp16,
//               swizzled staging in shared memory, TMA stores clipped to
//               M_g x N.
//   warp 6      (raw-scale path only) permutes raw 128-row x 16-byte scale
//               tiles into the 512-byte atoms the scale copy expects.
// A work unit is (group, MT consecutive 128-row tiles, one BN-column strip):
// the MT row tiles share every B stage, so a B strip is streamed from HBM
// once for up to 2*128 rows of A. Units of all groups are numbered through
// the per-group prefix sums and dealt to CTAs round-robin.
//
// Every mbarrier wait is bounded by the plan's timeout: on expiry the waiter
// records (status, site, block) in the error word, raises a CTA-wide abort
// flag and leaves its loop; all warps then drain their own asynchronous
// work, TMEM is released and the kernel returns normally.
#include <cuda_fp16.h>

#include "ggemm_internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

using namespace ptx;

constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kNumEpiWarps = 4;
constexpr int kWarpPermute = 6;
constexpr int kThreads = 7 * 32;

constexpr int kATileBytes = kTileM * (kTileK / 2);  // 16384
constexpr int kSfTileBytes = 4 * kSfAtomBytes;       // 2048: 128 rows x 256 k of scales
constexpr int kStagingBytes = 32 * 128;              // 32 rows x 64 fp16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kStatusTimeout = 6;  // NVFP4_ERR_TIMEOUT

template <int BN, int MT, int NS, bool RAW>
struct Cfg {
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "one scale atom column group covers at most 128 rows");
    static_assert(MT >= 1 && MT <= 2, "at most two row tiles per unit");
    static constexpr int kBBytes = BN * (kTileK / 2);
    static constexpr int kOffA = 0;
    static constexpr int kOffB = MT * kATileBytes;
    static constexpr int kOffSfa = kOffB + kBBytes;
    static constexpr int kOffSfb = kOffSfa + MT * kSfTileBytes;
    static constexpr int kStageBytes = kOffSfb + kSfTileBytes;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
    static constexpr int kOffStaging = NS * kStageBytes;
    static constexpr int kOffBars = kOffStaging + kNumEpiWarps * 2 * kStagingBytes;
    static constexpr int kNumBars = 3 * NS + 2 + 2 + 1;
    static constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1024
    static constexpr int kAccCols = MT * BN;                  // fp32 accumulator columns per buffer
    static constexpr int kSfCols = (MT + 1) * 16;             // scale columns per buffer
    static constexpr int kNumAcc = (2 * kAccCols + 2 * kSfCols <= (int)kTmemCols) ? 2 : 1;
    static constexpr int kSfBase = kNumAcc * kAccCols;
    static_assert(kSfBase + 2 * kSfCols <= (int)kTmemCols, "TMEM budget");
    static constexpr uint32_t kIdesc = idesc_mxf4nvf4_m128(BN);
    static constexpr uint32_t kSfbBytes = RAW ? BN * 16 : kSfTileBytes;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct Unit {
    int g;
    int mtile0;  // first 128-row tile of the unit
    int mtu;     // row tiles in this unit (1..MT)
    int n0;      // first column
};

template <int BN, int MT>
__device__ __forceinline__ Unit decode_unit(const GemmParams &p, int u)
{
    int lo = 0, hi = p.G;  // prefix[lo] <= u < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.unit_prefix + mid) <= u) lo = mid;
        else hi = mid;
    }
    const GroupDesc *gd = p.groups + lo;
    const int l = u - __ldg(p.unit_prefix + lo);
    const int mg = gd->m_groups;
    Unit t;
    t.g = lo;
    t.mtile0 = (l % mg) * MT;
    t.n0 = (l / mg) * BN;
    t.mtu = min(MT, gd->m_tiles - t.mtile0);
    return t;
}

__device__ __forceinline__ void record_error(uint32_t *err, uint32_t status, uint32_t site)
{
    const uint32_t word = status | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16);
    atomicCAS(err, 0u, word);
}

// Bounded wait for phase `parity` of `bar`. False when another warp aborted
// or the timeout expired (then this thread records the error and aborts).
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                        const GemmParams &p, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
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

template <int c>
__device__ __forceinline__ uint32_t word_of(const uint4 &v)
{
    return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

// In-place permutation of one raw scale tile ([rows][16 B], row r at 16r)
// into four 512-byte atoms: atom c holds the 4 scales of k in [64c, 64c+64)
// of row r at byte (r%32)*16 + (r/32)*4. Lane i owns rows i, i+32, i+64, i+96.
__device__ __forceinline__ void permute_sf_tile(uint8_t *tile, int rows, int lane)
{
    uint4 w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        w[j] = (r < rows) ? *reinterpret_cast<const uint4 *>(tile + 16 * r) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
    *reinterpret_cast<uint4 *>(tile + 0 * 512 + 16 * lane) =
        make_uint4(word_of<0>(w[0]), word_of<0>(w[1]), word_of<0>(w[2]), word_of<0>(w[3]));
    *reinterpret_cast<uint4 *>(tile + 1 * 512 + 16 * lane) =
        make_uint4(word_of<1>(w[0]), word_of<1>(w[1]), word_of<1>(w[2]), word_of<1>(w[3]));
    *reinterpret_cast<uint4 *>(tile + 2 * 512 + 16 * lane) =
        make_uint4(word_of<2>(w[0]), word_of<2>(w[1]), word_of<2>(w[2]), word_of<2>(w[3]));
    *reinterpret_cast<uint4 *>(tile + 3 * 512 + 16 * lane) =
        make_uint4(word_of<3>(w[0]), word_of<3>(w[1]), word_of<3>(w[2]), word_of<3>(w[3]));
    __syncwarp();
}

template <int BN, int MT, int NS, bool RAW>
struct Roles {
    using C = Cfg<BN, MT, NS, RAW>;

    uint8_t *smem;
    uint32_t sbase;
    volatile int *abort_flag;
    const GemmParams &p;

    __device__ Roles(uint8_t *s, const GemmParams &params)
        : smem(s), sbase(smem_addr(s)), abort_flag(reinterpret_cast<volatile int *>(s + C::kOffAbort)), p(params)
    {
    }

    __device__ __forceinline__ uint32_t bar_full(int s) const { return sbase + C::kOffBars + 8 * s; }
    __device__ __forceinline__ uint32_t bar_empty(int s) const { return sbase + C::kOffBars + 8 * (NS + s); }
    __device__ __forceinline__ uint32_t bar_sf(int s) const { return sbase + C::kOffBars + 8 * (2 * NS + s); }
    __device__ __forceinline__ uint32_t bar_acc_full(int a) const { return sbase + C::kOffBars + 8 * (3 * NS + a); }
    __device__ __forceinline__ uint32_t bar_acc_empty(int a) const
    {
        return sbase + C::kOffBars + 8 * (3 * NS + 2 + a);
    }
    __device__ __forceinline__ uint32_t bar_drain() const { return sbase + C::kOffBars + 8 * (3 * NS + 4); }
    __device__ __forceinline__ uint32_t stage_addr(int s) const { return sbase + s * C::kStageBytes; }

    __device__ void init_barriers()
    {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
            mbar_init(bar_sf(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_acc_full(a), 1);
            mbar_init(bar_acc_empty(a), kNumEpiWarps);
        }
        mbar_init(bar_drain(), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }

    // ---------------------------------------------------------------- producer
    __device__ void producer()
    {
        const uint64_t pol_a = policy_evict_last();   // A tiles are re-read by every column strip
        const uint64_t pol_b = policy_evict_first();  // B streams through once
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        int last_g = -1;
        int loads = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
            const Unit t = decode_unit<BN, MT>(p, u);
            const GroupDesc *gd = p.groups + t.g;
            if (t.g != last_g) {
                fence_tensormap_acquire(&gd->tmA);
                fence_tensormap_acquire(&gd->tmB);
                if (RAW) {
                    fence_tensormap_acquire(&gd->tmSFA);
                    fence_tensormap_acquire(&gd->tmSFB);
                }
                last_g = t.g;
            }
            const uint32_t bytes = (uint32_t)t.mtu * (kATileBytes + kSfTileBytes) + C::kBBytes + C::kSfbBytes;
            const size_t katoms = (size_t)(p.K / 64);
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!wait_phase(bar_empty(stage), phase ^ 1u, abort_flag, p, kSiteEmpty)) {
                    ok = false;
                    break;
                }
                ++loads;
                const bool skip = (p.debug_skip_load > 0 && blockIdx.x == 0 && loads == p.debug_skip_load);
                if (!skip) {
                    const uint32_t bar = bar_full(stage);
                    const uint32_t st = stage_addr(stage);
                    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        if (mt < t.mtu)
                            tma_load_2d(st + C::kOffA + mt * kATileBytes, &gd->tmA, kt * (kTileK / 2),
                                        (t.mtile0 + mt) * kTileM, bar, pol_a);
                    tma_load_2d(st + C::kOffB, &gd->tmB, kt * (kTileK / 2), t.n0, bar, pol_b);
                    if (RAW) {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
                            if (mt < t.mtu)
                                tma_load_2d(st + C::kOffSfa + mt * kSfTileBytes, &gd->tmSFA, kt * (kTileK / 16),
                                            (t.mtile0 + mt) * kTileM, bar, pol_a);
                        tma_load_2d(st + C::kOffSfb, &gd->tmSFB, kt * (kTileK / 16), t.n0, bar, pol_b);
                    } else {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
                            if (mt < t.mtu)
                                bulk_load(st + C::kOffSfa + mt * kSfTileBytes,
                                          gd->sfa_atoms + ((size_t)(t.mtile0 + mt) * katoms + (size_t)kt * 4) *
                                                              kSfAtomBytes,
                                          kSfTileBytes, bar, pol_a);
                        bulk_load(st + C::kOffSfb,
                                  gd->sfb_atoms + ((size_t)(t.n0 / 128) * katoms + (size_t)kt * 4) * kSfAtomBytes,
                                  kSfTileBytes, bar, pol_b);
                    }
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                } else {
                    issued_mask &= ~(1u << stage);  // nothing in flight for this stage
                }
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Every load issued here must have landed before the CTA may exit.
        for (int s = 0; s < NS; ++s)
            if ((issued_mask >> s) & 1u) wait_drain(bar_full(s), (issued_parity >> s) & 1u, p, kSiteLoadDrain);
    }

    // ------------------------------------------------------------- MMA issuer
    __device__ void mma_issuer(uint32_t tmem)
    {
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t sf_buf = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
            const Unit t = decode_unit<BN, MT>(p, u);
            if (!wait_phase(bar_acc_empty(acc), acc_phase ^ 1u, abort_flag, p, kSiteAccEmpty)) break;
            tc_fence_after_sync();
            const uint32_t d0 = tmem + (uint32_t)(acc * C::kAccCols);
            // atom layout: a 64-row strip inside a 128-row atom uses its upper columns
            const uint32_t sfb_sub = RAW ? 0u : (uint32_t)((t.n0 % 128) / 32);
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                const bool got = RAW ? wait_phase(bar_sf(stage), phase, abort_flag, p, kSiteSfReady)
                                     : wait_phase(bar_full(stage), phase, abort_flag, p, kSiteFull);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = stage_addr(stage);
                const uint32_t sf = tmem + (uint32_t)(C::kSfBase + sf_buf * C::kSfCols);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                    if (mt < t.mtu)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_cp_sf_atom(sf + mt * 16 + kk * 4,
                                          desc_sf_atom(st + C::kOffSfa + mt * kSfTileBytes + kk * kSfAtomBytes));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_cp_sf_atom(sf + MT * 16 + kk * 4, desc_sf_atom(st + C::kOffSfb + kk * kSfAtomBytes));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bdesc = desc_sw128_kmajor(st + C::kOffB + kk * 32);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        if (mt < t.mtu)
                            tc_mma_nvf4(d0 + mt * BN, desc_sw128_kmajor(st + C::kOffA + mt * kATileBytes + kk * 32),
                                        bdesc, C::kIdesc, sf + mt * 16 + kk * 4, sf + MT * 16 + kk * 4 + sfb_sub,
                                        (kt | kk) != 0 ? 1u : 0u);
                }
                tc_commit(bar_empty(stage));  // frees the stage once these MMAs have read it
                sf_buf ^= 1u;
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit(bar_acc_full(acc));
            if (++acc == C::kNumAcc) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // All tcgen05 work issued by this thread completes before TMEM is released.
        tc_commit(bar_drain());
        wait_drain(bar_drain(), 0, p, kSiteMmaDrain);
    }

    // --------------------------------------------------------------- epilogue
    __device__ void epilogue(uint32_t tmem, int warp, int lane)
    {
        const int q = warp & 3;  // the TMEM lane quarter this warp may read
        const int e = warp - kWarpEpi0;
        uint8_t *stage_ptr = smem + C::kOffStaging + e * 2 * kStagingBytes;
        const uint32_t stage_sa = sbase + C::kOffStaging + e * 2 * kStagingBytes;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sb = 0;
        int last_g = -1;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            const Unit t = decode_unit<BN, MT>(p, u);
            const GroupDesc *gd = p.groups + t.g;
            if (t.g != last_g) {
                if (lane == 0) fence_tensormap_acquire(&gd->tmC);
                last_g = t.g;
            }
            if (!warp_wait_phase(bar_acc_full(acc), acc_phase, abort_flag, p, kSiteAccFull)) break;
            tc_fence_after_sync();
            const int M = gd->M;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int row0 = (t.mtile0 + mt) * kTileM + 32 * q;
                if (mt >= t.mtu || row0 >= M) continue;
#pragma unroll 1
                for (int cc = 0; cc < BN / 64; ++cc) {
                    const int col0 = t.n0 + cc * 64;
                    if (col0 >= p.N) break;
                    uint32_t v0[32], v1[32];
                    const uint32_t taddr =
                        tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * C::kAccCols + mt * BN + cc * 64);
                    tmem_ld_32x32b_x32(taddr, v0);
                    tmem_ld_32x32b_x32(taddr + 32, v1);
                    tmem_ld_wait();
                    // staging buffer sb is free once at most one store (the other buffer's) still reads smem
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    uint8_t *row_ptr = stage_ptr + sb * kStagingBytes + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t *src = (j < 4) ? &v0[8 * j] : &v1[8 * (j - 4)];
                        uint4 pk;
                        pk.x = pack_half2(src[0], src[1]);
                        pk.y = pack_half2(src[2], src[3]);
                        pk.z = pack_half2(src[4], src[5]);
                        pk.w = pack_half2(src[6], src[7]);
                        // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
                        *reinterpret_cast<uint4 *>(row_ptr + ((j ^ (lane & 7)) * 16)) = pk;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&gd->tmC, col0, row0, stage_sa + sb * kStagingBytes);
                        bulk_commit_group();
                    }
                    sb ^= 1;
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty(acc));
            if (++acc == C::kNumAcc) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ----------------------------------------------------------- scale permuter
    __device__ void sf_permuter(int lane)
    {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
            const Unit t = decode_unit<BN, MT>(p, u);
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!warp_wait_phase(bar_full(stage), phase, abort_flag, p, kSiteFull)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + stage * C::kStageBytes;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                    if (mt < t.mtu) permute_sf_tile(st + C::kOffSfa + mt * kSfTileBytes, kTileM, lane);
                permute_sf_tile(st + C::kOffSfb, BN, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sf(stage));
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
};

template <int BN, int MT, int NS, bool RAW>
__global__ void __launch_bounds__(kThreads, 1) ggemm_kernel(const __grid_constant__ GemmParams p)
{
    using C = Cfg<BN, MT, NS, RAW>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Roles<BN, MT, NS, RAW> r(smem, p);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) r.init_barriers();
    if (warp == kWarpMma) {
        tmem_alloc(r.sbase + C::kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kOffTmemSlot);

    if (warp == kWarpProducer) {
        if (lane == 0) r.producer();
    } else if (warp == kWarpMma) {
        if (lane == 0) r.mma_issuer(tmem);
    } else if (warp < kWarpEpi0 + kNumEpiWarps) {
        r.epilogue(tmem, warp, lane);
    } else if (RAW && warp == kWarpPermute) {
        r.sf_permuter(lane);
    }
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ scale re-layout

// One warp per item = (matrix, 128-row block, 16-byte column piece of the
// raw rows, i.e. 4 x 64 k). Lane i reads rows i, i+32, i+64, i+96 of the
// block (16 bytes each) and writes 16 contiguous bytes into each of the four
// atoms, so every atom is written as one 512-byte coalesced store.
__global__ void __launch_bounds__(256) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int pieces = p.K / 256;
    const int katoms = p.K / 64;
    const size_t row_bytes = (size_t)(p.K / 16);
    for (int item = blockIdx.x * wpb + (threadIdx.x >> 5); item < p.total_items; item += gridDim.x * wpb) {
        RelayoutJob job;
        if (p.jobs == nullptr) {
            job = p.single;
        } else {
            int lo = 0, hi = p.njobs;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.jobs[mid].item_begin <= item) lo = mid;
                else hi = mid;
            }
            job = p.jobs[lo];
        }
        const int l = item - job.item_begin;
        const int rb = l / pieces;
        const int pc = l % pieces;
        uint4 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = rb * 128 + 32 * j + lane;
            w[j] = (r < job.rows) ? __ldg(reinterpret_cast<const uint4 *>(job.src + (size_t)r * row_bytes + pc * 16))
                                  : make_uint4(0u, 0u, 0u, 0u);
        }
        uint8_t *dst = job.dst + ((size_t)rb * katoms + (size_t)pc * 4) * kSfAtomBytes + 16 * lane;
        *reinterpret_cast<uint4 *>(dst + 0 * kSfAtomBytes) =
            make_uint4(word_of<0>(w[0]), word_of<0>(w[1]), word_of<0>(w[2]), word_of<0>(w[3]));
        *reinterpret_cast<uint4 *>(dst + 1 * kSfAtomBytes) =
            make_uint4(word_of<1>(w[0]), word_of<1>(w[1]), word_of<1>(w[2]), word_of<1>(w[3]));
        *reinterpret_cast<uint4 *>(dst + 2 * kSfAtomBytes) =
            make_uint4(word_of<2>(w[0]), word_of<2>(w[1]), word_of<2>(w[2]), word_of<2>(w[3]));
        *reinterpret_cast<uint4 *>(dst + 3 * kSfAtomBytes) =
            make_uint4(word_of<3>(w[0]), word_of<3>(w[1]), word_of<3>(w[2]), word_of<3>(w[3]));
    }
}

// ------------------------------------------------------------------- variants

using KernelFn = void (*)(GemmParams);

struct VariantEntry {
    GemmVariant v;
    KernelFn fn;
    int smem;
};

template <int BN, int MT, int NS, bool RAW>
constexpr VariantEntry make_entry()
{
    return VariantEntry{GemmVariant{BN, MT, NS, RAW}, &ggemm_kernel<BN, MT, NS, RAW>, Cfg<BN, MT, NS, RAW>::kSmemBytes};
}

const VariantEntry kVariants[] = {
    make_entry<128, 2, 3, false>(),
    make_entry<128, 2, 3, true>(),
    make_entry<64, 2, 4, false>(),
    make_entry<64, 2, 4, true>(),
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

}  // namespace

int ggemm_variant_index(int tile_n, bool sf_raw)
{
    for (int i = 0; i < kNumVariants; ++i)
        if (kVariants[i].v.tile_n == tile_n && kVariants[i].v.sf_raw == sf_raw) return i;
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

cudaError_t ggemm_launch(int index, const GemmParams &p, int grid, cudaStream_t stream)
{
    kVariants[index].fn<<<grid, kThreads, kVariants[index].smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t relayout_launch(const RelayoutParams &p, int sm_count, cudaStream_t stream)
{
    if (p.total_items <= 0) return cudaSuccess;
    const int warps_per_block = 8;
    int blocks = (p.total_items + warps_per_block - 1) / warps_per_block;
    const int cap = sm_count * 8;
    if (blocks > cap) blocks = cap;
    sf_relayout_kernel<<<blocks, warps_per_block * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
