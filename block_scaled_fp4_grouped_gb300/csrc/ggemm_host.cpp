// Host side of the C ABI: argument validation, the work decomposition
// (prefix sums of column chunks, per-CTA ranges), per-group TMA tensor maps
// in a device-resident problem table, workspace for re-laid-out scales,
// kernel launches and the device error word.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cudaTypedefs.h>

#include "ggemm_internal.h"
#include "io_copy.h"
#include "nvfp4_ggemm.h"

using namespace nvfp4;

namespace {

constexpr int kVersion = 10200;  // 1.2.0: row_units, nvfp4_ggemm_schedule_units, plan_info.row_units/split_acc
constexpr int kMaxGroups = 1024;
constexpr int32_t kMaxM = 1 << 20;
constexpr int32_t kMaxN = 1 << 20;
constexpr int32_t kMaxK = 1 << 18;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kSlots = 4;  // problem-table ring: a table is rewritten only after its last kernel finished
constexpr int kDefaultTileN = 256;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

#ifdef NVFP4_TRACE
// Timeline build: launch i of the process stores its stamps in block
// i % g_trace_calls of g_trace (kMaxCtas x kTraceSlots entries each).
unsigned long long *g_trace = nullptr;
int g_trace_calls = 0;
long g_trace_next = 0;
#endif
std::once_flag g_encode_once;

bool load_encode()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Per-group N and K limits: 16-byte C rows; whole 64-k MMA slices (a last
// 256-k stage may be partial). Raw scale rows are 16-byte TMA rows only when
// K % 256 == 0; the kernel copies other raw rows with cp.async.
inline bool shape_ok(int32_t N, int32_t K)
{
    return N >= 8 && N <= kMaxN && N % 8 == 0 && K >= 64 && K <= kMaxK && K % 64 == 0;
}

inline bool raw_tma_ok(int32_t K) { return K % 256 == 0; }

uint64_t atom_bytes(int64_t rows, int64_t K)
{
    return (uint64_t)((rows + 127) / 128) * (uint64_t)(K / 64) * (uint64_t)kSfAtomBytes;
}

// 2-D tensor map over a row-major [rows][cols] matrix of `esize`-byte elements.
bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t cols, uint64_t rows,
               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tensor map over an atom-layout scale matrix: [blocks][katoms] atoms of
// 512 bytes (a 128-row block's atoms of successive 64-k slices contiguous),
// read as 8-byte elements; a box is the four atoms of one k tile of
// `box_blocks` consecutive 128-row blocks (2 KB each, one after another).
bool encode_atoms(CUtensorMap *map, const void *base, uint64_t katoms, uint64_t blocks, uint32_t box_blocks)
{
    cuuint64_t dims[3] = {kSfAtomBytes / 8, katoms, blocks};
    cuuint64_t strides[2] = {kSfAtomBytes, katoms * kSfAtomBytes};
    cuuint32_t box[3] = {kSfAtomBytes / 8, kTileK / 64, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Smallest kernel tile width (128 or 256) that holds `tile_n` columns.
int variant_width(int tile_n) { return tile_n <= 128 ? 128 : 256; }

struct Slot {
    uint8_t *h_table = nullptr;  // pinned staging
    uint8_t *d_table = nullptr;
    cudaEvent_t ev = nullptr;
    bool used = false;
    std::vector<const void *> key;
    GemmParams *params = nullptr;  // the kernel parameters for this table (built when it is filled)
};

}  // namespace

namespace nvfp4 {

TensorMapEncodeFn tensor_map_encoder()
{
    return load_encode() ? reinterpret_cast<TensorMapEncodeFn>(g_encode) : nullptr;
}

int pair_cap_chunks(int max_n) { return (max_n >= 192 ? 192 : max_n) / kChunkN; }

int schedule_ctas(const GroupShape *shapes, int G, int unit, int cap_single, int cap_pair, int max_ctas,
                  int32_t *cta_begin, int32_t *counts)
{
    max_ctas = std::max(1, std::min(max_ctas, kMaxCtas));
    // segments: units of `unit` row tiles; the last unit of a group may have fewer
    long nseg = 0, total = 0;
    for (int g = 0; g < G; ++g) {
        const long units = ceil_div(shapes[g].m_tiles, unit);
        nseg += units;
        total += units * shapes[g].n_chunks;
    }
    if (total == 0) {
        cta_begin[0] = 0;
        return 0;
    }
    if (nseg > max_ctas) {
        // more segments than CTAs: equal contiguous chunk ranges
        const int grid = (int)std::min<long>(total, max_ctas);
        for (int c = 0; c <= grid; ++c) cta_begin[c] = (int32_t)((long)c * total / grid);
        return grid;
    }
    auto seg_cap = [&](int g, int t) { return unit == 2 && (shapes[g].m_tiles - t) >= 2 ? cap_pair : cap_single; };
    // CTAs a segment needs when a CTA may spend `budget` k-stages on it (at
    // least one pass). A CTA that walks two or more tiles of two row tiles
    // takes them one chunk narrower: such tiles fill both accumulator halves,
    // so each tile boundary waits for the previous tile's epilogue; narrower
    // tiles shorten that wait and spread the pair over more CTAs.
    auto ctas_for = [&](int g, int t, long budget) {
        const long passes = std::max<long>(1, budget / shapes[g].k_tiles);
        const bool pair = unit == 2 && (shapes[g].m_tiles - t) >= 2;
        const long cap = seg_cap(g, t);
        const long per_cta = passes * (pair && passes > 1 && cap > 2 ? cap - 1 : cap);
        return (shapes[g].n_chunks + per_cta - 1) / per_cta;
    };
    auto need = [&](long budget) {
        long n = 0;
        for (int g = 0; g < G; ++g)
            for (int t = 0; t < shapes[g].m_tiles; t += unit) n += ctas_for(g, t, budget);
        return n;
    };
    // the smallest budget that fits (need() does not grow with the budget; a
    // budget of max(k) * max(n) gives one CTA per segment)
    long hi = 1;
    for (int g = 0; g < G; ++g) hi = std::max<long>(hi, (long)shapes[g].k_tiles * shapes[g].n_chunks);
    long lo = 1;
    while (lo < hi) {
        const long mid = lo + (hi - lo) / 2;
        if (need(mid) <= max_ctas) hi = mid;
        else lo = mid + 1;
    }
    int grid = 0;
    {
        long s = 0;
        for (int g = 0; g < G; ++g)
            for (int t = 0; t < shapes[g].m_tiles; t += unit, ++s) counts[s] = (int32_t)ctas_for(g, t, lo);
        for (long i = 0; i < nseg; ++i) grid += counts[i];
    }
    // spare CTAs shorten the longest ranges, measured in k-stages, then in chunks
    for (; grid < max_ctas; ++grid) {
        long best = -1, best_stages = 0, best_len = 0;
        long s = 0;
        for (int g = 0; g < G; ++g)
            for (int t = 0; t < shapes[g].m_tiles; t += unit, ++s) {
                const int n = shapes[g].n_chunks;
                if (counts[s] >= n) continue;
                const long len = (n + counts[s] - 1) / counts[s];  // longest range of this segment
                const long cap = seg_cap(g, t);
                const long stages = (len + cap - 1) / cap * shapes[g].k_tiles;
                if (best < 0 || stages > best_stages || (stages == best_stages && len > best_len)) {
                    best = s;
                    best_stages = stages;
                    best_len = len;
                }
            }
        if (best < 0) break;
        ++counts[best];
    }
    int c = 0;
    long s = 0, base = 0;
    for (int g = 0; g < G; ++g)
        for (int t = 0; t < shapes[g].m_tiles; t += unit, ++s) {
            const long n = shapes[g].n_chunks;
            for (int j = 0; j < counts[s]; ++j) cta_begin[c++] = (int32_t)(base + (long)j * n / counts[s]);
            base += n;
        }
    cta_begin[c] = (int32_t)total;
    return c;
}

void fill_cta_ranges(CtaRange *ranges, const int32_t *cta_begin, int grid, const int32_t *chunk_prefix,
                     const GroupShape *shapes, int G, int unit, int cap_single, int cap_pair)
{
    int g = 0;
    for (int c = 0; c < grid; ++c) {
        CtaRange &r = ranges[c];
        r = CtaRange{};
        r.begin = cta_begin[c];
        r.end = cta_begin[c + 1];
        while (g + 1 < G && chunk_prefix[g + 1] <= r.begin) ++g;  // ranges ascend, so g only moves forward
        r.g = g;
        r.g_base = chunk_prefix[g];
        r.g_tiles = shapes[g].m_tiles;
        r.g_rows = shapes[g].M;
        // the kernel's walk: the part of the range in each unit is cut into
        // ceil(len / cap) tiles of equal width (to within one chunk)
        int pos = r.begin, wg = g;
        r.max_chunks = 1;
        r.max_rows = 1;
        while (pos < r.end) {
            while (pos >= chunk_prefix[wg] + ceil_div(shapes[wg].m_tiles, unit) * shapes[wg].n_chunks) ++wg;
            const int n = shapes[wg].n_chunks;
            const int local = pos - chunk_prefix[wg];
            const int mp = local / n;
            const int ch0 = local - mp * n;
            const int mtu = std::min(unit, shapes[wg].m_tiles - mp * unit);
            const int plen = std::min(n - ch0, r.end - pos);
            const int cap = mtu == 2 ? cap_pair : cap_single;
            const int pt = ceil_div(plen, cap);
            r.max_chunks = std::max(r.max_chunks, ceil_div(plen, pt));
            r.max_rows = std::max(r.max_rows, mtu);
            pos += plen;
        }
    }
}

void order_ctas(uint8_t *order, const CtaRange *ranges, int grid, const int32_t *chunk_prefix, const GroupShape *shapes,
                int unit, int cap_single, int cap_pair)
{
    double cost[kMaxCtas];
    int wg = 0;  // ranges ascend, so the group walk only moves forward
    for (int c = 0; c < grid; ++c) {
        cost[c] = 0.0;
        int pos = ranges[c].begin;
        while (pos < ranges[c].end) {
            while (pos >= chunk_prefix[wg] + ceil_div(shapes[wg].m_tiles, unit) * shapes[wg].n_chunks) ++wg;
            const int n = shapes[wg].n_chunks;
            const int local = pos - chunk_prefix[wg];
            const int mp = local / n;
            const int ch0 = local - mp * n;
            const int mtu = std::min(unit, shapes[wg].m_tiles - mp * unit);
            const int plen = std::min(n - ch0, ranges[c].end - pos);
            const int pt = ceil_div(plen, mtu == 2 ? cap_pair : cap_single);
            const double b_bytes = (double)plen * kChunkN * shapes[wg].k_tiles * (kTileK / 2) * 9.0 / 8.0;
            const int rows = std::max(0, std::min(shapes[wg].M - mp * unit * kTileM, mtu * kTileM));
            const double c_bytes = (double)rows * plen * kChunkN * 2.0;
            const double wait = (mtu == 2 && pt >= 2) ? 4.0 * c_bytes * (pt - 1) / pt : 0.0;
            cost[c] += b_bytes + c_bytes + wait;
            pos += plen;
        }
    }
    int idx[kMaxCtas];
    for (int c = 0; c < grid; ++c) idx[c] = c;
    std::stable_sort(idx, idx + grid, [&](int a, int b) { return cost[a] > cost[b]; });
    for (int c = 0; c < grid; ++c) order[c] = (uint8_t)idx[c];
}

namespace {

// The kernel's walk of a schedule: the most tiles and k-stages any CTA
// walks, and the widest tile (chunks) of two row tiles and of one.
struct WalkStats {
    int max_tiles = 0;
    long max_stages = 0;
    int max_pair_chunks = 0;
    int max_single_chunks = 0;
};

WalkStats walk_stats(const GroupShape *shapes, int G, int unit, int cap_single, int cap_pair,
                     const int32_t *cta_begin, int grid)
{
    WalkStats w;
    int g = 0;
    long base = 0;  // first chunk of group g; ranges ascend, so g only moves forward
    for (int c = 0; c < grid; ++c) {
        long pos = cta_begin[c];
        int tiles = 0;
        long stages = 0;
        while (pos < cta_begin[c + 1]) {
            while (g < G && pos >= base + (long)ceil_div(shapes[g].m_tiles, unit) * shapes[g].n_chunks) {
                base += (long)ceil_div(shapes[g].m_tiles, unit) * shapes[g].n_chunks;
                ++g;
            }
            if (g >= G) break;
            const long n = shapes[g].n_chunks;
            const long mp = (pos - base) / n;
            const long len = std::min<long>(base + (mp + 1) * n, cta_begin[c + 1]) - pos;
            const int mtu = std::min<int>(unit, shapes[g].m_tiles - (int)mp * unit);
            const long cap = mtu == 2 ? cap_pair : cap_single;
            const long pt = (len + cap - 1) / cap;
            const int width = (int)((len + pt - 1) / pt);
            tiles += (int)pt;
            stages += pt * shapes[g].k_tiles;
            if (mtu == 2) w.max_pair_chunks = std::max(w.max_pair_chunks, width);
            else w.max_single_chunks = std::max(w.max_single_chunks, width);
            pos += len;
        }
        w.max_tiles = std::max(w.max_tiles, tiles);
        w.max_stages = std::max(w.max_stages, stages);
    }
    return w;
}

}  // namespace

UnitChoice choose_units(const GroupShape *shapes, int G, int cap_single, int cap_pair, int max_ctas, int forced)
{
    if (forced == 2) return UnitChoice{2, false};
    int32_t begin[kMaxCtas + 1];
    int32_t counts[kMaxCtas];
    const int grid1 = schedule_ctas(shapes, G, 1, cap_single, cap_pair, max_ctas, begin, counts);
    const WalkStats w1 = walk_stats(shapes, G, 1, cap_single, cap_pair, begin, grid1);
    // every CTA walks one tile: splitting a tile's accumulator over both
    // halves never stalls a next tile (the kernel splits those of at most
    // half the accumulator columns)
    const bool split = grid1 > 0 && w1.max_tiles == 1;
    if (forced == 1) return UnitChoice{1, split};
    const int grid2 = schedule_ctas(shapes, G, 2, cap_single, cap_pair, max_ctas, begin, counts);
    const WalkStats w2 = walk_stats(shapes, G, 2, cap_single, cap_pair, begin, grid2);
    if (w2.max_pair_chunks > 0 && w2.max_pair_chunks <= 4 && split && w1.max_stages <= w2.max_stages)
        return UnitChoice{1, true};
    return UnitChoice{2, false};
}

void pack_cta_starts(CtaStart *out, const CtaRange *ranges, int grid, int total_chunks, const GroupShape *shapes)
{
    for (int c = 0; c < grid; ++c) {
        const CtaRange &r = ranges[c];
        const GroupShape &sh = shapes[r.g];
        out[c].begin = r.begin;
        out[c].g_base = r.g_base;
        out[c].rows = cta_pack_rows(sh.M, sh.k_tiles);
        out[c].packed = cta_pack(r.g, std::max(r.max_chunks, 1), std::max(r.max_rows, 1), sh.k_last, sh.n_chunks);
    }
    out[grid] = CtaStart{total_chunks, 0, 0, 0};
}

bool fill_group_desc(GroupDesc &d, int M, int N, int K, const void *A, const void *B, const void *SFA,
                     const void *SFB, void *C, bool sf_raw, int unit, bool sfb_padded)
{
    if (!load_encode()) return false;
    const uint64_t Mg = (uint64_t)M;
    d.M = M;
    d.m_tiles = ceil_div(M, kTileM);
    d.m_units = ceil_div(d.m_tiles, unit);
    d.b_keep = d.m_units > 1 ? 1 : 0;
    d.N = N;
    d.k_tiles = k_tiles_of(K);
    d.k_last = k_last_of(K);
    d.n_chunks = ceil_div(N, kChunkN);
    d.ldc = N;
    d.C = static_cast<uint16_t *>(C);
    bool ok = true;
    for (int i = 0; i < 2 && ok; ++i)
        ok = encode_2d(&d.maps.tmA[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K / 2, Mg, K / 2, kTileK / 2, kTileM << i,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    for (int i = 0; i < kNumRowBoxes && ok; ++i)
        ok = encode_2d(&d.maps.tmB[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K / 2, N, K / 2, kTileK / 2, kChunkN << i,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return false;
    d.sf_row_bytes = 0;
    d.sfb_tma = 0;
    d.sfa_rows = d.sfb_rows = nullptr;
    if (sf_raw && !raw_tma_ok(K)) {
        // rows of K/16 bytes, not whole 16-byte units: no SFA maps, the
        // kernel's scale producer copies the rows with its lanes; SFB too,
        // unless it is a copy with padded rows, which the TMA loads
        d.sf_row_bytes = K / 16;
        d.sfa_rows = static_cast<const uint8_t *>(SFA);
        if (sfb_padded) {
            const uint32_t sf_box = kSfKTiles * (kTileK / 16);
            d.sfb_tma = 1;
            for (int i = 0; i < kNumRowBoxes && ok; ++i)
                ok = encode_2d(&d.maps.tmSFB[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, K / 16, N,
                               (uint64_t)sf_padded_row_bytes(K), sf_box, kChunkN << i, CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            d.sfb_rows = static_cast<const uint8_t *>(SFB);
        }
    } else if (sf_raw) {
        const uint32_t sf_box = kSfKTiles * (kTileK / 16);  // bytes of one scale row per box
        for (int i = 0; i < 2 && ok; ++i)
            ok = encode_2d(&d.maps.tmSFA[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, SFA, K / 16, Mg, K / 16, sf_box, kTileM << i,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
        for (int i = 0; i < kNumRowBoxes && ok; ++i)
            ok = encode_2d(&d.maps.tmSFB[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, K / 16, N, K / 16, sf_box, kChunkN << i,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        // atom layout: SFA boxes of the unit's 1 or 2 row tiles, SFB boxes of
        // 1, 2 or 3 (and, unused by the kernel variants, 4) 128-row blocks
        const uint64_t katoms = (uint64_t)K / 64;
        for (int i = 0; i < 2 && ok; ++i)
            ok = encode_atoms(&d.maps.tmSFA[i], SFA, katoms, (uint64_t)ceil_div(M, kTileM), (uint32_t)(i + 1));
        for (int i = 0; i < kNumRowBoxes && ok; ++i)
            ok = encode_atoms(&d.maps.tmSFB[i], SFB, katoms, (uint64_t)ceil_div(N, kTileM), (uint32_t)(i + 1));
    }
    return ok;
}

}  // namespace nvfp4

struct nvfp4_ggemm_plan_s {
    int device = 0;
    int sm_count = 0;
    int G = 0;
    std::vector<int32_t> M, N, K;  // per group
    nvfp4_ggemm_options_t opt{};
    int variant = -1;
    GemmVariant var{};
    int grid = 0;
    int total_chunks = 0;
    int cap_single = 8, cap_pair = 6;
    int unit = 2;        // 128-row tiles per unit of work
    bool split = false;  // one-row-tile tiles accumulate in two halves
    bool sf_lanes = false;  // FUSED path with some K_g % 256 != 0: the scale producer copies those raw rows
    std::vector<int32_t> m_tiles, m_units, chunk_prefix, cta_begin;
    std::vector<GroupShape> shapes;
    std::vector<CtaRange> ctas;
    size_t off_prefix = 0, off_jobs = 0, table_bytes = 0;
    Slot slots[kSlots];
    int cur = -1;
    uint32_t *d_err = nullptr;
    uint8_t *d_ws = nullptr;
    std::vector<size_t> ws_sfa, ws_sfb;  // workspace offsets of each group's atom-layout scales
    // prepare_b_scales job table
    RelayoutJob *d_prep_jobs = nullptr;
    RelayoutJob *h_prep_jobs = nullptr;
    cudaEvent_t ev_prep = nullptr;
    bool prep_used = false;
    bool b_prepared = false;
    // run_host device buffers
    int batch = 1;  // problems per group of nvfp4_ggemm_plan_batched (plan groups = groups * batch)
    uint8_t *d_io = nullptr;
    std::vector<size_t> io_a, io_b, io_sfa, io_sfb, io_c;
    size_t io_bytes = 0;
    // run_host through the SMs: the host pointers last checked, and for each
    // (5 per group: A, B, SFA, SFB, C) the address the GPU uses, or none
    std::vector<const void *> io_key;
    std::vector<const void *> io_dev;
    bool io_direct = false;

    bool raw() const { return opt.sf_layout == NVFP4_SF_RAW; }
    bool relayout() const { return raw() && opt.sf_path == NVFP4_SF_RELAYOUT; }
    bool fused() const { return raw() && opt.sf_path == NVFP4_SF_FUSED; }
    // FUSED with cache_b_scales: SFB is copied once (prepare_b_scales) into
    // rows padded to 16 bytes, which the TMA loads whatever K_g is
    bool sfb_padded() const { return fused() && opt.cache_b_scales; }
};

namespace {

void release(nvfp4_ggemm_plan_s *p)
{
    for (Slot &s : p->slots) {
        if (s.ev) {
            if (s.used) cudaEventSynchronize(s.ev);
            cudaEventDestroy(s.ev);
        }
        if (s.h_table) cudaFreeHost(s.h_table);
        if (s.d_table) cudaFree(s.d_table);
        delete s.params;
    }
    if (p->ev_prep) {
        if (p->prep_used) cudaEventSynchronize(p->ev_prep);
        cudaEventDestroy(p->ev_prep);
    }
    if (p->h_prep_jobs) cudaFreeHost(p->h_prep_jobs);
    if (p->d_prep_jobs) cudaFree(p->d_prep_jobs);
    if (p->d_err) cudaFree(p->d_err);
    if (p->d_ws) cudaFree(p->d_ws);
    if (p->d_io) cudaFree(p->d_io);
    delete p;
}

nvfp4_status_t validate_options(const nvfp4_ggemm_options_t *in, nvfp4_ggemm_options_t *out)
{
    nvfp4_ggemm_default_options(out);
    if (!in) return NVFP4_OK;
    if (in->struct_size != sizeof(nvfp4_ggemm_options_t)) return NVFP4_ERR_INVALID_ARG;
    *out = *in;
    if (out->sf_layout != NVFP4_SF_RAW && out->sf_layout != NVFP4_SF_ATOM) return NVFP4_ERR_INVALID_ARG;
    if (out->sf_path != NVFP4_SF_FUSED && out->sf_path != NVFP4_SF_RELAYOUT) return NVFP4_ERR_INVALID_ARG;
    if (out->cache_b_scales != 0 && out->cache_b_scales != 1) return NVFP4_ERR_INVALID_ARG;
    if (out->tile_n == 0) out->tile_n = kDefaultTileN;
    if (out->tile_n < kChunkN || out->tile_n > kMaxTileN || out->tile_n % kChunkN != 0) return NVFP4_ERR_INVALID_ARG;
    if (out->b_stages < 0 || out->a_stages < 0 || (out->b_stages == 0) != (out->a_stages == 0))
        return NVFP4_ERR_INVALID_ARG;
    const bool raw_fused = out->sf_layout == NVFP4_SF_RAW && out->sf_path == NVFP4_SF_FUSED;
    if (ggemm_variant_index(variant_width(out->tile_n), out->b_stages, out->a_stages, raw_fused, 2) < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (out->max_ctas < 0 || out->debug_skip_load < 0) return NVFP4_ERR_INVALID_ARG;
    if (out->serial_launch != 0 && out->serial_launch != 1) return NVFP4_ERR_INVALID_ARG;
    if (out->b_static < 0 || out->b_static > 2) return NVFP4_ERR_INVALID_ARG;
    if (out->row_units < 0 || out->row_units > 2) return NVFP4_ERR_INVALID_ARG;
    if (out->debug_check_fail != 0 && (out->debug_check_fail < kSiteCheckLoadB || out->debug_check_fail > kSiteCheckEpi))
        return NVFP4_ERR_INVALID_ARG;
    if (out->wait_timeout_ns == 0) out->wait_timeout_ns = kDefaultTimeoutNs;
    return NVFP4_OK;
}

bool fill_table(nvfp4_ggemm_plan_s *p, uint8_t *tab, uint8_t *dtab, const void *const *A, const void *const *B,
                const void *const *SFA, const void *const *SFB, void *const *C, const int32_t *ldc, bool force_sfb,
                int *njobs_out)
{
    std::memset(tab, 0, p->table_bytes);
    auto *groups = reinterpret_cast<GroupDesc *>(tab);
    auto *prefix = reinterpret_cast<int32_t *>(tab + p->off_prefix);
    auto *jobs = reinterpret_cast<RelayoutJob *>(tab + p->off_jobs);
    int njobs = 0, items = 0;
    for (int g = 0; g <= p->G; ++g) prefix[g] = p->chunk_prefix[g];
    for (int g = 0; g < p->G; ++g) {
        GroupDesc &d = groups[g];
        d.M = p->M[g];
        d.m_tiles = p->m_tiles[g];
        d.m_units = p->m_units[g];
        d.chunk_begin = p->chunk_prefix[g];
        if (p->M[g] == 0) continue;
        const int N = p->N[g], K = p->K[g];
        const void *sfa = SFA[g];
        const void *sfb = SFB ? SFB[g] : nullptr;
        const bool pad = p->sfb_padded() && !force_sfb;
        if (pad) sfb = p->d_ws + p->ws_sfb[g];
        if (p->relayout()) {
            sfa = p->d_ws + p->ws_sfa[g];
            sfb = p->d_ws + p->ws_sfb[g];
            jobs[njobs] = RelayoutJob{static_cast<const uint8_t *>(SFA[g]), p->d_ws + p->ws_sfa[g], p->M[g], K, items, 0};
            items += relayout_items_of(p->M[g], K);
            ++njobs;
        }
        if (!fill_group_desc(d, p->M[g], N, K, A[g], B[g], sfa, sfb, C[g], p->fused(), p->unit, pad)) return false;
        d.chunk_begin = p->chunk_prefix[g];
        if (ldc) d.ldc = ldc[g];
    }
    if (p->relayout() && (force_sfb || !p->opt.cache_b_scales)) {
        for (int g = 0; g < p->G; ++g) {
            if (p->M[g] == 0) continue;
            const int N = p->N[g], K = p->K[g];
            jobs[njobs] = RelayoutJob{static_cast<const uint8_t *>(SFB[g]), p->d_ws + p->ws_sfb[g], N, K, items, 0};
            items += relayout_items_of(N, K);
            ++njobs;
        }
    }
    (void)dtab;
    *njobs_out = njobs;
    return true;
}

// The address through which the GPU can read and write host buffer `h`
// (pinned or registered host memory), or nullptr (pageable memory).
const void *device_view(const void *h)
{
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return nullptr;
    return attr.devicePointer;
}

int relayout_items(nvfp4_ggemm_plan_s *p, bool with_sfb)
{
    int items = 0;
    for (int g = 0; g < p->G; ++g) {
        if (p->M[g] == 0) continue;
        items += relayout_items_of(p->M[g], p->K[g]);
        if (with_sfb) items += relayout_items_of(p->N[g], p->K[g]);
    }
    return items;
}

nvfp4_status_t check_group_ptrs(nvfp4_ggemm_plan_s *p, const void *const *A, const void *const *B,
                                const void *const *SFA, const void *const *SFB, void *const *C, bool need_sfb)
{
    if (!A || !B || !SFA || !C || (need_sfb && !SFB)) return NVFP4_ERR_INVALID_ARG;
    for (int g = 0; g < p->G; ++g) {
        if (p->M[g] == 0) continue;
        if (!A[g] || !B[g] || !SFA[g] || !C[g] || (need_sfb && !SFB[g])) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(A[g]) || !aligned16(B[g]) || !aligned16(SFA[g]) || !aligned16(C[g]) ||
            (need_sfb && !aligned16(SFB[g])))
            return NVFP4_ERR_ALIGNMENT;
    }
    return NVFP4_OK;
}

nvfp4_status_t run_device(nvfp4_ggemm_plan_s *p, const void *const *A, const void *const *B,
                          const void *const *SFA, const void *const *SFB, void *const *C, const int32_t *ldc,
                          cudaStream_t stream, bool force_sfb, bool early_ok = true)
{
    const bool sfb_cached = (p->relayout() || p->sfb_padded()) && p->opt.cache_b_scales && !force_sfb;
    if (sfb_cached && !p->b_prepared) return NVFP4_ERR_NOT_PREPARED;
    nvfp4_status_t st = check_group_ptrs(p, A, B, SFA, SFB, C, !sfb_cached);
    if (st != NVFP4_OK) return st;
    if (ldc) {
        for (int g = 0; g < p->G; ++g)
            if (p->M[g] > 0 && (ldc[g] < p->N[g] || ldc[g] % 8 != 0)) return NVFP4_ERR_INVALID_ARG;
    }
    if (p->total_chunks == 0) return NVFP4_OK;

    std::vector<const void *> key;
    key.reserve(5 * (size_t)p->G + 1);
    for (int g = 0; g < p->G; ++g) {
        const bool on = p->M[g] > 0;
        key.push_back(on ? A[g] : nullptr);
        key.push_back(on ? B[g] : nullptr);
        key.push_back(on ? SFA[g] : nullptr);
        key.push_back(on && !sfb_cached ? SFB[g] : nullptr);
        key.push_back(on ? C[g] : nullptr);
        key.push_back(reinterpret_cast<const void *>(static_cast<uintptr_t>(on && ldc ? ldc[g] : 0)));
    }
    key.push_back(reinterpret_cast<const void *>(static_cast<uintptr_t>(force_sfb ? 1 : 0)));

    int slot = p->cur;
    bool uploaded = false;
    if (slot < 0 || p->slots[slot].key != key) {
        slot = (p->cur + 1) % kSlots;
        Slot &s = p->slots[slot];
        if (s.used && cudaEventSynchronize(s.ev) != cudaSuccess) return NVFP4_ERR_CUDA;
        int njobs = 0;
        if (!fill_table(p, s.h_table, s.d_table, A, B, SFA, SFB, C, ldc, force_sfb, &njobs)) return NVFP4_ERR_CUDA;
        if (cudaMemcpyAsync(s.d_table, s.h_table, p->table_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        s.key = key;
        p->cur = slot;
        uploaded = true;
        // the kernel parameters of this table: start records, the first
        // groups' tensor maps, pointers into the device copy
        GemmParams &gp = *s.params;
        gp = GemmParams{};
        gp.groups = reinterpret_cast<const GroupDesc *>(s.d_table);
        gp.chunk_prefix = reinterpret_cast<const int32_t *>(s.d_table + p->off_prefix);
        pack_cta_starts(gp.cta, p->ctas.data(), p->grid, p->total_chunks, p->shapes.data());
        order_ctas(gp.order, p->ctas.data(), p->grid, p->chunk_prefix.data(), p->shapes.data(), p->unit,
                   p->cap_single, p->cap_pair);
        const GroupDesc *hg = reinterpret_cast<const GroupDesc *>(s.h_table);
        for (int g = 0; g < std::min(p->G, kParamGroups); ++g) gp.pmaps[g] = hg[g].maps;
        gp.err = p->d_err;
        gp.timeout_ns = p->opt.wait_timeout_ns;
        gp.G = p->G;
        gp.cap_single = p->cap_single;
        gp.cap_pair = p->cap_pair;
        gp.debug_skip_load = p->opt.debug_skip_load;
        gp.debug_check_fail = p->opt.debug_check_fail;
        gp.split_acc = p->split ? 1 : 0;
    }
    Slot &s = p->slots[slot];

    if (p->relayout()) {
        RelayoutParams rp{};
        rp.jobs = reinterpret_cast<const RelayoutJob *>(s.d_table + p->off_jobs);
        int nj = 0;
        for (int g = 0; g < p->G; ++g) nj += p->M[g] > 0 ? 1 : 0;
        rp.njobs = sfb_cached ? nj : 2 * nj;
        rp.total_items = relayout_items(p, !sfb_cached);
        if (relayout_launch(rp, p->sm_count, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    }

    GemmParams &gp = *s.params;
    // Loads that may start before the previous kernel completes (the caller's
    // b_static: 1 for B and SFB, 2 for every input): never the scales on the
    // re-layout path (the re-layout kernel just before the GEMM writes them),
    // and nothing behind run_host's own copy of the inputs.
    gp.early = 0;
    if (early_ok && p->opt.b_static) {
        // (the plan's own copies of the scales are written by this
        // library's kernels, so those are never loaded early)
        gp.early = kEarlyB | (p->relayout() || sfb_cached ? 0 : kEarlySfb);
        if (p->opt.b_static == 2) gp.early |= kEarlyA | (p->relayout() ? 0 : kEarlySfa);
    }
#ifdef NVFP4_TRACE
    gp.trace = g_trace ? g_trace + (size_t)(g_trace_next++ % g_trace_calls) * kMaxCtas * kTraceSlots : nullptr;
#endif
    // The GEMM may overlap its set-up with the previous kernel of the stream
    // (it reads only the problem table before that kernel completes). Not
    // right after a table upload: the copy, not a kernel, precedes it then.
    const bool overlap = !p->opt.serial_launch && (p->relayout() || !uploaded);
    if (ggemm_launch(p->variant, gp, p->grid, stream, overlap) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (cudaEventRecord(s.ev, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    s.used = true;
    return NVFP4_OK;
}

}  // namespace

extern "C" {

void nvfp4_ggemm_default_options(nvfp4_ggemm_options_t *opt)
{
    if (!opt) return;
    std::memset(opt, 0, sizeof(*opt));
    opt->struct_size = sizeof(nvfp4_ggemm_options_t);
    opt->sf_layout = NVFP4_SF_RAW;
    opt->sf_path = NVFP4_SF_FUSED;
    opt->cache_b_scales = 0;
    opt->wait_timeout_ns = kDefaultTimeoutNs;
    opt->tile_n = 0;
    opt->max_ctas = 0;
    opt->debug_skip_load = 0;
    opt->b_stages = 0;
    opt->a_stages = 0;
    opt->serial_launch = 0;
    opt->b_static = 0;
}

nvfp4_status_t nvfp4_ggemm_schedule_units(int num_groups, const int32_t *M, const int32_t *N, const int32_t *K,
                                          int32_t tile_n, int32_t max_ctas, int32_t row_units, int32_t *cta_begin,
                                          int32_t *grid, int32_t *units, int32_t *split_acc)
{
    if (!M || !N || !K || !cta_begin || !grid || num_groups < 1 || num_groups > kMaxGroups)
        return NVFP4_ERR_INVALID_ARG;
    if (max_ctas < 1 || max_ctas > kMaxCtas || row_units < 0 || row_units > 2) return NVFP4_ERR_INVALID_ARG;
    if (tile_n == 0) tile_n = kDefaultTileN;
    if (tile_n < kChunkN || tile_n > kMaxTileN || tile_n % kChunkN != 0) return NVFP4_ERR_INVALID_ARG;
    std::vector<GroupShape> shapes(num_groups);
    std::vector<int32_t> counts(kMaxCtas, 0);
    long total = 0;
    for (int g = 0; g < num_groups; ++g) {
        if (M[g] < 0 || M[g] > kMaxM) return NVFP4_ERR_INVALID_ARG;
        if (!shape_ok(N[g], K[g])) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        shapes[g] = group_shape(M[g], N[g], K[g]);
        total += (long)shapes[g].m_tiles * shapes[g].n_chunks;
    }
    if (total > 0x7FFFFFFF) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const int cap_single = tile_n / kChunkN;
    const int cap_pair = std::min(cap_single, pair_cap_chunks(variant_width(tile_n)));
    const UnitChoice uc = choose_units(shapes.data(), num_groups, cap_single, cap_pair, max_ctas, row_units);
    *grid = schedule_ctas(shapes.data(), num_groups, uc.unit, cap_single, cap_pair, max_ctas, cta_begin,
                          counts.data());
    if (units) *units = uc.unit;
    if (split_acc) *split_acc = uc.split ? 1 : 0;
    return NVFP4_OK;
}

nvfp4_status_t nvfp4_ggemm_schedule(int num_groups, const int32_t *M, const int32_t *N, const int32_t *K,
                                    int32_t tile_n, int32_t max_ctas, int32_t *cta_begin, int32_t *grid)
{
    return nvfp4_ggemm_schedule_units(num_groups, M, N, K, tile_n, max_ctas, 2, cta_begin, grid, nullptr, nullptr);
}

nvfp4_status_t nvfp4_ggemm_plan(nvfp4_ggemm_plan_t *out, int device, int num_groups, const int32_t *M, int32_t N,
                                int32_t K, const nvfp4_ggemm_options_t *opt_in)
{
    if (!out) return NVFP4_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_groups < 1 || num_groups > kMaxGroups || !M) return NVFP4_ERR_INVALID_ARG;
    if (!shape_ok(N, K)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    std::vector<int32_t> Ns(num_groups, N), Ks(num_groups, K);
    return nvfp4_ggemm_plan_shapes(out, device, num_groups, M, Ns.data(), Ks.data(), opt_in);
}

nvfp4_status_t nvfp4_ggemm_plan_shapes(nvfp4_ggemm_plan_t *out, int device, int num_groups, const int32_t *M,
                                       const int32_t *N, const int32_t *K, const nvfp4_ggemm_options_t *opt_in)
{
    if (!out) return NVFP4_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_groups < 1 || num_groups > kMaxGroups || !M || !N || !K || device < 0) return NVFP4_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; ++g)
        if (M[g] < 0 || M[g] > kMaxM) return NVFP4_ERR_INVALID_ARG;
    for (int g = 0; g < num_groups; ++g)
        if (!shape_ok(N[g], K[g])) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    nvfp4_ggemm_options_t opt;
    nvfp4_status_t st = validate_options(opt_in, &opt);
    if (st != NVFP4_OK) return st;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
        cudaGetLastError();
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    }
    DeviceGuard guard(device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (major != 10 || minor != 3) return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (!load_encode()) return NVFP4_ERR_CUDA;

    auto *p = new (std::nothrow) nvfp4_ggemm_plan_s();
    if (!p) return NVFP4_ERR_CUDA;
    p->device = device;
    p->sm_count = sms;
    p->G = num_groups;
    p->M.assign(M, M + num_groups);
    p->N.assign(N, N + num_groups);
    p->K.assign(K, K + num_groups);
    p->opt = opt;
    for (int g = 0; g < num_groups; ++g)
        if (!raw_tma_ok(K[g])) p->sf_lanes = p->fused();

    // raw scale rows the scale producer's lanes copy: the kernels built for
    // that (the widest tiles, default ring depths; the tile caps still follow
    // tile_n)
    p->variant = p->sf_lanes ? ggemm_variant_index(kMaxTileN, 0, 0, true, 2, true)
                             : ggemm_variant_index(variant_width(opt.tile_n), opt.b_stages, opt.a_stages, p->fused(), 2);
    if (p->variant < 0) {
        release(p);
        return NVFP4_ERR_INVALID_ARG;
    }
    p->var = ggemm_variant(p->variant);
    if (ggemm_configure(p->variant) != cudaSuccess) {
        release(p);
        return NVFP4_ERR_CUDA;
    }

    // Work decomposition: m_units_g x ceil(N_g/32) chunks per group, prefix-summed.
    p->cap_single = opt.tile_n / kChunkN;
    p->cap_pair = std::min(p->cap_single, pair_cap_chunks(p->var.max_n));
    p->chunk_prefix.assign(num_groups + 1, 0);
    p->m_tiles.assign(num_groups, 0);
    p->m_units.assign(num_groups, 0);
    p->shapes.assign(num_groups, GroupShape{});
    long total = 0;
    for (int g = 0; g < num_groups; ++g) {
        p->m_tiles[g] = ceil_div(M[g], kTileM);
        p->shapes[g] = group_shape(M[g], N[g], K[g]);
        total += (long)p->m_tiles[g] * p->shapes[g].n_chunks;  // the most chunks either unit gives
    }
    if (total > 0x7FFFFFFF) {
        release(p);
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    }
    const int cap = std::min(opt.max_ctas > 0 ? std::min(opt.max_ctas, sms) : sms, kMaxCtas);
    const UnitChoice uc = choose_units(p->shapes.data(), num_groups, p->cap_single, p->cap_pair, cap, opt.row_units);
    p->unit = uc.unit;
    p->split = uc.split;
    if (p->unit != 2) {  // the same ring configuration, built for single row tiles
        p->variant =
            ggemm_variant_index(p->var.max_n, p->var.b_stages, p->var.a_stages, p->var.sf_raw, p->unit, p->var.lanes);
        if (p->variant < 0) {
            release(p);
            return NVFP4_ERR_INVALID_ARG;
        }
        p->var = ggemm_variant(p->variant);
        if (ggemm_configure(p->variant) != cudaSuccess) {
            release(p);
            return NVFP4_ERR_CUDA;
        }
    }
    total = 0;
    for (int g = 0; g < num_groups; ++g) {
        p->m_units[g] = ceil_div(p->m_tiles[g], p->unit);
        p->chunk_prefix[g] = (int32_t)total;
        total += (long)p->m_units[g] * p->shapes[g].n_chunks;
    }
    p->chunk_prefix[num_groups] = (int32_t)total;
    p->total_chunks = (int)total;
    p->cta_begin.assign(cap + 1, 0);
    {
        std::vector<int32_t> counts(kMaxCtas, 0);
        p->grid = schedule_ctas(p->shapes.data(), num_groups, p->unit, p->cap_single, p->cap_pair, cap,
                                p->cta_begin.data(), counts.data());
    }
    p->cta_begin.resize(p->grid + 1);

    p->off_prefix = align_up(sizeof(GroupDesc) * (size_t)num_groups, 64);
    p->ctas.assign(std::max(p->grid, 1), CtaRange{});
    fill_cta_ranges(p->ctas.data(), p->cta_begin.data(), p->grid, p->chunk_prefix.data(), p->shapes.data(),
                    num_groups, p->unit, p->cap_single, p->cap_pair);
    p->off_jobs = align_up(p->off_prefix + sizeof(int32_t) * (size_t)(num_groups + 1), 64);
    p->table_bytes = align_up(p->off_jobs + sizeof(RelayoutJob) * 2 * (size_t)num_groups, 128);

    bool ok = cudaMalloc(&p->d_err, sizeof(uint32_t)) == cudaSuccess &&
              cudaMemset(p->d_err, 0, sizeof(uint32_t)) == cudaSuccess;
    for (Slot &s : p->slots) {
        s.params = new (std::nothrow) GemmParams();
        ok = ok && s.params && cudaMallocHost(&s.h_table, p->table_bytes) == cudaSuccess &&
             cudaMalloc(&s.d_table, p->table_bytes) == cudaSuccess &&
             cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming) == cudaSuccess;
    }
    if (ok && (p->relayout() || p->sfb_padded())) {
        // RELAYOUT: atom-layout SFA and SFB; FUSED with cache_b_scales: SFB
        // with rows padded to 16 bytes
        size_t off = 0;
        p->ws_sfa.assign(num_groups, 0);
        p->ws_sfb.assign(num_groups, 0);
        for (int g = 0; g < num_groups && p->relayout(); ++g) {
            p->ws_sfa[g] = off;
            off = align_up(off + atom_bytes(M[g], K[g]), 256);
        }
        for (int g = 0; g < num_groups; ++g) {
            p->ws_sfb[g] = off;
            off = align_up(off + (p->relayout() ? atom_bytes(N[g], K[g])
                                                : (uint64_t)N[g] * (uint64_t)sf_padded_row_bytes(K[g])),
                           256);
        }
        ok = cudaMalloc(&p->d_ws, std::max<size_t>(off, 256)) == cudaSuccess &&
             cudaMalloc(&p->d_prep_jobs, sizeof(RelayoutJob) * (size_t)num_groups) == cudaSuccess &&
             cudaMallocHost(&p->h_prep_jobs, sizeof(RelayoutJob) * (size_t)num_groups) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_prep, cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        release(p);
        return NVFP4_ERR_CUDA;
    }
    *out = p;
    return NVFP4_OK;
}

nvfp4_status_t nvfp4_ggemm_run(nvfp4_ggemm_plan_t plan, const void *const *A, const void *const *B,
                               const void *const *SFA, const void *const *SFB, void *const *C, void *stream)
{
    if (!plan) return NVFP4_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    nvfp4_status_t st = run_device(plan, A, B, SFA, SFB, C, nullptr, static_cast<cudaStream_t>(stream), false);
    if (st == NVFP4_ERR_CUDA) cudaGetLastError();
    return st;
}

nvfp4_status_t nvfp4_ggemm_plan_batched(nvfp4_ggemm_plan_t *out, int device, int num_groups, int32_t batch,
                                        const int32_t *M, const int32_t *N, const int32_t *K,
                                        const nvfp4_ggemm_options_t *opt)
{
    if (!out) return NVFP4_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_groups < 1 || batch < 1 || (long)num_groups * batch > kMaxGroups || !M || !N || !K)
        return NVFP4_ERR_INVALID_ARG;
    const int total = num_groups * batch;
    std::vector<int32_t> Me(total), Ne(total), Ke(total);
    for (int g = 0; g < num_groups; ++g)
        for (int b = 0; b < batch; ++b) {
            Me[g * batch + b] = M[g];
            Ne[g * batch + b] = N[g];
            Ke[g * batch + b] = K[g];
        }
    nvfp4_status_t st = nvfp4_ggemm_plan_shapes(out, device, total, Me.data(), Ne.data(), Ke.data(), opt);
    if (st == NVFP4_OK) (*out)->batch = batch;
    return st;
}

nvfp4_status_t nvfp4_ggemm_run_batched(nvfp4_ggemm_plan_t plan, const void *const *A, const void *const *B,
                                       const void *const *SFA, const void *const *SFB, void *const *C,
                                       const int64_t *batch_stride, void *stream)
{
    if (!plan || !batch_stride || plan->batch < 1 || !A || !B || !SFA || !C) return NVFP4_ERR_INVALID_ARG;
    const int L = plan->batch, G = plan->G / L;
    for (int g = 0; g < G; ++g) {
        if (plan->M[g * L] == 0) continue;  // an empty group's pointers and strides are not read
        for (int i = 5 * g; i < 5 * g + 5; ++i) {
            if (batch_stride[i] < 0) return NVFP4_ERR_INVALID_ARG;
            if (batch_stride[i] % 16 != 0) return NVFP4_ERR_ALIGNMENT;
        }
    }
    // problem g * L + b: group g's pointers advanced by b strides
    std::vector<const void *> a(plan->G), bb(plan->G), sa(plan->G), sb(plan->G);
    std::vector<void *> c(plan->G);
    auto at = [](const void *base, int64_t off) -> const void * {
        return base ? static_cast<const void *>(static_cast<const uint8_t *>(base) + off) : nullptr;
    };
    for (int g = 0; g < G; ++g)
        for (int b = 0; b < L; ++b) {
            const int e = g * L + b;
            if (plan->M[e] == 0) continue;  // left null: never read
            const int64_t *st = batch_stride + 5 * g;
            a[e] = at(A[g], b * st[0]);
            bb[e] = at(B[g], b * st[1]);
            sa[e] = at(SFA[g], b * st[2]);
            sb[e] = SFB ? at(SFB[g], b * st[3]) : nullptr;
            c[e] = const_cast<void *>(at(C[g], b * st[4]));
        }
    DeviceGuard guard(plan->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    nvfp4_status_t st = run_device(plan, a.data(), bb.data(), sa.data(), SFB ? sb.data() : nullptr, c.data(),
                                   nullptr, static_cast<cudaStream_t>(stream), false);
    if (st == NVFP4_ERR_CUDA) cudaGetLastError();
    return st;
}

nvfp4_status_t nvfp4_ggemm_run_strided(nvfp4_ggemm_plan_t plan, const void *const *A, const void *const *B,
                                       const void *const *SFA, const void *const *SFB, void *const *C,
                                       const int32_t *ldc, void *stream)
{
    if (!plan || !ldc) return NVFP4_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    nvfp4_status_t st = run_device(plan, A, B, SFA, SFB, C, ldc, static_cast<cudaStream_t>(stream), false);
    if (st == NVFP4_ERR_CUDA) cudaGetLastError();
    return st;
}

nvfp4_status_t nvfp4_ggemm_run_host(nvfp4_ggemm_plan_t plan, const void *const *A, const void *const *B,
                                    const void *const *SFA, const void *const *SFB, void *const *C, void *stream)
{
    if (!plan) return NVFP4_ERR_INVALID_ARG;
    if (!A || !B || !SFA || !SFB || !C) return NVFP4_ERR_INVALID_ARG;
    nvfp4_ggemm_plan_s *p = plan;
    for (int g = 0; g < p->G; ++g)
        if (p->M[g] > 0 && (!A[g] || !B[g] || !SFA[g] || !SFB[g] || !C[g])) return NVFP4_ERR_INVALID_ARG;
    DeviceGuard guard(p->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto sf_bytes = [&](size_t rows, size_t K) -> size_t {
        return p->raw() ? rows * K / 16 : (size_t)atom_bytes((int64_t)rows, (int64_t)K);
    };
    if (!p->d_io) {
        size_t off = 0;
        p->io_a.assign(p->G, 0);
        p->io_b.assign(p->G, 0);
        p->io_sfa.assign(p->G, 0);
        p->io_sfb.assign(p->G, 0);
        p->io_c.assign(p->G, 0);
        for (int g = 0; g < p->G; ++g) {
            const size_t m = (size_t)p->M[g], N = (size_t)p->N[g], K = (size_t)p->K[g];
            p->io_a[g] = off, off = align_up(off + m * K / 2, 256);
            p->io_b[g] = off, off = align_up(off + N * K / 2, 256);
            p->io_sfa[g] = off, off = align_up(off + sf_bytes(m, K), 256);
            p->io_sfb[g] = off, off = align_up(off + sf_bytes(N, K), 256);
            p->io_c[g] = off, off = align_up(off + m * N * 2, 256);
        }
        p->io_bytes = std::max<size_t>(off, 256);
        if (cudaMalloc(&p->d_io, p->io_bytes) != cudaSuccess) {
            p->d_io = nullptr;
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
    }
    std::vector<const void *> dA(p->G), dB(p->G), dSFA(p->G), dSFB(p->G);
    std::vector<void *> dC(p->G);
    for (int g = 0; g < p->G; ++g) {
        dA[g] = p->d_io + p->io_a[g];
        dB[g] = p->d_io + p->io_b[g];
        dSFA[g] = p->d_io + p->io_sfa[g];
        dSFB[g] = p->d_io + p->io_sfb[g];
        dC[g] = p->d_io + p->io_c[g];
    }
    // Host buffers the GPU can address, 16-byte aligned, in few enough jobs:
    // one launch moves every input in and one moves C out. Otherwise one
    // copy per buffer. The check is cached for the last set of pointers.
    {
        std::vector<const void *> key;
        key.reserve(5 * (size_t)p->G);
        for (int g = 0; g < p->G; ++g) {
            const bool on = p->M[g] > 0;
            key.push_back(on ? A[g] : nullptr);
            key.push_back(on ? B[g] : nullptr);
            key.push_back(on ? SFA[g] : nullptr);
            key.push_back(on ? SFB[g] : nullptr);
            key.push_back(on ? C[g] : nullptr);
        }
        if (key != p->io_key) {
            p->io_key = key;
            p->io_dev.assign(key.size(), nullptr);
            int jobs = 0;
            bool ok = true;
            for (size_t i = 0; i < key.size() && ok; ++i) {
                if (!key[i]) continue;
                p->io_dev[i] = device_view(key[i]);
                ok = p->io_dev[i] && aligned16(p->io_dev[i]);
                ++jobs;
            }
            p->io_direct = ok && jobs <= kMaxIoJobs;
        }
    }
    if (p->io_direct) {
        IoCopyParams in{}, out{};
        for (int g = 0; g < p->G; ++g) {
            const size_t m = (size_t)p->M[g], N = (size_t)p->N[g], K = (size_t)p->K[g];
            if (m == 0) continue;
            const void *const *v = &p->io_dev[5 * (size_t)g];
            const size_t bytes[4] = {m * K / 2, N * K / 2, sf_bytes(m, K), sf_bytes(N, K)};
            const void *dst[4] = {dA[g], dB[g], dSFA[g], dSFB[g]};
            for (int i = 0; i < 4; ++i)
                in.jobs[in.njobs++] = IoJob{static_cast<const uint8_t *>(v[i]),
                                            static_cast<uint8_t *>(const_cast<void *>(dst[i])), bytes[i]};
            out.jobs[out.njobs++] = IoJob{static_cast<const uint8_t *>(dC[g]),
                                          static_cast<uint8_t *>(const_cast<void *>(v[4])), m * N * 2};
        }
        if (io_copy_launch(in, p->sm_count, s) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
        nvfp4_status_t st = run_device(p, dA.data(), dB.data(), dSFA.data(), dSFB.data(), dC.data(), nullptr, s, true, false);
        if (st != NVFP4_OK) {
            cudaGetLastError();
            return st;
        }
        if (io_copy_launch(out, p->sm_count, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
        return NVFP4_OK;
    }
    for (int g = 0; g < p->G; ++g) {
        const size_t m = (size_t)p->M[g], N = (size_t)p->N[g], K = (size_t)p->K[g];
        if (m == 0) continue;
        if (cudaMemcpyAsync(const_cast<void *>(dA[g]), A[g], m * K / 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(const_cast<void *>(dB[g]), B[g], N * K / 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(const_cast<void *>(dSFA[g]), SFA[g], sf_bytes(m, K), cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaMemcpyAsync(const_cast<void *>(dSFB[g]), SFB[g], sf_bytes(N, K), cudaMemcpyHostToDevice, s) !=
                cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
    }
    nvfp4_status_t st = run_device(p, dA.data(), dB.data(), dSFA.data(), dSFB.data(), dC.data(), nullptr, s, true, false);
    if (st != NVFP4_OK) {
        cudaGetLastError();
        return st;
    }
    for (int g = 0; g < p->G; ++g) {
        const size_t m = (size_t)p->M[g], N = (size_t)p->N[g];
        if (m == 0) continue;
        if (cudaMemcpyAsync(C[g], dC[g], m * N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

nvfp4_status_t nvfp4_ggemm_prepare_b_scales(nvfp4_ggemm_plan_t plan, const void *const *SFB, void *stream)
{
    if (!plan || !SFB) return NVFP4_ERR_INVALID_ARG;
    nvfp4_ggemm_plan_s *p = plan;
    if (!(p->relayout() || p->sfb_padded()) || !p->opt.cache_b_scales) return NVFP4_ERR_INVALID_ARG;
    for (int g = 0; g < p->G; ++g) {
        if (p->M[g] == 0) continue;
        if (!SFB[g]) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(SFB[g])) return NVFP4_ERR_ALIGNMENT;
    }
    DeviceGuard guard(p->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->prep_used && cudaEventSynchronize(p->ev_prep) != cudaSuccess) return NVFP4_ERR_CUDA;
    // RELAYOUT: atom layout (items of 128 rows x 16 atoms); FUSED: padded
    // rows (one item per row)
    int nj = 0, items = 0;
    for (int g = 0; g < p->G; ++g) {
        if (p->M[g] == 0) continue;
        p->h_prep_jobs[nj++] =
            RelayoutJob{static_cast<const uint8_t *>(SFB[g]), p->d_ws + p->ws_sfb[g], p->N[g], p->K[g], items, 0};
        items += p->relayout() ? relayout_items_of(p->N[g], p->K[g]) : p->N[g];
    }
    if (nj > 0) {
        if (cudaMemcpyAsync(p->d_prep_jobs, p->h_prep_jobs, sizeof(RelayoutJob) * (size_t)nj, cudaMemcpyHostToDevice,
                            s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        RelayoutParams rp{};
        rp.jobs = p->d_prep_jobs;
        rp.njobs = nj;
        rp.total_items = items;
        if ((p->relayout() ? relayout_launch(rp, p->sm_count, s) : sf_pad_launch(rp, p->sm_count, s)) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
    }
    if (cudaEventRecord(p->ev_prep, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    p->prep_used = true;
    p->b_prepared = true;
    return NVFP4_OK;
}

nvfp4_status_t nvfp4_ggemm_sync_status(nvfp4_ggemm_plan_t plan, void *stream, uint32_t *detail)
{
    if (detail) *detail = 0;
    if (!plan) return NVFP4_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return NVFP4_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, plan->d_err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    if (detail) *detail = word;
    if (word == 0) return NVFP4_OK;
    if (cudaMemset(plan->d_err, 0, sizeof(uint32_t)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    const uint32_t code = word & 0xFFu;
    return (code == NVFP4_ERR_TIMEOUT) ? NVFP4_ERR_TIMEOUT : NVFP4_ERR_DEVICE_FAULT;
}

nvfp4_status_t nvfp4_ggemm_destroy(nvfp4_ggemm_plan_t plan)
{
    if (!plan) return NVFP4_OK;
    DeviceGuard guard(plan->device);
    release(plan);
    return NVFP4_OK;
}

nvfp4_status_t nvfp4_sf_relayout(const void *in, void *out, int32_t rows, int32_t K, void *stream)
{
    if (!in || !out || rows < 1 || rows > (1 << 24)) return NVFP4_ERR_INVALID_ARG;
    if (K < 64 || K > kMaxK || K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(in) || !aligned16(out)) return NVFP4_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    }
    RelayoutParams rp{};
    rp.jobs = nullptr;
    rp.single = RelayoutJob{static_cast<const uint8_t *>(in), static_cast<uint8_t *>(out), rows, K, 0, 0};
    rp.njobs = 1;
    rp.total_items = relayout_items_of(rows, K);
    if (relayout_launch(rp, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

uint64_t nvfp4_sf_atom_bytes(int32_t rows, int32_t K)
{
    if (rows < 0 || K < 64 || K % 64 != 0) return 0;
    return atom_bytes(rows, K);
}

nvfp4_status_t nvfp4_ggemm_plan_info(nvfp4_ggemm_plan_t plan, nvfp4_ggemm_plan_info_t *info)
{
    if (!plan || !info) return NVFP4_ERR_INVALID_ARG;
    info->tile_n = plan->cap_single * kChunkN;
    info->b_stages = plan->var.b_stages;
    info->a_stages = plan->var.a_stages;
    info->chunks = plan->total_chunks;
    info->grid = plan->grid;
    info->sm_count = plan->sm_count;
    info->smem_bytes = ggemm_smem_bytes(plan->variant);
    info->kernels_per_run = plan->total_chunks == 0 ? 0 : (plan->relayout() ? 2 : 1);
    info->sf_path = plan->relayout() ? NVFP4_SF_RELAYOUT : NVFP4_SF_FUSED;
    info->row_units = plan->unit;
    info->split_acc = plan->split ? 1 : 0;
    return NVFP4_OK;
}

const char *nvfp4_status_string(nvfp4_status_t status)
{
    switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case NVFP4_ERR_UNSUPPORTED_SHAPE:
        return "unsupported shape (need K % 64 == 0, N % 8 == 0, sizes in range; at most 64 groups without allocation)";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "no usable device (needs compute capability 10.3, GB300)";
    case NVFP4_ERR_CUDA: return "CUDA call failed";
    case NVFP4_ERR_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4_ERR_DEVICE_FAULT: return "device-side check failed";
    case NVFP4_ERR_NOT_PREPARED: return "B scales not prepared (call nvfp4_ggemm_prepare_b_scales)";
    }
    return "unknown status";
}

int nvfp4_ggemm_version(void) { return kVersion; }

#ifdef NVFP4_TRACE
// Timeline build only: device buffer of calls x kMaxCtas x kTraceSlots
// 64-bit entries (NULL: off); stamps of the next launches go to it in turn.
NVFP4_API void nvfp4_debug_trace(void *buf, int calls)
{
    g_trace = static_cast<unsigned long long *>(buf);
    g_trace_calls = calls > 0 ? calls : 1;
    g_trace_next = 0;
}
#endif

}  // extern "C"
