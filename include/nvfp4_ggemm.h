/*
 * nvfp4_ggemm.h - C ABI of the NVFP4 block-scaled grouped GEMM for GB300
 * (sm_103a).
 *
 * The operation (nvfp4_group_gemm leaderboard problem; custom_kernel
 * docstring and kernel-launch comment of kernelindex submission 503584):
 * for every group g = 0..G-1
 *
 *     C_g[m, n] = fp16( sum_{k<K} e2m1(A_g[m,k]) * e4m3(SFA_g[m, k/16])
 *                                * e2m1(B_g[n,k]) * e4m3(SFB_g[n, k/16]) )
 *
 * for m < M_g, n < N. Products accumulate in fp32 on the tensor cores and
 * the result is rounded to fp16 (round to nearest even) once. N and K are
 * shared by the groups here; nvfp4_ggemm_plan_shapes takes N_g and K_g per
 * group, and everything below then holds with N_g, K_g in place of N, K.
 *
 * Layouts (all dense, row-major, K-major for the inputs; device memory):
 *   A[g]    M_g x K/2 bytes. Two E2M1 codes per byte, the even k in the low
 *           nibble (the pages' float4e2m1fn_x2 tensors [m, k//2]).
 *   B[g]    N x K/2 bytes, same packing.
 *   SFA[g]  E4M3 (FN: bias 7, no infinity) scale codes, one per 16 k.
 *           NVFP4_SF_RAW: M_g x K/16 bytes, row-major.
 *           NVFP4_SF_ATOM: the 128x4 atom layout the tensor cores read
 *           (ceil(M_g/128) * (K/64) atoms of 512 bytes; see
 *           nvfp4_sf_relayout), as the pages' pre-reordered scale tensors.
 *   SFB[g]  N x K/16 bytes (raw) or ceil(N/128)*(K/64)*512 bytes (atom).
 *   C[g]    M_g x N fp16, row-major (row stride N elements).
 *
 * Requirements (checked before anything is enqueued): 1 <= G <= 1024,
 * 0 <= M_g <= 2^20, 8 <= N <= 2^20 with N % 8 == 0 (16-byte C rows), 64 <= K
 * <= 2^18 with K % 64 == 0 (one 64-k MMA slice; the kernel's k tile is 256
 * and a last partial tile is read with the TMA's zero fill, as the kernel of
 * submission 503584 counts its k tiles by a ceil-div of k), every pointer of
 * a group with M_g > 0 non-null and 16-byte aligned (the TMA rule). A group
 * with M_g == 0 is skipped and its pointers are not read. Raw scale rows (K/16 bytes) are rows
 * the TMA can load only when K % 256 == 0 (the rule the TMA helper of
 * submission 498317 enforces on K); on the NVFP4_SF_FUSED path the kernel's
 * scale producer copies the rows of a group with K_g % 256 != 0 itself
 * (cp.async pieces of 8 bytes when K_g % 128 == 0, else 4), so every
 * K_g % 64 == 0 runs as one kernel on either path the caller picks.
 *
 * Ownership: the caller owns every tensor and the host arrays of pointers;
 * the arrays are read during the call only. A plan owns its device problem
 * table, pinned staging, scale workspace and device error word.
 *
 * Execution: nvfp4_ggemm_run enqueues work on `stream` and returns; buffers
 * must stay valid until the stream reaches that point. One plan may be used
 * from one host thread at a time; calls on different streams must not
 * overlap on the device (the plan's workspace is shared between calls).
 *
 * Errors: every call returns a status; nothing throws or aborts across the
 * ABI. Argument errors return before any work is enqueued. Device-side
 * failures (a pipeline wait that ran past the plan's timeout) are recorded
 * in the plan's device error word and reported by nvfp4_ggemm_sync_status.
 */
#ifndef NVFP4_GGEMM_H
#define NVFP4_GGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null, negative or out-of-range argument */
    NVFP4_ERR_ALIGNMENT = 2,         /* a tensor pointer is not 16-byte aligned */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 3, /* K % 64 != 0, N % 8 != 0, size limits */
    NVFP4_ERR_UNSUPPORTED_DEVICE = 4,/* no device, or not compute capability 10.3 */
    NVFP4_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
    NVFP4_ERR_TIMEOUT = 6,           /* a device pipeline wait exceeded the timeout */
    NVFP4_ERR_DEVICE_FAULT = 7,      /* a device-side consistency check failed */
    NVFP4_ERR_NOT_PREPARED = 8       /* cache_b_scales set but scales not prepared */
} nvfp4_status_t;

/* Layout of the scale tensors passed to run / prepare. */
enum { NVFP4_SF_RAW = 0, NVFP4_SF_ATOM = 1 };

/* How raw scales reach the tensor cores. */
enum {
    NVFP4_SF_FUSED = 0,   /* one kernel: the raw scale rows of each stage are loaded into shared
                             memory (by TMA when K_g % 256 == 0, else copied by the scale
                             producer's lanes) and permuted into the atom layout on their way
                             to the tensor memory */
    NVFP4_SF_RELAYOUT = 1 /* the re-layout kernel writes atom-layout copies into the plan's
                             workspace, then the GEMM kernel reads those */
};

typedef struct {
    uint32_t struct_size;     /* sizeof(nvfp4_ggemm_options_t) */
    int32_t sf_layout;        /* NVFP4_SF_RAW (default) or NVFP4_SF_ATOM */
    int32_t sf_path;          /* NVFP4_SF_FUSED (default) or NVFP4_SF_RELAYOUT; raw scales only */
    int32_t cache_b_scales;   /* SFB is copied once by nvfp4_ggemm_prepare_b_scales and run
                                 skips it: re-laid out into the atom layout (RELAYOUT path),
                                 or into rows padded to 16 bytes that the TMA loads whatever
                                 K_g is (FUSED path) */
    uint64_t wait_timeout_ns; /* bound on every device pipeline wait (default 2e9) */
    int32_t tile_n;           /* widest output tile in columns: 0 = 256, else a multiple of 32
                                 up to 256 (kernels exist for 128 and 256; a smaller value
                                 caps the tiles of the next wider kernel). A tile covers one
                                 or two 128-row tiles of one group, which share every B
                                 stage; with two row tiles it is at most 192 columns wide
                                 (128 for the 128 kernel), as both accumulators share TMEM */
    int32_t max_ctas;         /* persistent grid size: 0 = number of SMs */
    int32_t debug_skip_load;  /* test only: 0 = off; n > 0 = the B producer of CTA 0 leaves its
                                 n-th stage load unissued, so the consumers' waits run into the
                                 timeout (exercises the error path) */
    int32_t b_stages;         /* shared-memory stages of the B ring; 0 (with a_stages 0) = the
                                 default for the tile width and scale path. Kernels exist for
                                 (tile width, b_stages, a_stages) = (256,3,3) (default),
                                 (256,4,2) and (128,8,2) (default) with raw scales, and the
                                 defaults (256,3,3), (128,8,2) with atom-layout scales. The
                                 stage counts size the A and B regions for the widest tile;
                                 each CTA cuts them into more slots when its tiles are
                                 narrower or have one row tile. A raw-scale FUSED plan with
                                 some K_g % 256 != 0 runs (256,3,3), built with the scale
                                 producer's row copies, whatever these ask (tile_n still
                                 caps its tiles) */
    int32_t a_stages;         /* shared-memory stages of the A ring (see b_stages) */
    int32_t serial_launch;    /* 0 (default): a GEMM launch that follows another kernel on its
                                 stream may start its set-up (barriers, TMEM, tensor-map
                                 prefetch, the walk to its first tile) while that kernel's last
                                 CTAs finish (programmatic dependent launch); its loads and
                                 stores still wait until that kernel has completed. 1: plain
                                 launches, every kernel starts after the previous one ends */
    int32_t b_static;         /* 0 (default): every load waits for the kernel before the GEMM on
                                 its stream to complete. 1: the caller guarantees that this
                                 kernel (the only one that may still run when the GEMM starts)
                                 writes neither B nor SFB, e.g. model weights in inference; the
                                 GEMM then starts streaming B and SFB during that kernel's last
                                 CTAs, while A, SFA and the C stores still wait for it. 2: the
                                 same guarantee for all four inputs (A, SFA, B, SFB), e.g. inputs
                                 produced two or more kernels earlier: every load may start
                                 early and only the C stores wait. On the re-layout path the
                                 scales always wait (the re-layout kernel just before the GEMM
                                 writes them). With serial_launch, and in nvfp4_ggemm_run_host,
                                 the option has no effect */
    int32_t debug_check_fail; /* test only, and only in the debug build of the library (compiled
                                 with -DNVFP4_DEBUG, whose kernel checks every shared-memory and
                                 TMEM range, TMA coordinate and alignment before the operation it
                                 guards): 0 = off; a check site (0x21..0x26) = that check reports
                                 a failure as if its condition were false, so the error path
                                 (NVFP4_ERR_DEVICE_FAULT with the site in bits 8-15 of the
                                 detail word, the operation skipped, the kernel ending through
                                 its abort flag) runs without any invalid operation. The
                                 release build ignores it */
    int32_t row_units;        /* 128-row tiles per unit of work: 0 (default) = the plan chooses,
                                 1 = one row tile, 2 = pairs of row tiles. A pair shares every
                                 B stage between its two row tiles, so each B strip is streamed
                                 from memory once. The plan keeps pairs unless their tiles
                                 would be at most 128 columns wide while single row tiles give
                                 every CTA one tile of at most 192 columns in no more 256-k
                                 stages (few tall groups and a narrow N, such as the two
                                 2-group workloads of the pages). Such tiles then add their
                                 even and odd 64-k slices into two accumulators, summed by the
                                 epilogue: each MMA into an accumulator waits for the one
                                 before it, so two chains take about half as long. Results
                                 agree with pairs within the rounding of that one fp32 sum */
} nvfp4_ggemm_options_t;

typedef struct nvfp4_ggemm_plan_s *nvfp4_ggemm_plan_t;

/* Fill `opt` with the defaults listed above. */
NVFP4_API void nvfp4_ggemm_default_options(nvfp4_ggemm_options_t *opt);

/*
 * Build a plan for G groups with row counts M[0..G-1] (host array), shared N
 * and K, on CUDA device `device`. Validates the shape, computes the tile
 * schedule (prefix sums of the per-group work units), and allocates the
 * device problem table, scale workspace and error word. `opt` may be NULL
 * (defaults). On success *out holds the plan; on failure *out is NULL.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_plan(nvfp4_ggemm_plan_t *out, int device, int num_groups,
                                const int32_t *M, int32_t N, int32_t K,
                                const nvfp4_ggemm_options_t *opt);

/*
 * The same with per-group N_g and K_g (host arrays N[0..G-1], K[0..G-1]):
 * group g computes C_g[M_g, N_g] = sum over K_g of the block-scaled products
 * of A_g[M_g, K_g] and B_g[N_g, K_g], every size meeting the per-group rules
 * above (N_g % 8 == 0, K_g % 64 == 0). The pages' own interface takes one
 * (m, n, k) per group; nvfp4_ggemm_plan is this call with N_g = N and
 * K_g = K. Everything else (layouts per group, run, run_host, prepare,
 * status) is as for nvfp4_ggemm_plan.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_plan_shapes(nvfp4_ggemm_plan_t *out, int device, int num_groups,
                                       const int32_t *M, const int32_t *N, const int32_t *K,
                                       const nvfp4_ggemm_options_t *opt);

/*
 * Grouped GEMM on device buffers. A, B, SFA, SFB, C are host arrays of G
 * device pointers (layouts above; scales in the plan's sf_layout). `stream`
 * is a cudaStream_t (NULL = legacy default stream). Encodes the per-group
 * TMA tensor maps when the pointers differ from the previous call, uploads
 * the problem table, and enqueues the kernels. Asynchronous.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_run(nvfp4_ggemm_plan_t plan, const void *const *A, const void *const *B,
                               const void *const *SFA, const void *const *SFB, void *const *C,
                               void *stream);

/*
 * Batched groups. The pages' tensors carry a batch dimension l (A_g
 * [m, k/2, l], C_g [m, n, l], ...; submission 503584's docstring, with l = 1
 * there): every group is l independent problems of its shape.
 * nvfp4_ggemm_plan_batched plans num_groups groups of `batch` problems each
 * (M, N, K: host arrays of num_groups entries, as for
 * nvfp4_ggemm_plan_shapes); internally problem b of group g is problem
 * g * batch + b of a plan over num_groups * batch problems (at most 1024,
 * else NVFP4_ERR_INVALID_ARG, as is batch < 1), so nvfp4_ggemm_run and the
 * other calls on such a plan take num_groups * batch pointers in that order.
 *
 * nvfp4_ggemm_run_batched takes one pointer per group, to its batch 0, and
 * batch_stride, a host array of 5 * num_groups byte strides: entries
 * 5g .. 5g+4 are the distances between consecutive batches of A_g, B_g,
 * SFA_g, SFB_g and C_g (a dense [l][rows][cols] tensor has stride rows *
 * cols bytes of its element). Each stride of a group with M_g > 0 must be
 * >= 0 (NVFP4_ERR_INVALID_ARG) and a multiple of 16 (NVFP4_ERR_ALIGNMENT); a
 * stride of 0 shares one buffer between the batches, which is allowed for
 * the inputs. SFB may be NULL when the
 * plan caches B scales (nvfp4_ggemm_prepare_b_scales with num_groups *
 * batch pointers). Otherwise as nvfp4_ggemm_run. A plan made by
 * nvfp4_ggemm_plan or nvfp4_ggemm_plan_shapes counts as batch 1.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_plan_batched(nvfp4_ggemm_plan_t *out, int device, int num_groups,
                                        int32_t batch, const int32_t *M, const int32_t *N,
                                        const int32_t *K, const nvfp4_ggemm_options_t *opt);

NVFP4_API nvfp4_status_t nvfp4_ggemm_run_batched(nvfp4_ggemm_plan_t plan, const void *const *A,
                                       const void *const *B, const void *const *SFA,
                                       const void *const *SFB, void *const *C,
                                       const int64_t *batch_stride, void *stream);

/*
 * nvfp4_ggemm_run with a row stride for every C_g: ldc is a host array of G
 * strides in fp16 elements, each >= N_g and a multiple of 8 (16-byte rows);
 * row m of C_g starts at C[g] + m * ldc[g], and columns N_g .. ldc[g]-1 are
 * not written. This covers output buffers that are column slices of a wider
 * matrix (the strided C of submission 498317). Returns NVFP4_ERR_INVALID_ARG
 * for a bad stride before anything is enqueued; otherwise as nvfp4_ggemm_run.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_run_strided(nvfp4_ggemm_plan_t plan, const void *const *A,
                                       const void *const *B, const void *const *SFA,
                                       const void *const *SFB, void *const *C, const int32_t *ldc,
                                       void *stream);

/*
 * The same operation on HOST buffers: copies every input to plan-owned
 * device buffers (allocated on the first call), runs, and copies C back,
 * all on `stream`; returns after the stream has drained. When every host
 * buffer is one the GPU can address (pinned or registered) and 16-byte
 * aligned, one kernel launch moves all the inputs over the host link and
 * one moves C back; otherwise each buffer is one copy (pageable buffers
 * then go through the driver's staging). Scales as in the plan's sf_layout
 * (cache_b_scales is ignored here).
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_run_host(nvfp4_ggemm_plan_t plan, const void *const *A,
                                    const void *const *B, const void *const *SFA,
                                    const void *const *SFB, void *const *C, void *stream);

/*
 * A plan with cache_b_scales: copy the G raw SFB tensors into the plan's
 * workspace once (B's scales are fixed, e.g. MoE expert weights): in the
 * atom layout on the RELAYOUT path, as rows padded to a multiple of 16
 * bytes on the FUSED path (so the TMA loads them even when K_g % 256 != 0,
 * instead of the scale producer's lanes copying them every call). Later
 * runs read the cached copy and ignore their SFB argument; a run before the
 * first prepare returns NVFP4_ERR_NOT_PREPARED. Asynchronous on `stream`.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_prepare_b_scales(nvfp4_ggemm_plan_t plan, const void *const *SFB,
                                            void *stream);

/*
 * Wait for `stream`, then read and clear the plan's device error word.
 * Returns NVFP4_OK, NVFP4_ERR_TIMEOUT or NVFP4_ERR_DEVICE_FAULT (or
 * NVFP4_ERR_CUDA when the synchronisation itself failed). `detail` (may be
 * NULL) receives the raw error word: bits 0-7 status, 8-15 wait site,
 * 16-31 block index.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_sync_status(nvfp4_ggemm_plan_t plan, void *stream, uint32_t *detail);

/* Release the plan and everything it owns. NULL is accepted. Synchronises the device. */
NVFP4_API nvfp4_status_t nvfp4_ggemm_destroy(nvfp4_ggemm_plan_t plan);

/*
 * Scale re-layout, one matrix: raw row-major E4M3 scales in[rows, K/16] ->
 * the 128x4 atom layout out[ceil(rows/128) * (K/64) * 512 bytes]. Atom
 * (rb, kb) covers rows [128rb, 128rb+128) and k in [64kb, 64kb+64) and sits
 * at byte (rb*(K/64) + kb)*512; inside it the scale of row r, index j = k/16
 * sits at byte (r%32)*16 + ((r%128)/32)*4 + j%4 (the scale-factor atom of
 * the CuTe kernel of submission 402102, tiled as in the TMA issue code of
 * submission 498317). Rows past `rows` are written as zero. in and out are
 * device pointers, 16-byte aligned; K % 64 == 0 (64 <= K <= 2^18); rows >= 1.
 * Asynchronous.
 */
NVFP4_API nvfp4_status_t nvfp4_sf_relayout(const void *in, void *out, int32_t rows, int32_t K, void *stream);

/* Bytes of the atom-layout copy of a [rows, K/16] scale matrix. */
NVFP4_API uint64_t nvfp4_sf_atom_bytes(int32_t rows, int32_t K);

/*
 * The work split of a plan whose units of work are pairs of row tiles
 * (row_units 2), computed on the host alone (no device, no allocation).
 * M, N and K are host arrays of the G per-group sizes (the
 * limits of nvfp4_ggemm_plan_shapes). Every group with M_g > 0 has
 * ceil(ceil(M_g/128)/2) pairs of 128-row tiles; each pair owns ceil(N_g/32)
 * consecutive 32-column chunks, numbered group by group. CTA c of the
 * persistent grid takes chunks [cta_begin[c], cta_begin[c+1]). tile_n (0 =
 * 256) and the kernel width it selects cap the tiles as in
 * nvfp4_ggemm_options_t; the kernel cuts a range into the fewest tiles within
 * the cap, of equal width to within one chunk. When there are no more pairs
 * than max_ctas, every range lies inside one pair: the split uses the
 * smallest budget of k-stages per CTA (tiles times K_g/256) that fits
 * max_ctas CTAs, and spare CTAs then shorten the longest ranges. Otherwise
 * the chunks are cut into equal contiguous ranges. cta_begin must hold
 * max_ctas + 1 entries (max_ctas 1..192); *grid receives the CTA count (0
 * when every M_g is 0). This is not an operation of the pages; it exposes
 * the scheduling step for inspection and testing.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_schedule(int num_groups, const int32_t *M, const int32_t *N,
                                    const int32_t *K, int32_t tile_n, int32_t max_ctas,
                                    int32_t *cta_begin, int32_t *grid);

/*
 * The same split for units of row_units 128-row tiles (1 or 2; 0 = the
 * choice a plan with default options makes, see row_units in
 * nvfp4_ggemm_options_t). Units of one row tile own ceil(N_g/32) chunks each
 * and their tiles are at most tile_n wide. *units (if not NULL) receives the
 * row tiles per unit used, *split_acc (if not NULL) 1 when such a plan adds
 * the even and odd 64-k slices of its one-row-tile tiles into two
 * accumulators. nvfp4_ggemm_schedule is this call with row_units = 2. Host
 * only; for inspection and testing.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_schedule_units(int num_groups, const int32_t *M, const int32_t *N,
                                          const int32_t *K, int32_t tile_n, int32_t max_ctas,
                                          int32_t row_units, int32_t *cta_begin, int32_t *grid,
                                          int32_t *units, int32_t *split_acc);

/* Plan introspection (for tests and benchmarks). */
typedef struct {
    int32_t tile_n;        /* widest output tile (columns) */
    int32_t b_stages;      /* shared-memory stages of the B ring */
    int32_t a_stages;      /* shared-memory stages of the A ring */
    int32_t chunks;        /* scheduling chunks: 32 columns of one 128-row tile */
    int32_t grid;          /* persistent CTAs launched */
    int32_t sm_count;
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t kernels_per_run; /* kernel launches enqueued by one run */
    int32_t sf_path;       /* the scale path runs take: NVFP4_SF_FUSED or NVFP4_SF_RELAYOUT (as asked) */
    int32_t row_units;     /* 128-row tiles per unit of work: 1 or 2 (see nvfp4_ggemm_options_t) */
    int32_t split_acc;     /* 1: one-row-tile tiles accumulate in two accumulators */
} nvfp4_ggemm_plan_info_t;

NVFP4_API nvfp4_status_t nvfp4_ggemm_plan_info(nvfp4_ggemm_plan_t plan, nvfp4_ggemm_plan_info_t *info);

/* Static string for a status code. */
NVFP4_API const char *nvfp4_status_string(nvfp4_status_t status);

/*
 * Grouped GEMM without any device allocation. There is no counterpart on the
 * pages: this entry point exists for callers that may not call cudaMalloc
 * (code under a fixed memory budget or its own device allocator, code in a
 * region where an allocation would synchronise the device, plugins that must
 * not grow the process's device footprint). It computes what
 * nvfp4_ggemm_run computes for raw row-major scales, with the same kernels
 * and the units of work a plan with default options would choose, but
 * needs no plan: the per-group tensor maps and the device error word it
 * needs live in a static device array of under 112 KB that every GPU loading
 * the library holds until the process exits.
 *
 * Arguments: as nvfp4_ggemm_plan + nvfp4_ggemm_run (M host array of G row
 * counts, A/B/SFA/SFB/C host arrays of G device pointers, raw scales), on
 * the current device. Limits: 1 <= num_groups <= 64, otherwise
 * NVFP4_ERR_UNSUPPORTED_SHAPE before anything is enqueued; the shape rules,
 * other checks and status codes are those of plan/run (K % 64 == 0: raw
 * scale rows that are not 16-byte units are copied by the kernel's scale
 * producer, as on the plan's FUSED path).
 *
 * The first call on a device looks up the array's device address and
 * configures the kernel; make that first call before any stream capture.
 * A call made while `stream` is being captured returns
 * NVFP4_ERR_INVALID_ARG and enqueues nothing (its table is staged in a host
 * buffer that the next call rewrites). Every call reuses the same array (it
 * keeps the last call's contents; the error word is cleared at the start of
 * each call), so calls whose work overlaps on the GPU (different streams, or
 * different host threads) race: serialise them on one stream. Asynchronous
 * on `stream`; if `status_out` is not NULL the call waits for the stream and
 * stores the device error word there (0 = fine), returning NVFP4_ERR_TIMEOUT
 * or NVFP4_ERR_DEVICE_FAULT when it is not 0. A device error of a call made
 * without `status_out` is not reported: the next call clears the word.
 * Never calls cudaMalloc, cudaFree or any other allocating routine.
 */
NVFP4_API nvfp4_status_t nvfp4_ggemm_run_noalloc(int num_groups, const int32_t *M, int32_t N, int32_t K,
                                                 const void *const *A, const void *const *B,
                                                 const void *const *SFA, const void *const *SFB,
                                                 void *const *C, void *stream, uint32_t *status_out);

/* Library version, major*10000 + minor*100 + patch. */
NVFP4_API int nvfp4_ggemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GGEMM_H */
