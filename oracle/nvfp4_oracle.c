/*
 * CPU oracle for the NVFP4 block-scaled grouped GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition of the nvfp4_group_gemm problem as
 * the custom_kernel docstring of kernelindex submission 503584 states it, and
 * the product of A, SFA, B and SFB that its kernel-launch comment names):
 *
 *   C_g[m, n] = RN_fp16( sum_{k=0}^{K-1} e2m1(A_g[m,k]) * e4m3(SFA_g[m, k/16])
 *                                      * e2m1(B_g[n,k]) * e4m3(SFB_g[n, k/16]) )
 *
 * with A_g [M_g, K/2] and B_g [N, K/2] holding two E2M1 codes per byte (low
 * nibble = even k), SFA_g [M_g, K/16] and SFB_g [N, K/16] one E4M3 code per
 * 16 consecutive k (the kernel configuration block of submission 503584 names
 * Float4E2M1FN data, Float8E4M3FN scales, sf_vec_size = 16, Float16 output).
 *
 * Steps, in this order:
 *   1. decode tables written from the two formats' definitions;
 *   2. every element decoded to fp64 with its scale applied (exact);
 *   3. the sum over k in fp64, ascending k;
 *   4. one rounding, fp64 -> fp16 round-to-nearest-even, never via fp32.
 *
 * The scale re-layout restated here is the 128x4 "block scaling factors"
 * atom that the CuTe kernel of submission 402102 builds (atom shape
 * ((32,4),(16,4)), stride ((16,4),(0,1))) tiled as in the TMA issue code of
 * submission 498317 (512-byte blocks, block index (row/128)*(K/64) + k/64).
 *
 * Building with -DORACLE_MUTANT=n plants one deliberate mistake (used only
 * by the test that shows the pins catch such mistakes).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- decode */

/* E2M1: bit 3 sign, bits 2:1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 2^(1-1) * 0.5. */
static double e2m1_from_fields(unsigned code)
{
#if ORACLE_MUTANT == 7
    unsigned s = (code >> 2) & 1u; /* planted: wrong sign bit */
#else
    unsigned s = (code >> 3) & 1u;
#endif
    unsigned e = (code >> 1) & 3u;
    unsigned m = code & 1u;
    double mag;
    if (e == 0) {
#if ORACLE_MUTANT == 6
        mag = (double)m; /* planted: subnormal read as 1.0 */
#else
        mag = 0.5 * (double)m;
#endif
    } else {
        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    }
    return s ? -mag : mag;
}

/* E4M3 (FN flavour): bit 7 sign, bits 6:3 exponent (bias 7), bits 2:0
 * mantissa. Exponent 0 is subnormal (m * 2^-9). S.1111.111 is NaN; there is
 * no infinity. */
static double e4m3_from_fields(unsigned code)
{
    unsigned s = (code >> 7) & 1u;
    unsigned e = (code >> 3) & 15u;
    unsigned m = code & 7u;
#if ORACLE_MUTANT == 4
    const int bias = 8; /* planted: FNUZ-style bias */
#else
    const int bias = 7;
#endif
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - bias);
    return s ? -mag : mag;
}

static double E2M1[16];
static double E4M3[256];
static int tables_ready = 0;

void oracle_init(void)
{
    if (tables_ready) return;
    for (unsigned c = 0; c < 16; ++c) E2M1[c] = e2m1_from_fields(c);
    for (unsigned c = 0; c < 256; ++c) E4M3[c] = e4m3_from_fields(c);
    tables_ready = 1;
}

double oracle_e2m1(int code) { oracle_init(); return E2M1[code & 15]; }
double oracle_e4m3(int code) { oracle_init(); return E4M3[code & 255]; }

/* ------------------------------------------------------- fp64 -> fp16 RNE */

/* Round a non-negative double q to the nearest integer, ties to even.
 * q is exact, so floor and the comparisons with 0.5 are exact. */
static double rne_int(double q)
{
    double f = floor(q);
    double r = q - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
#if ORACLE_MUTANT == 9
    return f + 1.0; /* planted: ties away from zero */
#else
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
#endif
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. Largest
 * finite 65504; the halfway point to the next binade, 65520, rounds to
 * infinity (65504 has an odd mantissa). Subnormals are multiples of 2^-24. */
uint16_t oracle_fp16_rne(double x)
{
    if (isnan(x)) return 0x7E00u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        double n = rne_int(ldexp(a, 24)); /* units of 2^-24; n == 1024 is the smallest normal */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int ex;
    (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;       /* a in [2^E, 2^(E+1)) */
    double n = rne_int(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (n >= 2048.0) { n = 1024.0; E += 1; }
    if (E + 15 >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* Element-wise oracle_fp16_rne over an array (for the rounding pins). */
void oracle_fp16_rne_array(long n, const double *in, uint16_t *out)
{
    for (long i = 0; i < n; ++i) out[i] = oracle_fp16_rne(in[i]);
}

/* ------------------------------------------------------ element decoding */

static unsigned nibble(const uint8_t *row, int k, int is_b)
{
    uint8_t byte = row[k >> 1];
#if ORACLE_MUTANT == 1
    if (is_b) return (k & 1) ? (byte & 15u) : (byte >> 4); /* planted: B nibble order swapped */
#else
    (void)is_b;
#endif
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);
}

static int scale_index(int k)
{
#if ORACLE_MUTANT == 2
    return k / 32; /* planted: 32-element scale blocks */
#else
    return k / 16;
#endif
}

/* Decode R rows of a [R, K/2] operand with its [R, K/16] scales into
 * out[R*K] fp64: value(k) = e2m1(code_k) * e4m3(scale[k/16]). Exact. */
static void decode_operand(int R, int K, const uint8_t *q, const uint8_t *sf, double *out, int is_b)
{
    for (int r = 0; r < R; ++r) {
        const uint8_t *qrow = q + (size_t)r * (size_t)(K / 2);
        const uint8_t *srow = sf + (size_t)r * (size_t)(K / 16);
        double *orow = out + (size_t)r * (size_t)K;
        for (int k = 0; k < K; ++k)
            orow[k] = E2M1[nibble(qrow, k, is_b)] * E4M3[srow[scale_index(k)]];
    }
}

static double dot_ascending(const double *a, const double *b, int K)
{
    double s = 0.0;
#if ORACLE_MUTANT == 3
    K -= 1; /* planted: last term dropped */
#endif
    for (int k = 0; k < K; ++k) s += a[k] * b[k];
    return s;
}

static uint16_t to_fp16(double s)
{
#if ORACLE_MUTANT == 5
    return oracle_fp16_rne((double)(float)s); /* planted: double rounding via fp32 */
#else
    return oracle_fp16_rne(s);
#endif
}

/* ----------------------------------------------------------- exactness */

/* Exponent of the lowest set bit of a finite non-zero double. */
static int lsb_exponent(double v)
{
    int ex;
    double f = frexp(fabs(v), &ex); /* f in [0.5,1): f*2^53 is an integer < 2^53 */
    uint64_t mant = (uint64_t)ldexp(f, 53);
    int tz = 0;
    while (((mant >> tz) & 1u) == 0u) ++tz;
    return ex - 53 + tz;
}

/* 1 when every partial sum of every dot product is representable in fp64,
 * so the fp64 sum is the exact real sum whatever its order. */
static int sum_is_exact(const double *ad, size_t na, const double *bd, size_t nb, int K)
{
    double amax = 0.0, bmax = 0.0;
    int alsb = 100000, blsb = 100000;
    for (size_t i = 0; i < na; ++i) {
        if (ad[i] != 0.0) {
            if (isnan(ad[i])) return 0;
            if (fabs(ad[i]) > amax) amax = fabs(ad[i]);
            int l = lsb_exponent(ad[i]);
            if (l < alsb) alsb = l;
        }
    }
    for (size_t i = 0; i < nb; ++i) {
        if (bd[i] != 0.0) {
            if (isnan(bd[i])) return 0;
            if (fabs(bd[i]) > bmax) bmax = fabs(bd[i]);
            int l = lsb_exponent(bd[i]);
            if (l < blsb) blsb = l;
        }
    }
    if (amax == 0.0 || bmax == 0.0) return 1;
    /* every term is a multiple of 2^(alsb+blsb); every partial sum is below K*amax*bmax */
    double span = log2((double)K * amax * bmax) - (double)(alsb + blsb);
#if ORACLE_MUTANT == 10
    (void)span;
    return 1; /* planted: every sum declared exact */
#elif ORACLE_MUTANT == 11
    return span < 54.0; /* planted: one bit more than fp64 holds */
#else
    return span < 52.0;
#endif
}

/* --------------------------------------------------------- one group GEMM */

struct rows_job {
    const double *ad, *bd;
    int m0, m1, N, K;
    uint16_t *C16;
    double *Cx;
};

static void *rows_worker(void *p)
{
    struct rows_job *j = (struct rows_job *)p;
    for (int m = j->m0; m < j->m1; ++m) {
        const double *a = j->ad + (size_t)m * (size_t)j->K;
        for (int n = 0; n < j->N; ++n) {
            double s = dot_ascending(a, j->bd + (size_t)n * (size_t)j->K, j->K);
            if (j->C16) j->C16[(size_t)m * (size_t)j->N + (size_t)n] = to_fp16(s);
            if (j->Cx) j->Cx[(size_t)m * (size_t)j->N + (size_t)n] = s;
        }
    }
    return NULL;
}

static int host_threads(int requested)
{
    if (requested > 0) return requested;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * C16 [M, N] fp16 bits (nullable), Cx [M, N] fp64 pre-rounding sums
 * (nullable). Rows are split across `nthreads` threads (0 = all host cores);
 * the result does not depend on the split. Returns 1 when the fp64 sums are
 * provably exact, 0 when they may carry fp64 rounding, -1 on a bad argument,
 * -2 when out of memory.
 */
int oracle_group_gemm(int M, int N, int K, const uint8_t *A, const uint8_t *B, const uint8_t *SFA,
                      const uint8_t *SFB, uint16_t *C16, double *Cx, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (K % 16) != 0) return -1;
    oracle_init();
    if (M == 0 || N == 0) return 1;
    double *ad = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    double *bd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    if (!ad || !bd) { free(ad); free(bd); return -2; }
    decode_operand(M, K, A, SFA, ad, 0);
    decode_operand(N, K, B, SFB, bd, 1);
    int exact = sum_is_exact(ad, (size_t)M * (size_t)K, bd, (size_t)N * (size_t)K, K);

    int T = host_threads(nthreads);
    if (T > M) T = M;
    pthread_t *tid = (pthread_t *)calloc((size_t)T, sizeof(pthread_t));
    struct rows_job *jobs = (struct rows_job *)calloc((size_t)T, sizeof(struct rows_job));
    if (!tid || !jobs) { free(tid); free(jobs); free(ad); free(bd); return -2; }
    for (int t = 0; t < T; ++t) {
        jobs[t].ad = ad; jobs[t].bd = bd; jobs[t].N = N; jobs[t].K = K;
        jobs[t].m0 = (int)((long)M * t / T);
        jobs[t].m1 = (int)((long)M * (t + 1) / T);
        jobs[t].C16 = C16; jobs[t].Cx = Cx;
    }
    int started = 0;
    for (int t = 1; t < T; ++t)
        if (pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) == 0) ++started; else rows_worker(&jobs[t]), tid[t] = 0;
    rows_worker(&jobs[0]);
    for (int t = 1; t < T; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    (void)started;
    free(tid); free(jobs); free(ad); free(bd);
    return exact;
}

/*
 * Individual entries (rows[i], cols[i]) of one group's C, each summed the same
 * way (fp64, ascending k, one rounding). For sampled checks at sizes where the
 * full product is too slow. Returns 0, or -1 on a bad argument.
 */
int oracle_group_entries(int M, int N, int K, const uint8_t *A, const uint8_t *B, const uint8_t *SFA,
                         const uint8_t *SFB, int count, const int32_t *rows, const int32_t *cols,
                         uint16_t *out16, double *outx)
{
    if (M < 0 || N < 0 || K < 0 || (K % 16) != 0 || count < 0) return -1;
    oracle_init();
    double *a = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!a || !b) { free(a); free(b); return -1; }
    for (int i = 0; i < count; ++i) {
        int m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) { free(a); free(b); return -1; }
        decode_operand(1, K, A + (size_t)m * (size_t)(K / 2), SFA + (size_t)m * (size_t)(K / 16), a, 0);
        decode_operand(1, K, B + (size_t)n * (size_t)(K / 2), SFB + (size_t)n * (size_t)(K / 16), b, 1);
        double s = dot_ascending(a, b, K);
        if (out16) out16[i] = to_fp16(s);
        if (outx) outx[i] = s;
    }
    free(a); free(b);
    return 0;
}

/* ------------------------------------------------------ scale re-layout */

/*
 * Raw row-major scales in[R, K/16] -> the 128x4-atom layout: for every block
 * of 128 rows and every 64 values of k (four scales) one 512-byte atom; atoms
 * ordered (row block, k/64) with k/64 fastest; inside an atom the scale of
 * (row r, scale index j) sits at byte (r%32)*16 + ((r%128)/32)*4 + (j%4).
 * Rows past R (up to the next multiple of 128) are written as zero.
 * out holds ceil(R/128) * (K/64) * 512 bytes. Returns 0, or -1 when K is not
 * a multiple of 64.
 */
int oracle_sf_relayout(int R, int K, const uint8_t *in, uint8_t *out)
{
    if (R < 0 || K <= 0 || (K % 64) != 0) return -1;
    int J = K / 16;
    int rblocks = (R + 127) / 128;
    for (int r = 0; r < rblocks * 128; ++r) {
        for (int j = 0; j < J; ++j) {
            uint8_t v = (r < R) ? in[(size_t)r * (size_t)J + (size_t)j] : 0;
#if ORACLE_MUTANT == 8
            size_t atom = (size_t)(j / 4) * (size_t)rblocks + (size_t)(r / 128); /* planted: atoms ordered row-block fastest */
#else
            size_t atom = (size_t)(r / 128) * (size_t)(K / 64) + (size_t)(j / 4);
#endif
            size_t off = (size_t)(r % 32) * 16 + (size_t)((r % 128) / 32) * 4 + (size_t)(j % 4);
            out[atom * 512 + off] = v;
        }
    }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
