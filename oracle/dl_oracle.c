/*
 * CPU oracle for the decode linear layer.  TEST INFRASTRUCTURE ONLY: nothing in
 * the library calls, links or includes this file; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg use it.  It shares no code, header
 * or table with the CUDA path.
 *
 * What it computes (the plain definition, nothing else):
 *
 *   y_ref[m][n] = bias[n] + sum_{k = k_begin}^{k_end - 1} X(m,k) * Wv(n,k)
 *
 * in IEEE double, with k ascending.  This is the linear layer y = x W^T of
 * "Multi-GPU Inference and Serving at Scale" (Example 2, a column split: a
 * linear layer computes y = x W) with W stored [N, K], the weight rows taken
 * as columns as in the TileLang loop of "9% faster GLM-5.3-Flash prefill with
 * GPU-to-GPU IPC", section "TileLang: twice as fast, and no faster").  A k sub-range gives the
 * partial sum one device holds under a row split (same page, Example 3).
 *
 *   X(m,k)  = the bf16 activation, decoded exactly (its 16 bits are the top
 *             half of an IEEE binary32).
 *   Wv(n,k) = the bf16 weight decoded exactly, or, for weight-only FP8,
 *             E4M3[q(n,k)] * S[n / 128][k / 128]: the e4m3 code decoded by an
 *             explicit 256-entry table and multiplied by the fp32 scale of its
 *             128x128 block (the dequantisation "B_h = B_s * S[nb, k // 128]"
 *             of the TileLang loop).  The product is exact in double (4-bit
 *             by 24-bit significands).
 *
 * Every product X*Wv is exact in double (at most 8 + 28 significant bits), so
 * the only rounding is the double-precision running sum.  The oracle also
 * returns A[m][n] = sum_k |X*Wv|, the scale of the parity tolerance.
 *
 * E4M3: the pages only say "FP8" / "weight-only FP8"; the workload clamps to
 * +-448 before the cast, which fixes the OCP E4M3FN variant: sign, 4-bit
 * exponent with bias 7, 3-bit mantissa, no infinities, S.1111.111 = NaN,
 * largest finite 448.  Normal: (-1)^s 2^(e-7) (1 + m/8), e = 1..15;
 * subnormal: (-1)^s 2^-6 (m/8).
 *
 * Rows are computed independently; the work is spread over POSIX threads by
 * whole output rows, which changes no arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BF16 0
#define ORACLE_FP8_B128 1

static double g_e4m3[256];
static int g_e4m3_ready = 0;
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

/* Closed form of one E4M3FN code. */
static double e4m3_closed_form(unsigned code) {
    unsigned s = (code >> 7) & 1u;
    unsigned e = (code >> 3) & 15u;
    unsigned m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;            /* S.1111.111 */
    if (e == 0u)
        mag = ldexp((double)m / 8.0, -6);           /* subnormal */
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

static void build_table(void) {
    for (unsigned c = 0; c < 256u; ++c) g_e4m3[c] = e4m3_closed_form(c);
    g_e4m3_ready = 1;
}

static void ensure_table(void) { pthread_once(&g_once, build_table); }

void dl_oracle_e4m3_table(double* out256) {
    ensure_table();
    memcpy(out256, g_e4m3, sizeof(g_e4m3));
}

/* Exact value of a bf16 bit pattern. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void dl_oracle_bf16_values(const uint16_t* bits, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(bits[i]);
}

/*
 * binary32 -> bf16, round to nearest, ties to even, on the bit pattern.
 * NaN stays NaN (quiet); infinities and overflow to infinity follow IEEE.
 */
uint16_t dl_oracle_round_f32_to_bf16(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

void dl_oracle_round_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = dl_oracle_round_f32_to_bf16(in[i]);
}

typedef struct {
    int dtype, M, N, K, k_begin, k_end;
    const uint16_t* x;
    const void* w;
    const float* scales;
    const uint16_t* bias;
    const int64_t* rows;   /* which n to compute; NULL = all */
    int64_t n_rows;
    double* y;             /* [M][n_rows] */
    double* a;             /* [M][n_rows] or NULL */
    int64_t r_begin, r_end;
} job_t;

static void* run_rows(void* arg) {
    const job_t* j = (const job_t*)arg;
    const int64_t kb_count = ((int64_t)j->K + 127) / 128;
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const int64_t n = j->rows ? j->rows[r] : r;
        for (int m = 0; m < j->M; ++m) {
            double sum = 0.0, asum = 0.0;
            const uint16_t* xm = j->x + (int64_t)m * j->K;
            for (int64_t k = j->k_begin; k < j->k_end; ++k) {
                double wv;
                if (j->dtype == ORACLE_BF16) {
                    wv = bf16_value(((const uint16_t*)j->w)[n * j->K + k]);
                } else {
                    uint8_t q = ((const uint8_t*)j->w)[n * j->K + k];
                    double s = (double)j->scales[(n / 128) * kb_count + k / 128];
                    wv = g_e4m3[q] * s;
                }
                double p = bf16_value(xm[k]) * wv;
                sum += p;
                asum += fabs(p);
            }
            if (j->bias) sum += bf16_value(j->bias[n]);
            j->y[(int64_t)m * j->n_rows + r] = sum;
            if (j->a) j->a[(int64_t)m * j->n_rows + r] = asum;
        }
    }
    return NULL;
}

/*
 * y[M][n_rows] (and a[M][n_rows] if non-NULL) for the output rows listed in
 * rows[0..n_rows) (rows == NULL: n_rows must equal N and all rows are
 * computed), summing k over [k_begin, k_end).  bias may be NULL.  x is bf16
 * bits [M][K]; w is bf16 bits [N][K] (dtype 0) or e4m3 codes [N][K] (dtype 1,
 * with scales [ceil(N/128)][ceil(K/128)]).  Returns 0, or -1 on bad arguments.
 */
int dl_oracle_linear(int dtype, int M, int N, int K, const uint16_t* x, const void* w,
                     const float* scales, const uint16_t* bias, int k_begin, int k_end,
                     const int64_t* rows, int64_t n_rows, double* y, double* a,
                     int n_threads) {
    ensure_table();
    if (M < 0 || N < 0 || K < 0 || k_begin < 0 || k_end > K || k_begin > k_end) return -1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_FP8_B128) return -1;
    if (dtype == ORACLE_FP8_B128 && !scales) return -1;
    if (!rows && n_rows != N) return -1;
    if (n_rows == 0 || M == 0) return 0;
    if (!x || !w || !y) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > n_rows) n_threads = (int)n_rows;

    job_t jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < n_threads; ++t) {
        job_t* j = &jobs[t];
        j->dtype = dtype; j->M = M; j->N = N; j->K = K;
        j->k_begin = k_begin; j->k_end = k_end;
        j->x = x; j->w = w; j->scales = scales; j->bias = bias;
        j->rows = rows; j->n_rows = n_rows; j->y = y; j->a = a;
        j->r_begin = n_rows * t / n_threads;
        j->r_end = n_rows * (t + 1) / n_threads;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) break;
        started = t;
    }
    run_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < n_threads; ++t) run_rows(&jobs[t]);
    return 0;
}
