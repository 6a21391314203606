/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the decode-step
 * skinny GEMV paths.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * bench's cpu_baseline / reference legs load this library.  It shares no code,
 * header, table or helper with the CUDA library under
 * quantized_skinny_gemm_gb300/csrc, and neither side includes the other.
 *
 * Notation (all operations):  W is [N][K] row-major (output features x input
 * features, K contiguous, the nn.Linear layout), x is [M][K], y is [M][N] and
 *      y[m][n] = sum_k W[n][k] * x[m][k].
 * Every floating-point sum runs in IEEE double in ascending k; every integer
 * sum runs in int64.  Rows may be evaluated for a subset (rows != NULL), in
 * which case outputs are laid out [M][nrows] in the order of `rows`.
 *
 * What each function follows (the pages give no formulas; the readings are
 * stated per function):
 *  - orc_gemv_fp: the M=1 vector-matrix product that the custom cube matmul of
 *    "MiniCPM-V on Orange Pi AIPro (Ascend 310B)" computes (paragraph on the
 *    custom M=1 cube matmul), written as its plain definition in fp64.
 *  - orc_gemv_w8a8: "vLLM Arm CPU optimizations", section "INT8 W8A8 (8-bit
 *    weights and activations)": signed int8 x int8 products, exact integer
 *    accumulation, then the per-output-channel weight scale and the per-token
 *    activation scale.
 *  - orc_gemv_w4: "vLLM Arm CPU optimizations", section "INT8 W4A8", and the
 *    fused INT4 dequantization named in the closing paragraph of the
 *    Orange Pi AIPro post: two's-complement nibbles, byte j of a row holding
 *    k = 2j in bits 0-3 and k = 2j+1 in bits 4-7, one fp16 scale per group of
 *    `group` consecutive k.  W4A16 takes fp16 activations, W4A8 int8
 *    activations with one fp32 scale per token.
 *  - orc_quant_act: per-token symmetric int8 activation quantization for the
 *    W8A8 / W4A8 paths (same page and sections), decided in IEEE fp32:
 *    s = amax/127, q = clamp(rne(x/s), -127, 127); s = 1, q = 0 when amax = 0.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared -pthread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---- scalar decoding, written from the formats' definitions ------------ */

/* IEEE binary16: sign bit 15, exponent bits 14-10 (bias 15), fraction bits
 * 9-0.  Exponent 0 is zero/subnormal (fraction * 2^-24); 31 is inf/NaN. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void orc_decode_f16(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(h[i]);
}

void orc_decode_bf16(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(h[i]);
}

/* One packed int4 byte -> its two codes.  Low nibble is the even k, high
 * nibble the odd k; a nibble c >= 8 stands for c - 16. */
static int nibble_value(int c) { return c >= 8 ? c - 16 : c; }

void orc_unpack_w4(const uint8_t* b, int64_t nbytes, int8_t* codes) {
    for (int64_t j = 0; j < nbytes; ++j) {
        int lo = b[j] & 0xF;
        int hi = (b[j] >> 4) & 0xF;
        codes[2 * j] = (int8_t)nibble_value(lo);
        codes[2 * j + 1] = (int8_t)nibble_value(hi);
    }
}

/* Inverse of orc_unpack_w4 for codes in [-8, 7]; returns -1 on a code out of
 * range. */
int orc_pack_w4(const int8_t* codes, int64_t ncodes, uint8_t* b) {
    if (ncodes % 2) return -1;
    for (int64_t j = 0; j < ncodes / 2; ++j) {
        int lo = codes[2 * j], hi = codes[2 * j + 1];
        if (lo < -8 || lo > 7 || hi < -8 || hi > 7) return -1;
        b[j] = (uint8_t)(((lo + 16) % 16) | (((hi + 16) % 16) << 4));
    }
    return 0;
}

/* Index of the largest value; on exactly equal values the lowest index wins.
 * NaN entries never win (they compare false).  Returns -1 for n == 0 or when
 * every entry is NaN. */
int64_t orc_argmax(const double* v, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best;
}

/* ---- row-partitioned threading ----------------------------------------- */

typedef struct {
    int64_t lo, hi;           /* slice of the row list */
    const void* job;
    void (*fn)(const void* job, int64_t lo, int64_t hi);
} slice_t;

static void* run_slice(void* arg) {
    slice_t* s = (slice_t*)arg;
    s->fn(s->job, s->lo, s->hi);
    return NULL;
}

static int resolve_threads(int nthreads, int64_t nrows) {
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
    return nthreads;
}

/* Runs fn over [0, nrows) split into nthreads contiguous slices.  Each row is
 * computed by exactly one thread with the same code, so the result does not
 * depend on the thread count. */
static int parallel_rows(const void* job, int64_t nrows, int nthreads,
                         void (*fn)(const void*, int64_t, int64_t)) {
    int t = resolve_threads(nthreads, nrows);
    if (t <= 1) {
        fn(job, 0, nrows);
        return 0;
    }
    pthread_t th[256];
    int live[256];
    slice_t sl[256];
    for (int i = 0; i < t; ++i) {
        sl[i].lo = nrows * i / t;
        sl[i].hi = nrows * (i + 1) / t;
        sl[i].job = job;
        sl[i].fn = fn;
        live[i] = pthread_create(&th[i], NULL, run_slice, &sl[i]) == 0;
        if (!live[i]) run_slice(&sl[i]); /* no thread: run this slice here */
    }
    for (int i = 0; i < t; ++i)
        if (live[i]) pthread_join(th[i], NULL);
    return 0;
}

static int64_t row_at(const int64_t* rows, int64_t i) { return rows ? rows[i] : i; }

/* ---- FP16 / BF16 GEMV --------------------------------------------------- */

typedef struct {
    const uint16_t* W;
    const double* xd; /* x decoded to double, [M][K] */
    int fmt;
    int64_t M, N, K, nrows;
    const int64_t* rows;
    double *y, *A;
} fp_job;

static void fp_rows(const void* vj, int64_t lo, int64_t hi) {
    const fp_job* j = (const fp_job*)vj;
    double* w = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    for (int64_t i = lo; i < hi; ++i) {
        int64_t n = row_at(j->rows, i);
        const uint16_t* wr = j->W + n * j->K;
        for (int64_t k = 0; k < j->K; ++k)
            w[k] = j->fmt == 0 ? orc_f16_to_f64(wr[k]) : orc_bf16_to_f64(wr[k]);
        for (int64_t m = 0; m < j->M; ++m) {
            const double* xm = j->xd + m * j->K;
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < j->K; ++k) {
                double p = w[k] * xm[k]; /* exact: both factors have <= 11 significant bits */
                s += p;
                a += fabs(p);
            }
            j->y[m * j->nrows + i] = s;
            if (j->A) j->A[m * j->nrows + i] = a;
        }
    }
    free(w);
}

/* y[m][i] = sum_k W[rows[i]][k] x[m][k] in fp64; A[m][i] = sum_k |W x|.
 * fmt 0 = fp16, 1 = bf16 (both W and x). */
int orc_gemv_fp(const uint16_t* W, const uint16_t* x, int fmt, int64_t M, int64_t N,
                int64_t K, const int64_t* rows, int64_t nrows, double* y, double* A,
                int nthreads) {
    if (!W || !x || !y || M < 0 || N < 0 || K < 0 || (fmt != 0 && fmt != 1)) return -1;
    if (!rows) nrows = N;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -2;
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -3;
    for (int64_t i = 0; i < M * K; ++i)
        xd[i] = fmt == 0 ? orc_f16_to_f64(x[i]) : orc_bf16_to_f64(x[i]);
    fp_job j = {W, xd, fmt, M, N, K, nrows, rows, y, A};
    parallel_rows(&j, nrows, nthreads, fp_rows);
    free(xd);
    return 0;
}

/* ---- W8A8 --------------------------------------------------------------- */

typedef struct {
    const int8_t* W;
    const float* s_w;
    const int8_t* xq;
    const float* s_x;
    int64_t M, N, K, nrows;
    const int64_t* rows;
    int64_t* acc;
    double *y, *A;
} w8_job;

static void w8_rows(const void* vj, int64_t lo, int64_t hi) {
    const w8_job* j = (const w8_job*)vj;
    for (int64_t i = lo; i < hi; ++i) {
        int64_t n = row_at(j->rows, i);
        const int8_t* wr = j->W + n * j->K;
        for (int64_t m = 0; m < j->M; ++m) {
            const int8_t* xm = j->xq + m * j->K;
            int64_t acc = 0, aabs = 0;
            for (int64_t k = 0; k < j->K; ++k) {
                int64_t p = (int64_t)wr[k] * (int64_t)xm[k];
                acc += p;
                aabs += p < 0 ? -p : p;
            }
            double scale = (double)j->s_w[n] * (double)j->s_x[m];
            if (j->acc) j->acc[m * j->nrows + i] = acc;
            j->y[m * j->nrows + i] = (double)acc * scale;
            if (j->A) j->A[m * j->nrows + i] = (double)aabs * fabs(scale);
        }
    }
}

/* acc[m][i] = sum_k W[n][k] xq[m][k] exactly (int64);
 * y[m][i] = acc * s_w[n] * s_x[m] in fp64; A = sum_k |W xq| * |s_w s_x|. */
int orc_gemv_w8a8(const int8_t* W, const float* s_w, const int8_t* xq, const float* s_x,
                  int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                  int64_t* acc, double* y, double* A, int nthreads) {
    if (!W || !s_w || !xq || !s_x || !y || M < 0 || N < 0 || K < 0) return -1;
    if (!rows) nrows = N;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -2;
    w8_job j = {W, s_w, xq, s_x, M, N, K, nrows, rows, acc, y, A};
    parallel_rows(&j, nrows, nthreads, w8_rows);
    return 0;
}

/* ---- W4A16 / W4A8 ------------------------------------------------------- */

typedef struct {
    const uint8_t* Wq;
    const uint16_t* scales; /* fp16 bits, [N][K/group] */
    int64_t group;
    const double* xd;    /* W4A16: x decoded to double [M][K]; NULL for W4A8 */
    const int8_t* xq;    /* W4A8 */
    const float* s_x;    /* W4A8 */
    int64_t M, N, K, nrows;
    const int64_t* rows;
    double *y, *A;
    int64_t* acc_groups; /* W4A8 optional: [M][nrows][K/group] */
} w4_job;

static void w4_rows(const void* vj, int64_t lo, int64_t hi) {
    const w4_job* j = (const w4_job*)vj;
    int64_t G = j->K / j->group;
    int8_t* q = (int8_t*)malloc((size_t)(j->K > 0 ? j->K : 1));
    for (int64_t i = lo; i < hi; ++i) {
        int64_t n = row_at(j->rows, i);
        orc_unpack_w4(j->Wq + n * (j->K / 2), j->K / 2, q);
        const uint16_t* sr = j->scales + n * G;
        for (int64_t m = 0; m < j->M; ++m) {
            double y = 0.0, a = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double s = orc_f16_to_f64(sr[g]);
                if (j->xd) { /* W4A16 */
                    const double* xm = j->xd + m * j->K;
                    double P = 0.0, Pa = 0.0;
                    for (int64_t k = g * j->group; k < (g + 1) * j->group; ++k) {
                        double p = (double)q[k] * xm[k];
                        P += p;
                        Pa += fabs(p);
                    }
                    y += s * P;
                    a += fabs(s) * Pa;
                } else { /* W4A8 */
                    const int8_t* xm = j->xq + m * j->K;
                    int64_t acc = 0, aabs = 0;
                    for (int64_t k = g * j->group; k < (g + 1) * j->group; ++k) {
                        int64_t p = (int64_t)q[k] * (int64_t)xm[k];
                        acc += p;
                        aabs += p < 0 ? -p : p;
                    }
                    if (j->acc_groups) j->acc_groups[(m * j->nrows + i) * G + g] = acc;
                    y += s * (double)acc;
                    a += fabs(s) * (double)aabs;
                }
            }
            if (!j->xd) {
                y *= (double)j->s_x[m];
                a *= fabs((double)j->s_x[m]);
            }
            j->y[m * j->nrows + i] = y;
            if (j->A) j->A[m * j->nrows + i] = a;
        }
    }
    free(q);
}

/* W4A16 when x16 != NULL:  y = sum_g s[n][g] * sum_{k in g} q[n][k] x[m][k].
 * W4A8 when x16 == NULL:   acc_g = sum_{k in g} q xq (exact),
 *                          y = s_x[m] * sum_g s[n][g] * acc_g.
 * A = sum_k |dequantized w * dequantized x|. */
int orc_gemv_w4(const uint8_t* Wq, const uint16_t* scales, int64_t group, const uint16_t* x16,
                const int8_t* xq, const float* s_x, int64_t M, int64_t N, int64_t K,
                const int64_t* rows, int64_t nrows, double* y, double* A,
                int64_t* acc_groups, int nthreads) {
    if (!Wq || !scales || !y || M < 0 || N < 0 || K < 0 || group <= 0) return -1;
    if (K % group || K % 2) return -1;
    if (!x16 && (!xq || !s_x)) return -1;
    if (!rows) nrows = N;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -2;
    double* xd = NULL;
    if (x16) {
        xd = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
        if (!xd) return -3;
        for (int64_t i = 0; i < M * K; ++i) xd[i] = orc_f16_to_f64(x16[i]);
    }
    w4_job j = {Wq, scales, group, xd, xq, s_x, M, N, K, nrows, rows, y, A,
                x16 ? NULL : acc_groups};
    parallel_rows(&j, nrows, nthreads, w4_rows);
    free(xd);
    return 0;
}

/* ---- per-token activation quantization (decided in IEEE fp32) ----------- */

int orc_quant_act(const uint16_t* x16, int64_t M, int64_t K, int8_t* q, float* s) {
    if (!x16 || !q || !s || M < 0 || K < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* xm = x16 + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = fabsf((float)orc_f16_to_f64(xm[k])); /* exact: fp16 is a subset of fp32 */
            if (v > amax) amax = v;
        }
        volatile float scale = amax > 0.0f ? amax / 127.0f : 1.0f;
        s[m] = scale;
        for (int64_t k = 0; k < K; ++k) {
            if (amax == 0.0f) {
                q[m * K + k] = 0;
                continue;
            }
            volatile float t = (float)orc_f16_to_f64(xm[k]) / scale; /* one IEEE fp32 division */
            float r = rintf(t); /* default rounding mode: to nearest, ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[m * K + k] = (int8_t)r;
        }
    }
    return 0;
}
