/*
 * fp8blk_oracle.c -- plain CPU oracle for the FP8 block-scaled decode GEMV,
 * its fused greedy argmax, and the NVFP4 routed-expert dequant + GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library: every decode here is written from the format definitions and
 * every sum is a sequential double-precision loop.
 *
 * Sources (docs.rs pages of the memra-engine crate):
 *   [dsv4_gpu]  "Module dsv4_gpu" page, struct Fp8Dense: an FP8-blk linear is
 *               e4m3 codes [rows, cols] plus a 128x128 grid of e8m0 block
 *               scales decoded to f32 on the host; every e8m0 code is a power
 *               of two and 0xFF is refused; a weight is e4m3(code) * scale.
 *   [dsv4_gpu]  same page, module header and enum ExpertArm: routed experts
 *               stay NVFP4 and each activated expert is dequantised into a
 *               reused bf16 scratch, exact in bf16, then a bf16 GEMM with f32
 *               accumulation runs.
 *   [Dsv4Gpu]   "Struct Dsv4Gpu" page, method decode_step_greedy: the argmax
 *               runs on the device and only the u32 token returns.
 *   [dflash.rs] "dflash.rs source" page, fn dflash2_walk_greedy: argmax scan
 *               ascending with a strict '>' from best = -inf, index 0, so the
 *               lowest index wins ties; fn bf16_to_f32: a bf16 is the top
 *               16 bits of an f32.
 *
 * Readings taken where the pages are silent:
 *   - e4m3 is OCP FP8 E4M3 (bias 7, no infinities, NaN only at 0x7F/0xFF).
 *   - e2m1 is OCP FP4 E2M1 (bias 1, values 0, .5, 1, 1.5, 2, 3, 4, 6, signed).
 *   - e8m0 code c is 2^(c-127); c = 0xFF is refused.
 *   - scale block (i, j) covers rows [128i, 128i+128) x cols [128j, 128j+128).
 *   - NVFP4: two codes per byte, element 2j in the low nibble; one e4m3 scale
 *     per 16 consecutive columns of a row; one f32 global scale per expert.
 *   - MXFP4 (OCP MX, the MTP block's routed experts per [dsv4_gpu]
 *     ExpertKind): the same e2m1 code layout; one e8m0 scale per 32
 *     consecutive columns of a row, a weight is e2m1 * 2^(s-127); scale 0xFF
 *     is the MX NaN and makes its block's weights NaN; no global scale.
 *   - activations x are used as f32 (never rounded to bf16).
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off fp8blk_oracle.c -lm -lpthread
 * (no -ffast-math: IEEE semantics, subnormals and NaN must survive).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Format decoders, written from the bit-field definitions.            */
/* ------------------------------------------------------------------ */

/* OCP FP8 E4M3: sign | 4-bit exponent (bias 7) | 3-bit mantissa.
 * E = 0 is subnormal: mant/8 * 2^-6.  E = 15 with mant = 7 is NaN; there is
 * no infinity. */
double oracle_e4m3_value(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, mant = code & 7u;
    double mag;
    if (e == 15u && mant == 7u) return NAN;
    if (e == 0u)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* OCP FP4 E2M1: sign | 2-bit exponent (bias 1) | 1-bit mantissa.
 * E = 0 is subnormal: mant * 0.5.  All 16 codes are finite. */
double oracle_e2m1_value(unsigned nibble) {
    unsigned s = (nibble >> 3) & 1u, e = (nibble >> 1) & 3u, mant = nibble & 1u;
    double mag;
    if (e == 0u)
        mag = 0.5 * (double)mant;
    else
        mag = ldexp(1.0 + 0.5 * (double)mant, (int)e - 1);
    return s ? -mag : mag;
}

/* e8m0: an unsigned biased exponent, value 2^(c-127).  0xFF is refused at
 * load ([dsv4_gpu] Fp8Dense).  Returns 0 on success, -1 on refusal. */
int oracle_e8m0_value(unsigned code, double *out) {
    if ((code & 0xFFu) == 0xFFu) return -1;
    *out = ldexp(1.0, (int)(code & 0xFFu) - 127);
    return 0;
}

void oracle_e4m3_table(double *t256) {
    for (unsigned c = 0; c < 256u; ++c) t256[c] = oracle_e4m3_value(c);
}

void oracle_e2m1_table(double *t16) {
    for (unsigned c = 0; c < 16u; ++c) t16[c] = oracle_e2m1_value(c);
}

/* bf16 value of a bit pattern: the pattern is the top half of an f32
 * ([dflash.rs] bf16_to_f32). */
double oracle_bf16_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), from the bf16 format:
 * 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits, subnormal
 * spacing 2^-133 below 2^-126.  *inexact is set to 1 when the rounded value
 * differs from v. */
uint16_t oracle_bf16_rne(double v, int *inexact) {
    uint16_t sign;
    double a, quantum, n, r;
    int e;
    *inexact = 0;
    if (isnan(v)) {
        *inexact = 1;
        return (uint16_t)0x7FC0u;
    }
    sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0u;
    a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
    if (e - 1 < -126)
        quantum = ldexp(1.0, -133);
    else
        quantum = ldexp(1.0, (e - 1) - 7);
    n = rint(a / quantum); /* default rounding mode: nearest, ties to even */
    r = n * quantum;
    if (r != a) *inexact = 1;
    if (r >= ldexp(1.0, 128)) {
        *inexact = 1;
        return (uint16_t)(sign | 0x7F80u);
    }
    if (r < ldexp(1.0, -126)) /* subnormal (n <= 127) or rounded up to 2^-126 */
        return (uint16_t)(sign | (uint16_t)n);
    (void)frexp(r, &e);
    {
        int ub = e - 1;                               /* r = 1.m * 2^ub */
        double m = ldexp(r, -ub) - 1.0;               /* in [0, 1) */
        unsigned mant = (unsigned)(m * 128.0);        /* exact: 7 bits */
        return (uint16_t)(sign | (uint16_t)((unsigned)(ub + 127) << 7) | (uint16_t)mant);
    }
}

/* ------------------------------------------------------------------ */
/* FP8-blk GEMV: y[i][r] = sum_c e4m3(W[r][c]) * S[r/128][c/128] * x[i][c]  */
/* ------------------------------------------------------------------ */

/* Every job struct starts with its row range, so the thread runner can set it. */
typedef struct {
    int64_t r0, r1;
} row_range;

typedef struct {
    row_range range;
    const uint8_t *codes;   /* [rows, cols] e4m3 */
    const double *sgrid;    /* decoded scale grid [ceil(rows/128), ceil(cols/128)] */
    const float *x;         /* [m, cols] */
    double *y;              /* [m, rows] */
    double *abs_sum;        /* [m, rows], may be NULL */
    const double *e4m3;     /* 256-entry table */
    int m;
    int64_t rows, cols, gcols;
} gemv_job;

static void *gemv_rows(void *arg) {
    const gemv_job *j = (const gemv_job *)arg;
    for (int64_t r = j->range.r0; r < j->range.r1; ++r) {
        const uint8_t *wrow = j->codes + r * j->cols;
        const double *srow = j->sgrid + (r / 128) * j->gcols;
        for (int i = 0; i < j->m; ++i) {
            const float *xi = j->x + (int64_t)i * j->cols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t c = 0; c < j->cols; ++c) {
                double w = j->e4m3[wrow[c]] * srow[c / 128];
                double t = w * (double)xi[c];
                acc += t;
                aacc += fabs(t);
            }
            j->y[(int64_t)i * j->rows + r] = acc;
            if (j->abs_sum) j->abs_sum[(int64_t)i * j->rows + r] = aacc;
        }
    }
    return NULL;
}

/* Runs row ranges on `nthreads` POSIX threads.  Every output is computed by
 * the same sequential loop whatever the thread count, so results do not
 * depend on it. */
static int run_rows(void *(*fn)(void *), void *jobs, size_t job_size, int64_t rows, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!th) return -2;
    for (int t = 0; t < nthreads; ++t) {
        char *job = (char *)jobs + (size_t)t * job_size;
        row_range *range = (row_range *)job;
        range->r0 = rows * t / nthreads;
        range->r1 = rows * (t + 1) / nthreads;
        if (nthreads == 1) {
            fn(job);
        } else if (pthread_create(&th[t], NULL, fn, job) != 0) {
            for (int k = 0; k < t; ++k) pthread_join(th[k], NULL);
            free(th);
            return -2;
        }
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    return 0;
}

/* Returns 0 on success, -1 if a scale code is 0xFF (refused), -2 on a
 * resource failure, -3 on bad sizes. */
int oracle_fp8blk_gemv(const uint8_t *codes, const uint8_t *scale_e8m0, const float *x,
                       double *y, double *abs_sum, int m, int64_t rows, int64_t cols,
                       int nthreads) {
    double e4m3[256];
    int64_t grows, gcols;
    double *sgrid;
    if (m < 1 || rows < 0 || cols < 0) return -3;
    if (rows == 0) return 0;
    grows = (rows + 127) / 128;
    gcols = (cols + 127) / 128;
    oracle_e4m3_table(e4m3);
    sgrid = (double *)malloc((size_t)(grows * gcols > 0 ? grows * gcols : 1) * sizeof(double));
    if (!sgrid) return -2;
    for (int64_t k = 0; k < grows * gcols; ++k) {
        if (oracle_e8m0_value(scale_e8m0[k], &sgrid[k]) != 0) {
            free(sgrid);
            return -1;
        }
    }
    {
        int nt = nthreads < 1 ? 1 : nthreads;
        gemv_job *jobs = (gemv_job *)calloc((size_t)nt, sizeof(gemv_job));
        int rc;
        if (!jobs) {
            free(sgrid);
            return -2;
        }
        for (int t = 0; t < nt; ++t) {
            jobs[t].codes = codes;
            jobs[t].sgrid = sgrid;
            jobs[t].x = x;
            jobs[t].y = y;
            jobs[t].abs_sum = abs_sum;
            jobs[t].e4m3 = e4m3;
            jobs[t].m = m;
            jobs[t].rows = rows;
            jobs[t].cols = cols;
            jobs[t].gcols = gcols;
        }
        rc = run_rows(gemv_rows, jobs, sizeof(gemv_job), rows, nt);
        free(jobs);
        free(sgrid);
        return rc;
    }
}

/* ------------------------------------------------------------------ */
/* Greedy argmax: ascending scan, strict '>', best starts at -inf with    */
/* index 0.  Lowest index wins ties; NaN never wins.                       */
/* ------------------------------------------------------------------ */
int64_t oracle_argmax(const double *v, int64_t n) {
    double best = -INFINITY;
    int64_t bi = 0;
    for (int64_t k = 0; k < n; ++k) {
        if (v[k] > best) {
            best = v[k];
            bi = k;
        }
    }
    return bi;
}

/* ------------------------------------------------------------------ */
/* NVFP4 expert dequant to bf16: B[r][c] = bf16(e2m1(q) * e4m3(s) * g)    */
/* ------------------------------------------------------------------ */
int oracle_nvfp4_dequant_bf16(const uint8_t *codes, const uint8_t *scales, double g,
                              int64_t rows, int64_t cols, uint16_t *out, int64_t *n_inexact) {
    double e2m1[16], e4m3[256];
    int64_t inexact = 0;
    if (rows < 0 || cols < 0 || (cols % 16) != 0) return -3;
    oracle_e2m1_table(e2m1);
    oracle_e4m3_table(e4m3);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * (cols / 2) + c / 2];
            unsigned nib = (c % 2 == 0) ? (byte & 15u) : (unsigned)(byte >> 4);
            double v = e2m1[nib] * e4m3[scales[r * (cols / 16) + c / 16]] * g;
            int inx;
            out[r * cols + c] = oracle_bf16_rne(v, &inx);
            inexact += inx;
        }
    }
    if (n_inexact) *n_inexact = inexact;
    return 0;
}

/* ------------------------------------------------------------------ */
/* bf16 GEMV: y[r] = sum_c bf16(B[r][c]) * x[c], in double.                */
/* ------------------------------------------------------------------ */
typedef struct {
    row_range range;
    const uint16_t *b;
    const float *x;
    double *y;
    double *abs_sum;
    int m;
    int64_t rows, cols;
} bf16_job;

static void *bf16_rows(void *arg) {
    const bf16_job *j = (const bf16_job *)arg;
    for (int64_t r = j->range.r0; r < j->range.r1; ++r) {
        for (int i = 0; i < j->m; ++i) {
            const float *xi = j->x + (int64_t)i * j->cols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t c = 0; c < j->cols; ++c) {
                double t = oracle_bf16_value(j->b[r * j->cols + c]) * (double)xi[c];
                acc += t;
                aacc += fabs(t);
            }
            j->y[(int64_t)i * j->rows + r] = acc;
            if (j->abs_sum) j->abs_sum[(int64_t)i * j->rows + r] = aacc;
        }
    }
    return NULL;
}

int oracle_bf16_gemv(const uint16_t *b, const float *x, double *y, double *abs_sum, int m,
                     int64_t rows, int64_t cols, int nthreads) {
    int nt = nthreads < 1 ? 1 : nthreads;
    bf16_job *jobs;
    int rc;
    if (m < 1 || rows < 0 || cols < 0) return -3;
    if (rows == 0) return 0;
    jobs = (bf16_job *)calloc((size_t)nt, sizeof(bf16_job));
    if (!jobs) return -2;
    for (int t = 0; t < nt; ++t) {
        jobs[t].b = b;
        jobs[t].x = x;
        jobs[t].y = y;
        jobs[t].abs_sum = abs_sum;
        jobs[t].m = m;
        jobs[t].rows = rows;
        jobs[t].cols = cols;
    }
    rc = run_rows(bf16_rows, jobs, sizeof(bf16_job), rows, nt);
    free(jobs);
    return rc;
}

/* Routed experts: for each active id k, dequantise expert ids[k] to bf16,
 * then y[k] = B_k x.  codes [E, rows, cols/2], scales [E, rows, cols/16],
 * gscale [E].  scratch_out, when non-NULL, receives the LAST active expert's
 * bf16 matrix.  Returns -4 on a bad or repeated id. */
int oracle_nvfp4_expert_dequant_gemv(const uint8_t *codes, const uint8_t *scales,
                                     const float *gscale, int n_experts, const int32_t *ids,
                                     int n_active, const float *x, double *y, double *abs_sum,
                                     uint16_t *scratch_out, int64_t rows, int64_t cols,
                                     int nthreads) {
    uint16_t *b;
    int rc = 0;
    if (rows < 0 || cols < 0 || (cols % 32) != 0) return -3;
    for (int k = 0; k < n_active; ++k) {
        if (ids[k] < 0 || ids[k] >= n_experts) return -4;
        for (int q = 0; q < k; ++q)
            if (ids[q] == ids[k]) return -4;
    }
    b = (uint16_t *)malloc((size_t)(rows * cols > 0 ? rows * cols : 1) * sizeof(uint16_t));
    if (!b) return -2;
    for (int k = 0; k < n_active && rc == 0; ++k) {
        int64_t e = ids[k];
        int64_t nin = 0;
        rc = oracle_nvfp4_dequant_bf16(codes + e * rows * (cols / 2), scales + e * rows * (cols / 16),
                                       (double)gscale[e], rows, cols, b, &nin);
        if (rc == 0)
            rc = oracle_bf16_gemv(b, x, y + (int64_t)k * rows, abs_sum ? abs_sum + (int64_t)k * rows : NULL,
                                  1, rows, cols, nthreads);
        if (rc == 0 && scratch_out && k == n_active - 1)
            memcpy(scratch_out, b, (size_t)(rows * cols) * sizeof(uint16_t));
    }
    free(b);
    return rc;
}

/* ------------------------------------------------------------------ */
/* MXFP4 routed experts: y[k][r] = sum_c e2m1(q[e][r][c]) * 2^(s[e][r][c/32]-127) * x[c],  */
/* e = ids[k] (repeats allowed), each term in double, summed sequentially.  */
/* ------------------------------------------------------------------ */

typedef struct {
    row_range range;
    const uint8_t *codes;   /* [rows, cols/2] of one expert */
    const uint8_t *scales;  /* [rows, cols/32] e8m0 of one expert */
    const float *x;         /* [cols] */
    double *y;              /* [rows] */
    double *abs_sum;        /* [rows], may be NULL */
    const double *e2m1;     /* 16-entry table */
    int64_t rows, cols;
} mx_job;

static void *mx_rows(void *arg) {
    const mx_job *j = (const mx_job *)arg;
    for (int64_t r = j->range.r0; r < j->range.r1; ++r) {
        const uint8_t *crow = j->codes + r * (j->cols / 2);
        const uint8_t *srow = j->scales + r * (j->cols / 32);
        double acc = 0.0, aacc = 0.0;
        for (int64_t c = 0; c < j->cols; ++c) {
            const unsigned byte = crow[c / 2];
            const unsigned nib = (c % 2 == 0) ? (byte & 15u) : (byte >> 4);
            const unsigned sc = srow[c / 32];
            const double scale = sc == 0xFFu ? NAN : ldexp(1.0, (int)sc - 127);
            const double t = j->e2m1[nib] * scale * (double)j->x[c];
            acc += t;
            aacc += fabs(t);
        }
        j->y[r] = acc;
        if (j->abs_sum) j->abs_sum[r] = aacc;
    }
    return NULL;
}

/* Returns 0 on success, -2 on a resource failure, -3 on bad sizes, -4 on an
 * expert id outside [0, n_experts). */
int oracle_mxfp4_expert_gemv(const uint8_t *codes, const uint8_t *scales, int n_experts,
                             const int32_t *ids, int n_active, const float *x, double *y,
                             double *abs_sum, int64_t rows, int64_t cols, int nthreads) {
    double e2m1[16];
    if (rows < 0 || cols < 0 || (cols % 32) != 0 || n_active < 0) return -3;
    for (int k = 0; k < n_active; ++k)
        if (ids[k] < 0 || ids[k] >= n_experts) return -4;
    oracle_e2m1_table(e2m1);
    if (nthreads < 1) nthreads = 1;
    mx_job *jobs = (mx_job *)calloc((size_t)nthreads, sizeof(mx_job));
    if (!jobs) return -2;
    int rc = 0;
    for (int k = 0; k < n_active && rc == 0; ++k) {
        const int64_t e = ids[k];
        for (int t = 0; t < nthreads; ++t) {
            jobs[t].codes = codes + e * rows * (cols / 2);
            jobs[t].scales = scales + e * rows * (cols / 32);
            jobs[t].x = x;
            jobs[t].y = y + (int64_t)k * rows;
            jobs[t].abs_sum = abs_sum ? abs_sum + (int64_t)k * rows : NULL;
            jobs[t].e2m1 = e2m1;
            jobs[t].rows = rows;
            jobs[t].cols = cols;
        }
        rc = run_rows(mx_rows, jobs, sizeof(mx_job), rows, nthreads);
    }
    free(jobs);
    return rc;
}
