/*
 * bsg_oracle.c -- plain, slow CPU oracle for the block-scaled GEMM + Amax.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry point and the CPU-baseline leg of the benchmark may load or
 * call this code.  The product path (the CUDA library) never does, and this
 * file shares no code, table or constant with it.
 *
 * What it computes ("GEMM + Amax (SM100)", section "Equations"):
 *
 *     Ahat[m,k,l] = dec(A[m,k,l]) * sf(SFA, m, floor(k / sf_vec_size), l)
 *     Bhat[n,k,l] = dec(B[n,k,l]) * sf(SFB, n, floor(k / sf_vec_size), l)
 *     C[m,n,l]    = sum_k Ahat[m,k,l] * Bhat[n,k,l]
 *     Amax        = max_{m,n,l} |C[m,n,l]|
 *
 * The result has a plain definition, so the oracle is that definition
 * written out: decode every code through a table built from the format's bit
 * fields, look every scale up at its atom-layout offset, multiply and add in
 * IEEE double, k ascending.  No blocking, no reordering.  The rounding of the
 * double sum into the output dtype (round-to-nearest-even) and the per-element
 * tolerance are separate, explicit steps.
 *
 * Layouts (same page, "Parameters" / "Input/Output tensors"):
 *   A  (M, K, L), k-major, strides (K, 1, M*K): byte (l*M + m)*Kb + kb,
 *      Kb = K bytes (K/2 for FP4); or m-major (FP8 only), strides
 *      (1, M, M*K): byte (l*K + k)*M + m
 *   B  (N, K, L), k-major or n-major, likewise.
 *   FP4 (E2M1) is packed two per byte ("Support surface", "Layouts and
 *   strides"); element 2i sits in the low nibble, 2i+1 in the high nibble
 *   (the float4_e2m1fn_x2 convention; the pages do not spell it out).
 *   SFA/SFB logical (32, 4, ceil(MN/128), 4, ceil(K/(4*sfv)), L), stored as
 *   the C-contiguous physical (L, ceil(MN/128), ceil(K/(4*sfv)), 32, 4, 4)
 *   ("Using JAX arrays": the logical view is the physical one permuted by
 *   (3,4,1,5,2,0)).  Row mn of a 128-row block is split mn = m0 + 32*m1.
 *
 * Parity status: every function here is pinned by tests (hand-worked
 * examples, closed forms, invariants, brute force, library decodes), except
 * that the split of a row index into (m0, m1) inside an atom follows the
 * column-major convention of the atom's shape, which the pages do not state
 * beyond the shape and the permutation.
 */
#define _GNU_SOURCE
#include <fenv.h>
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* dtype codes of this oracle (its own numbering) */
enum {
    BSGO_E4M3 = 0,
    BSGO_E5M2 = 1,
    BSGO_E2M1 = 2,
    BSGO_UE8M0 = 3,
    BSGO_F32 = 4,
    BSGO_F16 = 5,
    BSGO_BF16 = 6
};

/* ---------------------------------------------------------------- decoding */

/* E4M3 ("fn"): sign | 4-bit exponent, bias 7 | 3-bit mantissa.  No infinity;
 * only S.1111.111 is NaN.  Exponent field 0 is subnormal: mant/8 * 2^(1-7). */
static double dec_e4m3(unsigned b)
{
    unsigned s = (b >> 7) & 1u, e = (b >> 3) & 0xFu, m = b & 7u;
    double v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) v = ldexp((double)m / 8.0, 1 - 7);
    else v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* E5M2: sign | 5-bit exponent, bias 15 | 2-bit mantissa, IEEE-like:
 * exponent 31 is infinity (mantissa 0) or NaN; exponent 0 is subnormal. */
static double dec_e5m2(unsigned b)
{
    unsigned s = (b >> 7) & 1u, e = (b >> 2) & 0x1Fu, m = b & 3u;
    double v;
    if (e == 31u) v = (m == 0u) ? INFINITY : NAN;
    else if (e == 0u) v = ldexp((double)m / 4.0, 1 - 15);
    else v = ldexp(1.0 + (double)m / 4.0, (int)e - 15);
    return s ? -v : v;
}

/* E2M1 (4 bits): sign | 2-bit exponent, bias 1 | 1-bit mantissa; no
 * infinity or NaN.  Exponent 0 is subnormal: mant/2 * 2^(1-1). */
static double dec_e2m1(unsigned c)
{
    unsigned s = (c >> 3) & 1u, e = (c >> 1) & 3u, m = c & 1u;
    double v;
    if (e == 0u) v = ldexp((double)m / 2.0, 1 - 1);
    else v = ldexp(1.0 + (double)m / 2.0, (int)e - 1);
    return s ? -v : v;
}

/* UE8M0: an unsigned biased exponent, value 2^(e-127); 0xFF is NaN. */
static double dec_ue8m0(unsigned b)
{
    if (b == 0xFFu) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Fill out[] with the value of every code of the format.  Returns the
 * number of codes (256, or 16 for E2M1), or -1 for an unknown dtype. */
int bsgo_decode_table(int dtype, double *out)
{
    unsigned i;
    switch (dtype) {
    case BSGO_E4M3:
        for (i = 0; i < 256u; i++) out[i] = dec_e4m3(i);
        return 256;
    case BSGO_E5M2:
        for (i = 0; i < 256u; i++) out[i] = dec_e5m2(i);
        return 256;
    case BSGO_E2M1:
        for (i = 0; i < 16u; i++) out[i] = dec_e2m1(i);
        return 16;
    case BSGO_UE8M0:
        for (i = 0; i < 256u; i++) out[i] = dec_ue8m0(i);
        return 256;
    default:
        return -1;
    }
}

/* ------------------------------------------------------------ atom layout */

/* Byte offset of the scale for row (or column) mn, K-block kb, batch l, in
 * the physical (L, t_mn, t_k, 32, 4, 4) scale tensor.  With mn = 128*mt +
 * 32*m1 + m0 and kb = 4*kt + kin the logical index is (m0, m1, mt, kin, kt,
 * l), whose C-contiguous physical position is (l, mt, kt, m0, m1, kin). */
int64_t bsgo_sf_offset(int64_t mn, int64_t kb, int64_t l, int64_t t_mn, int64_t t_k)
{
    int64_t mt = mn / 128, r = mn % 128;
    int64_t m0 = r % 32, m1 = r / 32;
    int64_t kt = kb / 4, kin = kb % 4;
    return ((((l * t_mn + mt) * t_k + kt) * 32 + m0) * 4 + m1) * 4 + kin;
}

/* ------------------------------------------------------------- operands */

typedef struct {
    int64_t M, N, K, L;
    int a_mn, b_mn;               /* 1: the operand is m- (n-) major */
    int a_dtype, b_dtype, sf_dtype, sfv;
    const uint8_t *A, *B, *SFA, *SFB;
    double tab_a[256], tab_b[256], tab_sf[256];
} problem_t;

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* raw code of element (r, k) of batch l of an operand with `rows` rows,
 * stored k-major (mn == 0) or with the rows contiguous (mn == 1, FP8 only) */
static unsigned code_at(const uint8_t *X, int dtype, int mn, int64_t rows, int64_t K,
                        int64_t r, int64_t k, int64_t l)
{
    if (mn) return X[(l * K + k) * rows + r];
    if (dtype == BSGO_E2M1) {
        uint8_t byte = X[(l * rows + r) * (K / 2) + k / 2];
        return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xFu);
    }
    return X[(l * rows + r) * K + k];
}

/* Dequantized row r of batch l: out[k] = dec(X[r,k,l]) * sf(SF, r, k/sfv, l) */
static void dequant_row(const problem_t *p, const uint8_t *X, const uint8_t *SF,
                        const double *tab, int dtype, int mn, int64_t rows, int64_t r,
                        int64_t l, double *out)
{
    int64_t t_mn = ceil_div(rows, 128), t_k = ceil_div(p->K, 4 * (int64_t)p->sfv);
    int64_t k;
    for (k = 0; k < p->K; k++) {
        double scale = p->tab_sf[SF[bsgo_sf_offset(r, k / p->sfv, l, t_mn, t_k)]];
        out[k] = tab[code_at(X, dtype, mn, rows, p->K, r, k, l)] * scale;
    }
}

static int setup(problem_t *p, const int64_t *dims, int a_dtype, int b_dtype,
                 int sf_dtype, int sfv, const uint8_t *A, const uint8_t *B,
                 const uint8_t *SFA, const uint8_t *SFB)
{
    memset(p, 0, sizeof(*p));
    p->M = dims[0]; p->N = dims[1]; p->K = dims[2]; p->L = dims[3];
    p->a_mn = dims[4] != 0; p->b_mn = dims[5] != 0;
    p->a_dtype = a_dtype; p->b_dtype = b_dtype; p->sf_dtype = sf_dtype; p->sfv = sfv;
    p->A = A; p->B = B; p->SFA = SFA; p->SFB = SFB;
    if (p->M < 1 || p->N < 1 || p->K < 1 || p->L < 1 || sfv < 1) return -1;
    if ((a_dtype == BSGO_E2M1 || b_dtype == BSGO_E2M1) && (p->K % 2)) return -1;
    /* packed FP4 is k-major only ("Support surface and constraints") */
    if ((a_dtype == BSGO_E2M1 && p->a_mn) || (b_dtype == BSGO_E2M1 && p->b_mn)) return -1;
    if (bsgo_decode_table(a_dtype, p->tab_a) < 0) return -1;
    if (bsgo_decode_table(b_dtype, p->tab_b) < 0) return -1;
    /* the scales are UE8M0, or E4M3 read as a non-negative multiplier */
    if (sf_dtype != BSGO_UE8M0 && sf_dtype != BSGO_E4M3) return -1;
    if (bsgo_decode_table(sf_dtype, p->tab_sf) < 0) return -1;
    return 0;
}

/* Dequantize one whole operand into out[(l*rows + r)*K + k] (double). */
int bsgo_dequantize(const uint8_t *X, int dtype, const uint8_t *SF, int sf_dtype,
                    int sfv, int64_t rows, int64_t K, int64_t L, double *out)
{
    problem_t p;
    int64_t dims[6] = {rows, rows, K, L, 0, 0};
    int64_t l, r;
    if (setup(&p, dims, dtype, dtype, sf_dtype, sfv, X, X, SF, SF) != 0) return -1;
    for (l = 0; l < L; l++)
        for (r = 0; r < rows; r++)
            dequant_row(&p, X, SF, p.tab_a, dtype, 0, rows, r, l, out + (l * rows + r) * K);
    return 0;
}

/* ---------------------------------------------------------- thread pool */

int bsgo_num_threads(int requested)
{
    if (requested > 0) return requested;
#ifdef CPU_COUNT
    {
        cpu_set_t set;
        if (sched_getaffinity(0, sizeof(set), &set) == 0) {
            int c = CPU_COUNT(&set);
            if (c > 0) return c;
        }
    }
#endif
    {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        return c > 0 ? (int)c : 1;
    }
}

typedef struct {
    const problem_t *p;
    int64_t m_begin, m_end;       /* rows of A computed, every batch */
    const double *bhat;           /* dequantized B, (L, N, K) */
    double *C, *S;                /* (L, m_end-m_begin, N) */
    int64_t item_begin, item_end; /* work items: (l, m) pairs */
} rows_job_t;

static void *rows_worker(void *arg)
{
    rows_job_t *j = (rows_job_t *)arg;
    const problem_t *p = j->p;
    int64_t rows = j->m_end - j->m_begin;
    double *ahat = (double *)malloc(sizeof(double) * (size_t)p->K);
    int64_t it;
    if (!ahat) return (void *)1;
    for (it = j->item_begin; it < j->item_end; it++) {
        int64_t l = it / rows, m = j->m_begin + it % rows, n, k;
        dequant_row(p, p->A, p->SFA, p->tab_a, p->a_dtype, p->a_mn, p->M, m, l, ahat);
        for (n = 0; n < p->N; n++) {
            const double *bh = j->bhat + (l * p->N + n) * p->K;
            double acc = 0.0, sabs = 0.0;
            for (k = 0; k < p->K; k++) {
                double prod = ahat[k] * bh[k];
                acc += prod;
                sabs += fabs(prod);
            }
            j->C[(l * rows + (m - j->m_begin)) * p->N + n] = acc;
            if (j->S) j->S[(l * rows + (m - j->m_begin)) * p->N + n] = sabs;
        }
    }
    free(ahat);
    return NULL;
}

/*
 * C[l][m - m_begin][n] = sum_k Ahat[m,k,l] * Bhat[n,k,l]   for m_begin <= m < m_end
 * S[l][m - m_begin][n] = sum_k |Ahat[m,k,l] * Bhat[n,k,l]| (S may be NULL)
 * dims = {M, N, K, L, a_mn, b_mn} (a_mn / b_mn: 1 for an m- / n-major
 * operand, 0 for k-major).  Returns the number of threads used, or -1.
 */
int bsgo_gemm_rows(const int64_t *dims, int a_dtype, int b_dtype, int sf_dtype, int sfv,
                   const uint8_t *A, const uint8_t *B, const uint8_t *SFA,
                   const uint8_t *SFB, int64_t m_begin, int64_t m_end, double *C,
                   double *S, int nthreads)
{
    problem_t p;
    double *bhat;
    pthread_t *tid;
    rows_job_t *jobs;
    int64_t items, t, l, n;
    int nt, rc = 0;
    if (setup(&p, dims, a_dtype, b_dtype, sf_dtype, sfv, A, B, SFA, SFB) != 0) return -1;
    if (m_begin < 0 || m_end > p.M || m_begin >= m_end) return -1;
    bhat = (double *)malloc(sizeof(double) * (size_t)(p.L * p.N * p.K));
    if (!bhat) return -1;
    for (l = 0; l < p.L; l++)
        for (n = 0; n < p.N; n++)
            dequant_row(&p, p.B, p.SFB, p.tab_b, p.b_dtype, p.b_mn, p.N, n, l,
                        bhat + (l * p.N + n) * p.K);
    items = p.L * (m_end - m_begin);
    nt = bsgo_num_threads(nthreads);
    if (nt > items) nt = (int)items;
    tid = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    jobs = (rows_job_t *)calloc((size_t)nt, sizeof(rows_job_t));
    if (!tid || !jobs) { free(bhat); free(tid); free(jobs); return -1; }
    for (t = 0; t < nt; t++) {
        jobs[t].p = &p;
        jobs[t].m_begin = m_begin;
        jobs[t].m_end = m_end;
        jobs[t].bhat = bhat;
        jobs[t].C = C;
        jobs[t].S = S;
        jobs[t].item_begin = items * t / nt;
        jobs[t].item_end = items * (t + 1) / nt;
        if (pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) != 0) {
            /* run the rest inline */
            rows_worker(&jobs[t]);
            tid[t] = 0;
        }
    }
    for (t = 0; t < nt; t++) {
        void *ret = NULL;
        if (tid[t]) pthread_join(tid[t], &ret);
        if (ret) rc = -1;
    }
    free(bhat); free(tid); free(jobs);
    return rc == 0 ? nt : -1;
}

/* Whole problem: C and S are (L, M, N). */
int bsgo_gemm(const int64_t *dims, int a_dtype, int b_dtype, int sf_dtype, int sfv,
              const uint8_t *A, const uint8_t *B, const uint8_t *SFA, const uint8_t *SFB,
              double *C, double *S, int nthreads)
{
    return bsgo_gemm_rows(dims, a_dtype, b_dtype, sf_dtype, sfv, A, B, SFA, SFB, 0,
                          dims[0], C, S, nthreads);
}

typedef struct {
    const problem_t *p;
    const int64_t *mnl;
    double *C, *S;
    int64_t begin, end;
} sample_job_t;

static void *sample_worker(void *arg)
{
    sample_job_t *j = (sample_job_t *)arg;
    const problem_t *p = j->p;
    double *ah = (double *)malloc(sizeof(double) * (size_t)p->K * 2);
    double *bh;
    int64_t i, k;
    if (!ah) return (void *)1;
    bh = ah + p->K;
    for (i = j->begin; i < j->end; i++) {
        int64_t m = j->mnl[3 * i], n = j->mnl[3 * i + 1], l = j->mnl[3 * i + 2];
        double acc = 0.0, sabs = 0.0;
        dequant_row(p, p->A, p->SFA, p->tab_a, p->a_dtype, p->a_mn, p->M, m, l, ah);
        dequant_row(p, p->B, p->SFB, p->tab_b, p->b_dtype, p->b_mn, p->N, n, l, bh);
        for (k = 0; k < p->K; k++) {
            double prod = ah[k] * bh[k];
            acc += prod;
            sabs += fabs(prod);
        }
        j->C[i] = acc;
        if (j->S) j->S[i] = sabs;
    }
    free(ah);
    return NULL;
}

/* The same sums at `count` chosen points mnl[3*i .. 3*i+2] = (m, n, l). */
int bsgo_gemm_sample(const int64_t *dims, int a_dtype, int b_dtype, int sf_dtype, int sfv,
                     const uint8_t *A, const uint8_t *B, const uint8_t *SFA,
                     const uint8_t *SFB, const int64_t *mnl, int64_t count, double *C,
                     double *S, int nthreads)
{
    problem_t p;
    pthread_t *tid;
    sample_job_t *jobs;
    int64_t i, t;
    int nt, rc = 0;
    if (setup(&p, dims, a_dtype, b_dtype, sf_dtype, sfv, A, B, SFA, SFB) != 0) return -1;
    for (i = 0; i < count; i++) {
        if (mnl[3 * i] < 0 || mnl[3 * i] >= p.M || mnl[3 * i + 1] < 0 ||
            mnl[3 * i + 1] >= p.N || mnl[3 * i + 2] < 0 || mnl[3 * i + 2] >= p.L)
            return -1;
    }
    if (count == 0) return 0;
    nt = bsgo_num_threads(nthreads);
    if (nt > count) nt = (int)count;
    tid = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    jobs = (sample_job_t *)calloc((size_t)nt, sizeof(sample_job_t));
    if (!tid || !jobs) { free(tid); free(jobs); return -1; }
    for (t = 0; t < nt; t++) {
        jobs[t].p = &p;
        jobs[t].mnl = mnl;
        jobs[t].C = C;
        jobs[t].S = S;
        jobs[t].begin = count * t / nt;
        jobs[t].end = count * (t + 1) / nt;
        if (pthread_create(&tid[t], NULL, sample_worker, &jobs[t]) != 0) {
            sample_worker(&jobs[t]);
            tid[t] = 0;
        }
    }
    for (t = 0; t < nt; t++) {
        void *ret = NULL;
        if (tid[t]) pthread_join(tid[t], &ret);
        if (ret) rc = -1;
    }
    free(tid); free(jobs);
    return rc == 0 ? nt : -1;
}

/* ------------------------------------------------ output rounding, tolerance */

/* significand bits p (with the hidden bit), smallest normal exponent, largest
 * exponent, of the output formats */
/* precision p (with the hidden bit), smallest normal exponent, largest
 * exponent of each output format */
static int out_format(int c_dtype, int *p, int *emin, int *emax)
{
    switch (c_dtype) {
    case BSGO_F32: *p = 24; *emin = -126; *emax = 127; return 0;
    case BSGO_F16: *p = 11; *emin = -14; *emax = 15; return 0;
    case BSGO_BF16: *p = 8; *emin = -126; *emax = 127; return 0;
    case BSGO_E4M3: *p = 4; *emin = -6; *emax = 8; return 0;
    case BSGO_E5M2: *p = 3; *emin = -14; *emax = 15; return 0;
    case BSGO_E2M1: *p = 2; *emin = 0; *emax = 2; return 0;
    default: return -1;
    }
}

static int quant_format(int dtype, int *emax, unsigned *maxc, unsigned *sign, unsigned *nanc);
static unsigned nearest_code(double y, const double *tab, unsigned maxc, unsigned sign);

/* Low-precision C ("GEMM + Amax (SM100)", "Parameters": C may be
 * float8_e4m3fn, float8_e5m2 or packed float4_e2m1fn_x2, with no scale; the
 * page does not say how the fp32 result is converted).  The reading used:
 * round to nearest even, magnitudes past the largest finite value (and
 * infinities) saturate to it, NaN stays NaN in E4M3 / E5M2 and becomes +0 in
 * E2M1, which has no NaN. */
static double round_low_precision(double x, int c_dtype)
{
    int emax;
    unsigned maxc, sign, nanc;
    double tab[256];
    if (quant_format(c_dtype, &emax, &maxc, &sign, &nanc) != 0) return NAN;
    bsgo_decode_table(c_dtype, tab);
    if (isnan(x)) return c_dtype == BSGO_E2M1 ? 0.0 : NAN;
    if (isinf(x)) return copysign(tab[maxc], x);
    return tab[nearest_code(x, tab, maxc, sign)];
}

/* Round x to the nearest value of the output format, ties to even, overflow
 * to infinity (IEEE round-to-nearest-even, non-saturating). */
double bsgo_round(double x, int c_dtype)
{
    int p, emin, emax, E;
    double q, r;
    if (out_format(c_dtype, &p, &emin, &emax) != 0) return NAN;
    if (c_dtype == BSGO_E4M3 || c_dtype == BSGO_E5M2 || c_dtype == BSGO_E2M1)
        return round_low_precision(x, c_dtype);
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    frexp(fabs(x), &E);            /* |x| = f * 2^E, f in [0.5, 1) */
    E -= 1;                        /* |x| in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;        /* subnormal spacing below the normal range */
    q = ldexp(1.0, E - (p - 1));   /* spacing of the format at |x| */
    r = nearbyint(x / q) * q;      /* default rounding mode: ties to even */
    if (fabs(r) >= ldexp(1.0, emax + 1)) return copysign(INFINITY, x);
    return r;
}

/* Spacing of the output format at |x|: 2^(max(floor(log2|x|), emin) - (p-1));
 * a saturating format caps floor(log2|x|) at its largest exponent. */
double bsgo_ulp(double x, int c_dtype)
{
    int p, emin, emax, E;
    if (out_format(c_dtype, &p, &emin, &emax) != 0) return NAN;
    if (isnan(x) || isinf(x)) return INFINITY;
    if (x == 0.0) return ldexp(1.0, emin - (p - 1));
    frexp(fabs(x), &E);
    E -= 1;
    if (E < emin) E = emin;
    if (E > emax) E = emax;
    return ldexp(1.0, E - (p - 1));
}

int bsgo_round_array(const double *x, int64_t n, int c_dtype, double *out)
{
    int64_t i;
    int p, emin, emax;
    if (out_format(c_dtype, &p, &emin, &emax) != 0) return -1;
    if (fegetround() != FE_TONEAREST) return -1;
    for (i = 0; i < n; i++) out[i] = bsgo_round(x[i], c_dtype);
    return 0;
}

/* tau = rel * S + ulp_c(|Cref|), elementwise */
int bsgo_tolerance(const double *cref, const double *S, int64_t n, int c_dtype,
                   double rel, double *tau)
{
    int64_t i;
    int p, emin, emax;
    if (out_format(c_dtype, &p, &emin, &emax) != 0) return -1;
    for (i = 0; i < n; i++) tau[i] = rel * S[i] + bsgo_ulp(cref[i], c_dtype);
    return 0;
}

/* ----------------------------------------------------------- MX quantizer */
/*
 * The row upstream of the GEMM: real values X (rows, cols, L), cols
 * contiguous, become element codes of out_dtype plus one E8M0 scale per
 * sf_vec_size consecutive elements of a row, the scales written in the atom
 * layout of bsgo_sf_offset.  "GEMM + RoPE + MXFP8 Projection (SM100)",
 * section "Equations", names the operation (MXFP8 quantize: an E8M0 scale per
 * block of 32, E4M3 data); "GEMM + Amax (SM100)" gives the scale layout and
 * the E5M2 / packed E2M1 element formats the GEMM consumes.  The pages do not
 * spell out how a block's scale is chosen.  The reading used here (and by the
 * CUDA path) takes the block's largest magnitude to the top binade of the
 * element format:
 *   amax  = max |x| over the block
 *   e     = floor(log2 amax) - emax(out_dtype)      (E4M3 8, E5M2 15, E2M1 2)
 *   e     clamped to [-127, 127]; scale = 2^e; scale byte = e + 127
 *   code  = the value of out_dtype nearest to x / scale, ties to the even
 *           code; magnitudes past the largest finite value saturate to it;
 *           the sign of x is kept (a negative value rounding to zero is -0)
 * Special blocks: all zeros -> byte 127 (scale 1); any NaN or infinity ->
 * byte 0xFF (E8M0 NaN) and every code of the block the format's NaN code
 * (E4M3 0x7F, E5M2 0x7F; E2M1 has none, so its codes are 0).  Scale bytes of
 * padding positions (rows past `rows`, blocks past cols/sfv inside the last
 * atoms) are 127.
 * Parity: pinned by hand-worked blocks, by torch's float8 conversions of the
 * scaled values, by an exhaustive E2M1 grid, and by invariants (rounding
 * error bound, scale invariance, sign symmetry, exact round trips).
 */

static int quant_format(int dtype, int *emax, unsigned *maxc, unsigned *sign, unsigned *nanc)
{
    switch (dtype) {
    case BSGO_E4M3: *emax = 8;  *maxc = 0x7Eu; *sign = 0x80u; *nanc = 0x7Fu; return 0;
    case BSGO_E5M2: *emax = 15; *maxc = 0x7Bu; *sign = 0x80u; *nanc = 0x7Fu; return 0;
    case BSGO_E2M1: *emax = 2;  *maxc = 0x7u;  *sign = 0x8u;  *nanc = 0x0u;  return 0;
    default: return -1;
    }
}

/* Code of the out_dtype value nearest to y (finite), ties to the even code,
 * saturating; the non-negative codes 0..maxc decode in increasing order. */
static unsigned nearest_code(double y, const double *tab, unsigned maxc, unsigned sign)
{
    double a = fabs(y);
    unsigned lo = 0u, hi = maxc, c;
    if (a >= tab[maxc]) {
        c = maxc;
    } else {
        /* largest c with tab[c] <= a (tab[0] = 0 <= a) */
        while (lo < hi) {
            unsigned mid = (lo + hi + 1u) / 2u;
            if (tab[mid] <= a) lo = mid; else hi = mid - 1u;
        }
        c = lo;
        if (tab[c] != a) {
            double d_lo = a - tab[c], d_hi = tab[c + 1u] - a;
            if (d_hi < d_lo || (d_hi == d_lo && ((c + 1u) & 1u) == 0u)) c = c + 1u;
        }
    }
    return signbit(y) ? (c | sign) : c;
}

/* One element: the code of y under out_dtype (after scaling), or -1. */
int bsgo_quantize_value(double y, int out_dtype)
{
    int emax;
    unsigned maxc, sign, nanc;
    double tab[256];
    if (quant_format(out_dtype, &emax, &maxc, &sign, &nanc) != 0) return -1;
    bsgo_decode_table(out_dtype, tab);
    if (isnan(y) || isinf(y)) return (int)nanc;
    return (int)nearest_code(y, tab, maxc, sign);
}

/* X: rows*cols*L doubles, element (l, r, k) at (l*rows + r)*cols + k.
 * codes: (l*rows + r)*cols + k bytes for FP8; for E2M1 two per byte, element
 * k in the low nibble of byte k/2 when k is even.  sf: the whole padded atom
 * tensor, L * ceil(rows/128) * ceil(cols/sfv/4) * 512 bytes.  Returns 0, or -1
 * for an unsupported request (unknown dtype, sfv not 16/32, cols not a
 * multiple of sfv). */
int bsgo_quantize(const double *X, int64_t rows, int64_t cols, int64_t L, int out_dtype,
                  int sfv, uint8_t *codes, uint8_t *sf)
{
    int emax;
    unsigned maxc, sign, nanc;
    double tab[256];
    int64_t nblk, t_r, t_k, l, r, b, k;
    if (quant_format(out_dtype, &emax, &maxc, &sign, &nanc) != 0) return -1;
    if ((sfv != 16 && sfv != 32) || rows < 1 || cols < 1 || L < 1 || cols % sfv != 0) return -1;
    bsgo_decode_table(out_dtype, tab);
    nblk = cols / sfv;
    t_r = ceil_div(rows, 128);
    t_k = ceil_div(nblk, 4);
    memset(sf, 127, (size_t)(L * t_r * t_k * 512));
    for (l = 0; l < L; l++)
        for (r = 0; r < rows; r++)
            for (b = 0; b < nblk; b++) {
                const double *x = X + (l * rows + r) * cols + b * sfv;
                double amax = 0.0, scale = 1.0;
                int nonfinite = 0, e = 0, E;
                unsigned byte = 127u;
                for (k = 0; k < sfv; k++) {
                    if (isnan(x[k]) || isinf(x[k])) nonfinite = 1;
                    else if (fabs(x[k]) > amax) amax = fabs(x[k]);
                }
                if (nonfinite) {
                    byte = 0xFFu;
                } else if (amax > 0.0) {
                    frexp(amax, &E);            /* amax = f * 2^E, f in [0.5, 1) */
                    e = (E - 1) - emax;         /* floor(log2 amax) - emax */
                    if (e < -127) e = -127;
                    if (e > 127) e = 127;
                    byte = (unsigned)(e + 127);
                    scale = ldexp(1.0, e);
                }
                sf[bsgo_sf_offset(r, b, l, t_r, t_k)] = (uint8_t)byte;
                for (k = 0; k < sfv; k++) {
                    const int64_t idx = (l * rows + r) * cols + b * sfv + k;
                    unsigned c = nonfinite ? nanc : nearest_code(x[k] / scale, tab, maxc, sign);
                    if (out_dtype == BSGO_E2M1) {
                        uint8_t *p = codes + idx / 2;
                        if ((idx & 1) == 0) *p = (uint8_t)((*p & 0xF0u) | c);
                        else *p = (uint8_t)((*p & 0x0Fu) | (c << 4));
                    } else {
                        codes[idx] = (uint8_t)c;
                    }
                }
            }
    return 0;
}

/* ------------------------------------------------ MX quantizer, columnwise */
/*
 * The columnwise direction of the same quantizer ("GEMM + RoPE + MXFP8
 * Projection (SM100)", sections "Overview" and "Equations": the output is
 * quantized in both the rowwise (D-direction) and the columnwise
 * (S-direction) layouts; MXFP8_S has its blocks along the tokens, the
 * non-contiguous dimension).  X is (rows, cols, L), cols contiguous, as for
 * the rowwise form, but a block is sf_vec_size consecutive ROWS of one
 * column.  The codes keep X's layout (element (l, r, c) at
 * (l*rows + r)*cols + c), which is the GEMM's MN-major operand layout when
 * rows play K and cols play M (or N): strides (1, cols, cols*rows).  The
 * scale of column c, block b = r / sfv sits where the GEMM reads the scale
 * of row mn = c, K-block kb = b: bsgo_sf_offset(c, b, l, ceil(cols/128),
 * ceil(rows/sfv/4)).  The pages print the S-direction scales as a plain
 * (tokens/32, ..., HEAD_DIM) array; this library writes them in the atom
 * layout its GEMM consumes (the same bytes, rearranged).
 * Per block the rule is the rowwise one: amax, e = floor(log2 amax) - emax,
 * clamp, nearest code ties to even, saturate, specials as above.  FP8 codes
 * only (E4M3 / E5M2): the GEMM takes MN-major operands in FP8 alone.
 * Returns 0, or -1 for an unsupported request (not FP8, sfv not 32, rows
 * not a multiple of sfv).
 */
int bsgo_quantize_colwise(const double *X, int64_t rows, int64_t cols, int64_t L,
                          int out_dtype, int sfv, uint8_t *codes, uint8_t *sf)
{
    int emax;
    unsigned maxc, sign, nanc;
    double tab[256];
    int64_t nblk, t_c, t_k, l, c, b, r;
    if (out_dtype != BSGO_E4M3 && out_dtype != BSGO_E5M2) return -1;
    if (quant_format(out_dtype, &emax, &maxc, &sign, &nanc) != 0) return -1;
    if (sfv != 32 || rows < 1 || cols < 1 || L < 1 || rows % sfv != 0) return -1;
    bsgo_decode_table(out_dtype, tab);
    nblk = rows / sfv;
    t_c = ceil_div(cols, 128);
    t_k = ceil_div(nblk, 4);
    memset(sf, 127, (size_t)(L * t_c * t_k * 512));
    for (l = 0; l < L; l++)
        for (c = 0; c < cols; c++)
            for (b = 0; b < nblk; b++) {
                /* the block: rows b*sfv .. b*sfv + sfv - 1 of column c */
                const double *x0 = X + (l * rows + b * sfv) * cols + c;
                double amax = 0.0, scale = 1.0;
                int nonfinite = 0, e = 0, E;
                unsigned byte = 127u;
                for (r = 0; r < sfv; r++) {
                    const double v = x0[r * cols];
                    if (isnan(v) || isinf(v)) nonfinite = 1;
                    else if (fabs(v) > amax) amax = fabs(v);
                }
                if (nonfinite) {
                    byte = 0xFFu;
                } else if (amax > 0.0) {
                    frexp(amax, &E);            /* amax = f * 2^E, f in [0.5, 1) */
                    e = (E - 1) - emax;         /* floor(log2 amax) - emax */
                    if (e < -127) e = -127;
                    if (e > 127) e = 127;
                    byte = (unsigned)(e + 127);
                    scale = ldexp(1.0, e);
                }
                sf[bsgo_sf_offset(c, b, l, t_c, t_k)] = (uint8_t)byte;
                for (r = 0; r < sfv; r++) {
                    const double v = x0[r * cols];
                    codes[(l * rows + b * sfv + r) * cols + c] =
                        (uint8_t)(nonfinite ? nanc : nearest_code(v / scale, tab, maxc, sign));
                }
            }
    return 0;
}
