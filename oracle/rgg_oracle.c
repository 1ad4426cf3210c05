/*
 * rgg_oracle.c -- the fp64 CPU oracle for the ragged-M grouped GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, the smoke check in __graft_entry__ and the
 * cpu_baseline / reference legs of bench.py use it.  It shares no code, no
 * header and no constant with the CUDA library; it is plain C on purpose so a
 * reader can check every loop against the pages by eye.
 *
 * What it computes (sources, by page title and section):
 *
 *  - "Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog",
 *    "What I am measuring" and section 2 ("The Grouped Problem and the flat
 *    tile list"): after routing, the rows of X are grouped by expert, and
 *    expert e computes the independent product  Y_e = X_e . W_e  with
 *    X_e = rows [off[e], off[e+1]) of X  ([m_e, K]) and W_e = W[e] ([K, N]).
 *    K and N are fixed, m_e is known only at run time and may be zero.
 *  - "Grouped GEMM" (InferenceX glossary), "Technical definition": a set of
 *    independent matrix multiplications with different row counts.
 *
 * The method (bf16 operands, fp32 accumulation, bf16 result) reaches this
 * definition up to rounding, so the oracle is the definition written out:
 *
 *     Y[i, j] = sum_{k=0}^{K-1} double(X[i, k]) * double(W[e, k, j])
 *
 * summed in fp64 in increasing k, for every row i of every expert e, from the
 * same bf16-rounded inputs the GPU receives (bf16 -> double is exact).  The
 * result is NOT rounded to bf16.
 *
 * Readings of points the pages leave open (each listed in the design notes):
 *  - valid offsets: 0 <= off[0] <= off[1] <= ... <= off[E] <= M_tot; rows of Y
 *    outside [off[0], off[E]) belong to no expert and are left untouched.
 *  - the tile list follows the worklog's host enumeration (section 2,
 *    "Source -- k1/common.cuh . k1/harness.cu"): expert-major, then M tile,
 *    then N tile, with rows = min(BM, m_e - mt*BM).
 *  - row utilisation eta (worklog section 2.1, whose displayed formula did not
 *    survive extraction) is read as  sum_e m_e / (BM * sum_e ceil(m_e/BM)),
 *    which reproduces the section's printed 10.2% / 22.0% waste figures.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (fp-contract off so
 * no multiply-add is fused and the k-ordered fp64 sum is the same on every
 * host architecture).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_BAD_OFFSETS 4
#define ORACLE_ERR_BAD_ROW_INDEX 7

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
static double bf16_bits_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Offsets validity, as read above. */
int rgg_oracle_check_offsets(const int32_t* off, int E, int64_t M_tot) {
    if (off == NULL || E < 1 || M_tot < 0) return ORACLE_ERR_INVALID_ARG;
    if (off[0] < 0) return ORACLE_ERR_BAD_OFFSETS;
    for (int e = 0; e < E; ++e)
        if (off[e + 1] < off[e]) return ORACLE_ERR_BAD_OFFSETS;
    if ((int64_t)off[E] > M_tot) return ORACLE_ERR_BAD_OFFSETS;
    return ORACLE_OK;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int rgg_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full grouped product.  X: bf16 bits [M_tot, K] row-major; W: bf16 bits
 * [E, K, N] row-major; off: int32 [E+1]; Y: double [M_tot, N] row-major.
 * Only rows of some expert are written.  Returns 0, or an error code with Y
 * untouched.
 */
int rgg_oracle_grouped_gemm(const uint16_t* X, const uint16_t* W, const int32_t* off,
                            int E, int64_t M_tot, int K, int N, double* Y, int nthreads) {
    if (X == NULL || W == NULL || Y == NULL || K < 1 || N < 1) return ORACLE_ERR_INVALID_ARG;
    int rc = rgg_oracle_check_offsets(off, E, M_tot);
    if (rc != ORACLE_OK) return rc;
    set_threads(nthreads);
    for (int e = 0; e < E; ++e) {
        const int64_t row_begin = off[e], row_end = off[e + 1];
        const uint16_t* We = W + (int64_t)e * K * N;
        #pragma omp parallel
        {
            double* acc = (double*)malloc(sizeof(double) * (size_t)N);
            #pragma omp for schedule(dynamic, 1)
            for (int64_t i = row_begin; i < row_end; ++i) {
                for (int j = 0; j < N; ++j) acc[j] = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double x = bf16_bits_to_f64(X[i * K + k]);
                    const uint16_t* wrow = We + (int64_t)k * N;
                    for (int j = 0; j < N; ++j) acc[j] += x * bf16_bits_to_f64(wrow[j]);
                }
                for (int j = 0; j < N; ++j) Y[i * N + j] = acc[j];
            }
            free(acc);
        }
    }
    return ORACLE_OK;
}

/*
 * The same definition evaluated at chosen output positions (rows[p], cols[p])
 * only, for full-size inputs the full product would take too long on.  The
 * expert of a row is found by a linear scan of the offsets.  A position whose
 * row belongs to no expert gets NaN (that output is left untouched by the
 * method).
 */
int rgg_oracle_grouped_gemm_points(const uint16_t* X, const uint16_t* W, const int32_t* off,
                                   int E, int64_t M_tot, int K, int N,
                                   const int64_t* rows, const int32_t* cols, int64_t npts,
                                   double* out, int nthreads) {
    if (X == NULL || W == NULL || rows == NULL || cols == NULL || out == NULL || K < 1 || N < 1)
        return ORACLE_ERR_INVALID_ARG;
    int rc = rgg_oracle_check_offsets(off, E, M_tot);
    if (rc != ORACLE_OK) return rc;
    for (int64_t p = 0; p < npts; ++p)
        if (rows[p] < 0 || rows[p] >= M_tot || cols[p] < 0 || cols[p] >= N) return ORACLE_ERR_INVALID_ARG;
    set_threads(nthreads);
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npts; ++p) {
        const int64_t i = rows[p];
        const int j = cols[p];
        int e = -1;
        for (int q = 0; q < E; ++q)
            if (i >= off[q] && i < off[q + 1]) { e = q; break; }
        if (e < 0) {
            uint64_t nan_bits = 0x7ff8000000000000ULL;
            memcpy(&out[p], &nan_bits, sizeof(double));
            continue;
        }
        const uint16_t* We = W + (int64_t)e * K * N;
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += bf16_bits_to_f64(X[i * K + k]) * bf16_bits_to_f64(We[(int64_t)k * N + j]);
        out[p] = acc;
    }
    return ORACLE_OK;
}

/*
 * The fused gate-up projection of an expert FFN with its activation: the
 * worklog ("What I am measuring"; section 7 "Scope of these results") leaves
 * out "the activation" that follows the grouped GEMM, and the Pearl article
 * ("What the 15% measures") benchmarks the gate and up projections of
 * GLM 5.3, DeepSeek V4 Pro and Kimi K3, models whose experts gate with SiLU
 * (SwiGLU).  Reading: W13 is bf16 [E, K, 2N] whose columns [0, N) are the
 * gate projection and [N, 2N) the up projection, and for every row i of
 * expert e and column j < N
 *
 *     g = sum_k x[i,k] w13[e,k,j],  u = sum_k x[i,k] w13[e,k,N+j]   (fp64, k increasing)
 *     H[i, j] = silu(g) * u,        silu(z) = z / (1 + exp(-z)).
 *
 * H is double [M_tot, N]; rows of no expert are untouched.
 */
static double silu_f64(double z) { return z / (1.0 + exp(-z)); }

double rgg_oracle_silu(double z) { return silu_f64(z); }

int rgg_oracle_grouped_swiglu(const uint16_t* X, const uint16_t* W13, const int32_t* off, int E, int64_t M_tot,
                              int K, int N, double* H, int nthreads) {
    if (X == NULL || W13 == NULL || H == NULL || K < 1 || N < 1) return ORACLE_ERR_INVALID_ARG;
    int rc = rgg_oracle_check_offsets(off, E, M_tot);
    if (rc != ORACLE_OK) return rc;
    set_threads(nthreads);
    const int64_t N2 = 2 * (int64_t)N;
    for (int e = 0; e < E; ++e) {
        const int64_t row_begin = off[e], row_end = off[e + 1];
        const uint16_t* We = W13 + (int64_t)e * K * N2;
        #pragma omp parallel
        {
            double* acc = (double*)malloc(sizeof(double) * (size_t)N2);
            #pragma omp for schedule(dynamic, 1)
            for (int64_t i = row_begin; i < row_end; ++i) {
                for (int64_t j = 0; j < N2; ++j) acc[j] = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double x = bf16_bits_to_f64(X[i * K + k]);
                    const uint16_t* wrow = We + (int64_t)k * N2;
                    for (int64_t j = 0; j < N2; ++j) acc[j] += x * bf16_bits_to_f64(wrow[j]);
                }
                for (int j = 0; j < N; ++j) H[i * N + j] = silu_f64(acc[j]) * acc[N + j];
            }
            free(acc);
        }
    }
    return ORACLE_OK;
}

/*
 * FP8 grouped GEMM.  The Pearl article ("What the 15% measures") says the
 * optimized kernel will be released with Pearl's FP8 scheme but does not
 * describe it.  Reading taken (the plainest one that keeps the K loop free of
 * scales): X and W hold FP8 E4M3 codes, X with one fp32 scale per row and W
 * with one fp32 scale per (expert, output column), so that
 *
 *     Y[i, j] = sx[i] * sw[e, j] * sum_k x8[i, k] * w8[e, k, j]      (fp64, k increasing)
 *
 * for every row i of expert e.  E4M3 (sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 = NaN): a code with exponent
 * field 0 is the subnormal m/8 * 2^-6, otherwise (1 + m/8) * 2^(e-7); decoding
 * to double is exact.
 */
static double e4m3_to_f64(uint8_t b) {
    const int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    if (e == 0xF && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

double rgg_oracle_e4m3_to_f64(uint8_t code) { return e4m3_to_f64(code); }

int rgg_oracle_grouped_gemm_fp8(const uint8_t* X8, const uint8_t* W8, const float* sx, const float* sw,
                                const int32_t* off, int E, int64_t M_tot, int K, int N, double* Y, int nthreads) {
    if (X8 == NULL || W8 == NULL || sx == NULL || sw == NULL || Y == NULL || K < 1 || N < 1)
        return ORACLE_ERR_INVALID_ARG;
    int rc = rgg_oracle_check_offsets(off, E, M_tot);
    if (rc != ORACLE_OK) return rc;
    set_threads(nthreads);
    for (int e = 0; e < E; ++e) {
        const int64_t row_begin = off[e], row_end = off[e + 1];
        const uint8_t* We = W8 + (int64_t)e * K * N;
        const float* swe = sw + (int64_t)e * N;
        #pragma omp parallel
        {
            double* acc = (double*)malloc(sizeof(double) * (size_t)N);
            #pragma omp for schedule(dynamic, 1)
            for (int64_t i = row_begin; i < row_end; ++i) {
                for (int j = 0; j < N; ++j) acc[j] = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double x = e4m3_to_f64(X8[i * K + k]);
                    const uint8_t* wrow = We + (int64_t)k * N;
                    for (int j = 0; j < N; ++j) acc[j] += x * e4m3_to_f64(wrow[j]);
                }
                for (int j = 0; j < N; ++j) Y[i * N + j] = (double)sx[i] * (double)swe[j] * acc[j];
            }
            free(acc);
        }
    }
    return ORACLE_OK;
}

/*
 * Token gather ahead of the grouped product.  The worklog starts after
 * routing, with the rows already grouped by expert ("What I am measuring"),
 * and names the permutation of rows and the scatter/gather of tokens among the
 * MoE work its kernel leaves out ("Scope of these results"); the InferenceX
 * glossary entry "Grouped GEMM" ("Engineering details") describes that token
 * permutation, which turns each expert's ragged group of tokens into operand
 * rows.  Reading: routed row i of the grouped operand is token row_index[i] of
 * an ungrouped token matrix X_tok [T, K],
 *
 *     Xg[i, k] = X_tok[row_index[i], k]        for begin <= i < end,
 *
 * and the gathered grouped product is the grouped product of Xg.  Only the
 * rows [begin, end) are gathered (the rows some expert owns); every index read
 * must lie in [0, T), otherwise nothing is written and the call fails.  Rows
 * of Xg outside [begin, end) are left as they were.
 */
int rgg_oracle_gather_rows(const uint16_t* Xtok, int64_t T, int K, const int32_t* row_index, int64_t begin,
                           int64_t end, uint16_t* Xg) {
    if (Xtok == NULL || row_index == NULL || Xg == NULL || T < 1 || K < 1 || begin < 0 || end < begin)
        return ORACLE_ERR_INVALID_ARG;
    for (int64_t i = begin; i < end; ++i)
        if (row_index[i] < 0 || (int64_t)row_index[i] >= T) return ORACLE_ERR_BAD_ROW_INDEX;
    for (int64_t i = begin; i < end; ++i) {
        const int64_t r = row_index[i];
        for (int k = 0; k < K; ++k) Xg[i * K + k] = Xtok[r * K + k];
    }
    return ORACLE_OK;
}

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * The worklog's flat tile list, section 2: for each expert e, for each M tile
 * mt < ceil(m_e/BM), for each N tile nt < ceil(N/BN), one descriptor
 * {expert, row0 = off[e] + mt*BM, rows = min(BM, m_e - mt*BM), col0 = nt*BN}.
 * Writes the first `cap` descriptors (4 int32 each) to desc (may be NULL when
 * cap is 0) and returns the total count, or -1 on bad arguments / offsets.
 */
int64_t rgg_oracle_tile_list(const int32_t* off, int E, int N, int BM, int BN,
                             int32_t* desc, int64_t cap) {
    if (off == NULL || E < 1 || N < 1 || BM < 1 || BN < 1 || cap < 0) return -1;
    if (cap > 0 && desc == NULL) return -1;
    if (off[0] < 0) return -1;
    for (int e = 0; e < E; ++e)
        if (off[e + 1] < off[e]) return -1;
    int64_t count = 0;
    const int64_t n_tiles = ceil_div64(N, BN);
    for (int e = 0; e < E; ++e) {
        const int64_t m_e = (int64_t)off[e + 1] - off[e];
        const int64_t m_tiles = ceil_div64(m_e, BM);
        for (int64_t mt = 0; mt < m_tiles; ++mt) {
            for (int64_t nt = 0; nt < n_tiles; ++nt) {
                if (count < cap) {
                    const int64_t left = m_e - mt * BM;
                    desc[4 * count + 0] = e;
                    desc[4 * count + 1] = (int32_t)(off[e] + mt * BM);
                    desc[4 * count + 2] = (int32_t)(left < BM ? left : BM);
                    desc[4 * count + 3] = (int32_t)(nt * BN);
                }
                ++count;
            }
        }
    }
    return count;
}

/*
 * Row utilisation eta, worklog section 2.1: the fraction of scheduled tile
 * rows that hold routed rows, sum_e m_e / (BM * sum_e ceil(m_e/BM)).  Returns
 * 1.0 when nothing is scheduled (no padding is introduced), -1.0 on bad input.
 */
double rgg_oracle_row_utilisation(const int32_t* off, int E, int BM) {
    if (off == NULL || E < 1 || BM < 1) return -1.0;
    int64_t used = 0, scheduled_tiles = 0;
    for (int e = 0; e < E; ++e) {
        const int64_t m_e = (int64_t)off[e + 1] - off[e];
        if (m_e < 0) return -1.0;
        used += m_e;
        scheduled_tiles += ceil_div64(m_e, BM);
    }
    if (scheduled_tiles == 0) return 1.0;
    return (double)used / ((double)BM * (double)scheduled_tiles);
}
