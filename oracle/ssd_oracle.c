/*
 * ssd_oracle.c -- CPU oracle for the Mamba-2 SSD forward scan.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library.  The product path (the CUDA library and its Python
 * binding) never links, loads or calls it, and this file includes nothing from the product.
 *
 * What it computes: the selective state-space recurrence, written out in float64 exactly as
 * the pages define it, one (batch, head) problem at a time, token by token.
 *
 *   Abar_t = exp(dt_t * A)                    (discretised transition, scalar A per head)
 *   Bbar_t = dt_t * B_t                       (discretised input matrix)
 *   h_t    = Abar_t * h_{t-1} + Bbar_t x_t^T  (h is a P x N matrix per head)
 *   y_t    = C_t^T h_t + D * x_t              (read after the token-t update)
 *
 * Sources:
 *   - youngju.dev "Mamba / selective SSM" article, section "LTIからSelectionへの切り替え":
 *     the four displayed equations for Abar_t, Bbar_t, h_t, y_t.
 *   - same article, the SelectiveSSM code listing: the skip term y += D * x.
 *   - Qiita "Mamba-2 / SSD" article, section 4.2 (SSD block pseudocode): A = -exp(A_log) is one
 *     scalar per head in Mamba-2.
 *   - same article, section 4.1 table and "ngroups" config keys: B and C are shared by groups
 *     of heads.  Reading used here: head h uses group h / (H / G) (contiguous head blocks).
 *
 * Precision: every input arrives already upcast to float64 (the stored bf16 / fp32 values,
 * exactly), every operation is float64, exp() is libm's.
 *
 * There is no chunking, blocking or reordering: the loop over t is the recurrence itself.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One independent (batch, head) problem.
 *   x  [L][P], dt [L], B [L][N], C [L][N], h0 [P][N] (NULL = zeros)
 *   y  [L][P] (output), hT [P][N] (output, may be NULL), h scratch [P][N]. */
static void scan_one_problem(int64_t L, int64_t P, int64_t N,
                             const double* x, const double* dt, double A,
                             const double* B, const double* C, double D,
                             const double* h0, double* y, double* hT, double* h)
{
    if (h0) memcpy(h, h0, (size_t)(P * N) * sizeof(double));
    else memset(h, 0, (size_t)(P * N) * sizeof(double));

    for (int64_t t = 0; t < L; ++t) {
        const double abar = exp(dt[t] * A);     /* Abar_t = exp(dt_t A) */
        const double* xt = x + t * P;
        const double* Bt = B + t * N;
        const double* Ct = C + t * N;
        double* yt = y + t * P;
        for (int64_t p = 0; p < P; ++p) {
            const double bx = dt[t] * xt[p];    /* Bbar_t x_t = dt_t B_t x_t */
            double* hp = h + p * N;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                hp[n] = abar * hp[n] + bx * Bt[n];   /* h_t = Abar_t h_{t-1} + Bbar_t x_t */
                acc += Ct[n] * hp[n];                /* y_t = C_t^T h_t (after the update) */
            }
            yt[p] = acc + D * xt[p];
        }
    }
    if (hT) memcpy(hT, h, (size_t)(P * N) * sizeof(double));
}

/*
 * ssd_oracle_scan: run n_problems independent (batch, head) recurrences.
 *
 *   x  [n][L][P]   dt [n][L]   A [n]   B [n][L][N]   C [n][L][N]
 *   D  [n] or NULL (no skip term)      h0 [n][P][N] or NULL (zero initial state)
 *   y  [n][L][P] (written)             hT [n][P][N] or NULL (final state, written)
 *   n_threads: OpenMP threads to use (<= 0: the runtime default).
 *
 * Returns the number of threads the parallel loop ran with (>= 1), or -1 on a bad argument
 * or an allocation failure.
 */
int ssd_oracle_scan(int64_t n_problems, int64_t L, int64_t P, int64_t N,
                    const double* x, const double* dt, const double* A,
                    const double* B, const double* C, const double* D,
                    const double* h0, double* y, double* hT, int n_threads)
{
    if (n_problems < 0 || L < 0 || P <= 0 || N <= 0) return -1;
    if (!x || !dt || !A || !B || !C || !y) return -1;
    int used = 1;
    int failed = 0;
#ifdef _OPENMP
    const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
#endif
#pragma omp parallel num_threads(nt) reduction(max : used) reduction(| : failed)
    {
#ifdef _OPENMP
        used = omp_get_num_threads();
#endif
        double* h = (double*)malloc((size_t)(P * N) * sizeof(double));
        if (!h) failed = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_problems; ++i) {
            if (!h) continue;
            scan_one_problem(L, P, N, x + i * L * P, dt + i * L, A[i],
                             B + i * L * N, C + i * L * N, D ? D[i] : 0.0,
                             h0 ? h0 + i * P * N : NULL, y + i * L * P,
                             hT ? hT + i * P * N : NULL, h);
        }
        free(h);
    }
    return failed ? -1 : used;
}

/* ABI version of this oracle library (bumped when the signature above changes). */
int ssd_oracle_version(void) { return 1; }
