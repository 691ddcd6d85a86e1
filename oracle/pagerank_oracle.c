/*
 * PageRank power-iteration oracle: plain, slow, single-threaded, fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the test suite, the package's smoke check and the CPU
 * baseline leg of the benchmark do. It shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it computes (from "Day 40 - PageRank on a real graph in CUDA",
 * section "One iteration, three shapes of work", the update formula):
 *
 *   x'[v] = (1 - d)/n + d * ( sum over u with an edge u->v of x[u]/outdeg[u]
 *                             + D/n ),
 *   D     = sum of x[u] over dangling u (outdeg[u] == 0),
 *
 * starting from x0[v] = 1/n (Meerkat, section on PageRank, Algorithm 5: the
 * static case initialises every entry to 1/vertex_n) and stopping after the
 * first update whose L1 distance sum_v |x'[v] - x[v]| is below tol (same
 * section of Meerkat: delta is the L1 norm of successive vectors; Day 40,
 * "Keep the dangling mass on the device": the residual is what the host tests).
 *
 * The transpose is the counting sort the Day 40 page describes in "One
 * iteration, three shapes of work": a histogram of in-degrees, an exclusive
 * prefix sum, and a scatter that visits sources in increasing order, so each
 * in-row lists its sources in ascending order (multiplicity kept).
 *
 * Readings taken where the pages leave a step open:
 *  - an edge listed k times counts k times (in the sum and in outdeg);
 *  - the contribution is divided per edge, as the formula is written, not
 *    precomputed once per vertex;
 *  - tol <= 0 means "run exactly max_iter updates" (the fixed-iteration mode
 *    the Day 40 page times and uses for its correctness cases);
 *  - the iteration count is the number of updates performed, including the
 *    one that met the tolerance;
 *  - no renormalisation of x is ever done.
 *
 * Parity pins (tests that tie this file to the pages and to mathematics
 * rather than to itself) live in the test suite: the sum-to-1 invariant after
 * every update, the 1 - d*D total when the dangling term is dropped, the
 * broken fixed point and its proportionality, closed forms on cycles,
 * circulants, stars, chains and a single node, a dense brute-force power
 * method and linear solve on graphs with n <= 64, and an independent
 * lexicographic sort for the transpose.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_NOT_CONVERGED 1
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_GRAPH (-2)
#define ORACLE_ERR_OOM (-4)

/* Checks that (row_ptr, col_idx) is a well-formed out-edge CSR over n vertices. */
int oracle_check_csr(int64_t n, int64_t m, const int64_t *row_ptr,
                     const int32_t *col_idx)
{
    if (n < 1 || m < 0 || m > INT32_MAX || row_ptr == NULL)
        return ORACLE_ERR_ARG;
    if (m > 0 && col_idx == NULL)
        return ORACLE_ERR_ARG;
    if (row_ptr[0] != 0 || row_ptr[n] != m)
        return ORACLE_ERR_GRAPH;
    for (int64_t u = 0; u < n; ++u)
        if (row_ptr[u + 1] < row_ptr[u])
            return ORACLE_ERR_GRAPH;
    for (int64_t j = 0; j < m; ++j)
        if (col_idx[j] < 0 || (int64_t)col_idx[j] >= n)
            return ORACLE_ERR_GRAPH;
    return ORACLE_OK;
}

/*
 * Out-edge CSR -> in-edge CSR by counting sort (Day 40, "One iteration, three
 * shapes of work": histogram, prefix sum, scatter).
 * in_ptr has n+1 entries, in_col has m entries; both are caller-owned.
 */
int oracle_transpose(int64_t n, int64_t m, const int64_t *row_ptr,
                     const int32_t *col_idx, int64_t *in_ptr, int32_t *in_col)
{
    int rc = oracle_check_csr(n, m, row_ptr, col_idx);
    if (rc != ORACLE_OK)
        return rc;
    if (in_ptr == NULL || (m > 0 && in_col == NULL))
        return ORACLE_ERR_ARG;

    int64_t *count = (int64_t *)calloc((size_t)n, sizeof(int64_t));
    int64_t *cursor = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    if (count == NULL || cursor == NULL) {
        free(count);
        free(cursor);
        return ORACLE_ERR_OOM;
    }

    /* 1. histogram: number of edges that point at each vertex */
    for (int64_t j = 0; j < m; ++j)
        count[col_idx[j]] += 1;

    /* 2. exclusive prefix sum: where each in-row starts */
    in_ptr[0] = 0;
    for (int64_t v = 0; v < n; ++v)
        in_ptr[v + 1] = in_ptr[v] + count[v];

    /* 3. scatter, sources visited in increasing order */
    for (int64_t v = 0; v < n; ++v)
        cursor[v] = in_ptr[v];
    for (int64_t u = 0; u < n; ++u) {
        for (int64_t j = row_ptr[u]; j < row_ptr[u + 1]; ++j) {
            int32_t v = col_idx[j];
            in_col[cursor[v]] = (int32_t)u;
            cursor[v] += 1;
        }
    }

    free(count);
    free(cursor);
    return ORACLE_OK;
}

/*
 * The power iteration. Arguments:
 *   d, tol, max_iter  damping factor in [0, 1]; L1 tolerance (<= 0: run
 *                     exactly max_iter updates); cap on updates (>= 1)
 *   drop_dangling     0 for the method; 1 replaces D by 0 in the update (the
 *                     broken variant of the Day 40 exercise, used only by tests)
 *   x_init            NULL for the uniform 1/n start, else n start values
 *   x_out             n doubles, the last iterate
 *   iters_out, l1_out number of updates performed; L1 distance of the last one
 *   sum_log, dmass_log, l1_log
 *                     optional (NULL or max_iter doubles): after update k
 *                     (0-based) they hold sum_v x_{k+1}[v], the dangling mass
 *                     D of the vector that update k read (always the true
 *                     mass, even with drop_dangling), and that update's L1.
 * Returns ORACLE_OK, ORACLE_NOT_CONVERGED (tol > 0 and max_iter reached;
 * outputs valid) or a negative error code.
 */
int oracle_pagerank(int64_t n, int64_t m, const int64_t *row_ptr,
                    const int32_t *col_idx, double d, double tol,
                    int32_t max_iter, int32_t drop_dangling,
                    const double *x_init, double *x_out, int32_t *iters_out,
                    double *l1_out, double *sum_log, double *dmass_log,
                    double *l1_log)
{
    if (!(d >= 0.0 && d <= 1.0) || max_iter < 1 || isnan(tol) || x_out == NULL)
        return ORACLE_ERR_ARG;
    int rc = oracle_check_csr(n, m, row_ptr, col_idx);
    if (rc != ORACLE_OK)
        return rc;

    int64_t *in_ptr = (int64_t *)malloc((size_t)(n + 1) * sizeof(int64_t));
    int32_t *in_col = (int32_t *)malloc((size_t)(m > 0 ? m : 1) * sizeof(int32_t));
    int64_t *outdeg = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    double *x = (double *)malloc((size_t)n * sizeof(double));
    double *x_next = (double *)malloc((size_t)n * sizeof(double));
    if (!in_ptr || !in_col || !outdeg || !x || !x_next) {
        free(in_ptr); free(in_col); free(outdeg); free(x); free(x_next);
        return ORACLE_ERR_OOM;
    }
    rc = oracle_transpose(n, m, row_ptr, col_idx, in_ptr, in_col);
    if (rc != ORACLE_OK) {
        free(in_ptr); free(in_col); free(outdeg); free(x); free(x_next);
        return rc;
    }

    /* out-degrees; a vertex with none is dangling */
    for (int64_t u = 0; u < n; ++u)
        outdeg[u] = row_ptr[u + 1] - row_ptr[u];

    const double nd = (double)n;
    for (int64_t v = 0; v < n; ++v)
        x[v] = (x_init != NULL) ? x_init[v] : 1.0 / nd;

    int32_t it = 0;
    double l1 = 0.0;
    int converged = 0;
    while (it < max_iter) {
        /* dangling mass of the current vector */
        double D = 0.0;
        for (int64_t u = 0; u < n; ++u)
            if (outdeg[u] == 0)
                D += x[u];
        if (dmass_log != NULL)
            dmass_log[it] = D;
        if (drop_dangling)
            D = 0.0;

        /* the update, one vertex at a time, pulling over in-edges */
        for (int64_t v = 0; v < n; ++v) {
            double s = 0.0;
            for (int64_t j = in_ptr[v]; j < in_ptr[v + 1]; ++j) {
                int32_t u = in_col[j];
                s += x[u] / (double)outdeg[u];
            }
            x_next[v] = (1.0 - d) / nd + d * (s + D / nd);
        }

        /* L1 distance between successive vectors, and the total */
        l1 = 0.0;
        double total = 0.0;
        for (int64_t v = 0; v < n; ++v) {
            l1 += fabs(x_next[v] - x[v]);
            total += x_next[v];
        }
        if (sum_log != NULL)
            sum_log[it] = total;
        if (l1_log != NULL)
            l1_log[it] = l1;

        double *t = x;
        x = x_next;
        x_next = t;
        it += 1;
        if (tol > 0.0 && l1 < tol) {
            converged = 1;
            break;
        }
    }

    memcpy(x_out, x, (size_t)n * sizeof(double));
    if (iters_out != NULL)
        *iters_out = it;
    if (l1_out != NULL)
        *l1_out = l1;

    free(in_ptr); free(in_col); free(outdeg); free(x); free(x_next);
    if (tol > 0.0 && !converged)
        return ORACLE_NOT_CONVERGED;
    return ORACLE_OK;
}
