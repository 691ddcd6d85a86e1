/* Multi-core CPU PageRank: the power iteration as a pull over the in-edge
 * CSR, parallelised with OpenMP over all host cores.
 *
 * A measured baseline that bench.py times beside the GPU path, in the way
 * "A Reproducible Empirical Study of GPU Graph-Analytics Strategies on
 * Irregular Security Graphs" reports its GPU numbers against the full
 * multi-core CPU (its T1 OpenMP tier). It is neither
 * the oracle (which
 * stays single-threaded and plain) nor part of the product: the CUDA library
 * never links or calls it, and it shares no code with either.
 *
 * What it computes is the update of "Day 40 - PageRank on a real graph in
 * CUDA" (section "One iteration, three shapes of work", the update formula):
 * x'[v] = (1 - d)/n + d * (sum over in-edges
 * u->v of x[u]/outdeg[u] + D/n), D the rank mass on dangling vertices,
 * x0 = 1/n, stopping after the first update whose L1 distance is below tol
 * (tol <= 0: exactly max_iter updates). All in fp64.
 *
 * The transpose is the counting sort of Day 40's section "One iteration,
 * three shapes of work" done in parallel: in-degrees by atomic increments, a
 * two-level prefix sum, a scatter through per-destination atomic cursors,
 * and then each in-row sorted by source. The scatter order is not
 * deterministic, but the sorted rows are the unique in-CSR (sources
 * ascending, multiplicity kept), so the result is bit-for-bit the
 * single-threaded counting sort's.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { PO_OK = 0, PO_NOT_CONVERGED = 1, PO_ERR_ARG = -1, PO_ERR_GRAPH = -2, PO_ERR_OOM = -4 };

static int cmp_i32(const void *a, const void *b)
{
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static void sort_row(int32_t *r, int64_t len)
{
    if (len > 32) {
        qsort(r, (size_t)len, sizeof(int32_t), cmp_i32);
        return;
    }
    for (int64_t i = 1; i < len; ++i) {   /* insertion sort for short rows */
        const int32_t v = r[i];
        int64_t j = i - 1;
        while (j >= 0 && r[j] > v) {
            r[j + 1] = r[j];
            --j;
        }
        r[j + 1] = v;
    }
}

/* Exclusive prefix sum of cnt[0..n) into out[0..n], in parallel: each thread
 * sums its block, the block totals are scanned, each thread writes its block. */
static void scan_excl(int64_t n, const int64_t *cnt, int64_t *out, int threads)
{
    int64_t *part = (int64_t *)calloc((size_t)threads + 1, sizeof(int64_t));
#pragma omp parallel num_threads(threads)
    {
        const int t = omp_get_thread_num(), nt = omp_get_num_threads();
        const int64_t lo = n * t / nt, hi = n * (t + 1) / nt;
        int64_t s = 0;
        for (int64_t i = lo; i < hi; ++i)
            s += cnt[i];
        part[t + 1] = s;
#pragma omp barrier
#pragma omp single
        for (int k = 1; k <= nt; ++k)
            part[k] += part[k - 1];
        s = part[t];
        for (int64_t i = lo; i < hi; ++i) {
            out[i] = s;
            s += cnt[i];
        }
        if (t == nt - 1)
            out[n] = s;
    }
    free(part);
}

/* In-edge CSR of an out-edge CSR. Returns PO_OK or PO_ERR_GRAPH (a col_idx
 * entry outside [0, n)); in_ptr has n + 1 entries, in_col m. */
int po_transpose(int64_t n, int64_t m, const int64_t *row_ptr, const int32_t *col_idx, int threads,
                 int64_t *in_ptr, int32_t *in_col)
{
    if (n < 1 || m < 0 || threads < 1)
        return PO_ERR_ARG;
    int64_t *cnt = (int64_t *)calloc((size_t)n, sizeof(int64_t));
    int64_t *cursor = (int64_t *)malloc((size_t)(n + 1) * sizeof(int64_t));
    if (!cnt || !cursor) {
        free(cnt);
        free(cursor);
        return PO_ERR_OOM;
    }
    int bad = 0;
#pragma omp parallel for num_threads(threads) schedule(static) reduction(| : bad)
    for (int64_t j = 0; j < m; ++j) {
        const int32_t v = col_idx[j];
        if (v < 0 || (int64_t)v >= n) {
            bad = 1;
            continue;
        }
#pragma omp atomic
        cnt[v] += 1;
    }
    if (bad) {
        free(cnt);
        free(cursor);
        return PO_ERR_GRAPH;
    }
    scan_excl(n, cnt, in_ptr, threads);
    memcpy(cursor, in_ptr, (size_t)(n + 1) * sizeof(int64_t));
#pragma omp parallel for num_threads(threads) schedule(dynamic, 4096)
    for (int64_t u = 0; u < n; ++u) {
        for (int64_t j = row_ptr[u]; j < row_ptr[u + 1]; ++j) {
            const int32_t v = col_idx[j];
            int64_t pos;
#pragma omp atomic capture
            pos = cursor[v]++;
            in_col[pos] = (int32_t)u;
        }
    }
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1024)
    for (int64_t v = 0; v < n; ++v)
        sort_row(in_col + in_ptr[v], in_ptr[v + 1] - in_ptr[v]);
    free(cnt);
    free(cursor);
    return PO_OK;
}

/* The power iteration. x_out gets the ranks (n doubles); times are wall
 * seconds of the transpose and of the update loop. */
int po_pagerank(int64_t n, int64_t m, const int64_t *row_ptr, const int32_t *col_idx, double d, double tol,
                int32_t max_iter, int threads, double *x_out, int32_t *iters_out, double *l1_out,
                double *t_transpose, double *t_loop)
{
    if (n < 1 || m < 0 || max_iter < 1 || threads < 1 || !(d >= 0.0 && d <= 1.0) || !x_out)
        return PO_ERR_ARG;
    int64_t *in_ptr = (int64_t *)malloc((size_t)(n + 1) * sizeof(int64_t));
    int32_t *in_col = (int32_t *)malloc((size_t)(m > 0 ? m : 1) * sizeof(int32_t));
    double *c = (double *)malloc((size_t)n * sizeof(double));
    double *xn = (double *)malloc((size_t)n * sizeof(double));
    int32_t *deg = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    int st = (in_ptr && in_col && c && xn && deg) ? PO_OK : PO_ERR_OOM;
    const double t0 = omp_get_wtime();
    if (st == PO_OK)
        st = po_transpose(n, m, row_ptr, col_idx, threads, in_ptr, in_col);
    const double t1 = omp_get_wtime();
    int32_t it = 0;
    double l1 = 0.0;
    if (st == PO_OK) {
        const double nd = (double)n;
        double *x = x_out;
        double dm = 0.0;   /* D: rank on dangling vertices */
#pragma omp parallel for num_threads(threads) schedule(static) reduction(+ : dm)
        for (int64_t u = 0; u < n; ++u) {
            deg[u] = (int32_t)(row_ptr[u + 1] - row_ptr[u]);
            x[u] = 1.0 / nd;
            c[u] = deg[u] ? x[u] / (double)deg[u] : 0.0;
            if (!deg[u])
                dm += x[u];
        }
        st = (tol > 0.0) ? PO_NOT_CONVERGED : PO_OK;
        while (it < max_iter) {
            l1 = 0.0;
            double dnext = 0.0;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 2048) reduction(+ : l1)
            for (int64_t v = 0; v < n; ++v) {
                double y = 0.0;
                for (int64_t j = in_ptr[v]; j < in_ptr[v + 1]; ++j)
                    y += c[in_col[j]];
                xn[v] = (1.0 - d) / nd + d * (y + dm / nd);
                l1 += fabs(xn[v] - x[v]);
            }
#pragma omp parallel for num_threads(threads) schedule(static) reduction(+ : dnext)
            for (int64_t u = 0; u < n; ++u) {
                x[u] = xn[u];
                c[u] = deg[u] ? x[u] / (double)deg[u] : 0.0;
                if (!deg[u])
                    dnext += x[u];
            }
            dm = dnext;
            ++it;
            if (tol > 0.0 && l1 < tol) {
                st = PO_OK;
                break;
            }
        }
    }
    const double t2 = omp_get_wtime();
    if (iters_out)
        *iters_out = it;
    if (l1_out)
        *l1_out = l1;
    if (t_transpose)
        *t_transpose = t1 - t0;
    if (t_loop)
        *t_loop = t2 - t1;
    free(in_ptr);
    free(in_col);
    free(c);
    free(xn);
    free(deg);
    return st;
}

int po_max_threads(void) { return omp_get_max_threads(); }
