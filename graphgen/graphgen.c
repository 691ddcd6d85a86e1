/*
 * Seeded synthetic directed graphs, written as out-edge CSR
 * (row_ptr int64[n+1], col_idx int32[m]).
 *
 * This file holds input generation only: no PageRank arithmetic. Both the
 * CUDA library's tests and the oracle's tests draw their inputs from here.
 *
 * Randomness is counter based: every value is a pure function of
 * (seed, stream, counter) through the SplitMix64 output mix (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), so a
 * graph is identical for any thread count and on any host.
 *
 * Recipes (sizes and shapes follow the workloads the PageRank pages measure):
 *  - gg_rmat: Graph500-style recursive matrix edges (quadrant probabilities
 *    a, b, c, d = 1-a-b-c; the source takes the row bit), edge_factor * 2^scale
 *    draws, self-loops and duplicates removed, no top-up, no relabelling.
 *  - gg_er: exactly round(f * n) dangling vertices chosen uniformly; every
 *    other vertex gets `deg` distinct uniform targets other than itself.
 *  - gg_citation: a growing citation network. Vertex 0 plus round(f * n) - 1
 *    others chosen uniformly are dangling. Every other vertex u, visited in id
 *    order, draws an out-degree from a power law k^-s on [kmin, kmax] (capped
 *    at u) and cites that many distinct earlier vertices (ids < u) by
 *    preferential attachment: probability proportional to in-degree so far + 1.
 * Every output row is sorted ascending.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GG_OK 0
#define GG_ERR_ARG (-1)
#define GG_ERR_OOM (-4)

enum { ST_DANGLING = 1, ST_DEGREE = 2, ST_TARGET = 3 };

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* k-th 64-bit value of stream `stream` under `seed` */
static inline uint64_t draw(uint64_t seed, uint64_t stream, uint64_t k)
{
    uint64_t key = mix64(seed * 0x9E3779B97F4A7C15ULL + stream + 1);
    return mix64(key + (k + 1) * 0x9E3779B97F4A7C15ULL);
}

/* uniform integer in [0, bound) from a 64-bit value (multiply-high) */
static inline uint64_t below(uint64_t r, uint64_t bound)
{
    return (uint64_t)(((unsigned __int128)r * bound) >> 64);
}

static inline double unit(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }

static void sort_i32(int32_t *a, int64_t len);

static int cmp_i32(const void *x, const void *y)
{
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return (a > b) - (a < b);
}

static void sort_i32(int32_t *a, int64_t len)
{
    if (len <= 24) {
        for (int64_t i = 1; i < len; ++i) {
            int32_t v = a[i];
            int64_t j = i - 1;
            while (j >= 0 && a[j] > v) {
                a[j + 1] = a[j];
                --j;
            }
            a[j + 1] = v;
        }
    } else {
        qsort(a, (size_t)len, sizeof(int32_t), cmp_i32);
    }
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* marks exactly k of the vertices first..n-1 as dangling (partial
 * Fisher-Yates shuffle); vertices below `first` are left unmarked */
static int pick_dangling(int64_t n, int64_t first, int64_t k, uint64_t seed,
                         uint8_t *is_dangling)
{
    int64_t pool = n - first;
    if (k > pool)
        return GG_ERR_ARG;
    int32_t *perm = (int32_t *)malloc((size_t)(pool > 0 ? pool : 1) * sizeof(int32_t));
    if (perm == NULL)
        return GG_ERR_OOM;
    for (int64_t i = 0; i < pool; ++i)
        perm[i] = (int32_t)(first + i);
    memset(is_dangling, 0, (size_t)n);
    for (int64_t i = 0; i < k; ++i) {
        int64_t j = i + (int64_t)below(draw(seed, ST_DANGLING, (uint64_t)i), (uint64_t)(pool - i));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
        is_dangling[perm[i]] = 1;
    }
    free(perm);
    return GG_OK;
}

int gg_rmat(int32_t scale, int64_t edge_factor, double a, double b, double c,
            uint64_t seed, int32_t nthreads, int64_t *row_ptr, int32_t *col_idx,
            int64_t *m_out)
{
    if (scale < 1 || scale > 30 || edge_factor < 1 || a < 0 || b < 0 || c < 0 ||
        a + b + c > 1.0 || row_ptr == NULL || col_idx == NULL || m_out == NULL)
        return GG_ERR_ARG;
    const int64_t n = (int64_t)1 << scale;
    const int64_t E = edge_factor * n;
    if (E > INT32_MAX)
        return GG_ERR_ARG;
    set_threads(nthreads);

    const uint64_t ta = (uint64_t)(a * 4294967296.0);
    const uint64_t tab = (uint64_t)((a + b) * 4294967296.0);
    const uint64_t tabc = (uint64_t)((a + b + c) * 4294967296.0);

    int32_t *src = (int32_t *)malloc((size_t)E * sizeof(int32_t));
    int32_t *dst = (int32_t *)malloc((size_t)E * sizeof(int32_t));
    int32_t *tmp = (int32_t *)malloc((size_t)E * sizeof(int32_t));
    int64_t *cnt = (int64_t *)calloc((size_t)n + 1, sizeof(int64_t));
    int64_t *cur = (int64_t *)malloc(((size_t)n + 1) * sizeof(int64_t));
    int64_t *ndeg = (int64_t *)malloc(((size_t)n + 1) * sizeof(int64_t));
    if (!src || !dst || !tmp || !cnt || !cur || !ndeg) {
        free(src); free(dst); free(tmp); free(cnt); free(cur); free(ndeg);
        return GG_ERR_OOM;
    }

    /* 1. draw every edge independently */
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < E; ++e) {
        uint32_t s = 0, t = 0;
        for (int32_t l = 0; l < scale; l += 2) {
            uint64_t r = draw(seed, (uint64_t)e, (uint64_t)l);
            for (int32_t h = 0; h < 2 && l + h < scale; ++h) {
                uint64_t u32 = (h == 0) ? (r & 0xFFFFFFFFULL) : (r >> 32);
                uint32_t sb, tb;
                if (u32 < ta) { sb = 0; tb = 0; }
                else if (u32 < tab) { sb = 0; tb = 1; }
                else if (u32 < tabc) { sb = 1; tb = 0; }
                else { sb = 1; tb = 1; }
                s = (s << 1) | sb;
                t = (t << 1) | tb;
            }
        }
        src[e] = (s == t) ? -1 : (int32_t)s;  /* self-loops dropped */
        dst[e] = (int32_t)t;
    }

    /* 2. bucket by source */
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < E; ++e)
        if (src[e] >= 0)
            __atomic_fetch_add(&cnt[src[e]], 1, __ATOMIC_RELAXED);
    int64_t acc = 0;
    for (int64_t u = 0; u < n; ++u) {
        int64_t k = cnt[u];
        cur[u] = acc;
        cnt[u] = acc;
        acc += k;
    }
    cnt[n] = acc;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < E; ++e) {
        if (src[e] >= 0) {
            int64_t p = __atomic_fetch_add(&cur[src[e]], 1, __ATOMIC_RELAXED);
            tmp[p] = dst[e];
        }
    }
    free(src);
    free(dst);

    /* 3. sort each row and drop duplicates */
#pragma omp parallel for schedule(dynamic, 4096)
    for (int64_t u = 0; u < n; ++u) {
        int32_t *r = tmp + cnt[u];
        int64_t len = cnt[u + 1] - cnt[u];
        sort_i32(r, len);
        int64_t k = 0;
        for (int64_t i = 0; i < len; ++i)
            if (k == 0 || r[i] != r[k - 1])
                r[k++] = r[i];
        ndeg[u] = k;
    }
    row_ptr[0] = 0;
    for (int64_t u = 0; u < n; ++u)
        row_ptr[u + 1] = row_ptr[u] + ndeg[u];
#pragma omp parallel for schedule(dynamic, 4096)
    for (int64_t u = 0; u < n; ++u)
        memcpy(col_idx + row_ptr[u], tmp + cnt[u], (size_t)ndeg[u] * sizeof(int32_t));

    *m_out = row_ptr[n];
    free(tmp); free(cnt); free(cur); free(ndeg);
    return GG_OK;
}

int gg_er(int64_t n, int32_t deg, double dangling_frac, uint64_t seed,
          int32_t nthreads, int64_t *row_ptr, int32_t *col_idx, int64_t *m_out)
{
    if (n < 2 || deg < 0 || (int64_t)deg > n - 1 || !(dangling_frac >= 0.0 && dangling_frac <= 1.0) ||
        row_ptr == NULL || m_out == NULL || (int64_t)deg * n > INT32_MAX)
        return GG_ERR_ARG;
    set_threads(nthreads);
    uint8_t *dang = (uint8_t *)malloc((size_t)n);
    if (dang == NULL)
        return GG_ERR_OOM;
    int64_t k = (int64_t)llround(dangling_frac * (double)n);
    int rc = pick_dangling(n, 0, k, seed, dang);
    if (rc != GG_OK) {
        free(dang);
        return rc;
    }
    row_ptr[0] = 0;
    for (int64_t u = 0; u < n; ++u)
        row_ptr[u + 1] = row_ptr[u] + (dang[u] ? 0 : deg);
    if (row_ptr[n] > 0 && col_idx == NULL) {
        free(dang);
        return GG_ERR_ARG;
    }

#pragma omp parallel for schedule(static, 4096)
    for (int64_t u = 0; u < n; ++u) {
        if (dang[u])
            continue;
        int32_t *r = col_idx + row_ptr[u];
        int32_t have = 0;
        uint64_t ctr = 0;
        while (have < deg) {
            int64_t t = (int64_t)below(draw(seed ^ 0x5EEDULL, (uint64_t)u, ctr++), (uint64_t)(n - 1));
            if (t >= u)
                t += 1;
            int dup = 0;
            for (int32_t i = 0; i < have; ++i)
                if (r[i] == (int32_t)t) { dup = 1; break; }
            if (!dup)
                r[have++] = (int32_t)t;
        }
        sort_i32(r, have);
    }
    *m_out = row_ptr[n];
    free(dang);
    return GG_OK;
}

int gg_citation(int64_t n, double zipf_s, int32_t kmin, int32_t kmax,
                double dangling_frac, uint64_t seed, int64_t *row_ptr,
                int32_t *col_idx, int64_t capacity, int64_t *m_out)
{
    if (n < 2 || kmin < 1 || kmax < kmin || !(dangling_frac >= 0.0 && dangling_frac <= 1.0) ||
        row_ptr == NULL || col_idx == NULL || m_out == NULL)
        return GG_ERR_ARG;
    if ((int64_t)kmax > n - 1)
        kmax = (int32_t)(n - 1);
    if (kmin > kmax)
        kmin = kmax;
    uint8_t *dang = (uint8_t *)malloc((size_t)n);
    double *cdf = (double *)malloc((size_t)(kmax - kmin + 1) * sizeof(double));
    int32_t *degs = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    if (!dang || !cdf || !degs) {
        free(dang); free(cdf); free(degs);
        return GG_ERR_OOM;
    }
    /* vertex 0 has nobody earlier to cite: it is one of the dangling set */
    int64_t k = (int64_t)llround(dangling_frac * (double)n);
    int rc = pick_dangling(n, 1, k > 0 ? k - 1 : 0, seed, dang);
    if (rc != GG_OK) {
        free(dang); free(cdf); free(degs);
        return rc;
    }
    dang[0] = 1;

    /* power-law out-degree table on [kmin, kmax] */
    double total = 0.0;
    for (int32_t q = kmin; q <= kmax; ++q) {
        total += pow((double)q, -zipf_s);
        cdf[q - kmin] = total;
    }
    int64_t m = 0;
    for (int64_t u = 0; u < n; ++u) {
        if (dang[u]) {
            degs[u] = 0;
            continue;
        }
        double r = unit(draw(seed, ST_DEGREE, (uint64_t)u)) * total;
        int32_t lo = 0, hi = kmax - kmin;
        while (lo < hi) {
            int32_t mid = (lo + hi) / 2;
            if (cdf[mid] > r) hi = mid; else lo = mid + 1;
        }
        degs[u] = kmin + lo;
        if ((int64_t)degs[u] > u)
            degs[u] = (int32_t)u;
        m += degs[u];
    }
    free(cdf);
    if (m > capacity || m > INT32_MAX) {
        free(dang); free(degs);
        return GG_ERR_ARG;
    }

    /* urn of earlier vertex ids: one entry per visited vertex plus one per
     * placed in-edge; vertex u joins the urn after its own citations */
    int32_t *urn = (int32_t *)malloc((size_t)(n + m) * sizeof(int32_t));
    if (urn == NULL) {
        free(dang); free(degs);
        return GG_ERR_OOM;
    }
    int64_t urn_len = 0;

    row_ptr[0] = 0;
    uint64_t ctr = 0;
    for (int64_t u = 0; u < n; ++u) {
        int32_t *r = col_idx + row_ptr[u];
        int32_t have = 0;
        while (have < degs[u]) {
            int32_t cand = urn[below(draw(seed, ST_TARGET, ctr++), (uint64_t)urn_len)];
            int dup = 0;
            for (int32_t i = 0; i < have; ++i)
                if (r[i] == cand) { dup = 1; break; }
            if (!dup)
                r[have++] = cand;
        }
        for (int32_t i = 0; i < have; ++i)
            urn[urn_len++] = r[i];
        urn[urn_len++] = (int32_t)u;
        sort_i32(r, have);
        row_ptr[u + 1] = row_ptr[u] + have;
    }
    *m_out = row_ptr[n];
    free(urn); free(dang); free(degs);
    return GG_OK;
}
