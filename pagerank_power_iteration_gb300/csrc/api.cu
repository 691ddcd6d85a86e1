// The C ABI (include/pagerank.h): argument checks, host/device pointer
// handling, ownership of device memory, and error reporting. The compute is
// in transpose.cu (pr_graph_create) and iterate.cu (pr_run).
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "pr_internal.cuh"

#define PR_API extern "C" __attribute__((visibility("default")))

namespace prk {

static thread_local char g_last_error[512] = "";

pr_status set_error(pr_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

pr_status cuda_status(cudaError_t e, const char *what)
{
    cudaGetLastError();   // clear a non-sticky error
    return set_error(e == cudaErrorMemoryAllocation ? PR_ERR_OOM : PR_ERR_CUDA, "%s: %s (%s)",
                     what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// Device memory comes from one stream-ordered pool per device, owned by the
// library, that keeps freed blocks for reuse (release threshold: never). A
// graph built after another one was destroyed reuses its memory instead of
// paying cudaMalloc and cudaFree (which synchronises the device) again. The
// pool holds its peak size until the process exits.
static std::mutex g_pool_mu;
static cudaMemPool_t g_pools[kMaxDevices] = {};

static pr_status device_pool(cudaMemPool_t *out)
{
    std::mutex &mu = g_pool_mu;
    cudaMemPool_t *pools = g_pools;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(PR_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (pools[dev] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaMemPoolCreate");
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaMemPoolSetAttribute");
        pools[dev] = pool;
    }
    *out = pools[dev];
    return PR_OK;
}

// Test hook: the k-th pool allocation from now fails (0: none does).
static std::atomic<int64_t> g_fail_countdown{0};

void fail_alloc_after(int64_t k) { g_fail_countdown.store(k > 0 ? k : 0); }

pr_status pool_used_bytes(int64_t *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(PR_ERR_CUDA, "device ordinal %d out of range", dev);
    // frees are stream ordered: let every pending one reach the pool
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_status(e, "cudaDeviceSynchronize");
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lock(g_pool_mu);
        pool = g_pools[dev];
    }
    if (pool == nullptr) {   // never created: nothing allocated
        *out = 0;
        return PR_OK;
    }
    uint64_t used = 0;
    e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &used);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaMemPoolGetAttribute");
    *out = (int64_t)used;
    return PR_OK;
}

pr_status pool_alloc(void **p, size_t bytes, cudaStream_t s)
{
    if (bytes == 0)
        bytes = 16;
    for (int64_t k = g_fail_countdown.load(); k > 0; k = g_fail_countdown.load()) {
        if (g_fail_countdown.compare_exchange_weak(k, k - 1)) {
            if (k == 1) {
                *p = nullptr;
                return set_error(PR_ERR_OOM, "device allocation of %zu bytes failed (injected by "
                                             "pr_test_fail_alloc_after)", bytes);
            }
            break;
        }
    }
    cudaMemPool_t pool;
    pr_status st = device_pool(&pool);
    if (st != PR_OK)
        return st;
    cudaError_t e = cudaMallocFromPoolAsync(p, bytes, pool, s);
    if (e != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        return set_error(e == cudaErrorMemoryAllocation ? PR_ERR_OOM : PR_ERR_CUDA,
                         "device allocation of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
    }
    return PR_OK;
}

void pool_free(void *p, cudaStream_t s)
{
    if (p)
        cudaFreeAsync(p, s);
}

pr_status graph_alloc(pr_graph *g, void **p, size_t bytes, cudaStream_t s)
{
    pr_status st = pool_alloc(p, bytes, s);
    if (st != PR_OK)
        return st;
    g->allocs.push_back(*p);
    g->device_bytes += (int64_t)(bytes ? bytes : 16);
    return PR_OK;
}

PtrKind pointer_kind(const void *p, int device)
{
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return kPtrHost;
    }
    if (attr.type == cudaMemoryTypeManaged)
        return kPtrDevice;
    if (attr.type == cudaMemoryTypeDevice)
        return attr.device == device ? kPtrDevice : kPtrOtherDevice;
    return kPtrHost;
}

}  // namespace prk

namespace {

constexpr int64_t kMaxN = ((int64_t)1 << 31) - 2;
constexpr int64_t kMaxM = ((int64_t)1 << 31) - 1;
// The work CSR pads every row that has in-edges to a multiple of 4 entries
// (at most 3 more per row, and at most min(n, m) such rows), and the few
// thread-class blocks that mix row lengths pad their rows to the block's
// longest (under 8192 entries in all); its offsets are int32.
constexpr int64_t kLayoutSlack = PR_LAYOUT_SLACK;

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            prev = -1;
        }
        if (dev >= 0 && dev != prev)
            cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        if (prev >= 0)
            cudaSetDevice(prev);
    }
};

void free_graph(pr_graph *g)
{
    if (!g)
        return;
    prk::release_dtype_state(g);
    for (cudaEvent_t &ev : g->ev)
        if (ev)
            cudaEventDestroy(ev);
    // no work on the handle is in flight (its calls synchronised their
    // streams), so the blocks can go back to the pool in default-stream order
    for (void *p : g->allocs)
        prk::pool_free(p, 0);
    delete g->h_scal;
    delete g;
}

}  // namespace

using prk::set_error;

PR_API pr_status pr_graph_create(int64_t n, int64_t m, const int64_t *row_ptr,
                                 const int32_t *col_idx, void *stream, pr_graph **out)
{
    return pr_graph_create_ex(n, m, row_ptr, col_idx, nullptr, stream, out);
}

PR_API pr_status pr_graph_create_ex(int64_t n, int64_t m, const int64_t *row_ptr,
                                    const int32_t *col_idx, const pr_options *opts, void *stream,
                                    pr_graph **out)
{
    const pr_options o = opts ? *opts : pr_options PR_OPTIONS_DEFAULT;
    if (o.thread_max < 1 || o.thread_max > prk::kThreadMaxLimit)
        return set_error(PR_ERR_INVALID_ARG, "thread_max must be in [1, %d] (got %d)", prk::kThreadMaxLimit,
                         (int)o.thread_max);
    if (o.warp_max < o.thread_max || o.warp_max > prk::kWarpMaxLimit)
        return set_error(PR_ERR_INVALID_ARG, "warp_max must be in [thread_max, %d] (got %d)", prk::kWarpMaxLimit,
                         (int)o.warp_max);
    if (out == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "out is NULL");
    if (n < 1)
        return set_error(PR_ERR_INVALID_ARG, "n must be >= 1 (got %lld)", (long long)n);
    if (m < 0)
        return set_error(PR_ERR_INVALID_ARG, "m must be >= 0 (got %lld)", (long long)m);
    if (n > kMaxN)
        return set_error(PR_ERR_TOO_LARGE, "n = %lld exceeds 2^31 - 2", (long long)n);
    if (m > kMaxM)
        return set_error(PR_ERR_TOO_LARGE, "m = %lld exceeds 2^31 - 1", (long long)m);
    if (m + 3 * (n < m ? n : m) + kLayoutSlack > kMaxM)
        return set_error(PR_ERR_TOO_LARGE,
                         "m + 3 min(n, m) + %lld = %lld exceeds 2^31 - 1 (the padded work layout keeps "
                         "int32 offsets)", (long long)kLayoutSlack,
                         (long long)(m + 3 * (n < m ? n : m) + kLayoutSlack));
    if (row_ptr == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "row_ptr is NULL");
    if (m > 0 && col_idx == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "col_idx is NULL but m > 0");

    cudaStream_t s = (cudaStream_t)stream;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return prk::cuda_status(e, "cudaGetDevice");

    prk::NvtxRange range("pr_graph_create");
    pr_graph *g = new (std::nothrow) pr_graph();
    if (!g)
        return set_error(PR_ERR_OOM, "host allocation failed");
    g->n = n;
    g->m = m;
    g->device = dev;
    g->thread_max = o.thread_max;
    g->warp_max = o.warp_max;
    g->stage_timing = o.stage_timing != 0;
    pr_status st = PR_OK;

    do {
        e = cudaDeviceGetAttribute(&g->num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) { st = prk::cuda_status(e, "device query"); break; }
        for (cudaEvent_t &ev : g->ev) {
            e = cudaEventCreate(&ev);
            if (e != cudaSuccess) break;
        }
        if (e != cudaSuccess) { st = prk::cuda_status(e, "cudaEventCreate"); break; }
        // a plain host copy: pr_run reads it once per run, right after the
        // stream synchronisation it waits for anyway, and pinning a buffer per
        // handle cost about 0.16 ms in pr_graph_create and 0.2 ms in
        // pr_graph_destroy (cudaMallocHost / cudaFreeHost)
        g->h_scal = new (std::nothrow) prk::Scalars();
        if (!g->h_scal) { st = set_error(PR_ERR_OOM, "host allocation failed"); break; }
        if ((st = prk::graph_alloc(g, (void **)&g->scal, sizeof(prk::Scalars), s)) != PR_OK) break;
        if ((st = prk::graph_alloc(g, (void **)&g->err, sizeof(unsigned), s)) != PR_OK) break;
        e = cudaMemsetAsync(g->scal, 0, sizeof(prk::Scalars), s);
        if (e != cudaSuccess) { st = prk::cuda_status(e, "memset"); break; }

        // inputs on the device (borrowed, or staged copies freed below)
        const prk::PtrKind rp_kind = prk::pointer_kind(row_ptr, dev);
        const prk::PtrKind ci_kind = m == 0 ? prk::kPtrDevice : prk::pointer_kind(col_idx, dev);
        if (rp_kind == prk::kPtrOtherDevice || ci_kind == prk::kPtrOtherDevice) {
            st = set_error(PR_ERR_INVALID_ARG, "row_ptr and col_idx must be host memory or memory of "
                                               "the current device (%d)", dev);
            break;
        }
        const bool rp_dev = rp_kind == prk::kPtrDevice;
        const bool ci_dev = ci_kind == prk::kPtrDevice;
        int64_t ends[2];
        if (rp_dev) {
            e = cudaMemcpyAsync(&ends[0], row_ptr, sizeof(int64_t), cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(&ends[1], row_ptr + n, sizeof(int64_t), cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess)
                e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) { st = prk::cuda_status(e, "reading row_ptr"); break; }
        } else {
            ends[0] = row_ptr[0];
            ends[1] = row_ptr[n];
        }
        if (ends[0] != 0) {
            st = set_error(PR_ERR_INVALID_GRAPH, "row_ptr[0] = %lld, expected 0", (long long)ends[0]);
            break;
        }
        if (ends[1] != m) {
            st = set_error(PR_ERR_INVALID_GRAPH, "row_ptr[n] = %lld, expected m = %lld",
                           (long long)ends[1], (long long)m);
            break;
        }
        void *rp_stage = nullptr, *ci_stage = nullptr;
        const int64_t *d_rp = row_ptr;
        const int32_t *d_ci = col_idx;
        if (!rp_dev) {
            st = prk::pool_alloc(&rp_stage, (size_t)(n + 1) * sizeof(int64_t), s);
            if (st == PR_OK)
                e = cudaMemcpyAsync(rp_stage, row_ptr, (size_t)(n + 1) * sizeof(int64_t),
                                    cudaMemcpyHostToDevice, s);
            d_rp = (const int64_t *)rp_stage;
        }
        // a host col_idx is copied by the build itself, beside its first steps
        if (st == PR_OK && e == cudaSuccess && !ci_dev) {
            st = prk::pool_alloc(&ci_stage, (size_t)m * sizeof(int32_t), s);
            d_ci = (const int32_t *)ci_stage;
        }
        if (st == PR_OK && e != cudaSuccess)
            st = prk::cuda_status(e, "staging the input CSR");
        if (st == PR_OK)
            st = prk::build_graph(g, d_rp, d_ci, ci_dev ? nullptr : col_idx, s);
        prk::pool_free(rp_stage, s);
        prk::pool_free(ci_stage, s);
        cudaError_t se = cudaStreamSynchronize(s);
        if (st == PR_OK && se != cudaSuccess)
            st = prk::cuda_status(se, "pr_graph_create");
    } while (0);

    if (st != PR_OK) {
        free_graph(g);
        return st;
    }
    *out = g;
    return PR_OK;
}

PR_API pr_status pr_run(pr_graph *g, double d, double tol, int32_t max_iter, pr_dtype dtype,
                        void *ranks_out, const void *x_init, int32_t *iters_out, double *l1_out,
                        void *stream)
{
    if (g == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "graph is NULL");
    if (!(d >= 0.0 && d <= 1.0))
        return set_error(PR_ERR_INVALID_ARG, "d must be in [0, 1] (got %g)", d);
    if (tol != tol)
        return set_error(PR_ERR_INVALID_ARG, "tol is NaN");
    if (max_iter < 1)
        return set_error(PR_ERR_INVALID_ARG, "max_iter must be >= 1 (got %d)", (int)max_iter);
    if (dtype != PR_F32 && dtype != PR_F64)
        return set_error(PR_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (ranks_out == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "ranks_out is NULL");
    DeviceGuard guard(g->device);
    return prk::run(g, d, tol, max_iter, (int)dtype, ranks_out, x_init, iters_out, l1_out,
                    (cudaStream_t)stream);
}

PR_API pr_status pr_get_in_csr(const pr_graph *g, int32_t *in_ptr, int32_t *in_col, void *stream)
{
    if (g == nullptr || in_ptr == nullptr || (g->m > 0 && in_col == nullptr))
        return set_error(PR_ERR_INVALID_ARG, "NULL argument");
    DeviceGuard guard(g->device);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(in_ptr, g->in_ptr, (size_t)(g->n + 1) * sizeof(int32_t),
                                    cudaMemcpyDefault, s);
    if (e == cudaSuccess && g->m > 0)
        e = cudaMemcpyAsync(in_col, g->in_col, (size_t)g->m * sizeof(int32_t), cudaMemcpyDefault, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? PR_OK : prk::cuda_status(e, "pr_get_in_csr");
}

PR_API pr_status pr_graph_get_info(const pr_graph *g, pr_graph_info *info)
{
    if (g == nullptr || info == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "NULL argument");
    memset(info, 0, sizeof(*info));
    info->n = g->n;
    info->m = g->m;
    info->n_dangling = g->n_dangling;
    info->rows_zero = g->n_z;
    info->rows_thread = g->n_t;
    info->rows_warp = g->n_w;
    info->rows_cta = g->n_c;
    info->edges_thread = g->e_t;
    info->edges_warp = g->e_w;
    info->edges_cta = g->e_c;
    info->cta_chunks = g->n_chunks;
    info->cta_chunk_edges = prk::kChunkEdges;
    info->iterate_grid = g->st[0].ready ? g->st[0].grid : g->st[1].grid;
    info->device_bytes = g->device_bytes;
    info->build_launches = g->build_launches;
    info->edges_hot_f32 = g->e_hot[0];
    info->edges_hot_f64 = g->e_hot[1];
    info->thread_max = g->thread_max;
    info->warp_max = g->warp_max;
    info->build_ms = g->build_ms;
    for (int k = 0; k < PR_BUILD_STAGES; ++k)
        info->build_stage_ms[k] = g->build_stage_ms[k];
    return PR_OK;
}

PR_API pr_status pr_measure_gather_rate(int64_t n, pr_dtype dtype, int64_t gathers, pr_gather_path path,
                                        double *gathers_per_s, void *stream)
{
    if (path != PR_GATHER_LOAD && path != PR_GATHER_TMA && path != PR_GATHER_BOTH)
        return set_error(PR_ERR_INVALID_ARG, "unknown gather path %d", (int)path);
    if (gathers_per_s == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "gathers_per_s is NULL");
    if (n < 1 || n > kMaxN)
        return set_error(PR_ERR_INVALID_ARG, "n must be in [1, 2^31 - 2] (got %lld)", (long long)n);
    if (gathers < 1 || gathers > ((int64_t)1 << 30))
        return set_error(PR_ERR_INVALID_ARG, "gathers must be in [1, 2^30] (got %lld)",
                         (long long)gathers);
    if (dtype != PR_F32 && dtype != PR_F64)
        return set_error(PR_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    return prk::measure_gather_rate(n, (int)dtype, gathers, (int)path, gathers_per_s, (cudaStream_t)stream);
}

PR_API pr_status pr_graph_last_run(const pr_graph *g, pr_run_stats *stats)
{
    if (g == nullptr || stats == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "NULL argument");
    *stats = g->last;
    return PR_OK;
}

PR_API void pr_graph_destroy(pr_graph *g)
{
    if (!g)
        return;
    DeviceGuard guard(g->device);
    free_graph(g);
}

PR_API pr_status pr_exclusive_scan_noalloc(const int32_t *counts, int32_t *offsets, int64_t count,
                                           void *stream)
{
    return prk::exclusive_scan_noalloc(counts, offsets, count, (cudaStream_t)stream);
}

PR_API void pr_test_fail_alloc_after(int64_t k) { prk::fail_alloc_after(k); }

PR_API pr_status pr_test_pool_used_bytes(int64_t *used)
{
    if (used == nullptr)
        return set_error(PR_ERR_INVALID_ARG, "used is NULL");
    return prk::pool_used_bytes(used);
}

PR_API pr_status pr_test_scan_timeout(int64_t count, int32_t spin_limit, void *stream)
{
    return prk::scan_timeout_probe(count, spin_limit, (cudaStream_t)stream);
}

PR_API const char *pr_last_error(void) { return prk::g_last_error; }

PR_API const char *pr_version(void) { return "pagerank-gb300 0.1 (sm_103a)"; }
