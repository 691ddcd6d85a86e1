// The power iteration on the device.
//
// One update ("Day 40 - PageRank on a real graph in CUDA", section "One
// iteration, three shapes of work"):
//   x'[v] = (1 - d)/n + d * (y[v] + D/n),  y[v] = sum over in-edges u->v of x[u]/outdeg[u]
// is one launch of k_iterate, a persistent kernel that fuses the four stages
// the page runs as separate launches:
//   - the contribution x[u]/outdeg[u] is not recomputed per update: the state
//     vector s holds it (s[u] = x[u]/outdeg[u], or x[u] for a dangling u),
//     written by the update that produced x[u] (the contribution cache of
//     Meerkat's PageRank, Algorithm 5, and "Precomputed inverse out-degree" of
//     gpu-graph-study's T3 tier);
//   - the pull SpMV over the in-edge CSR gathers s, by in-degree class:
//     one thread per row (<= 32 in-edges), one warp per row (33..1024), and
//     CTA-sized chunks of 4096 edges for larger rows, whose partial sums the
//     CTA finishing the row's last chunk adds up in chunk order;
//   - the combine reads D from device memory (Day 40, "Keep the dangling mass
//     on the device"), writes s' and accumulates the L1 distance and the next
//     dangling mass;
//   - the two reductions go thread -> warp -> CTA -> one fp64 partial per CTA,
//     and the last CTA to arrive sums the partials in CTA order (Day 40 budget
//     of gridDim.x + 1 global writes per reduction; gpu-graph-study T3's "one
//     atomic per block" ticket).
// The last CTA also advances the update counter and, when L1 < tol or the
// cap is reached, ends the CUDA graph's WHILE loop with
// cudaGraphSetConditional, so a whole run is one graph launch and the host
// never waits between updates (Meerkat Algorithm 5's loop while delta >
// error_margin and it < max_iter).
//
// No kernel here waits on another CTA: the chunk and last-CTA hand-offs use
// arrival counters only, so nothing can spin.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pr_internal.cuh"

namespace prk {
namespace {

template <typename T>
struct IterArgs {
    const int32_t *in_ptr;
    const int32_t *in_col;
    const int32_t *deg_out;
    const int32_t *rows_z, *rows_t, *rows_w, *rows_c;
    const int32_t *chunk_row, *chunk_first;
    uint32_t *hub_arrivals;
    T *s0, *s1;
    T *hub_partial;
    double *block_partials;
    Scalars *scal;
    int64_t n, n_z, n_t, n_w, n_chunks;
};

// streaming (evict-first) loads of the index stream
__device__ __forceinline__ int32_t ld_stream(const int32_t *p) { return __ldcs(p); }
__device__ __forceinline__ int4 ld_stream4(const int4 *p) { return __ldcs(p); }

template <typename T>
__device__ __forceinline__ T warp_sum(T v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide sum; the result is valid in thread 0. `red` holds 32 entries.
template <typename T>
__device__ __forceinline__ T block_sum(T v, T *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    T t = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : T(0);
    if (warp == 0)
        t = warp_sum(t);
    __syncthreads();
    return t;
}

// Sum of s[in_col[j]] for j in [b, e) over `lanes` cooperating threads
// (`lane` in [0, lanes)): an unaligned head of at most 3 edges, a body of
// 16-byte index loads, and a tail of at most 3 edges.
template <typename T, int kLanes>
__device__ __forceinline__ T gather_range(const int32_t *__restrict__ col, const T *__restrict__ s,
                                          int64_t b, int64_t e, int lane)
{
    T acc0 = T(0), acc1 = T(0);
    const int64_t a0 = (b + 3) & ~int64_t(3);
    const int64_t a1 = e & ~int64_t(3);
    if (a0 >= a1) {
        for (int64_t j = b + lane; j < e; j += kLanes)
            acc0 += __ldg(s + ld_stream(col + j));
        return acc0;
    }
    if (b + lane < a0)
        acc0 += __ldg(s + ld_stream(col + b + lane));
    if (a1 + lane < e)
        acc1 += __ldg(s + ld_stream(col + a1 + lane));
    const int4 *cv = reinterpret_cast<const int4 *>(col + a0);
    const int64_t nv = (a1 - a0) >> 2;
    int64_t k = lane;
    for (; k + kLanes < nv; k += 2 * kLanes) {
        const int4 q = ld_stream4(cv + k);
        const int4 r = ld_stream4(cv + k + kLanes);
        acc0 += __ldg(s + q.x);
        acc1 += __ldg(s + q.y);
        acc0 += __ldg(s + q.z);
        acc1 += __ldg(s + q.w);
        acc0 += __ldg(s + r.x);
        acc1 += __ldg(s + r.y);
        acc0 += __ldg(s + r.z);
        acc1 += __ldg(s + r.w);
    }
    if (k < nv) {
        const int4 q = ld_stream4(cv + k);
        acc0 += __ldg(s + q.x);
        acc1 += __ldg(s + q.y);
        acc0 += __ldg(s + q.z);
        acc1 += __ldg(s + q.w);
    }
    return acc0 + acc1;
}

__device__ __forceinline__ float abs_t(float x) { return fabsf(x); }
__device__ __forceinline__ double abs_t(double x) { return ::fabs(x); }

// The combine for one row: new rank, new state, L1 and dangling-mass terms.
template <typename T>
__device__ __forceinline__ void finish_row(int32_t v, T y, const int32_t *__restrict__ deg_out,
                                           const T *__restrict__ s_old, T *__restrict__ s_new,
                                           T base, T d, T &l1, T &dm)
{
    const int32_t deg = deg_out[v];
    const T so = s_old[v];
    const T x_old = deg ? so * T(deg) : so;
    const T x_new = base + d * y;
    l1 += abs_t(x_new - x_old);
    if (deg) {
        __stcs(s_new + v, x_new / T(deg));
    } else {
        __stcs(s_new + v, x_new);
        dm += x_new;
    }
}

template <typename T>
__global__ void __launch_bounds__(kBlock)
k_iterate(IterArgs<T> a, cudaGraphConditionalHandle cond)
{
    __shared__ T s_red[32];
    __shared__ double s_redd[32];
    __shared__ int s_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t G = gridDim.x;

    // run scalars, read once (the last CTA rewrites them after every other
    // CTA has passed its arrival)
    const volatile Scalars *vs = a.scal;
    const int it = vs->it;
    const double dd = vs->d, inv_n = vs->inv_n, D = vs->dmass;
    const T *__restrict__ s_old = (it & 1) ? a.s1 : a.s0;
    T *__restrict__ s_new = (it & 1) ? a.s0 : a.s1;
    const T d = T(dd);
    const T base = T((1.0 - dd) * inv_n + dd * D * inv_n);

    T l1 = T(0), dm = T(0);

    // rows with more than 1024 in-edges, in chunks of kChunkEdges
    for (int64_t c = blockIdx.x; c < a.n_chunks; c += G) {
        const int32_t r = a.chunk_row[c];
        const int32_t v = a.rows_c[r];
        const int32_t first = a.chunk_first[r];
        const int32_t nch = a.chunk_first[r + 1] - first;
        const int64_t rb = a.in_ptr[v], re = a.in_ptr[v + 1];
        const int64_t cb = rb + (int64_t)(c - first) * kChunkEdges;
        const int64_t ce = min(cb + (int64_t)kChunkEdges, re);
        T part = gather_range<T, kBlock>(a.in_col, s_old, cb, ce, tid);
        part = block_sum(part, s_red);
        if (tid == 0) {
            __stcg(a.hub_partial + c, part);
            __threadfence();
            const uint32_t prev = atomicAdd(a.hub_arrivals + r, 1u);
            s_flag = (prev == (uint32_t)(nch - 1));
        }
        __syncthreads();
        if (s_flag && tid == 0) {
            __threadfence();
            T y = T(0);
            for (int32_t k = 0; k < nch; ++k)
                y += __ldcg(a.hub_partial + first + k);
            a.hub_arrivals[r] = 0u;
            finish_row(v, y, a.deg_out, s_old, s_new, base, d, l1, dm);
        }
        __syncthreads();
    }

    // 33..1024 in-edges: one warp per row
    for (int64_t i = (int64_t)blockIdx.x * (kBlock / 32) + warp; i < a.n_w; i += G * (kBlock / 32)) {
        const int32_t v = a.rows_w[i];
        T y = gather_range<T, 32>(a.in_col, s_old, a.in_ptr[v], a.in_ptr[v + 1], lane);
        y = warp_sum(y);
        if (lane == 0)
            finish_row(v, y, a.deg_out, s_old, s_new, base, d, l1, dm);
    }

    // 1..32 in-edges: one thread per row
    for (int64_t i = (int64_t)blockIdx.x * kBlock + tid; i < a.n_t; i += G * kBlock) {
        const int32_t v = a.rows_t[i];
        const int32_t b = a.in_ptr[v], e = a.in_ptr[v + 1];
        T y0 = T(0), y1 = T(0);
        int32_t j = b;
        for (; j + 1 < e; j += 2) {
            const int32_t u0 = ld_stream(a.in_col + j);
            const int32_t u1 = ld_stream(a.in_col + j + 1);
            y0 += __ldg(s_old + u0);
            y1 += __ldg(s_old + u1);
        }
        if (j < e)
            y0 += __ldg(s_old + ld_stream(a.in_col + j));
        finish_row(v, y0 + y1, a.deg_out, s_old, s_new, base, d, l1, dm);
    }

    // no in-edges
    for (int64_t i = (int64_t)blockIdx.x * kBlock + tid; i < a.n_z; i += G * kBlock)
        finish_row(a.rows_z[i], T(0), a.deg_out, s_old, s_new, base, d, l1, dm);

    // reductions: one fp64 partial pair per CTA, the last CTA sums them
    const double l1_blk = block_sum((double)l1, s_redd);
    const double dm_blk = block_sum((double)dm, s_redd);
    if (tid == 0) {
        __stcg(a.block_partials + 2 * blockIdx.x, l1_blk);
        __stcg(a.block_partials + 2 * blockIdx.x + 1, dm_blk);
        __threadfence();
        const uint32_t t = atomicAdd(&a.scal->ticket, 1u);
        s_flag = (t == (uint32_t)(G - 1));
    }
    __syncthreads();
    if (!s_flag)
        return;
    __threadfence();
    double L = 0.0, M = 0.0;
    for (int64_t b = tid; b < G; b += kBlock) {
        L += __ldcg(a.block_partials + 2 * b);
        M += __ldcg(a.block_partials + 2 * b + 1);
    }
    L = block_sum(L, s_redd);
    M = block_sum(M, s_redd);
    if (tid == 0) {
        Scalars *sc = a.scal;
        const int it1 = it + 1;
        const bool conv = (sc->tol > 0.0) && (L < sc->tol);
        sc->l1 = L;
        sc->dmass = M;
        sc->it = it1;
        sc->converged = conv ? 1 : 0;
        sc->ticket = 0u;
        __threadfence();
        if (conv || it1 >= sc->max_iter)
            cudaGraphSetConditional(cond, 0);
    }
}

// Start vector (1/n, or the caller's x_init), its state and dangling mass,
// and the run scalars.
template <typename T>
__global__ void __launch_bounds__(kBlock)
k_init(IterArgs<T> a, const T *__restrict__ x_init, double d, double tol, int32_t max_iter)
{
    __shared__ double s_redd[32];
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    const int64_t G = gridDim.x;
    const T x_uniform = T(1.0 / (double)a.n);
    T dm = T(0);
    for (int64_t v = (int64_t)blockIdx.x * kBlock + tid; v < a.n; v += G * kBlock) {
        const T x = x_init ? x_init[v] : x_uniform;
        const int32_t deg = a.deg_out[v];
        if (deg) {
            a.s0[v] = x / T(deg);
        } else {
            a.s0[v] = x;
            dm += x;
        }
    }
    const double dm_blk = block_sum((double)dm, s_redd);
    if (tid == 0) {
        __stcg(a.block_partials + 2 * blockIdx.x + 1, dm_blk);
        __threadfence();
        const uint32_t t = atomicAdd(&a.scal->ticket, 1u);
        s_flag = (t == (uint32_t)(G - 1));
    }
    __syncthreads();
    if (!s_flag)
        return;
    __threadfence();
    double M = 0.0;
    for (int64_t b = tid; b < G; b += kBlock)
        M += __ldcg(a.block_partials + 2 * b + 1);
    M = block_sum(M, s_redd);
    if (tid == 0) {
        Scalars *sc = a.scal;
        sc->dmass = M;
        sc->l1 = 0.0;
        sc->d = d;
        sc->tol = tol;
        sc->inv_n = 1.0 / (double)a.n;
        sc->it = 0;
        sc->max_iter = max_iter;
        sc->converged = 0;
        sc->ticket = 0u;
    }
}

// Ranks from the final state: x = s * outdeg, or s for a dangling vertex.
template <typename T>
__global__ void k_output(IterArgs<T> a, T *__restrict__ out)
{
    const int it = ((const volatile Scalars *)a.scal)->it;
    const T *s = (it & 1) ? a.s1 : a.s0;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < a.n;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int32_t deg = a.deg_out[v];
        const T sv = s[v];
        out[v] = deg ? sv * T(deg) : sv;
    }
}

template <typename T>
IterArgs<T> make_args(pr_graph *g)
{
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    IterArgs<T> a;
    a.in_ptr = g->in_ptr;
    a.in_col = g->in_col;
    a.deg_out = g->deg_out;
    a.rows_z = g->rows_z;
    a.rows_t = g->rows_t;
    a.rows_w = g->rows_w;
    a.rows_c = g->rows_c;
    a.chunk_row = g->chunk_row;
    a.chunk_first = g->chunk_first;
    a.hub_arrivals = g->hub_arrivals;
    a.s0 = (T *)st.s[0];
    a.s1 = (T *)st.s[1];
    a.hub_partial = (T *)st.hub_partial;
    a.block_partials = st.block_partials;
    a.scal = g->scal;
    a.n = g->n;
    a.n_z = g->n_z;
    a.n_t = g->n_t;
    a.n_w = g->n_w;
    a.n_chunks = g->n_chunks;
    return a;
}

// Allocates a precision's state and builds its graph: one conditional WHILE
// node whose body is one k_iterate launch.
template <typename T>
pr_status prepare(pr_graph *g)
{
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    if (st.ready)
        return PR_OK;
    pr_status r;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_iterate<T>, kBlock, 0);
    if (e != cudaSuccess)
        return cuda_status(e, "occupancy query");
    if (per_sm < 1)
        per_sm = 1;
    st.grid = per_sm * g->num_sms;
    st.init_grid = st.grid;
    const size_t n = (size_t)g->n;
    if ((r = graph_alloc(g, &st.s[0], n * sizeof(T))) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.s[1], n * sizeof(T))) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.stage, n * sizeof(T))) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.hub_partial, (size_t)(g->n_chunks + 1) * sizeof(T))) != PR_OK) return r;
    if ((r = graph_alloc(g, (void **)&st.block_partials, (size_t)st.grid * 2 * sizeof(double))) != PR_OK)
        return r;

    IterArgs<T> args = make_args<T>(g);
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaGraphConditionalHandle handle;
    cudaGraphNodeParams cp = {};
    cudaGraphNode_t cnode, knode;
    cudaKernelNodeParams kp = {};
    void *kargs[] = {&args, &handle};

    e = cudaGraphCreate(&graph, 0);
    if (e == cudaSuccess)
        e = cudaGraphConditionalHandleCreate(&handle, graph, 1, cudaGraphCondAssignDefault);
    if (e == cudaSuccess) {
        cp.type = cudaGraphNodeTypeConditional;
        cp.conditional.handle = handle;
        cp.conditional.type = cudaGraphCondTypeWhile;
        cp.conditional.size = 1;
        e = cudaGraphAddNode(&cnode, graph, nullptr, nullptr, 0, &cp);
    }
    if (e == cudaSuccess) {
        kp.func = (void *)k_iterate<T>;
        kp.gridDim = dim3((unsigned)st.grid);
        kp.blockDim = dim3(kBlock);
        kp.sharedMemBytes = 0;
        kp.kernelParams = kargs;
        e = cudaGraphAddKernelNode(&knode, cp.conditional.phGraph_out[0], nullptr, 0, &kp);
    }
    if (e == cudaSuccess)
        e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        if (graph)
            cudaGraphDestroy(graph);
        return cuda_status(e, "building the iteration graph");
    }
    st.graph = graph;
    st.exec = exec;
    st.ready = true;
    return PR_OK;
}

template <typename T>
pr_status run_typed(pr_graph *g, double d, double tol, int32_t max_iter, void *ranks_out,
                    const void *x_init, int32_t *iters_out, double *l1_out, cudaStream_t s)
{
    pr_status r = prepare<T>(g);
    if (r != PR_OK)
        return r;
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    IterArgs<T> args = make_args<T>(g);
    const size_t bytes = (size_t)g->n * sizeof(T);
    cudaError_t e = cudaSuccess;

    const T *xi = nullptr;
    if (x_init) {
        if (is_device_pointer(x_init)) {
            xi = (const T *)x_init;
        } else {
            e = cudaMemcpyAsync(st.stage, x_init, bytes, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess)
                return cuda_status(e, "copying x_init");
            xi = (const T *)st.stage;
        }
    }
    const bool out_dev = is_device_pointer(ranks_out);
    T *out = out_dev ? (T *)ranks_out : (T *)st.stage;

    e = cudaEventRecord(g->ev[0], s);
    if (e == cudaSuccess) {
        k_init<T><<<st.init_grid, kBlock, 0, s>>>(args, xi, d, tol, max_iter);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(g->ev[1], s);
    if (e == cudaSuccess)
        e = cudaGraphLaunch(st.exec, s);
    if (e == cudaSuccess)
        e = cudaEventRecord(g->ev[2], s);
    if (e == cudaSuccess) {
        const int og = (int)((g->n + kBlock - 1) / kBlock < 8 * g->num_sms
                                 ? (g->n + kBlock - 1) / kBlock : 8 * g->num_sms);
        k_output<T><<<og, kBlock, 0, s>>>(args, out);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && !out_dev)
        e = cudaMemcpyAsync(ranks_out, st.stage, bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(g->h_scal, g->scal, sizeof(Scalars), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_status(e, "pr_run");

    const Scalars hs = *g->h_scal;
    float loop_ms = 0.f, total_ms = 0.f;
    cudaEventElapsedTime(&loop_ms, g->ev[1], g->ev[2]);
    cudaEventElapsedTime(&total_ms, g->ev[0], g->ev[2]);
    g->last.iterations = hs.it;
    g->last.converged = hs.converged;
    g->last.l1 = hs.l1;
    g->last.dangling_mass = hs.dmass;
    g->last.loop_ms = loop_ms;
    g->last.total_ms = total_ms;
    g->last.launches = hs.it + 2;
    if (iters_out)
        *iters_out = hs.it;
    if (l1_out)
        *l1_out = hs.l1;
    if (tol > 0.0 && !hs.converged)
        return PR_NOT_CONVERGED;
    return PR_OK;
}

}  // namespace

pr_status run(pr_graph *g, double d, double tol, int32_t max_iter, int dtype, void *ranks_out,
              const void *x_init, int32_t *iters_out, double *l1_out, cudaStream_t s)
{
    if (dtype == PR_F64)
        return run_typed<double>(g, d, tol, max_iter, ranks_out, x_init, iters_out, l1_out, s);
    return run_typed<float>(g, d, tol, max_iter, ranks_out, x_init, iters_out, l1_out, s);
}

void release_dtype_state(pr_graph *g)
{
    for (auto &st : g->st) {
        if (st.exec)
            cudaGraphExecDestroy(st.exec);
        if (st.graph)
            cudaGraphDestroy(st.graph);
        st.exec = nullptr;
        st.graph = nullptr;
        st.ready = false;
    }
}

}  // namespace prk
