// One-time preprocessing on the device: out-edge CSR -> in-edge CSR, and the
// split of in-rows into in-degree classes.
//
// The transpose is the counting sort of "Day 40 - PageRank on a real graph in
// CUDA" (section "One iteration, three shapes of work": a histogram, a prefix
// sum and a scatter), done on the GPU:
//   1. k_outdeg     out-degrees, row_ptr validation, dangling count
//   2. k_expand     source id of every edge, col_idx validation, and the
//                   in-degree histogram (global atomics)
//   3. k_scan_excl  in_ptr = exclusive prefix sum of the in-degrees, one pass
//                   with decoupled look-back between tiles
//   4. the stable scatter, as a least-significant-digit radix sort of the
//      edges by destination with 8-bit digits: each pass is itself a counting
//      sort over 256 bins (per-tile shared-memory digit counts, decoupled
//      look-back across tiles, rank-preserving scatter), so the edges into
//      one vertex keep the order of the out-edge CSR, i.e. ascending sources.
//      A 2^24-vertex graph needs 3 passes; a single counting sort over n bins
//      would need n-entry histograms that no shared memory holds.
// Then k_scan_excl over class flags and k_compact build the row lists of the
// four in-degree classes (gpu-graph-study, "PageRank T4": <= 32, 33..1024,
// > 1024; in-degree 0 gathers nothing), and the rows above 1024 are cut into
// fixed-size edge chunks.
//
// Every wait in this file (the look-back) is bounded: after kSpinLimit polls
// it sets kErrTimeout in the error word and moves on, so no launch can hang.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pr_internal.cuh"

namespace prk {
namespace {

constexpr unsigned long long kFlagA = 1ull << 62;   // tile aggregate published
constexpr unsigned long long kFlagP = 2ull << 62;   // inclusive prefix published
constexpr unsigned long long kValueMask = (1ull << 62) - 1;
constexpr int kSpinLimit = 1 << 20;

__device__ __forceinline__ unsigned long long load_desc(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void store_desc(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Waits (bounded) for a published descriptor; returns 0 on timeout.
__device__ __forceinline__ unsigned long long wait_desc(const unsigned long long *p, unsigned *err)
{
    unsigned long long v = load_desc(p);
    int spins = 0;
    unsigned ns = 32;
    while ((v >> 62) == 0) {
        if (++spins > kSpinLimit) {
            atomicOr(err, kErrTimeout);
            return 0;
        }
        __nanosleep(ns);
        if (ns < 1024)
            ns <<= 1;
        v = load_desc(p);
    }
    return v;
}

// Sum of everything published before `tile` for one descriptor column (walks
// back until an inclusive prefix is found). Tile 0 always publishes kFlagP.
__device__ long long look_back(const unsigned long long *desc, int64_t tile, int64_t stride,
                               unsigned *err)
{
    long long prefix = 0;
    for (int64_t p = tile - 1; p >= 0; --p) {
        unsigned long long v = wait_desc(desc + p * stride, err);
        if (v == 0)
            break;  // timed out: error already flagged
        prefix += (long long)(v & kValueMask);
        if ((v >> 62) == 2)
            break;
    }
    return prefix;
}

// ---------------------------------------------------------------- step 1 --

__global__ void k_outdeg(int64_t n, const int64_t *__restrict__ row_ptr,
                         int32_t *__restrict__ deg_out, unsigned long long *n_dangling,
                         unsigned *err)
{
    unsigned dangling = 0;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < n;
         u += (int64_t)gridDim.x * blockDim.x) {
        int64_t len = row_ptr[u + 1] - row_ptr[u];
        if (len < 0) {
            atomicOr(err, kErrRowPtr);
            len = 0;
        }
        if (len > INT32_MAX)
            len = INT32_MAX;
        deg_out[u] = (int32_t)len;
        dangling += (len == 0);
    }
    for (int o = 16; o > 0; o >>= 1)
        dangling += __shfl_xor_sync(0xffffffffu, dangling, o);
    if ((threadIdx.x & 31) == 0 && dangling)
        atomicAdd(n_dangling, (unsigned long long)dangling);
}

// ---------------------------------------------------------------- step 2 --

// First index i in [0, len) with a[i] > key (len if none).
__device__ __forceinline__ int64_t upper_bound_i64(const int64_t *a, int64_t len, int64_t key)
{
    int64_t lo = 0, hi = len;
    while (lo < hi) {
        int64_t mid = (lo + hi) >> 1;
        if (a[mid] <= key)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

constexpr int kExpandItems = 8;

// Source of every edge, range check of the targets and the in-degree
// histogram. Requires row_ptr[0] == 0 and row_ptr[n] == m (checked on the
// host before launch), which keeps every index below in range even when
// row_ptr is not monotone (that case is flagged by k_outdeg and the build
// stops before the sources are used).
__global__ void __launch_bounds__(kBlock)
k_expand(int64_t n, int64_t m, const int64_t *__restrict__ row_ptr,
         const int32_t *__restrict__ col, int32_t *__restrict__ src,
         int32_t *__restrict__ in_deg, unsigned *err)
{
    __shared__ int64_t s_lo, s_hi;
    const int64_t tile = (int64_t)kBlock * kExpandItems;
    for (int64_t j0 = blockIdx.x * tile; j0 < m; j0 += (int64_t)gridDim.x * tile) {
        const int64_t j1 = min(j0 + tile, m);
        if (threadIdx.x == 0) {
            s_lo = upper_bound_i64(row_ptr, n + 1, j0) - 1;
            s_hi = upper_bound_i64(row_ptr, n + 1, j1 - 1);
        }
        __syncthreads();
        const int64_t lo0 = s_lo, hi0 = s_hi;
#pragma unroll
        for (int k = 0; k < kExpandItems; ++k) {
            const int64_t j = j0 + (int64_t)k * kBlock + threadIdx.x;
            if (j < j1) {
                int64_t lo = lo0, hi = hi0;   // row_ptr[lo] <= j < row_ptr[hi]
                while (hi - lo > 1) {
                    int64_t mid = (lo + hi) >> 1;
                    if (row_ptr[mid] <= j)
                        lo = mid;
                    else
                        hi = mid;
                }
                src[j] = (int32_t)lo;
                const int32_t v = col[j];
                if (v < 0 || (int64_t)v >= n)
                    atomicOr(err, kErrColIdx);
                else
                    atomicAdd(&in_deg[v], 1);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- step 3 --

constexpr int kScanItems = 16;
constexpr int kScanTile = kBlock * kScanItems;

struct LoadCount {   // element i of an int32 array
    const int32_t *p;
    __device__ int32_t operator()(int64_t i) const { return p[i]; }
};

__device__ __forceinline__ int row_class(int32_t deg)
{
    return deg == 0 ? kClassZero : deg <= kThreadMax ? kClassThread
                                   : deg <= kWarpMax ? kClassWarp : kClassCta;
}

struct LoadClassFlag {   // 1 if row i is in class cls
    const int32_t *in_ptr;
    int cls;
    __device__ int32_t operator()(int64_t i) const
    {
        return row_class(in_ptr[i + 1] - in_ptr[i]) == cls ? 1 : 0;
    }
};

struct LoadChunkCount {   // number of edge chunks of CTA row i
    const int32_t *in_ptr;
    const int32_t *rows_c;
    __device__ int32_t operator()(int64_t i) const
    {
        const int32_t v = rows_c[i];
        const int64_t deg = (int64_t)in_ptr[v + 1] - in_ptr[v];
        return (int32_t)((deg + kChunkEdges - 1) / kChunkEdges);
    }
};

// out[i] = sum of load(k) for k < i, for i in [0, count]; out[count] is the
// total. Single pass: tiles are taken in launch order from a counter and each
// finds its prefix by decoupled look-back over its predecessors' descriptors.
template <class Load>
__global__ void __launch_bounds__(kBlock)
k_scan_excl(Load load, int32_t *__restrict__ out, int64_t count,
            unsigned long long *desc, unsigned *tile_counter, unsigned *err)
{
    __shared__ int32_t s_items[kScanTile];
    __shared__ long long s_warp[kBlock / 32];
    __shared__ long long s_prefix;
    __shared__ unsigned s_tile;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        s_tile = atomicAdd(tile_counter, 1u);
    __syncthreads();
    const int64_t tile = s_tile;
    const int64_t base = tile * kScanTile;

    for (int k = 0; k < kScanItems; ++k) {
        const int64_t i = base + (int64_t)k * kBlock + tid;
        s_items[k * kBlock + tid] = (i < count) ? load(i) : 0;
    }
    __syncthreads();

    int32_t v[kScanItems];
    long long local = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = s_items[tid * kScanItems + k];
        local += v[k];
    }
    // block-wide exclusive scan of the per-thread sums
    long long incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        s_warp[warp] = incl;
    __syncthreads();
    long long warp_base = 0, total = 0;
    for (int w = 0; w < kBlock / 32; ++w) {
        if (w < warp)
            warp_base += s_warp[w];
        total += s_warp[w];
    }
    const long long thread_excl = warp_base + incl - local;

    if (tid == 0) {
        long long prefix = 0;
        if (tile == 0) {
            store_desc(desc, kFlagP | (unsigned long long)total);
        } else {
            store_desc(desc + tile, kFlagA | (unsigned long long)total);
            prefix = look_back(desc, tile, 1, err);
            store_desc(desc + tile, kFlagP | (unsigned long long)(prefix + total));
        }
        s_prefix = prefix;
        if (base + kScanTile >= count)   // the last tile writes the total
            out[count] = (int32_t)(prefix + total);
    }
    __syncthreads();
    long long run = s_prefix + thread_excl;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        s_items[tid * kScanItems + k] = (int32_t)run;
        run += v[k];
    }
    __syncthreads();
    for (int k = 0; k < kScanItems; ++k) {
        const int64_t i = base + (int64_t)k * kBlock + tid;
        if (i < count)
            out[i] = s_items[k * kBlock + tid];
    }
}

// ---------------------------------------------------------------- step 4 --

constexpr int kRadixBits = 8;
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kRadixItems = 16;
constexpr int kRadixTile = kBlock * kRadixItems;
constexpr int kMaxPasses = 4;

// Digit counts of every pass at once (one read of the keys).
__global__ void __launch_bounds__(kBlock)
k_digit_hist(const int32_t *__restrict__ keys, int64_t count, int passes,
             unsigned *__restrict__ hist)
{
    __shared__ unsigned s_h[kMaxPasses][kRadixBins];
    for (int i = threadIdx.x; i < kMaxPasses * kRadixBins; i += kBlock)
        (&s_h[0][0])[i] = 0;
    __syncthreads();
    for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * kBlock) {
        const unsigned k = (unsigned)keys[i];
        for (int p = 0; p < passes; ++p)
            atomicAdd(&s_h[p][(k >> (p * kRadixBits)) & (kRadixBins - 1)], 1u);
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p) {
        const unsigned c = s_h[p][threadIdx.x];
        if (c)
            atomicAdd(&hist[p * kRadixBins + threadIdx.x], c);
    }
}

// Exclusive scan of each pass's 256 digit counts: where each digit's bucket starts.
__global__ void k_digit_base(const unsigned *__restrict__ hist, int passes,
                             unsigned *__restrict__ base)
{
    __shared__ unsigned s[kRadixBins];
    for (int p = 0; p < passes; ++p) {
        s[threadIdx.x] = hist[p * kRadixBins + threadIdx.x];
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned run = 0;
            for (int d = 0; d < kRadixBins; ++d) {
                unsigned c = s[d];
                s[d] = run;
                run += c;
            }
        }
        __syncthreads();
        base[p * kRadixBins + threadIdx.x] = s[threadIdx.x];
        __syncthreads();
    }
}

// One stable counting-sort pass over digit (key >> shift) & 255.
// Tile layout: warp w owns tile positions [w*32*ITEMS, (w+1)*32*ITEMS) and
// walks them in 32-key rounds, so "earlier round, then lower lane" is input
// order. Within a warp, __match_any_sync groups equal digits of a round and a
// per-warp shared counter carries the running count across rounds; per-warp
// counts are then scanned across warps, and across tiles by look-back (one
// thread per digit).
template <bool kWriteKeys>
__global__ void __launch_bounds__(kBlock)
k_radix_pass(const int32_t *__restrict__ keys_in, const int32_t *__restrict__ vals_in,
             int32_t *__restrict__ keys_out, int32_t *__restrict__ vals_out, int64_t count,
             int shift, const unsigned *__restrict__ digit_base, unsigned long long *desc,
             unsigned *tile_counter, unsigned *err)
{
    constexpr int kWarps = kBlock / 32;
    constexpr int kWarpSpan = 32 * kRadixItems;
    __shared__ unsigned s_wh[kWarps][kRadixBins];
    __shared__ unsigned s_base[kRadixBins];
    __shared__ unsigned s_tile;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        s_tile = atomicAdd(tile_counter, 1u);
    for (int w = 0; w < kWarps; ++w)
        s_wh[w][tid] = 0;
    __syncthreads();
    const int64_t tile = s_tile;
    const int64_t base = tile * kRadixTile + (int64_t)warp * kWarpSpan;

    int32_t key[kRadixItems], val[kRadixItems];
    unsigned rank[kRadixItems], dig[kRadixItems];
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        const int64_t i = base + r * 32 + lane;
        const bool ok = i < count;
        key[r] = ok ? keys_in[i] : 0;
        val[r] = ok ? vals_in[i] : 0;
        dig[r] = ok ? (((unsigned)key[r] >> shift) & (kRadixBins - 1)) : kRadixBins;
    }
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        const unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        const bool ok = dig[r] < kRadixBins;
        const unsigned before = ok ? s_wh[warp][dig[r]] : 0u;
        __syncwarp();
        rank[r] = before + __popc(peers & below);
        if (ok && (peers >> lane) == 1u)   // highest lane of the group
            s_wh[warp][dig[r]] = before + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // thread tid owns digit tid: offsets of each warp, the tile's count, and
    // the count of all earlier tiles
    unsigned tot = 0;
    for (int w = 0; w < kWarps; ++w) {
        const unsigned c = s_wh[w][tid];
        s_wh[w][tid] = tot;
        tot += c;
    }
    long long prefix = 0;
    unsigned long long *my = desc + tile * kRadixBins + tid;
    if (tile == 0) {
        store_desc(my, kFlagP | tot);
    } else {
        store_desc(my, kFlagA | tot);
        prefix = look_back(desc + tid, tile, kRadixBins, err);
        store_desc(my, kFlagP | (unsigned long long)(prefix + tot));
    }
    s_base[tid] = digit_base[tid] + (unsigned)prefix;
    __syncthreads();

#pragma unroll
    for (int r = 0; r < kRadixItems; ++r) {
        if (dig[r] < kRadixBins) {
            const unsigned pos = s_base[dig[r]] + s_wh[warp][dig[r]] + rank[r];
            if ((int64_t)pos >= count)   // only reachable after a look-back timeout
                continue;
            vals_out[pos] = val[r];
            if (kWriteKeys)
                keys_out[pos] = key[r];
        }
    }
}

// ------------------------------------------------------------ classes ---

struct ClassLists {
    const int32_t *pos[4];   // exclusive scans of the class flags
    int32_t *rows[4];        // compacted row ids
    int64_t count[4];        // list lengths
};

__global__ void k_compact(int64_t n, const int32_t *__restrict__ in_ptr, ClassLists L)
{
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int c = row_class(in_ptr[v + 1] - in_ptr[v]);
        const int32_t p = L.pos[c][v];
        if (p >= 0 && p < L.count[c])
            L.rows[c][p] = (int32_t)v;
    }
}

__global__ void k_fill_chunks(int64_t n_c, int64_t n_chunks, const int32_t *__restrict__ chunk_first,
                              int32_t *__restrict__ chunk_row)
{
    for (int64_t r = blockIdx.x; r < n_c; r += gridDim.x)
        for (int32_t c = chunk_first[r] + threadIdx.x; c < chunk_first[r + 1]; c += blockDim.x)
            if (c >= 0 && c < n_chunks)
                chunk_row[c] = (int32_t)r;
}

// Edges per class (for reporting): sum of in-degrees over each list.
__global__ void k_class_edges(const int32_t *__restrict__ in_ptr, const int32_t *__restrict__ rows,
                              int64_t count, unsigned long long *out)
{
    unsigned long long s = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = rows[i];
        s += (unsigned long long)(in_ptr[v + 1] - in_ptr[v]);
    }
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0 && s)
        atomicAdd(out, s);
}

// ------------------------------------------------------------- host side --

int grid_for(int64_t items, int per_block, int cap)
{
    int64_t g = (items + per_block - 1) / per_block;
    if (g < 1)
        g = 1;
    if (g > cap)
        g = cap;
    return (int)g;
}

// Scratch of one build, released when the build returns.
struct Scratch {
    std::vector<void *> ptrs;
    ~Scratch()
    {
        for (void *p : ptrs)
            cudaFree(p);
    }
    pr_status alloc(void **p, size_t bytes)
    {
        if (bytes == 0)
            bytes = 16;
        cudaError_t e = cudaMalloc(p, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return set_error(e == cudaErrorMemoryAllocation ? PR_ERR_OOM : PR_ERR_CUDA,
                             "cudaMalloc of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
        }
        ptrs.push_back(*p);
        return PR_OK;
    }
};

template <class Load>
pr_status launch_scan(Load load, int32_t *out, int64_t count, unsigned long long *desc,
                      unsigned *counter, unsigned *err, int32_t *launches, cudaStream_t s)
{
    if (count == 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, sizeof(int32_t), s);
        return e == cudaSuccess ? PR_OK : cuda_status(e, "scan memset");
    }
    const int64_t tiles = (count + kScanTile - 1) / kScanTile;
    cudaError_t e = cudaMemsetAsync(desc, 0, (size_t)tiles * sizeof(unsigned long long), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(counter, 0, sizeof(unsigned), s);
    if (e != cudaSuccess)
        return cuda_status(e, "scan state reset");
    k_scan_excl<Load><<<(unsigned)tiles, kBlock, 0, s>>>(load, out, count, desc, counter, err);
    ++*launches;
    e = cudaGetLastError();
    return e == cudaSuccess ? PR_OK : cuda_status(e, "k_scan_excl launch");
}

pr_status read_err(pr_graph *g, cudaStream_t s, unsigned *out)
{
    cudaError_t e = cudaMemcpyAsync(out, g->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? PR_OK : cuda_status(e, "reading the error word");
}

}  // namespace

pr_status build_graph(pr_graph *g, const int64_t *d_row_ptr, const int32_t *d_col, cudaStream_t s)
{
    const int64_t n = g->n, m = g->m;
    const int cap = g->num_sms * 32;
    pr_status st;
    cudaError_t e;
    Scratch tmp;

#define PRK_TRY(expr)             \
    do {                          \
        st = (expr);              \
        if (st != PR_OK)          \
            return st;            \
    } while (0)
#define PRK_CUDA(expr, what)                         \
    do {                                             \
        e = (expr);                                  \
        if (e != cudaSuccess)                        \
            return cuda_status(e, what);             \
    } while (0)

    // handle-owned buffers
    PRK_TRY(graph_alloc(g, (void **)&g->in_ptr, (size_t)(n + 1) * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->in_col, (size_t)(m + 4) * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->deg_out, (size_t)n * sizeof(int32_t)));

    // scratch
    int32_t *src = nullptr, *in_deg = nullptr;
    unsigned long long *counters = nullptr;   // [0] = dangling, [1..3] = class edges
    unsigned *tile_counter = nullptr, *hist = nullptr, *dbase = nullptr;
    unsigned long long *desc = nullptr;
    PRK_TRY(tmp.alloc((void **)&src, (size_t)m * sizeof(int32_t)));
    PRK_TRY(tmp.alloc((void **)&in_deg, (size_t)n * sizeof(int32_t)));
    PRK_TRY(tmp.alloc((void **)&counters, 8 * sizeof(unsigned long long)));
    PRK_TRY(tmp.alloc((void **)&tile_counter, sizeof(unsigned)));
    PRK_TRY(tmp.alloc((void **)&hist, 2 * kMaxPasses * kRadixBins * sizeof(unsigned)));
    dbase = hist + kMaxPasses * kRadixBins;

    const int64_t scan_tiles = (n + 1 + kScanTile - 1) / kScanTile;
    const int64_t radix_tiles = (m + kRadixTile - 1) / kRadixTile;
    const int64_t desc_words = scan_tiles > radix_tiles * kRadixBins ? scan_tiles
                                                                     : radix_tiles * kRadixBins;
    PRK_TRY(tmp.alloc((void **)&desc, (size_t)(desc_words + 1) * sizeof(unsigned long long)));

    PRK_CUDA(cudaMemsetAsync(g->err, 0, sizeof(unsigned), s), "memset");
    PRK_CUDA(cudaMemsetAsync(in_deg, 0, (size_t)n * sizeof(int32_t), s), "memset");
    PRK_CUDA(cudaMemsetAsync(counters, 0, 8 * sizeof(unsigned long long), s), "memset");
    PRK_CUDA(cudaMemsetAsync(hist, 0, kMaxPasses * kRadixBins * sizeof(unsigned), s), "memset");

    // 1 + 2: degrees, sources, validation, in-degree histogram
    k_outdeg<<<grid_for(n, kBlock, cap), kBlock, 0, s>>>(n, d_row_ptr, g->deg_out, counters, g->err);
    ++g->build_launches;
    if (m > 0)
        k_expand<<<grid_for(m, kBlock * kExpandItems, cap), kBlock, 0, s>>>(
            n, m, d_row_ptr, d_col, src, in_deg, g->err);
    g->build_launches += (m > 0);
    PRK_CUDA(cudaGetLastError(), "validation launch");
    unsigned herr = 0;
    PRK_TRY(read_err(g, s, &herr));
    if (herr & kErrRowPtr)
        return set_error(PR_ERR_INVALID_GRAPH, "row_ptr is not non-decreasing");
    if (herr & kErrColIdx)
        return set_error(PR_ERR_INVALID_GRAPH, "col_idx has an entry outside [0, n)");

    // a look-back that gave up leaves garbage offsets: stop before they are used
    auto check_timeout = [&]() -> pr_status {
        unsigned w = 0;
        pr_status r = read_err(g, s, &w);
        if (r != PR_OK)
            return r;
        if (w & kErrTimeout)
            return set_error(PR_ERR_TIMEOUT, "a look-back wait in the transpose gave up");
        return PR_OK;
    };

    // 3: in_ptr = exclusive scan of the in-degrees (n + 1 outputs)
    PRK_TRY(launch_scan(LoadCount{in_deg}, g->in_ptr, n, desc, tile_counter, g->err, &g->build_launches, s));

    // 4: stable scatter by destination (LSD radix over 8-bit digits)
    int bits = 0;
    while (bits < 31 && ((int64_t)1 << bits) < n)
        ++bits;
    const int passes = (bits + kRadixBits - 1) / kRadixBits;
    if (m > 0 && passes == 0) {
        PRK_CUDA(cudaMemcpyAsync(g->in_col, src, (size_t)m * sizeof(int32_t),
                                 cudaMemcpyDeviceToDevice, s), "copy");
    } else if (m > 0) {
        int32_t *kb[2] = {nullptr, nullptr}, *vb[2] = {nullptr, nullptr};
        for (int i = 0; i < 2 && i < passes - 1; ++i) {
            PRK_TRY(tmp.alloc((void **)&kb[i], (size_t)m * sizeof(int32_t)));
            PRK_TRY(tmp.alloc((void **)&vb[i], (size_t)m * sizeof(int32_t)));
        }
        k_digit_hist<<<grid_for(m, kBlock * 16, cap), kBlock, 0, s>>>(d_col, m, passes, hist);
        k_digit_base<<<1, kRadixBins, 0, s>>>(hist, passes, dbase);
        g->build_launches += 2;
        PRK_CUDA(cudaGetLastError(), "digit histogram launch");
        for (int p = 0; p < passes; ++p) {
            const int32_t *kin = p == 0 ? d_col : kb[(p - 1) & 1];
            const int32_t *vin = p == 0 ? src : vb[(p - 1) & 1];
            const bool last = p == passes - 1;
            int32_t *vout = last ? g->in_col : vb[p & 1];
            int32_t *kout = last ? nullptr : kb[p & 1];
            PRK_CUDA(cudaMemsetAsync(desc, 0, (size_t)radix_tiles * kRadixBins * sizeof(unsigned long long), s),
                     "memset");
            PRK_CUDA(cudaMemsetAsync(tile_counter, 0, sizeof(unsigned), s), "memset");
            if (last)
                k_radix_pass<false><<<(unsigned)radix_tiles, kBlock, 0, s>>>(
                    kin, vin, kout, vout, m, p * kRadixBits, dbase + p * kRadixBins, desc,
                    tile_counter, g->err);
            else
                k_radix_pass<true><<<(unsigned)radix_tiles, kBlock, 0, s>>>(
                    kin, vin, kout, vout, m, p * kRadixBits, dbase + p * kRadixBins, desc,
                    tile_counter, g->err);
            PRK_CUDA(cudaGetLastError(), "k_radix_pass launch");
            ++g->build_launches;
        }
    }

    PRK_TRY(check_timeout());

    // classes: flags -> exclusive scans -> compaction
    int32_t *pos[4];
    for (int c = 0; c < 4; ++c) {
        PRK_TRY(tmp.alloc((void **)&pos[c], (size_t)(n + 1) * sizeof(int32_t)));
        PRK_TRY(launch_scan(LoadClassFlag{g->in_ptr, c}, pos[c], n, desc, tile_counter, g->err, &g->build_launches, s));
    }
    int32_t h_cnt[4];
    for (int c = 0; c < 4; ++c)
        PRK_CUDA(cudaMemcpyAsync(&h_cnt[c], pos[c] + n, sizeof(int32_t), cudaMemcpyDeviceToHost, s),
                 "class counts");
    PRK_TRY(check_timeout());
    g->n_z = h_cnt[0];
    g->n_t = h_cnt[1];
    g->n_w = h_cnt[2];
    g->n_c = h_cnt[3];
    PRK_TRY(graph_alloc(g, (void **)&g->rows_z, (size_t)g->n_z * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->rows_t, (size_t)g->n_t * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->rows_w, (size_t)g->n_w * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->rows_c, (size_t)g->n_c * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->chunk_first, (size_t)(g->n_c + 1) * sizeof(int32_t)));
    PRK_TRY(graph_alloc(g, (void **)&g->hub_arrivals, (size_t)(g->n_c + 1) * sizeof(uint32_t)));
    PRK_CUDA(cudaMemsetAsync(g->hub_arrivals, 0, (size_t)(g->n_c + 1) * sizeof(uint32_t), s), "memset");
    ClassLists lists;
    int32_t *rows[4] = {g->rows_z, g->rows_t, g->rows_w, g->rows_c};
    for (int c = 0; c < 4; ++c) {
        lists.pos[c] = pos[c];
        lists.rows[c] = rows[c];
        lists.count[c] = h_cnt[c];
    }
    k_compact<<<grid_for(n, kBlock, cap), kBlock, 0, s>>>(n, g->in_ptr, lists);
    ++g->build_launches;
    PRK_CUDA(cudaGetLastError(), "k_compact launch");

    // CTA rows -> chunks
    PRK_TRY(launch_scan(LoadChunkCount{g->in_ptr, g->rows_c}, g->chunk_first, g->n_c, desc,
                        tile_counter, g->err, &g->build_launches, s));
    int32_t h_chunks = 0;
    PRK_CUDA(cudaMemcpyAsync(&h_chunks, g->chunk_first + g->n_c, sizeof(int32_t),
                             cudaMemcpyDeviceToHost, s), "chunk count");
    PRK_TRY(check_timeout());
    g->n_chunks = h_chunks;
    PRK_TRY(graph_alloc(g, (void **)&g->chunk_row, (size_t)g->n_chunks * sizeof(int32_t)));
    g->build_launches += (g->n_c > 0);
    if (g->n_c > 0)
        k_fill_chunks<<<grid_for(g->n_c, 1, cap), kBlock, 0, s>>>(g->n_c, g->n_chunks, g->chunk_first,
                                                                   g->chunk_row);

    // class edge counts (reporting only)
    g->build_launches += (g->n_t > 0) + (g->n_w > 0) + (g->n_c > 0);
    if (g->n_t)
        k_class_edges<<<grid_for(g->n_t, kBlock, cap), kBlock, 0, s>>>(g->in_ptr, g->rows_t, g->n_t, counters + 1);
    if (g->n_w)
        k_class_edges<<<grid_for(g->n_w, kBlock, cap), kBlock, 0, s>>>(g->in_ptr, g->rows_w, g->n_w, counters + 2);
    if (g->n_c)
        k_class_edges<<<grid_for(g->n_c, kBlock, cap), kBlock, 0, s>>>(g->in_ptr, g->rows_c, g->n_c, counters + 3);
    PRK_CUDA(cudaGetLastError(), "class launch");
    unsigned long long h_counters[4];
    PRK_CUDA(cudaMemcpyAsync(h_counters, counters, sizeof(h_counters), cudaMemcpyDeviceToHost, s),
             "counters");
    PRK_TRY(read_err(g, s, &herr));
    if (herr & kErrTimeout)
        return set_error(PR_ERR_TIMEOUT, "a look-back wait in the transpose gave up");
    g->n_dangling = (int64_t)h_counters[0];
    g->e_t = (int64_t)h_counters[1];
    g->e_w = (int64_t)h_counters[2];
    g->e_c = (int64_t)h_counters[3];
    return PR_OK;
#undef PRK_TRY
#undef PRK_CUDA
}

}  // namespace prk
