// One-time preprocessing on the device: out-edge CSR -> in-edge CSR, the split
// of in-rows into in-degree classes, and the class-major work layout the
// iteration runs on.
//
// The transpose is the counting sort of "Day 40 - PageRank on a real graph in
// CUDA" (section "One iteration, three shapes of work": a histogram, a prefix
// sum and a scatter), done on the GPU:
//   1. k_outdeg      out-degrees, row_ptr validation, dangling count
//   2. + 3. the stable scatter, as a least-significant-digit radix sort of
//      the edges by destination with 8-bit digits. Each pass is itself a
//      counting sort over 256 bins in reduce-then-scan form: k_radix_upsweep
//      counts the digits of every tile (the first one also checks col_idx),
//      one exclusive scan of those counts in digit-major order gives every
//      (digit, tile) its output position, and k_radix_pass ranks each tile
//      with per-warp shared-memory counters and scatters it, staged through
//      shared memory so that the stores are coalesced. No tile waits for
//      another. Stable passes keep the edges into one vertex in out-edge CSR
//      order, i.e. with ascending sources. The first pass's values, the
//      edges' sources, come from k_edge_sources (row_ptr spread over the
//      edges); the last pass also produces the in-degree histogram, one
//      atomic per run of equal destinations in a tile. A 2^24-vertex graph
//      takes 3 passes: one counting sort over n bins would need n-entry
//      histograms that no shared memory holds.
//   4. k_scan_excl   in_ptr = exclusive prefix sum of the in-degrees, in one
//                    pass with decoupled look-back between tiles
//
// Classes (gpu-graph-study, "PageRank T4": in-degree > 1024, 33..1024, 1..32,
// and 0) give the class-major work order: one more stable counting-sort pass
// over the vertices, keyed by class (CTA rows first, then warp, thread and
// zero rows) and, inside a class, by half-octave bucket of the out-degree,
// largest first; thread-class rows by padded length first, longest first,
// then by a coarse out-degree bucket (ties by id; see k_order_keys).
//
// Work layout. The iteration does not run on the in-edge CSR above (which is
// kept, bit for bit, for pr_get_in_csr) but on the same graph relabelled by
// that class-major order: vertex v becomes perm[v], row i of the work CSR
// (w_ptr, w_col) is the in-row of order[i] with every source u replaced by
// perm[u], padded with kPadSource entries to a multiple of 4. Each class is then a contiguous range of rows and of edges, the
// per-row state is read and written in order, and, since the order leads with
// in-degree hubs sorted by out-degree, the most gathered values of skewed
// graphs sit together at the start of the state vector (where the iteration
// keeps a copy in shared memory). Rows above 1024 in-edges are cut into
// fixed-size edge chunks.
//
// Every wait in this file (the scans' look-backs) is bounded: after
// kSpinLimit polls it sets kErrTimeout in the error word and moves on, the
// host stops the build at the next check, and every store whose offset came
// out of a scan is range-checked, so no launch can hang or write out of
// bounds.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "pr_internal.cuh"

namespace prk {
namespace {

constexpr unsigned long long kFlagA = 1ull << 62;   // tile aggregate published
constexpr unsigned long long kFlagP = 2ull << 62;   // inclusive prefix published
constexpr unsigned long long kValueMask = (1ull << 62) - 1;
constexpr int kSpinLimit = 1 << 22;

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

// Waits (bounded: at most spin_limit polls) for a published descriptor;
// returns 0 on timeout. Polls back to back first (the predecessor is usually
// moments away), then backs off.
__device__ __forceinline__ unsigned long long wait_desc(const unsigned long long *p, unsigned *err,
                                                        int spin_limit)
{
    unsigned long long v = load_desc(p);
    int spins = 0;
    while ((v >> 62) == 0) {
        if (++spins > spin_limit) {
            atomicOr(err, kErrTimeout);
            return 0;
        }
        if (spins > 64)
            __nanosleep(spins > 4096 ? 256 : 32);
        v = load_desc(p);
    }
    return v;
}

// Sum of everything published before `tile` in one descriptor column (walks
// back until an inclusive prefix is found). Tile 0 always publishes kFlagP.
// Four predecessors are read per step, so a walk over aggregate-only tiles
// costs a quarter of the round trips; a descriptor still unpublished is
// waited for (bounded) before it is used.
__device__ long long look_back(const unsigned long long *desc, int64_t tile, int64_t stride,
                               unsigned *err, int spin_limit)
{
    long long prefix = 0;
    int64_t p = tile - 1;
    while (p >= 0) {
        unsigned long long v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = (p - k >= 0) ? load_desc(desc + (p - k) * stride) : 0ull;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (p - k < 0)
                return prefix;
            if ((v[k] >> 62) == 0) {
                v[k] = wait_desc(desc + (p - k) * stride, err, spin_limit);
                if (v[k] == 0)
                    return prefix;   // timed out: error already flagged
            }
            prefix += (long long)(v[k] & kValueMask);
            if ((v[k] >> 62) == 2)
                return prefix;
        }
        p -= 4;
    }
    return prefix;
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += t;
    }
    return v;
}

// First index i in [0, len) with a[i] > key (len if none).
template <typename I>
__device__ __forceinline__ int64_t upper_bound(const I *a, int64_t len, int64_t key)
{
    int64_t lo = 0, hi = len;
    while (lo < hi) {
        int64_t mid = (lo + hi) >> 1;
        if ((int64_t)a[mid] <= key)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Advances row r (off[r] <= i) to the row holding offset i: galloping (1, 2,
// 4, ... rows) then bisection, so runs of empty rows cost O(log gap).
// `last` is the index of the final offset; requires off[last] > i, so no
// index beyond `last` is read.
template <typename I>
__device__ __forceinline__ int64_t advance_row(const I *off, int64_t r, int64_t i, int64_t last)
{
    if ((int64_t)off[r + 1] > i)
        return r;
    int64_t lo = r + 1, step = 1;   // off[lo] <= i
    int64_t hi = min(lo + step, last);
    while ((int64_t)off[hi] <= i) {
        lo = hi;
        step <<= 1;
        hi = min(lo + step, last);
    }
    while (hi - lo > 1) {   // off[lo] <= i < off[hi]
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)off[mid] <= i)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Row of offset i in a CSR offset array: the r with off[r] <= i < off[r+1],
// searched in (lo, hi) where off[lo] <= i < off[hi].
template <typename I>
__device__ __forceinline__ int64_t row_of(const I *off, int64_t lo, int64_t hi, int64_t i)
{
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)off[mid] <= i)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
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

constexpr int kRadixBits = 8;
constexpr int kRadixBins = 1 << kRadixBits;
// Keys per thread of a counting-sort tile (256 threads). Measured on the
// transpose of RMAT-24 / ER-24 / RMAT-22 with four CTAs per SM: 8 keys 9.25 /
// 10.95 / 2.68 ms per pr_graph_create, 12 keys 8.86 / 10.11 / 2.60 ms; 16 keys
// need fewer CTAs per SM (registers) and lost (three per SM 9.20 / 10.13 /
// 2.67, two per SM 10.54 / 10.71 / 3.00).
constexpr int kRadixItems = 12;
constexpr int kRadixTile = kBlock * kRadixItems;

// Tiles [tile_lo(c), tile_lo(c + 1)) of a pass belong to CTA c of `ctas`:
// contiguous ranges, so that a CTA's output for each digit is one run.
__device__ __forceinline__ int64_t tile_lo(int64_t c, int64_t tiles, int64_t ctas)
{
    return tiles * c / ctas;
}

// Block-wide inclusive max-scan of the kRadixTile entries of `a` (16-byte
// aligned, unpadded), kRadixItems consecutive entries per thread, read and
// written as whole int4s.
__device__ __forceinline__ void block_max_scan(int32_t *a, int32_t *s_wmax)
{
    static_assert(kRadixItems % 4 == 0, "whole int4s per thread");
    constexpr int kQ = kRadixItems / 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int4 *a4 = reinterpret_cast<int4 *>(a) + kQ * tid;
    int4 q[kQ];
    int32_t run = INT32_MIN;
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
        q[k] = a4[k];
        run = max(run, max(max(q[k].x, q[k].y), max(q[k].z, q[k].w)));
    }
    int32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl = max(incl, t);
    }
    if (lane == 31)
        s_wmax[warp] = incl;
    __syncthreads();
    int32_t carry = INT32_MIN;
    for (int w = 0; w < warp; ++w)
        carry = max(carry, s_wmax[w]);
    const int32_t up = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane > 0)
        carry = max(carry, up);
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
        q[k].x = carry = max(carry, q[k].x);
        q[k].y = carry = max(carry, q[k].y);
        q[k].z = carry = max(carry, q[k].z);
        q[k].w = carry = max(carry, q[k].w);
        a4[k] = q[k];
    }
    __syncthreads();
}

// Upsweep of one counting-sort pass: the 256 digit counts of each CTA's tile
// range (key i at keys[i * stride]: stride 2 reads the keys of (key, value)
// pairs), written digit-major (counts[d * ctas + c]), so that one exclusive
// scan of the whole array gives every (digit, CTA) its output position. With
// n > 0 every key is also checked against [0, n); a bad key is still
// counted, so the downsweep's positions stay a permutation of [0, count) and
// the build stops on the error flag before any later step reads them.
__global__ void __launch_bounds__(kBlock)
k_radix_upsweep(const int32_t *__restrict__ keys, int stride, int64_t count, int64_t n, int shift,
                int32_t *__restrict__ counts, int64_t tiles, int64_t ctas, unsigned *err)
{
    constexpr int kWarps = kBlock / 32;
    __shared__ unsigned s_h[kWarps][kRadixBins];
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int w = 0; w < kWarps; ++w)
        s_h[w][tid] = 0;
    __syncthreads();
    const int64_t c = blockIdx.x;
    const int64_t i_end = min(count, tile_lo(c + 1, tiles, ctas) * kRadixTile);
    bool bad = false;
    for (int64_t b = tile_lo(c, tiles, ctas) * kRadixTile; b < i_end; b += kRadixTile) {
        int32_t v[kRadixItems];
#pragma unroll
        for (int k = 0; k < kRadixItems; ++k) {
            const int64_t i = b + (int64_t)k * kBlock + tid;
            v[k] = i < i_end ? keys[i * stride] : 0;
        }
#pragma unroll
        for (int k = 0; k < kRadixItems; ++k) {
            if (b + (int64_t)k * kBlock + tid < i_end) {
                bad |= n > 0 && (v[k] < 0 || (int64_t)v[k] >= n);
                atomicAdd(&s_h[warp][((unsigned)v[k] >> shift) & (kRadixBins - 1)], 1u);
            }
        }
    }
    if (bad)
        atomicOr(err, kErrColIdx);
    __syncthreads();
    unsigned t = 0;
    for (int w = 0; w < kWarps; ++w)
        t += s_h[w][tid];
    counts[(int64_t)tid * ctas + c] = (int32_t)t;
}

// The source of every edge of the out-edge CSR: src[i] = the row r with
// row_ptr[r] <= i < row_ptr[r+1], for i in [0, m), so that the first radix
// pass reads its values like every later one. One CTA per tile of
// kRadixTile edges (grid-stride): the rows that start inside the tile are
// marked at their first position in shared memory and a block max-scan
// spreads each row over its edges. tile_rows holds the row of every tile's
// first position (k_tile_rows), so rows (tile_rows[t], tile_rows[t+1]] are
// the only ones that can start inside tile t.
__global__ void __launch_bounds__(kBlock)
k_edge_sources(const int64_t *__restrict__ row_ptr, const int32_t *__restrict__ tile_rows, int64_t m,
               int64_t tiles, int32_t *__restrict__ src)
{
    constexpr int kWarps = kBlock / 32;
    __shared__ __align__(16) int32_t s_rmap[kRadixTile];
    __shared__ int32_t s_wmax[kWarps];
    const int tid = threadIdx.x;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t b = t * kRadixTile;
        const int64_t rlo = tile_rows[t], rhi = tile_rows[t + 1];
        const int tile_count = (int)min((int64_t)kRadixTile, m - b);
        const int4 none = make_int4(INT32_MIN, INT32_MIN, INT32_MIN, INT32_MIN);
#pragma unroll
        for (int k = 0; k < kRadixItems / 4; ++k)
            reinterpret_cast<int4 *>(s_rmap)[(kRadixItems / 4) * tid + k] = none;
        __syncthreads();
        if (tid == 0)
            s_rmap[0] = (int32_t)rlo;
        for (int64_t r = rlo + 1 + tid; r <= rhi; r += kBlock) {
            const int64_t p = row_ptr[r] - b;   // rows starting past the tile are skipped
            if (p > 0 && p < tile_count)
                atomicMax(&s_rmap[(int)p], (int32_t)r);
        }
        __syncthreads();
        block_max_scan(s_rmap, s_wmax);
#pragma unroll
        for (int k = 0; k < kRadixItems; ++k) {
            const int j = k * kBlock + tid;
            if (j < tile_count)
                src[b + j] = s_rmap[j];
        }
        __syncthreads();   // the row map is read before the next tile's marks
    }
}

// ---------------------------------------------------------------- step 3 --

// Downsweep of one stable counting-sort pass over digit (key >> shift) & 255.
// CTA c sorts its tile range in order. `offsets` is the exclusive scan of the
// upsweep's digit-major counts: offsets[d * ctas + c] is where CTA c's keys of
// digit d start, and the CTA keeps each digit's running position in shared
// memory from tile to tile, so no CTA waits for another.
//
// Tile layout: warp w owns tile positions [w*32*ITEMS, (w+1)*32*ITEMS) and
// walks them in 32-key rounds, so "earlier round, then lower lane" is input
// order. In each round, one ballot per digit bit gives every lane the mask of
// lanes with its digit (the native match instruction was slower, its cost
// growing with the number of distinct digits in the warp); a per-warp shared
// counter carries each digit's running count across rounds. Per-warp counts
// are then scanned across warps (and across digits for the tile-local order)
// and the tile is staged in shared memory in (digit, input) order, as (key,
// value) pairs. The write-out walks the staged tile linearly, so a warp
// stores consecutive addresses of one bucket, and a CTA's stores of one digit
// continue where its previous tile's ended. The next tile's keys are loaded
// while the current one is written out.
//
// Between passes each key travels with its value as one int2, so a staged
// entry is one shared-memory store and one global store: the write-out's
// stores scatter over a few buckets per warp, and with separate key and value
// arrays every entry cost two such scattered stores.
//
// kFlags:
//   kPairsIn   the input is (key, value) pairs; else two arrays (first pass).
//   kPairsOut  the output is (key, value) pairs; else the values only (last pass).
//   kHistogram the last pass of the edge sort: the tile, ordered by full key
//              within each digit bucket, adds each run of equal keys to the
//              in-degree histogram once.
enum : unsigned { kPairsIn = 1u, kPairsOut = 2u, kHistogram = 4u };

__device__ __forceinline__ int spad(int i) { return i + (i >> 5); }   // bank-conflict padding

template <unsigned kFlags>
__global__ void __launch_bounds__(kBlock, 4)
k_radix_pass(const int32_t *__restrict__ keys_in, const int32_t *__restrict__ vals_in,
             const int2 *__restrict__ pairs_in, int64_t n, int2 *__restrict__ pairs_out,
             int32_t *__restrict__ vals_out, int32_t *__restrict__ in_deg, int64_t count,
             int shift, const int32_t *__restrict__ offsets, int64_t tiles, int64_t ctas)
{
    constexpr int kWarps = kBlock / 32;
    constexpr int kWarpSpan = 32 * kRadixItems;
    constexpr int kPadTile = kRadixTile + kRadixTile / 32;
    __shared__ unsigned s_wh[kWarps][kRadixBins];   // per-warp counts, then staged offsets
    __shared__ unsigned s_run[kRadixBins];          // next output position of each digit
    __shared__ unsigned s_delta[kRadixBins];        // output position - staged position, per digit
    __shared__ unsigned s_wsum[kWarps];
    __shared__ int32_t s_wmax[kWarps];
    __shared__ __align__(16) int2 s_kv[kPadTile];   // staged (key, value) pairs

    // positions are below count <= 2^31 - 1: 32-bit indexing throughout
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    const int32_t t_first = (int32_t)tile_lo(c, tiles, ctas), t_last = (int32_t)tile_lo(c + 1, tiles, ctas);
    const int32_t n_keys = (int32_t)count;
    s_run[tid] = (unsigned)offsets[(int64_t)tid * ctas + c];

    int32_t key[kRadixItems], val[kRadixItems];
    unsigned rank[kRadixItems];
    // keys (and values) of tile t into registers
    auto load_tile = [&](int32_t t) {
        const int32_t base = t * kRadixTile + warp * kWarpSpan;
#pragma unroll
        for (int r = 0; r < kRadixItems; ++r) {
            const int32_t i = base + r * 32 + lane;
            const bool ok = i < n_keys;
            if (kFlags & kPairsIn) {
                const int2 kv = ok ? pairs_in[i] : make_int2(0, 0);
                key[r] = kv.x;
                val[r] = kv.y;
            } else {
                key[r] = ok ? keys_in[i] : 0;
                val[r] = ok ? vals_in[i] : 0;
            }
        }
    };
    if (t_first < t_last)
        load_tile(t_first);

    // One tile; kFull (every tile but the last) drops the bounds checks.
    auto process = [&](int32_t tile, auto full) {
        constexpr bool kFull = decltype(full)::value;
        const int32_t tile_begin = tile * kRadixTile;
        const int tile_count = kFull ? kRadixTile : min(kRadixTile, n_keys - tile_begin);
        const int32_t base = tile_begin + warp * kWarpSpan;
        // each round's lanes with an equal digit, one ballot per digit bit;
        // rank[] holds the masks until the ranks replace them
#pragma unroll
        for (int r = 0; r < kRadixItems; ++r) {
            const bool ok = kFull || base + r * 32 + lane < n_keys;
            const unsigned dig = ok ? (((unsigned)key[r] >> shift) & (kRadixBins - 1)) : kRadixBins;
            unsigned peers = 0xffffffffu;
#pragma unroll
            for (int b = 0; b < (kFull ? 8 : 9); ++b) {
                const bool bit = (dig >> b) & 1u;
                const unsigned m = __ballot_sync(0xffffffffu, bit);
                peers &= bit ? m : ~m;
            }
            rank[r] = peers;
        }
        __syncthreads();   // the previous tile's shared-memory reads are done
        for (int w = 0; w < kWarps; ++w)
            s_wh[w][tid] = 0;
        __syncthreads();   // s_wh cleared

        const unsigned below = (1u << lane) - 1u;
#pragma unroll
        for (int r = 0; r < kRadixItems; ++r) {
            const bool ok = kFull || base + r * 32 + lane < n_keys;
            const unsigned dig = ok ? (((unsigned)key[r] >> shift) & (kRadixBins - 1)) : kRadixBins;
            const unsigned peers = rank[r];
            const unsigned before = ok ? s_wh[warp][dig] : 0u;
            __syncwarp();
            rank[r] = before + __popc(peers & below);
            if (ok && (peers >> lane) == 1u)   // highest lane of the group
                s_wh[warp][dig] = before + __popc(peers);
            __syncwarp();
        }
        __syncthreads();

        // thread tid owns digit tid: the tile's count of the digit, its
        // tile-local start (exclusive scan over the 256 digits), and, per
        // warp, where that warp's keys of the digit are staged
        unsigned tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            tot += s_wh[w][tid];
        const unsigned incl = warp_incl_scan(tot, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        unsigned woff = 0;
        for (int w = 0; w < warp; ++w)
            woff += s_wsum[w];
        const unsigned start = woff + incl - tot;
        unsigned run = start;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const unsigned cnt = s_wh[w][tid];
            s_wh[w][tid] = run;
            run += cnt;
        }
        // staged position j of digit tid goes to s_run + (j - start); positions
        // are below count <= 2^31 - 1, so unsigned 32-bit arithmetic is exact
        s_delta[tid] = s_run[tid] - start;
        s_run[tid] += tot;
        __syncthreads();

        // stage the tile in (digit, input) order
#pragma unroll
        for (int r = 0; r < kRadixItems; ++r) {
            if (kFull || base + r * 32 + lane < n_keys) {
                const unsigned dig = ((unsigned)key[r] >> shift) & (kRadixBins - 1);
                const int lp = (int)(s_wh[warp][dig] + rank[r]);
                s_kv[spad(lp)] = make_int2(key[r], val[r]);
            }
        }
        __syncthreads();

        // the next tile's loads overlap this tile's write-out
        if (tile + 1 < t_last)
            load_tile(tile + 1);

        // write-out: consecutive staged entries of one digit go to consecutive addresses
#pragma unroll
        for (int k = 0; k < kRadixItems; ++k) {
            const int i = k * kBlock + tid;
            if (kFull || i < tile_count) {
                const int2 kv = s_kv[spad(i)];
                const unsigned dig = ((unsigned)kv.x >> shift) & (kRadixBins - 1);
                const unsigned pos = s_delta[dig] + (unsigned)i;
                if (pos >= (unsigned)n_keys)   // only reachable if the offsets scan failed
                    continue;
                if (kFlags & kPairsOut)
                    pairs_out[pos] = kv;
                else
                    vals_out[pos] = kv.y;
            }
        }

        if (kFlags & kHistogram) {
            // thread t owns staged entries [t*ITEMS, (t+1)*ITEMS); each run of
            // equal keys adds its length once, at its last entry. The head of
            // the run an entry belongs to comes from a max-scan of run heads.
            const int j0 = tid * kRadixItems;
            int head_local = -1;
            for (int j = j0; j < j0 + kRadixItems && j < tile_count; ++j)
                if (j == 0 || s_kv[spad(j)].x != s_kv[spad(j - 1)].x)
                    head_local = j;
            int carry = head_local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, carry, o);
                if (lane >= o)
                    carry = max(carry, t);
            }
            if (lane == 31)
                s_wmax[warp] = carry;
            __syncthreads();
            int head = -1;
            for (int w = 0; w < warp; ++w)
                head = max(head, s_wmax[w]);
            const int up = __shfl_up_sync(0xffffffffu, carry, 1);
            if (lane > 0)
                head = max(head, up);   // last run head before this thread's entries
            for (int j = j0; j < j0 + kRadixItems && j < tile_count; ++j) {
                const int32_t kv = s_kv[spad(j)].x;
                if (j == 0 || kv != s_kv[spad(j - 1)].x)
                    head = j;
                if ((j == tile_count - 1 || s_kv[spad(j + 1)].x != kv) && kv >= 0 && (int64_t)kv < n)
                    atomicAdd(&in_deg[kv], j - head + 1);
            }
        }
    };
    for (int32_t tile = t_first; tile < t_last; ++tile) {
        if (n_keys - tile * kRadixTile >= kRadixTile)
            process(tile, std::true_type{});
        else
            process(tile, std::false_type{});
    }
}

// Row of the first position of every radix tile (tile_rows[tiles] = the row
// of the last edge), one bisection per tile, all in parallel.
__global__ void k_tile_rows(const int64_t *__restrict__ row_ptr, int64_t n, int64_t m, int64_t tiles,
                            int32_t *__restrict__ tile_rows)
{
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t <= tiles;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = min(t * kRadixTile, m - 1);
        tile_rows[t] = (int32_t)(upper_bound(row_ptr, n + 1, pos) - 1);
    }
}

// ---------------------------------------------------------------- step 4 --

constexpr int kScanItems = 32;
constexpr int kScanTile = kBlock * kScanItems;

struct LoadCount {   // element i of an int32 array
    const int32_t *p;
    __device__ int32_t operator()(int64_t i) const { return p[i]; }
};

// Length of work row i: the in-degree of order[i] rounded up to a multiple
// of 4, so that every row starts 16-byte aligned and is read in whole int4s.
__device__ __forceinline__ int32_t padded_degree(int32_t deg)
{
    return (deg + 3) & ~3;
}

// Padded length of work row i, from pdeg (the padded in-degrees in work
// order). Thread-class rows (work rows [t_begin, t_end)) are stored in
// interleaved blocks of 32 and take the padded length of their block's first
// row, the longest of the block (the work order sorts them by length,
// longest first), so every row of a block has one length.
struct LoadWorkDeg {
    const int32_t *pdeg;
    int64_t t_begin, t_end;
    __device__ int32_t operator()(int64_t i) const
    {
        if (i >= t_begin && i < t_end)
            i = t_begin + ((i - t_begin) & ~(int64_t)31);
        return pdeg[i];
    }
};

struct LoadChunkCount {   // number of edge chunks of work row i
    const int32_t *w_ptr;
    __device__ int32_t operator()(int64_t i) const
    {
        const int64_t deg = (int64_t)w_ptr[i + 1] - w_ptr[i];
        return (int32_t)((deg + kChunkEdges - 1) / kChunkEdges);
    }
};

// out[i] = sum of load(k) for k < i, for i in [0, count]; out[count] is the
// total. Single pass: tiles are taken in launch order from a counter and each
// finds its prefix by decoupled look-back over its predecessors' descriptors
// (each wait at most spin_limit polls). A negative count is added as 0 and
// sets kErrNegative; a total above INT32_MAX sets kErrOverflow (the offsets
// are then not meaningful). Both keep every descriptor a valid non-negative
// sum below 2^62, so the look-back stays well formed.
template <class Load>
__global__ void __launch_bounds__(kBlock)
k_scan_excl(Load load, int32_t *__restrict__ out, int64_t count,
            unsigned long long *desc, unsigned *tile_counter, unsigned *err, int spin_limit)
{
    __shared__ int32_t s_items[kScanTile + kScanTile / 32];   // padded: no bank conflicts
    __shared__ long long s_warp[kBlock / 32];
    __shared__ long long s_prefix;
    __shared__ unsigned s_tile;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        s_tile = atomicAdd(tile_counter, 1u);
    __syncthreads();
    const int64_t tile = s_tile;
    const int64_t base = tile * kScanTile;
    auto pad = [](int i) { return i + (i >> 5); };

    // every load of the thread in flight before the first store (the loads
    // of the work layout's scans are dependent gathers)
    bool negative = false;
    {
        int32_t ld[kScanItems];
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int64_t i = base + (int64_t)k * kBlock + tid;
            ld[k] = (i < count) ? load(i) : 0;
        }
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            negative |= ld[k] < 0;
            s_items[pad(k * kBlock + tid)] = max(ld[k], 0);
        }
    }
    if (negative)
        atomicOr(err, kErrNegative);
    __syncthreads();

    int32_t v[kScanItems];
    long long local = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = s_items[pad(tid * kScanItems + k)];
        local += v[k];
    }
    const long long incl = warp_incl_scan(local, lane);
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
            prefix = look_back(desc, tile, 1, err, spin_limit);
            store_desc(desc + tile, kFlagP | (unsigned long long)(prefix + total));
        }
        s_prefix = prefix;
        if (base + kScanTile >= count) {   // the last tile writes the total
            out[count] = (int32_t)(prefix + total);
            if (prefix + total > (long long)INT32_MAX)
                atomicOr(err, kErrOverflow);
        }
    }
    __syncthreads();
    long long run = s_prefix + thread_excl;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        s_items[pad(tid * kScanItems + k)] = (int32_t)run;
        run += v[k];
    }
    __syncthreads();
    for (int k = 0; k < kScanItems; ++k) {
        const int64_t i = base + (int64_t)k * kBlock + tid;
        if (i < count)
            out[i] = s_items[pad(k * kBlock + tid)];
    }
}

// ------------------------------------------------------------ classes ---

// Position of a class in the class-major order: CTA rows, warp rows, thread
// rows, then rows without in-edges (thresholds thread_max <= 32 <= ... as set
// by the handle's options).
__device__ __forceinline__ int class_slot(int32_t deg, int32_t thread_max, int32_t warp_max)
{
    return deg > warp_max ? 0 : deg > thread_max ? 1 : deg > 0 ? 2 : 3;
}

// Half-octave bucket of an out-degree: 2*floor(log2(d+1)) plus the next bit.
__device__ __forceinline__ int degree_bucket(int32_t deg)
{
    const unsigned x = (unsigned)deg + 1u;
    const int b = 31 - __clz(x);
    const int half = b > 0 ? (int)((x >> (b - 1)) & 1u) : 0;
    return min(63, 2 * b + half);
}

// Sort key of the work order (8 bits): the class slot, then, within the
// class, out-degree bucket, largest first (the most gathered vertices lead).
// Thread-class rows are keyed by their length in int4s first (longest first,
// 8 lengths) and then by a coarse out-degree bucket (8 levels), so that the
// 32 rows one warp takes together mostly have the same length. Ties go by
// vertex id (the sort is stable over vals = ids).
__global__ void k_order_keys(int64_t n, const int32_t *__restrict__ in_ptr,
                             const int32_t *__restrict__ deg_out, int32_t thread_max, int32_t warp_max,
                             int32_t *__restrict__ keys, int32_t *__restrict__ vals)
{
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int32_t indeg = in_ptr[v + 1] - in_ptr[v];
        const int slot = class_slot(indeg, thread_max, warp_max);
        const int ob = degree_bucket(deg_out[v]);
        const int sub = slot == 2 ? (8 - ((indeg + 3) >> 2)) * 8 + (7 - min(7, ob >> 2)) : 63 - ob;
        keys[v] = slot * 64 + sub;
        vals[v] = (int32_t)v;
    }
}

// The inverse of the work order (perm[order[i]] = i), and, in work order, the
// out-degrees (w_deg) and the in-degrees padded to whole int4s (pdeg, the
// lengths the work CSR's offsets are scanned from). An entry of order outside
// [0, n) (only if a scan before it failed) is skipped, and its row gets 0s.
__global__ void k_invert(int64_t n, const int32_t *__restrict__ order, const int32_t *__restrict__ in_deg,
                         const int32_t *__restrict__ deg_out, int32_t *__restrict__ perm,
                         int32_t *__restrict__ w_deg, int32_t *__restrict__ pdeg)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = order[i];
        int32_t dout = 0, din = 0;
        if (v >= 0 && (int64_t)v < n) {
            perm[v] = (int32_t)i;
            dout = deg_out[v];
            din = in_deg[v];
        }
        w_deg[i] = dout;
        pdeg[i] = padded_degree(din);
    }
}

// The work CSR: w_col[w_ptr[i] + k] = perm[in_col[in_ptr[order[i]] + k]] for
// k below the in-degree, and kPadSource (gathers 0) in the padding. CTA-class rows
// are copied in their kChunkEdges chunks, one warp per chunk; warp-class rows
// by one warp each; thread-class rows by one thread each. Rows without
// in-edges have nothing to copy.
//
// Thread-class rows are interleaved by blocks of 32 consecutive work rows
// (the last block may hold fewer, cnt): all rows of a block have the same
// padded length L int4s (see LoadOrderDeg), the block occupies the int4s
// [w_ptr[r0] / 4, w_ptr[r0] / 4 + cnt * L), and int4 k of the block's row j
// sits at w_ptr[r0] / 4 + k * cnt + j, so that the lanes of a warp, one row
// each, read consecutive int4s.
//
// The kernel also counts, for reporting, the true in-edges of the CTA, warp
// and thread classes (class_edges[0..2]) and the edges whose relabelled
// source falls in the head of the state vector that the update keeps in
// shared memory, for fp32 (kHotF32 vertices) and fp64 (kHotF64) runs: hot[0]
// and hot[1]. All five counters are zeroed by the caller. Each thread counts
// the entries it writes in 32 bits (a thread writes far fewer than 2^32 of
// the m < 2^31 entries).
//
// Two launches: kWide = true copies the CTA and warp classes (warps stream
// rows, four entries per lane in flight; held to 32 registers, because their
// perm gathers need every warp an SM can hold in flight, 8 CTAs per SM),
// kWide = false the thread class (one thread per row, 16 perm gathers in
// flight; more registers).
template <bool kWide>
__global__ void __launch_bounds__(kBlock, kWide ? 8 : 1)
k_relabel(int64_t n, int64_t n_c, int64_t n_chunks, int64_t wide_end, int64_t rows_end,
          const int32_t *__restrict__ chunk_row, const int32_t *__restrict__ chunk_first,
          const int32_t *__restrict__ w_ptr, const int32_t *__restrict__ order,
          const int32_t *__restrict__ perm, const int32_t *__restrict__ in_ptr,
          const int32_t *__restrict__ in_col, int32_t *__restrict__ w_col,
          unsigned long long *__restrict__ class_edges, unsigned long long *__restrict__ hot)
{
    const int lane = threadIdx.x & 31;
    const int64_t gtid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gwarp = gtid >> 5, nwarps = nthreads >> 5;
    unsigned h32 = 0, h64 = 0;             // entries with a hot source
    unsigned e_cta = 0, e_warp = 0, e_thr = 0;   // true entries written, per class
    auto relabel = [&](int32_t u) {
        const int32_t w = perm[u];
        h32 += (w < kHotF32);
        h64 += (w < kHotF64);
        return w;
    };
    // entries [k0, k1) of one row, four loads of in_col, then four perm
    // gathers, in flight per lane
    auto copy = [&](int32_t src, int32_t deg, int32_t dst, int32_t k0, int32_t k1, unsigned &e) {
        for (int32_t kb = k0; kb < k1; kb += 4 * 32) {
            int32_t u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t k = kb + q * 32 + lane;
                u[q] = (k < k1 && k < deg) ? in_col[src + k] : -1;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                u[q] = u[q] >= 0 ? relabel(u[q]) : kPadSource;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t k = kb + q * 32 + lane;
                if (k < k1) {
                    e += (k < deg);
                    w_col[dst + k] = u[q];
                }
            }
        }
    };
    for (int64_t c = gwarp; kWide && c < n_chunks; c += nwarps) {
        const int32_t r = chunk_row[c];
        const int32_t v = order[r];
        const int32_t src = in_ptr[v], deg = in_ptr[v + 1] - src;
        const int32_t dst = w_ptr[r], len = w_ptr[r + 1] - dst;
        const int32_t k0 = (int32_t)(c - chunk_first[r]) * kChunkEdges;
        copy(src, deg, dst, k0, min(k0 + kChunkEdges, len), e_cta);
    }
    for (int64_t i = n_c + gwarp; kWide && i < wide_end; i += nwarps) {
        const int32_t v = order[i];
        const int32_t src = in_ptr[v], deg = in_ptr[v + 1] - src;
        const int32_t dst = w_ptr[i], len = w_ptr[i + 1] - dst;
        copy(src, deg, dst, 0, len, e_warp);
    }
    // thread-class rows: one thread per row, whole int4s, so the 32 lanes of
    // a warp (the 32 rows of one block) store 32 consecutive int4s
    int4 *w_col4 = reinterpret_cast<int4 *>(w_col);
    for (int64_t i = wide_end + gtid; !kWide && i < rows_end; i += nthreads) {
        const int32_t v = order[i];
        const int32_t src = in_ptr[v], deg = in_ptr[v + 1] - src;
        const int64_t r0 = wide_end + ((i - wide_end) & ~(int64_t)31);
        const int64_t cnt = min((int64_t)32, rows_end - r0);
        const int64_t j = i - r0;
        const int64_t blk4 = w_ptr[r0] >> 2;   // rows start 16-byte aligned
        const int32_t len4 = (w_ptr[i + 1] - w_ptr[i]) >> 2;
        e_thr += (unsigned)deg;
        // up to four int4s (16 entries) at a time: every load of in_col, then
        // every perm gather, then the stores, so that a row costs two round
        // trips to memory per 16 entries instead of two per int4
        for (int32_t q0 = 0; q0 < len4; q0 += 4) {
            int32_t u[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                u[k] = (4 * q0 + k < deg) ? in_col[src + 4 * q0 + k] : -1;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                u[k] = u[k] >= 0 ? relabel(u[k]) : kPadSource;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q0 + q < len4)
                    w_col4[blk4 + (int64_t)(q0 + q) * cnt + j] =
                        make_int4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
        }
    }
    // per CTA: 32-bit warp sums (a warp writes far fewer than 2^32 entries),
    // 64-bit CTA sums, one atomic per counter and CTA
    __shared__ unsigned long long s_cnt[5];
    if (threadIdx.x < 5)
        s_cnt[threadIdx.x] = 0ull;
    __syncthreads();
    unsigned v[5] = {h32, h64, e_cta, e_warp, e_thr};
#pragma unroll
    for (int q = 0; q < 5; ++q) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
        if (lane == 0 && v[q])
            atomicAdd(&s_cnt[q], (unsigned long long)v[q]);
    }
    __syncthreads();
    if (threadIdx.x < 5 && s_cnt[threadIdx.x])
        atomicAdd(threadIdx.x < 2 ? hot + threadIdx.x : class_edges + (threadIdx.x - 2), s_cnt[threadIdx.x]);
}

// First thread-class block (32 work rows from t_begin) whose rows span at
// most two int4s; t_blocks if there is none. Block lengths never increase
// (the work order sorts these rows by length, longest first), so one thread
// bisects.
__global__ void k_first_short_block(const int32_t *__restrict__ w_ptr, int64_t t_begin, int64_t t_blocks,
                                    unsigned long long *out)
{
    int64_t lo = 0, hi = t_blocks;
    while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        const int64_t r = t_begin + 32 * mid;
        if (w_ptr[r + 1] - w_ptr[r] <= 8)
            hi = mid;
        else
            lo = mid + 1;
    }
    *out = (unsigned long long)lo;
}

__global__ void k_fill_chunks(int64_t n_c, int64_t n_chunks, const int32_t *__restrict__ chunk_first,
                              int32_t *__restrict__ chunk_row)
{
    for (int64_t r = blockIdx.x; r < n_c; r += gridDim.x)
        for (int32_t c = chunk_first[r] + threadIdx.x; c < chunk_first[r + 1]; c += blockDim.x)
            if (c >= 0 && c < n_chunks)
                chunk_row[c] = (int32_t)r;
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

// Scratch of one build, returned to the pool in stream order when the build
// returns.
struct Scratch {
    cudaStream_t s;
    std::vector<void *> ptrs;
    explicit Scratch(cudaStream_t stream) : s(stream) {}
    ~Scratch()
    {
        for (void *p : ptrs)
            pool_free(p, s);
    }
    pr_status alloc(void **p, size_t bytes)
    {
        pr_status st = pool_alloc(p, bytes, s);
        if (st == PR_OK)
            ptrs.push_back(*p);
        return st;
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
    k_scan_excl<Load><<<(unsigned)tiles, kBlock, 0, s>>>(load, out, count, desc, counter, err, kSpinLimit);
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

// CTAs of a counting-sort pass over `tiles` tiles: four per SM (the
// downsweep's occupancy), each with a contiguous tile range.
int64_t sort_ctas(const pr_graph *g, int64_t tiles)
{
    const int64_t want = (int64_t)g->num_sms * 4;
    return tiles < want ? tiles : want;
}

// One counting-sort pass: upsweep (digit counts per CTA range), one
// exclusive scan of the digit-major counts, downsweep (rank and scatter).
template <unsigned kFlags>
pr_status sort_pass(pr_graph *g, cudaStream_t s, const int32_t *kin, const int32_t *vin, const int2 *pin,
                    int64_t n, int2 *pout, int32_t *vout, int32_t *in_deg, int64_t count, int shift,
                    int64_t validate_n, int32_t *counts, int32_t *offsets, unsigned long long *desc,
                    unsigned *counter)
{
    const int64_t tiles = (count + kRadixTile - 1) / kRadixTile;
    const int64_t ctas = sort_ctas(g, tiles);
    const int32_t *ukeys = (kFlags & kPairsIn) ? reinterpret_cast<const int32_t *>(pin) : kin;
    k_radix_upsweep<<<(unsigned)ctas, kBlock, 0, s>>>(ukeys, (kFlags & kPairsIn) ? 2 : 1, count, validate_n, shift,
                                                      counts, tiles, ctas, g->err);
    ++g->build_launches;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_status(e, "k_radix_upsweep launch");
    pr_status st = launch_scan(LoadCount{counts}, offsets, ctas * kRadixBins, desc, counter, g->err,
                               &g->build_launches, s);
    if (st != PR_OK)
        return st;
    k_radix_pass<kFlags><<<(unsigned)ctas, kBlock, 0, s>>>(kin, vin, pin, n, pout, vout, in_deg, count, shift,
                                                          offsets, tiles, ctas);
    ++g->build_launches;
    e = cudaGetLastError();
    return e == cudaSuccess ? PR_OK : cuda_status(e, "k_radix_pass launch");
}

// ------------------------------------------- allocation-free scan ---

// The scratch of pr_exclusive_scan_noalloc: the look-back descriptors of up
// to kNoAllocScanTiles tiles, then the tile counter, then the error word. It
// is a file-scope device array, so every device that loads the library holds
// these bytes until the process exits, and every call shares them.
constexpr int64_t kNoAllocScanMax = PR_SCAN_NOALLOC_MAX;
constexpr int64_t kNoAllocScanTiles = (kNoAllocScanMax + kScanTile - 1) / kScanTile;
static __device__ __align__(256) unsigned long long g_noalloc_scan_scratch[kNoAllocScanTiles + 2];

}  // namespace

// Device address of g_noalloc_scan_scratch on the current device, looked up
// once per device (the array's name is only a host-side stand-in in host code).
static pr_status noalloc_scratch(unsigned long long **out)
{
    static std::mutex mu;
    static unsigned long long *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(PR_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scan_scratch);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaGetSymbolAddress of the scan scratch");
        addr[dev] = static_cast<unsigned long long *>(p);
    }
    *out = addr[dev];
    return PR_OK;
}

pr_status exclusive_scan_noalloc(const int32_t *counts, int32_t *offsets, int64_t count,
                                 cudaStream_t s)
{
    if (count < 0)
        return set_error(PR_ERR_INVALID_ARG, "count must be >= 0 (got %lld)", (long long)count);
    if (count > kNoAllocScanMax)
        return set_error(PR_ERR_TOO_LARGE,
                         "count = %lld exceeds the %lld elements the static scratch of "
                         "pr_exclusive_scan_noalloc is sized for",
                         (long long)count, (long long)kNoAllocScanMax);
    if (offsets == nullptr || (count > 0 && counts == nullptr))
        return set_error(PR_ERR_INVALID_ARG, "NULL pointer");
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess)
        return cuda_status(de, "cudaGetDevice");
    if (pointer_kind(offsets, dev) != kPtrDevice || (count > 0 && pointer_kind(counts, dev) != kPtrDevice))
        return set_error(PR_ERR_INVALID_ARG, "counts and offsets must be memory of the current device (%d)",
                         dev);
    unsigned long long *scratch = nullptr;
    pr_status st = noalloc_scratch(&scratch);
    if (st != PR_OK)
        return st;
    cudaError_t e;
    if (count == 0) {
        e = cudaMemsetAsync(offsets, 0, sizeof(int32_t), s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        return e == cudaSuccess ? PR_OK : cuda_status(e, "pr_exclusive_scan_noalloc");
    }
    const int64_t tiles = (count + kScanTile - 1) / kScanTile;
    unsigned long long *desc = scratch;
    unsigned *counter = reinterpret_cast<unsigned *>(scratch + kNoAllocScanTiles);
    unsigned *err = reinterpret_cast<unsigned *>(scratch + kNoAllocScanTiles + 1);
    // what the scan expects to start at zero: the descriptors it will use,
    // the tile counter and the error word (the previous call's values remain)
    e = cudaMemsetAsync(desc, 0, (size_t)tiles * sizeof(unsigned long long), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(scratch + kNoAllocScanTiles, 0, 2 * sizeof(unsigned long long), s);
    if (e != cudaSuccess)
        return cuda_status(e, "clearing the scan scratch");
    k_scan_excl<LoadCount><<<(unsigned)tiles, kBlock, 0, s>>>(LoadCount{counts}, offsets, count, desc,
                                                             counter, err, kSpinLimit);
    e = cudaGetLastError();
    unsigned herr = 0;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&herr, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_status(e, "pr_exclusive_scan_noalloc");
    if (herr & kErrTimeout)
        return set_error(PR_ERR_TIMEOUT, "a look-back wait in the scan gave up");
    if (herr & kErrNegative)
        return set_error(PR_ERR_INVALID_ARG, "counts has a negative entry (offsets are not valid)");
    if (herr & kErrOverflow)
        return set_error(PR_ERR_TOO_LARGE, "the sum of counts exceeds INT32_MAX (offsets are not valid)");
    return PR_OK;
}

pr_status scan_timeout_probe(int64_t count, int spin_limit, cudaStream_t s)
{
    if (count <= kScanTile || count > ((int64_t)1 << 24))
        return set_error(PR_ERR_INVALID_ARG, "count must be in (%d, 2^24] (got %lld)", kScanTile,
                         (long long)count);
    if (spin_limit < 1 || spin_limit > (1 << 20))
        return set_error(PR_ERR_INVALID_ARG, "spin_limit must be in [1, 2^20] (got %d)", spin_limit);
    const int64_t tiles = (count + kScanTile - 1) / kScanTile;
    Scratch tmp(s);
    int32_t *counts = nullptr, *out = nullptr;
    unsigned long long *desc = nullptr;
    unsigned *words = nullptr;   // [0] tile counter, [1] error word
    pr_status st;
    if ((st = tmp.alloc((void **)&counts, (size_t)count * sizeof(int32_t))) != PR_OK ||
        (st = tmp.alloc((void **)&out, (size_t)(count + 1) * sizeof(int32_t))) != PR_OK ||
        (st = tmp.alloc((void **)&desc, (size_t)tiles * sizeof(unsigned long long))) != PR_OK ||
        (st = tmp.alloc((void **)&words, 2 * sizeof(unsigned))) != PR_OK)
        return st;
    // tile 0 never runs: its descriptor stays unpublished, so tile 1 (and
    // any tile that walks back to it) waits until its spin limit runs out.
    // Every CTA still reads and writes only inside the buffers above.
    const unsigned first_tile = 1;
    cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)count * sizeof(int32_t), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(desc, 0, (size_t)tiles * sizeof(unsigned long long), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(words, 0, 2 * sizeof(unsigned), s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(words, &first_tile, sizeof(unsigned), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) {
        k_scan_excl<LoadCount><<<(unsigned)(tiles - 1), kBlock, 0, s>>>(LoadCount{counts}, out, count, desc,
                                                                        words, words + 1, spin_limit);
        e = cudaGetLastError();
    }
    unsigned herr = 0;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&herr, words + 1, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_status(e, "scan timeout probe");
    if (herr & kErrTimeout)
        return set_error(PR_ERR_TIMEOUT, "a look-back wait in the scan gave up");
    return PR_OK;
}

// A second stream per device (non-blocking, created on first use, kept until
// exit) for build work that runs beside the build's own stream. Calls from
// several threads share it; each forks and joins with events of its own.
static pr_status side_stream(cudaStream_t *out)
{
    static std::mutex mu;
    static cudaStream_t streams[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(PR_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (streams[dev] == nullptr) {
        e = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            streams[dev] = nullptr;
            return cuda_status(e, "cudaStreamCreateWithFlags");
        }
    }
    *out = streams[dev];
    return PR_OK;
}

// Work forked from stream `main` onto stream `side` and joined back: fork()
// makes side wait for main's work so far; the join (join(), or the
// destructor on any early return) makes main wait for everything issued on
// side since, so that nothing main does afterwards (freeing the build's
// scratch, say) overtakes it. The events are destroyed with the guard (a
// recorded event may be destroyed before it completes).
struct ForkJoin {
    cudaStream_t main = nullptr, side = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    bool forked = false;
    pr_status fork(cudaStream_t m, cudaStream_t sd)
    {
        main = m;
        side = sd;
        cudaError_t e = cudaEventCreateWithFlags(&fork_ev, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&join_ev, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventRecord(fork_ev, main);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(side, fork_ev, 0);
        if (e != cudaSuccess)
            return cuda_status(e, "forking the build onto a second stream");
        forked = true;
        return PR_OK;
    }
    pr_status join()
    {
        if (!forked)
            return PR_OK;
        forked = false;
        cudaError_t e = cudaEventRecord(join_ev, side);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(main, join_ev, 0);
        return e == cudaSuccess ? PR_OK : cuda_status(e, "joining the build's second stream");
    }
    ~ForkJoin()
    {
        if (forked && join() != PR_OK)
            cudaStreamSynchronize(side);   // the join itself failed: wait outright
        if (fork_ev)
            cudaEventDestroy(fork_ev);
        if (join_ev)
            cudaEventDestroy(join_ev);
    }
};

// CUDA events at the boundaries of the build's stages (PR_STAGE_*), on the
// build's stream, when the handle asks for them; destroyed with the build.
struct StageClock {
    cudaEvent_t ev[PR_BUILD_STAGES + 1] = {};
    bool on = false;
    pr_status start(bool wanted, cudaStream_t s)
    {
        on = wanted;
        if (!on)
            return PR_OK;
        for (cudaEvent_t &e : ev) {
            const cudaError_t r = cudaEventCreate(&e);
            if (r != cudaSuccess)
                return cuda_status(r, "cudaEventCreate");
        }
        const cudaError_t r = cudaEventRecord(ev[0], s);
        return r == cudaSuccess ? PR_OK : cuda_status(r, "cudaEventRecord");
    }
    // end of stage k (0-based)
    void mark(int k, cudaStream_t s)
    {
        if (on)
            cudaEventRecord(ev[k + 1], s);
    }
    // per-stage times once the stream has passed every mark
    void read(float *ms) const
    {
        if (!on)
            return;
        for (int k = 0; k < PR_BUILD_STAGES; ++k)
            if (cudaEventElapsedTime(&ms[k], ev[k], ev[k + 1]) != cudaSuccess)
                ms[k] = 0.f;
        cudaGetLastError();
    }
    ~StageClock()
    {
        for (cudaEvent_t e : ev)
            if (e)
                cudaEventDestroy(e);
    }
};

pr_status build_graph(pr_graph *g, const int64_t *d_row_ptr, const int32_t *d_col, const int32_t *h_col,
                      cudaStream_t s)
{
    const int64_t n = g->n, m = g->m;
    const int cap = g->num_sms * 32;
    pr_status st;
    cudaError_t e;
    Scratch tmp(s);
    StageClock clock;

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

    // the build's device time (always) and its stages (when asked for)
    PRK_CUDA(cudaEventRecord(g->ev[0], s), "cudaEventRecord");
    PRK_TRY(clock.start(g->stage_timing, s));

    // A host col_idx goes to its device buffer on the second stream while the
    // steps that read only row_ptr (degrees, tile rows, edge sources) run on
    // s; s waits for the copy before the first radix pass, and on any early
    // return (the guard's destructor), so the buffer outlives the copy.
    ForkJoin staging;
    if (h_col != nullptr && m > 0) {
        cudaStream_t side = s;
        PRK_TRY(side_stream(&side));
        PRK_TRY(staging.fork(s, side));
        PRK_CUDA(cudaMemcpyAsync(const_cast<int32_t *>(d_col), h_col, (size_t)m * sizeof(int32_t),
                                 cudaMemcpyHostToDevice, side),
                 "staging col_idx");
    }

    // handle-owned buffers: the in-edge CSR and the work layout
    PRK_TRY(graph_alloc(g, (void **)&g->in_ptr, (size_t)(n + 1) * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->in_col, (size_t)(m + 4) * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->deg_out, (size_t)n * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->order, (size_t)n * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->perm, (size_t)n * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->w_ptr, (size_t)(n + 1) * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->w_deg, (size_t)n * sizeof(int32_t), s));

    int bits = 0;
    while (bits < 31 && ((int64_t)1 << bits) < n)
        ++bits;
    int passes = (bits + kRadixBits - 1) / kRadixBits;
    if (passes < 1)
        passes = 1;

    // scratch
    int32_t *in_deg = nullptr;
    unsigned long long *counters = nullptr;   // [0] dangling, [1..3] class edges, [4] t_short,
                                              // [5..6] edges with a hot source (fp32, fp64)
    unsigned *tile_counter = nullptr;
    unsigned long long *desc = nullptr;
    int32_t *counts = nullptr, *offsets = nullptr;   // digit-major tile counts and their scan
    PRK_TRY(tmp.alloc((void **)&in_deg, (size_t)n * sizeof(int32_t)));
    PRK_TRY(tmp.alloc((void **)&counters, 8 * sizeof(unsigned long long)));
    PRK_TRY(tmp.alloc((void **)&tile_counter, sizeof(unsigned)));
    const int64_t radix_tiles = (m + kRadixTile - 1) / kRadixTile;
    const int64_t order_tiles = (n + kRadixTile - 1) / kRadixTile;
    const int64_t max_tiles = radix_tiles > order_tiles ? radix_tiles : order_tiles;
    const int64_t count_words = sort_ctas(g, max_tiles) * kRadixBins;
    PRK_TRY(tmp.alloc((void **)&counts, (size_t)count_words * sizeof(int32_t)));
    PRK_TRY(tmp.alloc((void **)&offsets, (size_t)(count_words + 1) * sizeof(int32_t)));
    int64_t desc_words = (n + 1 + kScanTile - 1) / kScanTile;
    if ((count_words + kScanTile - 1) / kScanTile > desc_words)
        desc_words = (count_words + kScanTile - 1) / kScanTile;
    PRK_TRY(tmp.alloc((void **)&desc, (size_t)(desc_words + 1) * sizeof(unsigned long long)));

    PRK_CUDA(cudaMemsetAsync(g->err, 0, sizeof(unsigned), s), "memset");
    PRK_CUDA(cudaMemsetAsync(in_deg, 0, (size_t)n * sizeof(int32_t), s), "memset");
    PRK_CUDA(cudaMemsetAsync(counters, 0, 8 * sizeof(unsigned long long), s), "memset");

    // 1: degrees and row_ptr validation (col_idx is checked by the first upsweep)
    k_outdeg<<<grid_for(n, kBlock, cap), kBlock, 0, s>>>(n, d_row_ptr, g->deg_out, counters, g->err);
    ++g->build_launches;
    PRK_CUDA(cudaGetLastError(), "validation launch");

    // The error word is read (one stream synchronisation) right after the
    // row_ptr check, since the row ranges of the edge-source kernel assume a
    // non-decreasing row_ptr; after that only where the host needs a size
    // anyway, and before any kernel that indexes an array through values an
    // earlier step computed: a bad col_idx, or a look-back that gave up,
    // stops the build there. Every kernel before such a check stays in
    // bounds and ends in time whatever the values: edge sources and radix
    // keys are only moved, radix write positions and histogram keys are
    // range-checked, and the vertex order is inverted with a range check.
    auto check = [&]() -> pr_status {
        unsigned w = 0;
        pr_status r = read_err(g, s, &w);
        if (r != PR_OK)
            return r;
        if (w & kErrRowPtr)
            return set_error(PR_ERR_INVALID_GRAPH, "row_ptr is not non-decreasing");
        if (w & kErrColIdx)
            return set_error(PR_ERR_INVALID_GRAPH, "col_idx has an entry outside [0, n)");
        if (w & kErrTimeout)
            return set_error(PR_ERR_TIMEOUT, "a look-back wait in the transpose gave up");
        return PR_OK;
    };
    PRK_TRY(check());
    clock.mark(PR_STAGE_DEGREES, s);

    // 2 + 3: stable scatter by destination (LSD radix over 8-bit digits),
    // which also yields the in-degree histogram
    if (m > 0) {
        int2 *pb[2] = {nullptr, nullptr};   // (key, value) pairs between passes
        for (int i = 0; i < 2 && i < passes - 1; ++i)
            PRK_TRY(tmp.alloc((void **)&pb[i], (size_t)m * sizeof(int2)));
        int32_t *tile_rows = nullptr;
        PRK_TRY(tmp.alloc((void **)&tile_rows, (size_t)(radix_tiles + 1) * sizeof(int32_t)));
        k_tile_rows<<<grid_for(radix_tiles + 1, kBlock, cap), kBlock, 0, s>>>(d_row_ptr, n, m, radix_tiles,
                                                                            tile_rows);
        ++g->build_launches;
        PRK_CUDA(cudaGetLastError(), "k_tile_rows launch");
        // the source of every edge, the first pass's values: a value buffer
        // that no pass before the second writes (with two passes, in_col,
        // which only the last pass writes)
        int32_t *src = nullptr;
        if (passes >= 3)
            src = reinterpret_cast<int32_t *>(pb[1]);
        else if (passes == 2)
            src = g->in_col;
        else
            PRK_TRY(tmp.alloc((void **)&src, (size_t)m * sizeof(int32_t)));
        k_edge_sources<<<grid_for(radix_tiles, 1, g->num_sms * 8), kBlock, 0, s>>>(d_row_ptr, tile_rows, m,
                                                                                 radix_tiles, src);
        ++g->build_launches;
        PRK_CUDA(cudaGetLastError(), "k_edge_sources launch");
        clock.mark(PR_STAGE_SOURCES, s);
        PRK_TRY(staging.join());   // col_idx is on the device from here on
        for (int p = 0; p < passes; ++p) {
            const bool first = p == 0, last = p == passes - 1;
            const int2 *pin = first ? nullptr : pb[(p - 1) & 1];
            int2 *pout = last ? nullptr : pb[p & 1];
            const int shift = p * kRadixBits;
            const int64_t vn = first ? n : 0;   // the first upsweep checks col_idx
            if (first && last)
                st = sort_pass<kHistogram>(g, s, d_col, src, nullptr, n, nullptr, g->in_col, in_deg, m, shift, vn,
                                           counts, offsets, desc, tile_counter);
            else if (first)
                st = sort_pass<kPairsOut>(g, s, d_col, src, nullptr, n, pout, nullptr, in_deg, m, shift, vn,
                                          counts, offsets, desc, tile_counter);
            else if (last)
                st = sort_pass<kPairsIn | kHistogram>(g, s, nullptr, nullptr, pin, n, nullptr, g->in_col, in_deg, m,
                                                      shift, vn, counts, offsets, desc, tile_counter);
            else
                st = sort_pass<kPairsIn | kPairsOut>(g, s, nullptr, nullptr, pin, n, pout, nullptr, in_deg, m,
                                                     shift, vn, counts, offsets, desc, tile_counter);
            if (st != PR_OK)
                return st;
        }
    }

    if (m == 0)
        clock.mark(PR_STAGE_SOURCES, s);

    // 4: in_ptr = exclusive scan of the in-degrees (n + 1 outputs), once the
    // input is known to be valid
    PRK_TRY(check());
    clock.mark(PR_STAGE_SORT, s);
    PRK_TRY(launch_scan(LoadCount{in_deg}, g->in_ptr, n, desc, tile_counter, g->err,
                        &g->build_launches, s));
    clock.mark(PR_STAGE_OFFSETS, s);

    // the work order: a stable counting sort of the vertices by (class,
    // out-degree bucket), its inverse, and the degrees in work order
    int32_t *pdeg = nullptr;
    PRK_TRY(tmp.alloc((void **)&pdeg, (size_t)n * sizeof(int32_t)));
    {
        int32_t *okeys = nullptr, *ovals = nullptr;
        PRK_TRY(tmp.alloc((void **)&okeys, (size_t)n * sizeof(int32_t)));
        PRK_TRY(tmp.alloc((void **)&ovals, (size_t)n * sizeof(int32_t)));
        k_order_keys<<<grid_for(n, kBlock, cap), kBlock, 0, s>>>(n, g->in_ptr, g->deg_out, g->thread_max,
                                                                 g->warp_max, okeys, ovals);
        ++g->build_launches;
        PRK_TRY(sort_pass<0u>(g, s, okeys, ovals, nullptr, n, nullptr, g->order, nullptr, n, 0, 0, counts, offsets,
                              desc, tile_counter));
        k_invert<<<grid_for(n, kBlock, cap), kBlock, 0, s>>>(n, g->order, in_deg, g->deg_out, g->perm, g->w_deg,
                                                             pdeg);
        ++g->build_launches;
        PRK_CUDA(cudaGetLastError(), "order launch");
    }
    // class sizes: the scanned counts at the digit boundaries 64, 128, 192, 256
    // (keys are class * 64 + bucket)
    int32_t h_cls[5];
    for (int q = 0; q < 4; ++q)
        PRK_CUDA(cudaMemcpyAsync(&h_cls[q], offsets + (int64_t)(q + 1) * 64 * sort_ctas(g, order_tiles), sizeof(int32_t),
                                 cudaMemcpyDeviceToHost, s), "class counts");
    // key 255 (no in-edges, out-degree bucket of 0) holds exactly the vertices
    // with neither in- nor out-edges: the tail of the order
    PRK_CUDA(cudaMemcpyAsync(&h_cls[4], offsets + (int64_t)255 * sort_ctas(g, order_tiles), sizeof(int32_t),
                             cudaMemcpyDeviceToHost, s), "isolated count");
    PRK_TRY(check());
    clock.mark(PR_STAGE_ORDER, s);
    g->n_c = h_cls[0];
    g->n_w = h_cls[1] - h_cls[0];
    g->n_t = h_cls[2] - h_cls[1];
    g->n_z = h_cls[3] - h_cls[2];
    g->n_iso = h_cls[3] - h_cls[4];

    // the work CSR's offsets in class-major order, and the chunks of the CTA
    // rows (work rows [0, n_c)); one read of both totals
    PRK_TRY(launch_scan(LoadWorkDeg{pdeg, g->n_c + g->n_w, g->n_c + g->n_w + g->n_t}, g->w_ptr, n, desc, tile_counter,
                        g->err, &g->build_launches, s));
    PRK_TRY(graph_alloc(g, (void **)&g->chunk_first, (size_t)(g->n_c + 1) * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->hub_arrivals, (size_t)(g->n_c + 1) * sizeof(uint32_t), s));
    PRK_CUDA(cudaMemsetAsync(g->hub_arrivals, 0, (size_t)(g->n_c + 1) * sizeof(uint32_t), s), "memset");
    PRK_TRY(launch_scan(LoadChunkCount{g->w_ptr}, g->chunk_first, g->n_c, desc, tile_counter, g->err,
                        &g->build_launches, s));
    if (g->n_t > 0) {
        k_first_short_block<<<1, 1, 0, s>>>(g->w_ptr, g->n_c + g->n_w, (g->n_t + 31) / 32, counters + 4);
        ++g->build_launches;
    }
    PRK_CUDA(cudaGetLastError(), "short-block launch");
    int32_t h_sizes[2] = {0, 0};   // work CSR entries, CTA-row chunks
    unsigned long long h_short = 0;
    PRK_CUDA(cudaMemcpyAsync(&h_sizes[0], g->w_ptr + n, sizeof(int32_t), cudaMemcpyDeviceToHost, s), "work size");
    PRK_CUDA(cudaMemcpyAsync(&h_sizes[1], g->chunk_first + g->n_c, sizeof(int32_t), cudaMemcpyDeviceToHost, s),
             "chunk count");
    PRK_CUDA(cudaMemcpyAsync(&h_short, counters + 4, sizeof(h_short), cudaMemcpyDeviceToHost, s), "short blocks");
    PRK_TRY(check());
    g->m_w = h_sizes[0];
    g->n_chunks = h_sizes[1];
    g->t_short = (int64_t)h_short;
    PRK_TRY(graph_alloc(g, (void **)&g->w_col, (size_t)(g->m_w + 4) * sizeof(int32_t), s));
    PRK_TRY(graph_alloc(g, (void **)&g->chunk_row, (size_t)g->n_chunks * sizeof(int32_t), s));
    clock.mark(PR_STAGE_LAYOUT, s);
    g->build_launches += (g->n_c > 0);
    if (g->n_c > 0)
        k_fill_chunks<<<grid_for(g->n_c, 1, cap), kBlock, 0, s>>>(g->n_c, g->n_chunks, g->chunk_first,
                                                                   g->chunk_row);
    PRK_CUDA(cudaGetLastError(), "chunk launch");
    if (g->m_w > 0) {
        // the two relabel launches run side by side: the thread-class one on
        // a second stream, forked from and joined back to the build's stream
        const int64_t wide_end = g->n_c + g->n_w, rows_end = wide_end + g->n_t;
        const bool both = wide_end > 0 && g->n_t > 0;
        cudaStream_t side = s;
        ForkJoin fj;
        if (both) {
            PRK_TRY(side_stream(&side));
            PRK_TRY(fj.fork(s, side));
        }
        if (g->n_t > 0) {
            k_relabel<false><<<grid_for(g->n_t, kBlock, g->num_sms * 4), kBlock, 0, side>>>(
                n, g->n_c, g->n_chunks, wide_end, rows_end, g->chunk_row, g->chunk_first, g->w_ptr, g->order,
                g->perm, g->in_ptr, g->in_col, g->w_col, counters + 1, counters + 5);
            ++g->build_launches;
        }
        if (wide_end > 0) {
            k_relabel<true><<<g->num_sms * 8, kBlock, 0, s>>>(n, g->n_c, g->n_chunks, wide_end, rows_end,
                                                               g->chunk_row, g->chunk_first, g->w_ptr, g->order,
                                                               g->perm, g->in_ptr, g->in_col, g->w_col,
                                                               counters + 1, counters + 5);
            ++g->build_launches;
        }
        PRK_TRY(fj.join());
    }
    PRK_CUDA(cudaGetLastError(), "relabel launch");
    clock.mark(PR_STAGE_RELABEL, s);

    // the fp32 run's state and iteration graph, built on the host while the
    // relabel runs (pr_run would otherwise build them with the device idle)
    PRK_TRY(prepare_dtype(g, PR_F32, s));

    unsigned long long h_counters[7] = {0, 0, 0, 0, 0, 0, 0};
    PRK_CUDA(cudaMemcpyAsync(h_counters, counters, sizeof(h_counters), cudaMemcpyDeviceToHost, s),
             "counters");
    clock.mark(PR_STAGE_FINISH, s);
    PRK_CUDA(cudaEventRecord(g->ev[1], s), "cudaEventRecord");
    PRK_TRY(check());
    cudaEventElapsedTime(&g->build_ms, g->ev[0], g->ev[1]);
    clock.read(g->build_stage_ms);
    g->n_dangling = (int64_t)h_counters[0];
    g->e_c = (int64_t)h_counters[1];
    g->e_w = (int64_t)h_counters[2];
    g->e_t = (int64_t)h_counters[3];
    g->e_hot[0] = (int64_t)h_counters[5];
    g->e_hot[1] = (int64_t)h_counters[6];
    return PR_OK;
#undef PRK_TRY
#undef PRK_CUDA
}

}  // namespace prk
