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
//   - the pull SpMV gathers s over the class-major work CSR (the in-edge CSR
//     relabelled so that each in-degree class is one contiguous range of rows
//     and edges, see transpose.cu), by class: rows above 1024 in-edges are
//     streamed in 256-edge chunks, each warp a contiguous range of chunks,
//     and the warp that completes a row adds its pieces in chunk order (no
//     CTA-wide barrier); rows of 33..1024 in-edges are taken 32 consecutive
//     rows at a time by one warp that streams their int4s flat and forms the
//     row sums with a segmented scan; rows of 1..32 in-edges one per lane,
//     sorted by length and stored interleaved by blocks of 32, each warp
//     reading where its next 32 blocks lie before it starts them; rows
//     without in-edges take the constant term only (after the first update,
//     those that have no out-edges either are not touched: they all add the
//     same L1 and dangling terms, counted once). Every row is padded to
//     whole 16-byte index loads. Each warp takes the three gathering classes
//     in its own order (starting at class warp % 3), so the classes run side
//     by side on every SM;
//   - the combine reads D from device memory (Day 40, "Keep the dangling mass
//     on the device"), writes s' and accumulates the L1 distance and the next
//     dangling mass;
//   - the two reductions go thread -> warp -> CTA -> one 64-bit fixed-point
//     partial per CTA (exact, so the totals do not depend on the order), and
//     the last CTA to arrive sums the partials (Day 40 budget
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
    const int32_t *w_ptr;     // work CSR offsets (class-major order)
    const int32_t *w_col;     // work sources; padding entries are kPadSource
    const int32_t *w_deg;     // out-degrees in work order
    const int32_t *chunk_row, *chunk_first;
    uint32_t *hub_arrivals;
    T *s0, *s1;               // state [n + 1], slot n is 0
    T *hub_partial;
    unsigned long long *block_partials;   // [grid][2] fixed-point L1 and D of each CTA
    Scalars *scal;
    const int32_t *perm;      // vertex id -> work position (start vector, output)
    const int32_t *order;     // work position -> vertex id
    const int32_t *deg_out;   // out-degrees by vertex id
    const int32_t *w_split;   // [warps + 1]: warp-class rows of each warp of the grid
    int64_t n, n_c, n_w, n_t, n_z, n_chunks;
    int64_t n_iso;            // the last rows of the zero class: no in- and no out-edges
    int64_t t_short;          // first thread-class block whose rows span at most two int4s
    int rotate;               // 1: warp w starts at gather class w % 3
};

// streaming (evict-first) loads of the index stream
__device__ __forceinline__ int4 ld_stream4(const int4 *p) { return __ldcs(p); }

// Asynchronous 16-byte global -> shared copies (cp.async, L2 only), their
// commit, and the wait for all of this thread's outstanding ones.
__device__ __forceinline__ void cp_async16(int4 *smem_dst, const int4 *gmem_src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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

// The gathered state: slots below `hot` come from the CTA's shared-memory
// copy of the head of the state vector, the rest from L2 (ld.global.cg: a
// random gather gains nothing from L1, and not allocating there leaves L1 to
// the loads in flight). A padding entry (kPadSource, negative) contributes 0.
template <typename T>
struct Gather {
    const T *__restrict__ s;   // global state (s_old)
    const T *h;                // shared copy of s[0, hot)
    int32_t hot;
    __device__ __forceinline__ T operator()(int32_t u) const
    {
        return u < 0 ? T(0) : u < hot ? h[u] : __ldcg(s + u);
    }
    __device__ __forceinline__ T four(int4 q) const
    {
        return ((*this)(q.x) + (*this)(q.y)) + ((*this)(q.z) + (*this)(q.w));
    }
};

// L1 and dangling-mass terms are summed as 64-bit fixed-point integers with
// kFixBits fraction bits: integer addition is exact and associative, so the
// totals do not depend on which thread, warp or CTA adds which term, and a run
// repeats bit for bit. Every term is in [0, 1] and each total is at most 2,
// so kFixBits = 61 cannot overflow; rounding each term to 2^-61 bounds the
// error of a total by n * 2^-62 (4e-12 for n = 2^24). The conversion works on
// the bit pattern (integer ALU only), which keeps fp64 runs off the FP64 pipe.
constexpr int kFixBits = 61;

__device__ __forceinline__ unsigned long long shift_round(unsigned long long mant, int sh)
{
    if (sh >= 0)
        return mant << sh;
    sh = -sh;
    if (sh >= 64)
        return 0ull;
    return (mant + (1ull << (sh - 1))) >> sh;
}

// x >= 0 (and <= 2) to fixed point
__device__ __forceinline__ unsigned long long to_fixed(float x)
{
    const unsigned bits = __float_as_uint(x);
    const int e = (int)((bits >> 23) & 0xFF);
    if (e == 0)
        return 0ull;   // zero or denormal (< 2^-126): below the resolution
    const unsigned long long mant = (bits & 0x7FFFFFu) | 0x800000u;   // value = mant * 2^(e-150)
    return shift_round(mant, e - 150 + kFixBits);
}

__device__ __forceinline__ unsigned long long to_fixed(double x)
{
    const unsigned long long bits = (unsigned long long)__double_as_longlong(x);
    const int e = (int)((bits >> 52) & 0x7FF);
    if (e == 0)
        return 0ull;
    const unsigned long long mant = (bits & 0xFFFFFFFFFFFFFull) | (1ull << 52);   // value = mant * 2^(e-1075)
    return shift_round(mant, e - 1075 + kFixBits);
}

__device__ __forceinline__ double from_fixed(unsigned long long f)
{
    return (double)f * 0x1p-61;
}

__device__ __forceinline__ float abs_t(float x) { return fabsf(x); }
__device__ __forceinline__ double abs_t(double x) { return ::fabs(x); }

// The combine for work row i, given its out-degree and old state: new rank,
// new state, L1 and dangling-mass terms.
template <typename T>
__device__ __forceinline__ void combine_row(int64_t i, T y, int32_t deg, T so, T *__restrict__ s_new,
                                            T base, T d, unsigned long long &l1,
                                            unsigned long long &dm)
{
    const T x_old = deg ? so * T(deg) : so;
    const T x_new = base + d * y;
    l1 += to_fixed(abs_t(x_new - x_old));
    if (deg) {
        __stcs(s_new + i, x_new / T(deg));
    } else {
        __stcs(s_new + i, x_new);
        dm += to_fixed(x_new);
    }
}

template <typename T>
__device__ __forceinline__ void finish_row(int64_t i, T y, const int32_t *__restrict__ w_deg,
                                           const T *__restrict__ s_old, T *__restrict__ s_new,
                                           T base, T d, unsigned long long &l1,
                                           unsigned long long &dm)
{
    combine_row(i, y, w_deg[i], s_old[i], s_new, base, d, l1, dm);
}

// Offsets of a block of up to 32 consecutive work rows [r0, r0 + cnt), in
// 16-byte units: lane j gets row j's start relative to the block's first
// int4 (rows past cnt get nvec).
struct RowBlock {
    int32_t seg0;   // first int4 of the block
    int32_t nvec;   // int4s in the block
    int32_t cs;     // this lane's row start, relative to seg0
};

__device__ __forceinline__ RowBlock load_row_block(const int32_t *__restrict__ w_ptr, int64_t r0, int cnt,
                                                   int lane)
{
    RowBlock b;
    const int32_t mine = lane < cnt ? w_ptr[r0 + lane] : 0;
    const int32_t end = w_ptr[r0 + cnt];
    b.seg0 = __shfl_sync(0xffffffffu, mine, 0) >> 2;
    b.nvec = (end >> 2) - b.seg0;
    b.cs = lane < cnt ? (mine >> 2) - b.seg0 : b.nvec;
    return b;
}

// Thread-class rows: lane j owns row j of a block of cnt <= 32 consecutive
// work rows. The rows of a block all span len int4s, stored interleaved
// (int4 k of row j at blk + k * cnt + j), so a warp's loads are coalesced.
template <typename T>
struct LaneRow {
    int32_t off;       // this lane's first int4 (index into the work CSR)
    int32_t len, cnt;  // int4s per row (0: no row in this lane), rows in the block
    int32_t deg;       // out-degree and old state, for the combine
    T so;
};

// Where a thread-class block lies in the work CSR: its first int4 and the
// length in int4s that all its rows share (the block's first row is its
// longest, and every row of the block is padded to that length).
struct BlockDesc {
    int32_t off4, len4;
};

// Lane j reads the descriptor of block b0 + j * stride (j < 32, blocks below
// nblocks; the others get an empty one). A warp reads the descriptors of its
// next 32 blocks at once, so the index loads of a block never wait on w_ptr.
__device__ __forceinline__ BlockDesc load_block_descs(const int32_t *__restrict__ w_ptr, int64_t t_begin,
                                                      int64_t b0, int64_t stride, int64_t nblocks, int lane)
{
    BlockDesc d{0, 0};
    const int64_t b = b0 + (int64_t)lane * stride;
    if (b < nblocks) {
        const int64_t r = t_begin + b * 32;
        const int32_t p = w_ptr[r];
        d.off4 = p >> 2;
        d.len4 = (w_ptr[r + 1] - p) >> 2;   // every thread-class row spans at least one int4
    }
    return d;
}

// Lane rows of the block at work row r0 (rows past t_end are inactive), the
// block's placement taken from lane k's descriptor.
template <typename T>
__device__ __forceinline__ LaneRow<T> lane_row_of(const IterArgs<T> &a, const T *__restrict__ s_old, int64_t r0,
                                                  int64_t t_end, const BlockDesc &desc, int k, int lane)
{
    LaneRow<T> r;
    const int64_t i = r0 + lane;
    const bool act = i < t_end;
    r.cnt = (int)min((int64_t)32, t_end - r0);
    r.off = __shfl_sync(0xffffffffu, desc.off4, k) + lane;
    const int32_t len = __shfl_sync(0xffffffffu, desc.len4, k);
    r.len = act ? len : 0;
    r.deg = 0;
    r.so = T(0);
    if (act) {
        r.deg = a.w_deg[i];
        r.so = s_old[i];
    }
    return r;
}

// Row sum of one lane row, up to four int4s (16 gathers) in flight.
template <typename T>
__device__ __forceinline__ T lane_row_sum(const LaneRow<T> &R, const int4 *__restrict__ cv, const Gather<T> &gat)
{
    T y = T(0);
    for (int32_t k = 0; k < R.len; k += 4) {
        int4 q[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (k + t < R.len)
                q[t] = ld_stream4(cv + R.off + (k + t) * R.cnt);
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (k + t < R.len)
                y += gat.four(q[t]);
    }
    return y;
}

// Row sums of two lane rows of at most two int4s each (A and B, from two
// blocks), all their loads in flight at once. Each row adds its int4s in order.
template <typename T>
__device__ __forceinline__ void short_row_sums2(const LaneRow<T> &A, const LaneRow<T> &B,
                                                const int4 *__restrict__ cv, const Gather<T> &gat, T &ya, T &yb)
{
    int4 qa0, qa1, qb0, qb1;
    const bool a0 = 0 < A.len, a1 = 1 < A.len, b0 = 0 < B.len, b1 = 1 < B.len;
    if (a0)
        qa0 = ld_stream4(cv + A.off);
    if (a1)
        qa1 = ld_stream4(cv + A.off + A.cnt);
    if (b0)
        qb0 = ld_stream4(cv + B.off);
    if (b1)
        qb1 = ld_stream4(cv + B.off + B.cnt);
    ya = T(0);
    yb = T(0);
    if (a0)
        ya += gat.four(qa0);
    if (a1)
        ya += gat.four(qa1);
    if (b0)
        yb += gat.four(qb0);
    if (b1)
        yb += gat.four(qb1);
}

// Row sums of a block of up to 32 consecutive work rows, each padded to
// whole int4s, lane j owning row j. The warp streams the block's int4s in
// coalesced 32-wide steps, U steps of loads (4U gathers per lane) in flight
// at once, so every lane has work whatever the row lengths. The row of each
// int4 comes from a bisection over the lanes' row starts, and a segmented
// scan forms each row's run within the step: the lane holding the run's last
// int4 hands the run sum to the row's owner. A row may span many steps. The
// order of every addition is fixed by the layout, so the sums repeat bit for
// bit.
template <int U, typename T>
__device__ __forceinline__ T block_row_sums(const RowBlock &b, int cnt, const int4 *__restrict__ cv,
                                            const Gather<T> &gat, int lane)
{
    int32_t ce = __shfl_down_sync(0xffffffffu, b.cs, 1);
    if (lane >= cnt - 1)
        ce = b.nvec;
    T acc = T(0);
    for (int32_t p0 = 0; p0 < b.nvec; p0 += 32 * U) {
        int4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int32_t p = p0 + 32 * u + lane;
            if (p < b.nvec)
                q[u] = ld_stream4(cv + b.seg0 + p);
        }
        T v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = (p0 + 32 * u + lane < b.nvec) ? gat.four(q[u]) : T(0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int32_t ps = p0 + 32 * u;   // warp-uniform
            if (ps < b.nvec) {
                const int32_t p = ps + lane;
                int32_t row = 0, rs = 0;   // largest j < cnt with cs_j <= p, and cs_j
#pragma unroll
                for (int step = 16; step >= 1; step >>= 1) {
                    const int32_t cand = row + step;
                    const int32_t c_cs = __shfl_sync(0xffffffffu, b.cs, cand & 31);
                    if (cand < cnt && c_cs <= p) {
                        row = cand;
                        rs = c_cs;
                    }
                }
                // lanes [lo, lane] of this step hold int4s of this lane's row
                const int lo = max(rs - ps, 0);
                T x = v[u];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const T t = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane - o >= lo)
                        x += t;
                }
                const int32_t last = min(ce, ps + 32) - 1;   // row's last int4 in this step
                const T got = __shfl_sync(0xffffffffu, x, (last - ps) & 31);
                if (lane < cnt && last >= max(b.cs, ps))
                    acc += got;
            }
        }
    }
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kIterBlock, 1)
k_iterate(IterArgs<T> a, int32_t hot, cudaGraphConditionalHandle cond)
{
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ unsigned long long s_redf[32];
    __shared__ int s_flag;
    constexpr int kWarps = kIterBlock / 32;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t G = gridDim.x;

    // run scalars, read once (the last CTA rewrites them after every other
    // CTA has passed its arrival). A launch that follows the update which
    // ended the loop, in the same trip of the WHILE body, does nothing.
    const volatile Scalars *vs = a.scal;
    if (vs->stop)
        return;
    const int it = vs->it;
    const double dd = vs->d, inv_n = vs->inv_n, D = vs->dmass;
    const T *__restrict__ s_old = (it & 1) ? a.s1 : a.s0;
    T *__restrict__ s_new = (it & 1) ? a.s0 : a.s1;
    const T d = T(dd);
    const T base = T((1.0 - dd) * inv_n + dd * D * inv_n);

    unsigned long long l1 = 0ull, dm = 0ull;   // fixed point, see to_fixed

    // The head of the state vector, where the work order puts the most
    // gathered vertices, is staged in shared memory for this update with
    // asynchronous 16-byte copies (cp.async; both buffers are 16-byte
    // aligned). The rows without in-edges, which gather nothing, are combined
    // while the copies land.
    T *s_hot = reinterpret_cast<T *>(s_dyn);
    {
        const int32_t hot4 = (int32_t)((int64_t)hot * (int64_t)sizeof(T) / 16);
        const int4 *src = reinterpret_cast<const int4 *>(s_old);
        int4 *dst = reinterpret_cast<int4 *>(s_hot);
        for (int32_t q = tid; q < hot4; q += kIterBlock)
            cp_async16(dst + q, src + q);
        cp_async_commit();
        for (int32_t u = (int32_t)(hot4 * 16 / (int32_t)sizeof(T)) + tid; u < hot; u += kIterBlock)
            s_hot[u] = s_old[u];
    }

    // rows without in-edges: x' = base; eight rows per thread in flight.
    // From the second update on, the isolated rows at the end of the class
    // (no out-edges either, so never gathered) are not touched: each had
    // x = the previous update's base, so together they add n_iso times one
    // L1 term and one dangling term, and the output takes their rank from
    // base_last. The integer sums are the same as row by row.
    {
        const int64_t z0 = a.n - a.n_z, stride = G * kIterBlock;
        const int64_t z_end = it == 0 ? a.n : a.n - a.n_iso;
        for (int64_t i = z0 + (int64_t)blockIdx.x * kIterBlock + tid; i < z_end; i += 8 * stride) {
            int32_t dg[8];
            T so[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (i + t * stride < z_end) {
                    dg[t] = a.w_deg[i + t * stride];
                    so[t] = s_old[i + t * stride];
                }
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (i + t * stride < z_end)
                    combine_row(i + t * stride, T(0), dg[t], so[t], s_new, base, d, l1, dm);
        }
        if (it > 0 && a.n_iso > 0 && blockIdx.x == 0 && tid == 0) {
            const T prev = T(vs->base_last);
            l1 += (unsigned long long)a.n_iso * to_fixed(abs_t(base - prev));
            dm += (unsigned long long)a.n_iso * to_fixed(base);
        }
    }
    cp_async_wait_all();
    __syncthreads();
    const Gather<T> gat{s_old, s_hot, hot};

    // Work ranges are numbered warp-major across the grid (gw = warp * G +
    // CTA), so the 32 warps of a CTA take ranges spread evenly over each
    // class instead of 32 neighbouring ones: rows at the head of a class cost
    // more than rows at its tail, and every CTA gets the same mix.
    //
    // CTA class: rows with more than 1024 in-edges, cut into chunks of
    // kChunkEdges (whole int4s). Warp gw streams the contiguous chunk range
    // [gw * per, (gw + 1) * per). A warp sums each row's chunks in its range
    // in registers; a row that lies wholly in the range is combined at once. A row that
    // crosses a range boundary is handed off: each warp stores its piece's
    // sum at the piece's first chunk (the row's first chunk, or a multiple of
    // `per`), adds its chunk count to the row's arrival counter, and the warp
    // that completes the count adds the pieces in chunk order and combines
    // the row. No CTA-wide barrier, and no wait.
    const int64_t gw = (int64_t)warp * G + blockIdx.x;
    const int4 *cv = reinterpret_cast<const int4 *>(a.w_col);
    auto phase_hub = [&]() {
        const int64_t nwarps = G * kWarps;
        const int64_t per = (a.n_chunks + nwarps - 1) / nwarps;
        const int64_t c_end = min((gw + 1) * per, a.n_chunks);
        const int4 *cv_all = reinterpret_cast<const int4 *>(a.w_col);
        constexpr int kVecPerLane = kChunkEdges / 4 / 32;
        int64_t c = gw * per;
        while (c < c_end) {
            const int32_t r = a.chunk_row[c];
            const int32_t first = a.chunk_first[r];
            const int32_t nch = a.chunk_first[r + 1] - first;
            const int64_t stop = min((int64_t)first + nch, c_end);
            const int64_t row_b = a.w_ptr[r], row_e = a.w_ptr[r + 1];
            T acc = T(0);
            for (int64_t cc = c; cc < stop; ++cc) {
                const int64_t cb = row_b + (cc - first) * kChunkEdges;
                const int nv = (int)((min(cb + (int64_t)kChunkEdges, row_e) - cb) >> 2);
                const int4 *cv = cv_all + (cb >> 2);
                int4 q[kVecPerLane];
#pragma unroll
                for (int t = 0; t < kVecPerLane; ++t)
                    if (lane + 32 * t < nv)
                        q[t] = ld_stream4(cv + lane + 32 * t);
#pragma unroll
                for (int t = 0; t < kVecPerLane; ++t)
                    if (lane + 32 * t < nv)
                        acc += gat.four(q[t]);
            }
            acc = warp_sum(acc);
            const int32_t covered = (int32_t)(stop - c);
            if (covered == nch) {
                if (lane == 0)
                    finish_row(r, acc, a.w_deg, s_old, s_new, base, d, l1, dm);
            } else {
                uint32_t prev = 0;
                if (lane == 0) {
                    __stcg(a.hub_partial + c, acc);
                    __threadfence();
                    prev = atomicAdd(a.hub_arrivals + r, (uint32_t)covered);
                }
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev + (uint32_t)covered == (uint32_t)nch) {
                    __threadfence();
                    T y = T(0);
                    for (int32_t k = lane; k < nch; k += 32) {
                        const int64_t cc = (int64_t)first + k;
                        if (k == 0 || cc % per == 0)
                            y += __ldcg(a.hub_partial + cc);
                    }
                    y = warp_sum(y);
                    if (lane == 0) {
                        a.hub_arrivals[r] = 0u;
                        finish_row(r, y, a.w_deg, s_old, s_new, base, d, l1, dm);
                    }
                }
            }
            c = stop;
        }
    };

    // warp class (33..1024 in-edges) and thread class (1..32), in blocks of
    // 32 consecutive rows. Warp-class rows: each warp owns one contiguous
    // range of rows, cut so that every warp has about the same edges
    // (w_split), and streams each block's int4s (block_row_sums).
    // Thread-class rows: the warps of the grid sweep the blocks round-robin,
    // one row per lane, the blocks stored interleaved: blocks of long rows
    // one at a time (lane_row_sum), blocks of short rows two at a time
    // (short_row_sums2). The old state and out-degree of a block's
    // rows are loaded before its gathers; in the warp class, the next block's
    // offsets are loaded while they are in flight.
    auto phase_warp = [&]() {
        const int64_t r_begin = a.w_split[gw], r_end = a.w_split[gw + 1];
        if (r_begin < r_end) {
            RowBlock nb = load_row_block(a.w_ptr, r_begin, (int)min((int64_t)32, r_end - r_begin), lane);
            for (int64_t r0 = r_begin; r0 < r_end; r0 += 32) {
                const int cnt = (int)min((int64_t)32, r_end - r0);
                const RowBlock b = nb;
                int32_t deg = 0;
                T so = T(0);
                if (lane < cnt) {
                    deg = a.w_deg[r0 + lane];
                    so = s_old[r0 + lane];
                }
                const int64_t r1 = r0 + 32;
                if (r1 < r_end)
                    nb = load_row_block(a.w_ptr, r1, (int)min((int64_t)32, r_end - r1), lane);
                const T y = block_row_sums<4>(b, cnt, cv, gat, lane);
                if (lane < cnt)
                    combine_row(r0 + lane, y, deg, so, s_new, base, d, l1, dm);
            }
        }
    };
    auto phase_thread = [&]() {
        const int64_t t_begin = a.n_c + a.n_w, t_end = t_begin + a.n_t;
        const int64_t nw = G * kWarps;
        const int64_t t_blocks = (t_end - t_begin + 31) / 32;
        const int64_t t_short = min(a.t_short, t_blocks);
        // rows of three to eight int4s: one block per warp at a time (blocks
        // gw, gw + nw, ...), their descriptors read 32 blocks ahead
        for (int64_t b0 = gw; b0 < t_short; b0 += 32 * nw) {
            const BlockDesc desc = load_block_descs(a.w_ptr, t_begin, b0, nw, t_short, lane);
            for (int k = 0; k < 32; ++k) {
                const int64_t bb = b0 + k * nw;
                if (bb >= t_short)   // warp-uniform
                    break;
                const LaneRow<T> A = lane_row_of(a, s_old, t_begin + bb * 32, t_end, desc, k, lane);
                const T y = lane_row_sum(A, cv, gat);
                if (A.len > 0)
                    combine_row(t_begin + bb * 32 + lane, y, A.deg, A.so, s_new, base, d, l1, dm);
            }
        }
        // rows of one or two int4s: two blocks per warp at a time (blocks bb
        // and bb + nw, bb = t_short + gw, then every 2 nw), descriptors read
        // 16 pairs ahead
        for (int64_t b0 = t_short + gw; b0 < t_blocks; b0 += 32 * nw) {
            const BlockDesc desc = load_block_descs(a.w_ptr, t_begin, b0, nw, t_blocks, lane);
            for (int k = 0; k < 32; k += 2) {
                const int64_t bb = b0 + k * nw;
                if (bb >= t_blocks)   // warp-uniform
                    break;
                const bool has_b = bb + nw < t_blocks;   // warp-uniform
                const LaneRow<T> A = lane_row_of(a, s_old, t_begin + bb * 32, t_end, desc, k, lane);
                const LaneRow<T> B = has_b ? lane_row_of(a, s_old, t_begin + (bb + nw) * 32, t_end, desc, k + 1, lane)
                                           : LaneRow<T>{0, 0, 1, 0, T(0)};
                T ya, yb;
                short_row_sums2(A, B, cv, gat, ya, yb);
                if (A.len > 0)
                    combine_row(t_begin + bb * 32 + lane, ya, A.deg, A.so, s_new, base, d, l1, dm);
                if (B.len > 0)
                    combine_row(t_begin + (bb + nw) * 32 + lane, yb, B.deg, B.so, s_new, base, d, l1, dm);
            }
        }
    };
    // On graphs with many rows, each warp takes the three gather phases in
    // its own order: warp w of the CTA starts with phase w % 3 (hub,
    // warp-class, thread-class) and wraps around. Every SM then runs all
    // three at once, and the thread class, whose short rows leave few gathers
    // in flight per warp, overlaps the streaming classes instead of running
    // alone at the end of the update. On small graphs (a.rotate == 0), which
    // sit in L2 and are bound by fixed costs, every warp takes the classes in
    // one order. What a warp computes does not depend on the order (no phase
    // waits on another, and the L1 and D totals are exact).
    const int rot = a.rotate ? warp % 3 : 0;
    if (rot == 0) {
        phase_hub();
        phase_warp();
        phase_thread();
    } else if (rot == 1) {
        phase_warp();
        phase_thread();
        phase_hub();
    } else {
        phase_thread();
        phase_hub();
        phase_warp();
    }

    // reductions: one fp64 partial pair per CTA, the last CTA sums them
    const unsigned long long l1_blk = block_sum(l1, s_redf);
    const unsigned long long dm_blk = block_sum(dm, s_redf);
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
    unsigned long long Lf = 0ull, Mf = 0ull;
    for (int64_t b = tid; b < G; b += kIterBlock) {
        Lf += __ldcg(a.block_partials + 2 * b);
        Mf += __ldcg(a.block_partials + 2 * b + 1);
    }
    Lf = block_sum(Lf, s_redf);
    Mf = block_sum(Mf, s_redf);
    if (tid == 0) {
        const double L = from_fixed(Lf), M = from_fixed(Mf);
        Scalars *sc = a.scal;
        const int it1 = it + 1;
        const bool conv = (sc->tol > 0.0) && (L < sc->tol);
        sc->l1 = L;
        sc->dmass = M;
        sc->it = it1;
        sc->converged = conv ? 1 : 0;
        sc->ticket = 0u;
        sc->base_last = (double)base;
        if (conv || it1 >= sc->max_iter) {
            sc->stop = 1;
            cudaGraphSetConditional(cond, 0);
        }
        __threadfence();
    }
}

// Start vector (1/n, or the caller's x_init in vertex ids), its state in
// work order and its dangling mass, and the run scalars.
template <typename T>
__global__ void __launch_bounds__(kBlock)
k_init(IterArgs<T> a, const T *__restrict__ x_init, double d, double tol, int32_t max_iter)
{
    __shared__ unsigned long long s_redf[32];
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    const int64_t G = gridDim.x;
    const T x_uniform = T(1.0 / (double)a.n);
    unsigned long long dm = 0ull;   // fixed point, see to_fixed
    if (blockIdx.x == 0 && tid == 0) {
        a.s0[a.n] = T(0);   // slot n stays 0 (the shared copy may include it)
        a.s1[a.n] = T(0);
    }
    for (int64_t i = (int64_t)blockIdx.x * kBlock + tid; i < a.n; i += G * kBlock) {
        const T x = x_init ? x_init[a.order[i]] : x_uniform;
        const int32_t deg = a.w_deg[i];
        if (deg) {
            a.s0[i] = x / T(deg);
        } else {
            a.s0[i] = x;
            dm += to_fixed(x);
        }
    }
    const unsigned long long dm_blk = block_sum(dm, s_redf);
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
    unsigned long long Mf = 0ull;
    for (int64_t b = tid; b < G; b += kBlock)
        Mf += __ldcg(a.block_partials + 2 * b + 1);
    Mf = block_sum(Mf, s_redf);
    if (tid == 0) {
        Scalars *sc = a.scal;
        sc->dmass = from_fixed(Mf);
        sc->l1 = 0.0;
        sc->d = d;
        sc->tol = tol;
        sc->inv_n = 1.0 / (double)a.n;
        sc->it = 0;
        sc->max_iter = max_iter;
        sc->converged = 0;
        sc->ticket = 0u;
        sc->stop = 0;
        sc->base_last = 0.0;
    }
}

// Ranks from the final state, in vertex ids: x[v] = s[perm[v]] * outdeg[v],
// or s[perm[v]] for a dangling vertex.
template <typename T>
__global__ void k_output(IterArgs<T> a, T *__restrict__ out)
{
    const volatile Scalars *vs = a.scal;
    const int it = vs->it;
    const T base_last = T(vs->base_last);
    const int64_t iso0 = a.n - a.n_iso;   // isolated rows keep no state after the first update
    const T *s = (it & 1) ? a.s1 : a.s0;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < a.n;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int32_t deg = a.deg_out[v];
        const int32_t p = a.perm[v];
        const T sv = p >= iso0 ? base_last : s[p];
        out[v] = deg ? sv * T(deg) : sv;
    }
}

// Cuts rows [lo, hi) into `parts` contiguous ranges of about equal cost,
// cost(i) = edges of rows lo..i-1 + row_cost * (i - lo): split[p] is the first
// row whose cost reaches p/parts of the total (split[0] = lo, split[parts] = hi).
__global__ void k_split(const int32_t *__restrict__ w_ptr, int64_t lo, int64_t hi, int64_t parts,
                        int64_t row_cost, int32_t *__restrict__ split)
{
    const int64_t base_e = w_ptr[lo];
    const double total = (double)(w_ptr[hi] - base_e) + (double)row_cost * (double)(hi - lo);
    for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p <= parts;
         p += (int64_t)gridDim.x * blockDim.x) {
        const double target = total * (double)p / (double)parts;
        int64_t a = lo, b = hi;   // first i in [lo, hi] with cost(i) >= target
        while (a < b) {
            const int64_t mid = (a + b) >> 1;
            const double c = (double)(w_ptr[mid] - base_e) + (double)row_cost * (double)(mid - lo);
            if (c >= target)
                b = mid;
            else
                a = mid + 1;
        }
        split[p] = (int32_t)(p == parts ? hi : a);
    }
}

template <typename T>
IterArgs<T> make_args(pr_graph *g)
{
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    IterArgs<T> a;
    a.w_ptr = g->w_ptr;
    a.w_col = g->w_col;
    a.w_deg = g->w_deg;
    a.chunk_row = g->chunk_row;
    a.chunk_first = g->chunk_first;
    a.hub_arrivals = g->hub_arrivals;
    a.s0 = (T *)st.s[0];
    a.s1 = (T *)st.s[1];
    a.hub_partial = (T *)st.hub_partial;
    a.block_partials = st.block_partials;
    a.scal = g->scal;
    a.perm = g->perm;
    a.order = g->order;
    a.deg_out = g->deg_out;
    a.w_split = st.w_split;
    a.n = g->n;
    a.n_c = g->n_c;
    a.n_w = g->n_w;
    a.n_t = g->n_t;
    a.n_z = g->n_z;
    a.n_chunks = g->n_chunks;
    a.n_iso = g->n_iso;
    a.t_short = g->t_short;
    a.rotate = (g->n - g->n_z >= kRotateRows) ? 1 : 0;
    return a;
}

// Allocates a precision's state and builds its graph: one conditional WHILE
// node whose body is kUpdatesPerTrip chained k_iterate launches. Nothing here
// reads device results on the host, so the graph is built while the device
// still runs the work queued before it (for fp32, the end of pr_graph_create).
template <typename T>
pr_status prepare_once(pr_graph *g, cudaStream_t s);

// prepare_once, undone on failure: the blocks it took from the pool go back
// and the handle is as before, so a later pr_run can try again.
template <typename T>
pr_status prepare(pr_graph *g, cudaStream_t s)
{
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    if (st.ready)
        return PR_OK;
    const size_t n_allocs = g->allocs.size();
    const int64_t bytes = g->device_bytes;
    const pr_status r = prepare_once<T>(g, s);
    if (r != PR_OK) {
        for (size_t k = n_allocs; k < g->allocs.size(); ++k)
            pool_free(g->allocs[k], s);
        g->allocs.resize(n_allocs);
        g->device_bytes = bytes;
        st = DtypeState();
    }
    return r;
}

template <typename T>
pr_status prepare_once(pr_graph *g, cudaStream_t s)
{
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    pr_status r;
    const int64_t hot_cap = kHotBytes / (int64_t)sizeof(T);
    st.hot = (int32_t)(g->n + 1 < hot_cap ? g->n + 1 : hot_cap);
    st.smem = (size_t)st.hot * sizeof(T);
    // the kernel's limit is set to the largest copy any handle asks for, not
    // to this handle's: handles prepared from several host threads at once
    // then all write the same value, and no handle's graph is instantiated
    // while another thread has lowered the limit below its own size
    cudaError_t e = cudaFuncSetAttribute(k_iterate<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kHotBytes);
    if (e != cudaSuccess)
        return cuda_status(e, "shared memory attribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_iterate<T>, kIterBlock, st.smem);
    if (e != cudaSuccess)
        return cuda_status(e, "occupancy query");
    if (per_sm < 1)
        return set_error(PR_ERR_CUDA, "the update kernel does not fit on an SM");
    st.grid = per_sm * g->num_sms;
    st.init_grid = 8 * g->num_sms;
    const size_t n = (size_t)g->n;
    if ((r = graph_alloc(g, &st.s[0], (n + 1) * sizeof(T), s)) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.s[1], (n + 1) * sizeof(T), s)) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.stage, n * sizeof(T), s)) != PR_OK) return r;
    if ((r = graph_alloc(g, &st.hub_partial, (size_t)(g->n_chunks + 1) * sizeof(T), s)) != PR_OK) return r;
    const int pgrid = st.grid > st.init_grid ? st.grid : st.init_grid;
    if ((r = graph_alloc(g, (void **)&st.block_partials, (size_t)pgrid * 2 * sizeof(unsigned long long), s)) != PR_OK)
        return r;

    // edge-balanced ranges of warp-class rows, one per warp
    const int64_t warps = (int64_t)st.grid * (kIterBlock / 32);
    if ((r = graph_alloc(g, (void **)&st.w_split, (size_t)(warps + 1) * sizeof(int32_t), s)) != PR_OK)
        return r;
    const int64_t w0 = g->n_c, w1 = w0 + g->n_w;
    const int sg = (int)((warps + 1 + kBlock - 1) / kBlock);
    k_split<<<sg, kBlock, 0, s>>>(g->w_ptr, w0, w1, warps, kWarpRowCost, st.w_split);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_status(e, "splitting the classes");

    IterArgs<T> args = make_args<T>(g);
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaGraphConditionalHandle handle;
    cudaGraphNodeParams cp = {};
    cudaGraphNode_t cnode, knode;
    cudaKernelNodeParams kp = {};
    int32_t hot = st.hot;
    void *kargs[] = {&args, &hot, &handle};

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
        kp.blockDim = dim3(kIterBlock);
        kp.sharedMemBytes = (unsigned)st.smem;
        kp.kernelParams = kargs;
        // the WHILE body: kUpdatesPerTrip update launches in a chain
        cudaGraphNode_t prev = nullptr;
        for (int k = 0; k < kUpdatesPerTrip && e == cudaSuccess; ++k) {
            e = cudaGraphAddKernelNode(&knode, cp.conditional.phGraph_out[0], prev ? &prev : nullptr, prev ? 1 : 0,
                                       &kp);
            prev = knode;
        }
    }
    if (e == cudaSuccess)
        e = cudaGraphInstantiate(&exec, graph, 0);
    // the graph's one-time upload to the device belongs to preparation, not
    // to the first run's loop
    if (e == cudaSuccess)
        e = cudaGraphUpload(exec, s);
    if (e != cudaSuccess) {
        if (exec)
            cudaGraphExecDestroy(exec);
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
    // the caller's buffers: host memory, or memory the graph's device may
    // dereference; memory of another GPU is refused before any work
    const PtrKind out_kind = pointer_kind(ranks_out, g->device);
    const PtrKind xi_kind = x_init ? pointer_kind(x_init, g->device) : kPtrHost;
    if (out_kind == kPtrOtherDevice || xi_kind == kPtrOtherDevice)
        return set_error(PR_ERR_INVALID_ARG, "ranks_out and x_init must be host memory or memory of "
                                             "the graph's device (%d)", g->device);
    pr_status r = prepare<T>(g, s);
    if (r != PR_OK)
        return r;
    DtypeState &st = g->st[sizeof(T) == 8 ? 1 : 0];
    IterArgs<T> args = make_args<T>(g);
    const size_t bytes = (size_t)g->n * sizeof(T);
    cudaError_t e = cudaSuccess;

    const T *xi = nullptr;
    if (x_init) {
        if (xi_kind == kPtrDevice) {
            xi = (const T *)x_init;
        } else {
            e = cudaMemcpyAsync(st.stage, x_init, bytes, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess)
                return cuda_status(e, "copying x_init");
            xi = (const T *)st.stage;
        }
    }
    const bool out_dev = out_kind == kPtrDevice;
    T *out = out_dev ? (T *)ranks_out : (T *)st.stage;

    e = cudaEventRecord(g->ev[0], s);
    if (e == cudaSuccess) {
        NvtxRange range("pr_init");
        k_init<T><<<st.init_grid, kBlock, 0, s>>>(args, xi, d, tol, max_iter);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(g->ev[1], s);
    if (e == cudaSuccess) {
        NvtxRange range("pr_iterate");
        e = cudaGraphLaunch(st.exec, s);
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(g->ev[2], s);
    if (e == cudaSuccess) {
        NvtxRange range("pr_output");
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
    // init, every update launch of the loop's trips (the last trip may end
    // with launches that do nothing), output
    g->last.launches = (hs.it + kUpdatesPerTrip - 1) / kUpdatesPerTrip * kUpdatesPerTrip + 2;
    if (iters_out)
        *iters_out = hs.it;
    if (l1_out)
        *l1_out = hs.l1;
    if (tol > 0.0 && !hs.converged)
        return PR_NOT_CONVERGED;
    return PR_OK;
}

}  // namespace

pr_status prepare_dtype(pr_graph *g, int dtype, cudaStream_t s)
{
    return dtype == PR_F64 ? prepare<double>(g, s) : prepare<float>(g, s);
}

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
