// The random-gather rate of the current GPU, the bound of the update's
// gathers that the shared-memory copy of the state's head does not serve.
//
// The update gathers one state value per in-edge from a source that is, for
// all but the hottest vertices, unrelated to its neighbours in the edge
// stream: a 4- or 8-byte load from a random address. Each such load that
// misses L1 costs one L2 request, and the rate of those requests, not HBM
// bandwidth, is what the update runs into. This file measures that rate with
// a kernel that does nothing but random gathers from a state vector of the
// run's size and type, so that a run's gather rate can be reported as a
// fraction of it.
//
// Three paths are measured:
//   - loads: ld.global.cg from the warps (the path the update uses);
//   - the tensor memory accelerator: cp.async.bulk.tensor tile::gather4
//     copies, each bringing four 16-byte rows of a 2-D view of the state
//     ([rows][16 bytes]) at four row coordinates into shared memory, issued
//     by the lanes themselves and completed on mbarriers. These requests do
//     not go through the warps' load path;
//   - both at once, the index stream split between them in the ratio of
//     their rates measured alone.
#include <cuda.h>   // CUtensorMap and its enums (types only: the encoder is looked up at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "pr_internal.cuh"

namespace prk {
namespace {

constexpr int kGatherBlock = 256;
constexpr int kGatherVecs = 2;   // int4 index loads in flight per thread

// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): the finalizer of a Weyl sequence.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// idx[i] uniform in [0, n), state[i] = 0 for i < n_state (the values do not matter).
template <typename T>
__global__ void k_fill(int32_t *__restrict__ idx, int64_t count, T *__restrict__ state, int64_t n, int64_t n_state)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
        idx[i] = (int32_t)(splitmix64((uint64_t)i) % (uint64_t)n);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_state; i += stride)
        state[i] = T(0);
}

// Gathers state[idx[i]] for every i (indices streamed as int4s, two in
// flight per thread; gathers through L2, as the update's cold gathers) and
// keeps the sum, which is written only if it takes an impossible value, so
// that the loads are not removed.
template <typename T>
__global__ void __launch_bounds__(kGatherBlock)
k_gather(const int4 *__restrict__ idx, int64_t nvec, const T *__restrict__ state, T *__restrict__ sink)
{
    T acc = T(0);
    const int64_t stride = (int64_t)gridDim.x * kGatherBlock * kGatherVecs;
    for (int64_t b = (int64_t)blockIdx.x * kGatherBlock * kGatherVecs + threadIdx.x; b < nvec; b += stride) {
        int4 q[kGatherVecs];
#pragma unroll
        for (int u = 0; u < kGatherVecs; ++u)
            q[u] = b + u * kGatherBlock < nvec ? __ldcs(idx + b + u * kGatherBlock) : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kGatherVecs; ++u)
            acc += (__ldcg(state + q[u].x) + __ldcg(state + q[u].y)) +
                   (__ldcg(state + q[u].z) + __ldcg(state + q[u].w));
    }
    if (acc == T(-1))
        *sink = acc;
}

// ------------------------------------------------ tensor-memory-accelerator gathers --

constexpr int kTmaSlots = 4;           // gather4 copies in flight per lane
constexpr int kTmaSlotBytes = 128;     // 4 rows x 16 bytes, in 128-byte aligned slots
constexpr int kTmaSpinLimit = 1 << 20; // polls of an mbarrier before a wait gives up

__device__ __forceinline__ unsigned smem_u32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete, at most
// kTmaSpinLimit polls; false if it did not.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity)
{
    for (int i = 0; i < kTmaSpinLimit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

// Four 16-byte rows (row coordinates r0..r3, column 0) of the tensor `map`
// into 64 bytes of shared memory at dst, completing `bar`'s transaction count.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int r0, int r1, int r2, int r3,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
          "r"(smem_u32(bar))
        : "memory");
}

// Random gathers through both paths. Warps [0, 8 - tma_warps) of each CTA
// gather idx_load (as k_gather does); the lanes of the last tma_warps warps
// take the groups of four indices of idx_tma, each lane with kTmaSlots
// gather4 copies in flight, and add the gathered element of each row. A
// wait that gives up sets bit 0 of *err; the lane then issues no more
// copies and waits (bounded) for the ones it has in flight before leaving.
template <typename T>
__global__ void __launch_bounds__(kGatherBlock)
k_gather_tma(const __grid_constant__ CUtensorMap map, const int4 *__restrict__ idx_load, int64_t nvec_load,
             const int4 *__restrict__ idx_tma, int64_t groups_tma, const T *__restrict__ state,
             T *__restrict__ sink, unsigned *err, int tma_warps)
{
    extern __shared__ __align__(128) unsigned char s_tma[];
    constexpr int kRow = 16 / (int)sizeof(T);   // elements per 16-byte row
    const int tid = threadIdx.x;
    const int load_threads = kGatherBlock - 32 * tma_warps;
    const int tma_lanes = 32 * tma_warps;
    T acc = T(0);
    if (tid < load_threads) {
        const int64_t stride = (int64_t)gridDim.x * load_threads;
        for (int64_t b = (int64_t)blockIdx.x * load_threads + tid; b < nvec_load; b += stride) {
            const int4 q = __ldcs(idx_load + b);
            acc += (__ldcg(state + q.x) + __ldcg(state + q.y)) + (__ldcg(state + q.z) + __ldcg(state + q.w));
        }
    } else {
        const int tl = tid - load_threads;
        unsigned char *slot = s_tma + (size_t)tl * kTmaSlots * kTmaSlotBytes;
        uint64_t *bar = reinterpret_cast<uint64_t *>(s_tma + (size_t)tma_lanes * kTmaSlots * kTmaSlotBytes) +
                        tl * kTmaSlots;
        for (int k = 0; k < kTmaSlots; ++k)
            mbar_init(bar + k, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const int64_t stride = (int64_t)gridDim.x * tma_lanes;
        const int64_t g0 = (int64_t)blockIdx.x * tma_lanes + tl;
        unsigned parity = 0, pending = 0;   // per slot: phase to wait for, copy in flight
        auto issue = [&](int k, int64_t g) {
            const int4 q = __ldcs(idx_tma + g);
            mbar_expect_tx(bar + k, 4 * 16);
            tma_gather4(slot + k * kTmaSlotBytes, &map, q.x / kRow, q.y / kRow, q.z / kRow, q.w / kRow, bar + k);
            pending |= 1u << k;
        };
        for (int k = 0; k < kTmaSlots; ++k)
            if (g0 + k * stride < groups_tma)
                issue(k, g0 + k * stride);
        int k = 0;
        bool ok = true;
        for (int64_t g = g0; g < groups_tma; g += stride) {
            if (!mbar_wait(bar + k, (parity >> k) & 1u)) {
                ok = false;
                break;
            }
            parity ^= 1u << k;
            pending &= ~(1u << k);
            const int4 q = __ldcs(idx_tma + g);
            const T *row = reinterpret_cast<const T *>(slot + k * kTmaSlotBytes);
            acc += (row[q.x % kRow] + row[kRow + q.y % kRow]) + (row[2 * kRow + q.z % kRow] + row[3 * kRow + q.w % kRow]);
            const int64_t gn = g + (int64_t)kTmaSlots * stride;
            if (gn < groups_tma) {
                // the slot's reads above are done before the next copy overwrites it
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(k, gn);
            }
            k = (k + 1) % kTmaSlots;
        }
        if (!ok) {
            atomicOr(err, 1u);
            for (int j = 0; j < kTmaSlots; ++j)
                if (pending & (1u << j))
                    mbar_wait(bar + j, (parity >> j) & 1u);
        }
    }
    if (acc == T(-1))
        *sink = acc;
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 2-D tensor map over `rows` 16-byte rows of `state`: box one row high and
// 16 bytes wide (the shape tile::gather4 loads), no swizzle, no fill.
template <typename T>
pr_status encode_rows(CUtensorMap *map, void *state, int64_t rows)
{
    static EncodeTiled encode = nullptr;
    if (encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return set_error(PR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        encode = reinterpret_cast<EncodeTiled>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)(16 / sizeof(T)), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {16};
    const cuuint32_t box[2] = {(cuuint32_t)(16 / sizeof(T)), 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, sizeof(T) == 8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT64 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                              state, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(PR_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PR_OK;
}

template <typename T>
pr_status measure(int64_t n, int64_t gathers, int path, double *rate, cudaStream_t s)
{
    const int64_t count = (gathers + 3) & ~(int64_t)3;
    // the state padded to whole 16-byte rows, for the tensor map
    const int64_t rows = ((n + 1) * (int64_t)sizeof(T) + 15) / 16;
    const int64_t state_elems = rows * (16 / (int64_t)sizeof(T));
    int dev = 0, sms = 0, per_sm = 0, per_sm_tma = 0, per_sm_both = 0;
    const int tma_only_warps = kGatherBlock / 32, both_warps = 1;
    const size_t smem_only = (size_t)32 * tma_only_warps * kTmaSlots * (kTmaSlotBytes + 8);
    const size_t smem_both = (size_t)32 * both_warps * kTmaSlots * (kTmaSlotBytes + 8);
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gather<T>, kGatherBlock, 0);
    if (e == cudaSuccess && path != PR_GATHER_LOAD) {
        e = cudaFuncSetAttribute(k_gather_tma<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_only);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_tma, k_gather_tma<T>, kGatherBlock, smem_only);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_both, k_gather_tma<T>, kGatherBlock, smem_both);
    }
    if (e != cudaSuccess)
        return cuda_status(e, "device query");
    void *idx = nullptr, *state = nullptr;
    unsigned *err = nullptr;
    pr_status st = pool_alloc(&idx, (size_t)count * sizeof(int32_t), s);
    if (st == PR_OK)
        st = pool_alloc(&state, (size_t)state_elems * sizeof(T), s);
    if (st == PR_OK)
        st = pool_alloc((void **)&err, sizeof(unsigned), s);
    CUtensorMap map;
    if (st == PR_OK && path != PR_GATHER_LOAD)
        st = encode_rows<T>(&map, state, rows);
    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (st == PR_OK) {
        e = cudaEventCreate(&ev[0]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&ev[1]);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(err, 0, sizeof(unsigned), s);
        if (e == cudaSuccess) {
            k_fill<T><<<sms * 8, kGatherBlock, 0, s>>>((int32_t *)idx, count, (T *)state, n, state_elems);
            e = cudaGetLastError();
        }
        T *sink = (T *)state + n;
        const int4 *idx4 = (const int4 *)idx;
        const int64_t nvec = count / 4;
        // one warm-up pass, then three timed ones; returns the rate in gathers/s
        auto timed = [&](auto launch) -> double {
            for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {
                if (rep == 1)
                    e = cudaEventRecord(ev[0], s);
                if (e == cudaSuccess) {
                    launch();
                    e = cudaGetLastError();
                }
            }
            if (e == cudaSuccess)
                e = cudaEventRecord(ev[1], s);
            if (e == cudaSuccess)
                e = cudaEventSynchronize(ev[1]);
            float ms = 0.f;
            if (e == cudaSuccess)
                e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
            return (e == cudaSuccess && ms > 0.f) ? 3.0 * (double)count / ((double)ms * 1e-3) : 0.0;
        };
        const int grid = (per_sm > 0 ? per_sm : 1) * sms;
        auto run_load = [&]() { k_gather<T><<<grid, kGatherBlock, 0, s>>>(idx4, nvec, (const T *)state, sink); };
        auto run_tma = [&]() {
            k_gather_tma<T><<<(per_sm_tma > 0 ? per_sm_tma : 1) * sms, kGatherBlock, smem_only, s>>>(
                map, idx4, 0, idx4, nvec, (const T *)state, sink, err, tma_only_warps);
        };
        if (path == PR_GATHER_LOAD) {
            *rate = timed(run_load);
        } else if (path == PR_GATHER_TMA) {
            *rate = timed(run_tma);
        } else {
            // both paths at once: the first nvec_load groups of four go
            // through the loads, the rest through the TMA, in the ratio of
            // the two rates measured alone
            const double r_load = timed(run_load);
            const double r_tma = timed(run_tma);
            const int64_t nvec_load = (r_load + r_tma > 0.0)
                                          ? (int64_t)((double)nvec * r_load / (r_load + r_tma))
                                          : nvec / 2;
            *rate = timed([&]() {
                k_gather_tma<T><<<(per_sm_both > 0 ? per_sm_both : 1) * sms, kGatherBlock, smem_both, s>>>(
                    map, idx4, nvec_load, idx4 + nvec_load, nvec - nvec_load, (const T *)state, sink, err,
                    both_warps);
            });
        }
        unsigned herr = 0;
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&herr, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        if (e != cudaSuccess)
            st = cuda_status(e, "measuring the gather rate");
        else if (herr)
            st = set_error(PR_ERR_TIMEOUT, "a gather4 copy did not complete within its wait limit");
    }
    for (cudaEvent_t x : ev)
        if (x)
            cudaEventDestroy(x);
    pool_free(idx, s);
    pool_free(state, s);
    pool_free(err, s);
    cudaError_t se = cudaStreamSynchronize(s);
    if (st == PR_OK && se != cudaSuccess)
        st = cuda_status(se, "measuring the gather rate");
    return st;
}

}  // namespace

pr_status measure_gather_rate(int64_t n, int dtype, int64_t gathers, int path, double *rate, cudaStream_t s)
{
    return dtype == PR_F64 ? measure<double>(n, gathers, path, rate, s) : measure<float>(n, gathers, path, rate, s);
}

}  // namespace prk
