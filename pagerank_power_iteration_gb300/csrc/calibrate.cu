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

// idx[i] uniform in [0, n), state[i] = 0 (the values do not matter).
template <typename T>
__global__ void k_fill(int32_t *__restrict__ idx, int64_t count, T *__restrict__ state, int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
        idx[i] = (int32_t)(splitmix64((uint64_t)i) % (uint64_t)n);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
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

template <typename T>
pr_status measure(int64_t n, int64_t gathers, double *rate, cudaStream_t s)
{
    const int64_t count = (gathers + 3) & ~(int64_t)3;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gather<T>, kGatherBlock, 0);
    if (e != cudaSuccess)
        return cuda_status(e, "device query");
    void *idx = nullptr, *state = nullptr;
    pr_status st = pool_alloc(&idx, (size_t)count * sizeof(int32_t), s);
    if (st == PR_OK)
        st = pool_alloc(&state, (size_t)(n + 1) * sizeof(T), s);
    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (st == PR_OK) {
        e = cudaEventCreate(&ev[0]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&ev[1]);
        if (e == cudaSuccess) {
            k_fill<T><<<sms * 8, kGatherBlock, 0, s>>>((int32_t *)idx, count, (T *)state, n);
            e = cudaGetLastError();
        }
        const int grid = (per_sm > 0 ? per_sm : 1) * sms;
        const int64_t nvec = count / 4;
        T *sink = (T *)state + n;
        // one warm-up pass, then three timed ones
        for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {
            if (rep == 1)
                e = cudaEventRecord(ev[0], s);
            if (e == cudaSuccess) {
                k_gather<T><<<grid, kGatherBlock, 0, s>>>((const int4 *)idx, nvec, (const T *)state, sink);
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
        if (e == cudaSuccess && ms > 0.f)
            *rate = 3.0 * (double)count / ((double)ms * 1e-3);
        if (e != cudaSuccess)
            st = cuda_status(e, "measuring the gather rate");
    }
    for (cudaEvent_t x : ev)
        if (x)
            cudaEventDestroy(x);
    pool_free(idx, s);
    pool_free(state, s);
    cudaError_t se = cudaStreamSynchronize(s);
    if (st == PR_OK && se != cudaSuccess)
        st = cuda_status(se, "measuring the gather rate");
    return st;
}

}  // namespace

pr_status measure_gather_rate(int64_t n, int dtype, int64_t gathers, double *rate, cudaStream_t s)
{
    return dtype == PR_F64 ? measure<double>(n, gathers, rate, s) : measure<float>(n, gathers, rate, s);
}

}  // namespace prk
