// Internal declarations shared by the library's translation units.
// Not part of the ABI: callers use include/pagerank.h only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "pagerank.h"

namespace prk {

// In-degree classes of the pull SpMV (gpu-graph-study, "PageRank T4 -
// degree-bucketed load balancing": thread per row up to 32, warp per row up
// to 1024, block per row above); pr_options can move both thresholds. Rows
// above the warp threshold are cut into chunks of kChunkEdges edges; each
// warp of the update kernel streams one contiguous range of chunks, so one
// hub is spread over many warps and CTAs. A thread-class row is one lane's
// work in at most eight int4s, so the thread threshold is at most 32.
constexpr int kDefaultThreadMax = 32;
constexpr int kDefaultWarpMax = 1024;
constexpr int kThreadMaxLimit = 32;
// A warp-class row is summed by one warp, each lane adding one int4 of it per
// 32-int4 step into one register; past a few dozen steps that sequential sum
// loses fp32 accuracy (a 70,000-edge row was off by 1.2e-5 relative), so the
// warp threshold is capped, and longer rows go to the chunked class.
constexpr int kWarpMaxLimit = 8192;
constexpr int kChunkEdges = 256;
constexpr int kBlock = 256;        // CTA size of the preprocessing kernels
constexpr int kIterBlock = 1024;   // CTA size of the update kernel (one CTA per SM)
constexpr int kHotBytes = 160 * 1024;   // shared-memory copy of the state's head
constexpr int32_t kHotF32 = kHotBytes / 4;   // state entries in that copy, fp32 runs
constexpr int32_t kHotF64 = kHotBytes / 8;   // and fp64 runs
// Per-row cost, in edges, added to the edges when warp-class rows are split
// over the warps of the update kernel. The flat 32-row blocks make the
// per-row work small: a pure edge balance (0) measured best (RMAT-24 update
// 0.754 ms at 32, 0.735 at 16, 0.711 at 0).
constexpr int kWarpRowCost = 0;
// Graphs with fewer rows that have in-edges than this take the gather
// classes in one order in every warp (small graphs sit in L2 and are bound
// by fixed costs); larger ones start each warp at its own class.
constexpr int64_t kRotateRows = (int64_t)1 << 20;
// Update launches per trip of the CUDA graph's WHILE loop: the loop's own
// turnaround costs more than the gap between two kernel nodes.
constexpr int kUpdatesPerTrip = 2;
// Work-CSR entry that pads a row to whole 16-byte loads; it gathers 0. (A
// pad pointing at a zero slot of the state instead makes every pad of every
// SM read one L2 line, a hot spot that was measured to cost 15 %.)
constexpr int32_t kPadSource = -1;

enum RowClass : int { kClassZero = 0, kClassThread = 1, kClassWarp = 2, kClassCta = 3 };

// Bits of the device error word.
enum : unsigned {
    kErrRowPtr = 1u,    // row_ptr decreases somewhere
    kErrColIdx = 2u,    // a col_idx entry is outside [0, n)
    kErrTimeout = 4u,   // a bounded look-back wait gave up
    kErrNegative = 8u,  // a scanned count was negative (counted as 0)
    kErrOverflow = 16u, // a scan's total exceeds INT32_MAX
};

// Device-resident scalars of a run. Written by the init kernel, read at the
// start of every update and rewritten by the last CTA of each update.
struct Scalars {
    double dmass;       // dangling mass D of the current vector
    double l1;          // L1 distance of the last update
    double d;           // damping factor
    double tol;         // L1 tolerance (<= 0: fixed number of updates)
    double inv_n;       // 1/n
    double base_last;   // the constant term (1-d)/n + d D/n of the last update, in the
                        // run's precision: the rank of every vertex without in-edges
    int32_t it;         // updates performed so far
    int32_t max_iter;
    int32_t converged;
    uint32_t ticket;    // arrival counter for the last-CTA reductions
    int32_t stop;       // 1 once an update has ended the loop (L1 < tol or the cap):
                        // a later update launch in the same loop body does nothing
    int32_t pad;
};

// Per-precision iteration state of a handle.
struct DtypeState {
    bool ready = false;
    void *s[2] = {nullptr, nullptr};   // ping-pong state [n + 1] in work order: x/outdeg,
                                       // or x for a dangling vertex; slot n stays 0
    void *hub_partial = nullptr;       // one partial row sum per CTA chunk
    void *stage = nullptr;             // staging for host x_init / ranks_out
    unsigned long long *block_partials = nullptr;  // [grid][2]: fixed-point L1 and D of each CTA
    int32_t *w_split = nullptr;        // [warps + 1] warp-class row ranges per warp
    int grid = 0;                      // CTAs of the persistent iteration kernel
    int init_grid = 0;
    int32_t hot = 0;                   // state slots staged in shared memory per update
    size_t smem = 0;                   // dynamic shared memory of the update kernel
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

}  // namespace prk

struct pr_graph {
    int64_t n = 0, m = 0;
    int device = 0;
    int num_sms = 0;
    int32_t thread_max = prk::kDefaultThreadMax;   // in-degree class thresholds
    int32_t warp_max = prk::kDefaultWarpMax;
    bool stage_timing = false;                      // record the build's stages
    float build_ms = 0.f;                           // device time of the build
    float build_stage_ms[PR_BUILD_STAGES] = {};     // per stage, if recorded

    // in-edge CSR in the caller's vertex ids (kept for pr_get_in_csr)
    int32_t *in_ptr = nullptr;     // [n + 1]
    int32_t *in_col = nullptr;     // [m]
    int32_t *deg_out = nullptr;    // [n] out-degrees, caller's ids

    // work layout: the graph relabelled in class-major order (CTA rows, warp
    // rows, thread rows, rows without in-edges; ascending ids in a class)
    int32_t *order = nullptr;      // [n] work position -> vertex id
    int32_t *perm = nullptr;       // [n] vertex id -> work position
    int32_t *w_ptr = nullptr;      // [n + 1] work CSR offsets; rows padded to a multiple
                                   // of 4 edges (16-byte aligned)
    int32_t *w_col = nullptr;      // [m_w] work sources; padding entries are kPadSource
    int32_t *w_deg = nullptr;      // [n] out-degrees in work order
    int64_t m_w = 0;               // edges in the work CSR, padding included

    // CTA rows (work rows [0, n_c)) are cut into chunks of kChunkEdges edges
    int32_t *chunk_row = nullptr;    // [n_chunks]: work row of each chunk
    int32_t *chunk_first = nullptr;  // [n_c + 1]: first chunk of each CTA row
    uint32_t *hub_arrivals = nullptr; // [n_c]: chunks of the row finished this update
    int64_t n_dangling = 0, n_z = 0, n_t = 0, n_w = 0, n_c = 0, n_chunks = 0;
    // the last n_iso work rows: vertices with neither in- nor out-edges
    int64_t n_iso = 0;
    // thread-class rows come in blocks of 32 sorted by length, longest first;
    // blocks [t_short, ...) have rows of at most two int4s
    int64_t t_short = 0;
    int64_t e_t = 0, e_w = 0, e_c = 0;
    int64_t e_hot[2] = {0, 0};     // in-edges with a source in the hot head, fp32 / fp64

    prk::Scalars *scal = nullptr;   // device
    unsigned *err = nullptr;        // device error word
    prk::Scalars *h_scal = nullptr; // host mirror (pageable), read after each run

    prk::DtypeState st[2];
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    pr_run_stats last = {};

    int32_t build_launches = 0;     // kernels launched by pr_graph_create
    std::vector<void *> allocs;     // every device allocation owned by the handle
    int64_t device_bytes = 0;
};

namespace prk {

// NVTX range for the duration of a scope (header-only NVTX; costs nothing
// unless a tool such as Nsight Compute is attached). Ranges: "pr_graph_create",
// "pr_init", "pr_iterate" (the CUDA-graph loop of updates), "pr_output".
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// Error reporting (api.cu).
pr_status set_error(pr_status st, const char *fmt, ...);
pr_status cuda_status(cudaError_t e, const char *what);

// Device memory from the library's stream-ordered pool (api.cu); graph_alloc
// records the block as owned by the handle (freed by pr_graph_destroy).
pr_status pool_alloc(void **p, size_t bytes, cudaStream_t s);
void pool_free(void *p, cudaStream_t s);
pr_status graph_alloc(pr_graph *g, void **p, size_t bytes, cudaStream_t s);

// Where a caller's pointer lives, seen from `device`: host memory (pageable
// or pinned), device memory that `device`'s kernels may dereference (its own
// memory, or managed memory), or memory of another GPU, which a kernel on
// `device` must not touch (that would be a peer access nobody enabled).
enum PtrKind : int { kPtrHost = 0, kPtrDevice = 1, kPtrOtherDevice = 2 };
PtrKind pointer_kind(const void *p, int device);

// Transpose + classification (transpose.cu). d_row_ptr/d_col are device
// pointers. With h_col non-null, d_col is a device buffer of m entries that
// the build fills from the host array h_col itself, on a second stream, while
// the steps that read only row_ptr run; the copy is joined back to s before
// the build returns, whatever it returns.
pr_status build_graph(pr_graph *g, const int64_t *d_row_ptr, const int32_t *d_col,
                      const int32_t *h_col, cudaStream_t s);

// A precision's state and iteration graph (iterate.cu), built once per handle:
// by pr_graph_create for fp32, by the first pr_run of fp64.
pr_status prepare_dtype(pr_graph *g, int dtype, cudaStream_t s);

// Allocation-free exclusive scan (transpose.cu).
pr_status exclusive_scan_noalloc(const int32_t *counts, int32_t *offsets, int64_t count,
                                 cudaStream_t s);

// Test hooks (api.cu, transpose.cu): make the k-th pool allocation from now
// fail with PR_ERR_OOM (k = 0: never); bytes of the current device's pool in
// use; a scan whose first tile never publishes, so its look-back waits run
// out after spin_limit polls.
void fail_alloc_after(int64_t k);
pr_status pool_used_bytes(int64_t *out);
pr_status scan_timeout_probe(int64_t count, int spin_limit, cudaStream_t s);
constexpr int kMaxDevices = 64;

// Random-gather rate of the current GPU (calibrate.cu).
pr_status measure_gather_rate(int64_t n, int dtype, int64_t gathers, int path, double *rate, cudaStream_t s);

// Iteration (iterate.cu).
pr_status run(pr_graph *g, double d, double tol, int32_t max_iter, int dtype,
              void *ranks_out, const void *x_init, int32_t *iters_out, double *l1_out,
              cudaStream_t s);
void release_dtype_state(pr_graph *g);

}  // namespace prk
