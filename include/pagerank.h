/*
 * pagerank.h - C ABI of the GB300 (sm_103a) PageRank power-iteration library.
 *
 * The library computes PageRank by power iteration on one GPU:
 *
 *   x'[v] = (1 - d)/n + d * ( sum over in-neighbours u of x[u]/outdeg[u]
 *                             + D/n ),     D = sum of x over dangling vertices
 *
 * ("Day 40 - PageRank on a real graph in CUDA", section "One iteration, three
 * shapes of work", update formula; a dangling vertex is one with no out-edge,
 * introduction of the same page), starting from x0 = 1/n (Meerkat, "Dynamic
 * graph algorithms on GPUs", PageRank section, Algorithm 5, static case) and
 * stopping after the first update whose L1 distance sum_v |x'[v] - x[v]| is
 * below tol (same Meerkat section; Day 40, "Keep the dangling mass on the
 * device").
 *
 * pr_graph_create transposes the caller's out-edge CSR into an in-edge CSR on
 * the device (Day 40, "One iteration, three shapes of work": histogram, prefix
 * sum, scatter) and splits the in-rows into in-degree classes (gpu-graph-study,
 * "PageRank T4 - degree-bucketed load balancing": <= 32, 33..1024, > 1024).
 * pr_run performs the whole iteration on the device inside one CUDA graph and
 * synchronises the stream once, at the end.
 *
 * Conventions shared by every entry point:
 *  - Vertex ids are int32 in [0, n); edge offsets are int64 on input and
 *    int32 inside the library, so 1 <= n <= 2^31 - 2 and 0 <= m <= 2^31 - 1.
 *  - A pointer argument may point to host memory (pageable or pinned) or to
 *    device memory of the current device (of the graph's device for pr_run);
 *    the library tells them apart with cudaPointerGetAttributes and copies as
 *    needed. Managed memory is treated as device memory. Device memory of
 *    any other GPU is rejected with PR_ERR_INVALID_ARG before any work, since
 *    a kernel that dereferenced it would make a peer access nobody enabled.
 *  - `stream` is a cudaStream_t passed as void* (for example
 *    torch.cuda.current_stream().cuda_stream); NULL means the legacy default
 *    stream. All device work of a call is ordered on that stream (work that
 *    pr_graph_create runs on a second, library-owned stream, such as the copy
 *    of a host col_idx, is forked from and joined back to it).
 *  - Every entry point that can fail returns a pr_status. Negative values are
 *    errors: nothing is written to the caller's output buffers and
 *    pr_last_error() returns a message (thread-local, valid until the next
 *    call on the same thread). Calls on one pr_graph are not thread-safe.
 */
#ifndef PAGERANK_GB300_H
#define PAGERANK_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle. Owns device memory: the in-edge CSR, per-vertex out-degrees,
 * the in-degree class lists, the fp32 iteration state with its instantiated
 * CUDA graph and, after the first fp64 pr_run, the same for fp64.
 *
 * Device memory (handle-owned and the build's scratch) comes from one
 * stream-ordered memory pool per device that the library creates on first
 * use and never trims: pr_graph_destroy returns a handle's memory to that
 * pool, where later handles reuse it, and the process keeps it until exit. */
typedef struct pr_graph pr_graph;

typedef enum pr_status {
    PR_OK = 0,
    PR_NOT_CONVERGED = 1,       /* tol > 0 and max_iter updates ran without L1 < tol;
                                   ranks, iterations and L1 are still written */
    PR_ERR_INVALID_ARG = -1,    /* bad scalar argument or NULL pointer */
    PR_ERR_INVALID_GRAPH = -2,  /* row_ptr[0] != 0, row_ptr[n] != m, row_ptr
                                   decreasing, or a col_idx entry outside [0, n) */
    PR_ERR_TOO_LARGE = -3,      /* n or m beyond the int32 limits above */
    PR_ERR_OOM = -4,            /* a device allocation failed */
    PR_ERR_CUDA = -5,           /* any other CUDA runtime error */
    PR_ERR_TIMEOUT = -6         /* a bounded device-side wait gave up (the
                                   transpose's scan look-back); the context
                                   stays usable, the handle is not created */
} pr_status;

typedef enum pr_dtype {
    PR_F32 = 0,                 /* ranks and contributions in fp32, row sums in fp32
                                   tree order, L1 and D totals in fp64 */
    PR_F64 = 1                  /* everything in fp64 */
} pr_dtype;

/* Stages of pr_graph_create, in order (pr_graph_info.build_stage_ms). */
#define PR_BUILD_STAGES 8
typedef enum pr_build_stage {
    PR_STAGE_DEGREES = 0,       /* out-degrees, dangling count, row_ptr check */
    PR_STAGE_SOURCES = 1,       /* the source of every edge, from row_ptr */
    PR_STAGE_SORT = 2,          /* the radix passes by destination (the stable
                                   scatter) and the in-degree histogram */
    PR_STAGE_OFFSETS = 3,       /* in_ptr, the exclusive scan of the in-degrees */
    PR_STAGE_ORDER = 4,         /* the class-major vertex order and its inverse */
    PR_STAGE_LAYOUT = 5,        /* the work CSR's offsets and the hub chunks */
    PR_STAGE_RELABEL = 6,       /* the work CSR's sources, relabelled */
    PR_STAGE_FINISH = 7         /* sizes for reporting */
} pr_build_stage;

/* Options of pr_graph_create_ex. A NULL pointer, or the values of
 * PR_OPTIONS_DEFAULT, give what pr_graph_create does. */
typedef struct pr_options {
    int32_t thread_max;         /* rows with 1..thread_max in-edges are the thread class
                                   (one lane per row); 1 <= thread_max <= 32. Default 32 */
    int32_t warp_max;           /* rows with thread_max+1..warp_max in-edges are the warp
                                   class (32-row blocks, one warp each); rows above are cut
                                   into chunks (the "CTA" class); thread_max <= warp_max
                                   <= 8192. Default 1024. A warp-class row's sum builds up
                                   in one register per lane, one int4 per 32-entry step, so
                                   the cap keeps fp32 row sums inside the parity tolerance
                                   (a 70,000-edge row summed that way was off by 1.2e-5) */
    int32_t stage_timing;       /* nonzero: record CUDA events between the build's stages
                                   (pr_graph_info.build_stage_ms); default 0 */
} pr_options;

#define PR_OPTIONS_DEFAULT {32, 1024, 0}

/* Sizes of the preprocessed graph (filled by pr_graph_get_info). */
typedef struct pr_graph_info {
    int64_t n, m;
    int64_t n_dangling;         /* vertices with out-degree 0 */
    int64_t rows_zero;          /* in-degree 0: no gather */
    int64_t rows_thread;        /* in-degree 1..32: one lane per row */
    int64_t rows_warp;          /* in-degree 33..1024: 32-row blocks, one warp each */
    int64_t rows_cta;           /* in-degree > 1024: split into chunks streamed by CTAs */
    int64_t edges_thread, edges_warp, edges_cta;
    int64_t cta_chunks;         /* number of CTA chunks */
    int32_t cta_chunk_edges;    /* edges per chunk of a CTA row, one warp each (the last
                                   chunk of a row may be shorter) */
    int32_t iterate_grid;       /* CTAs of the persistent iteration kernel */
    int64_t device_bytes;       /* device memory held by the handle */
    int32_t build_launches;     /* kernels pr_graph_create launched */
    int64_t edges_hot_f32;      /* in-edges whose source is in the head of the state
                                   vector that every update copies into each SM's
                                   shared memory (fp32 runs: 40,960 vertices); their
                                   gathers never reach L2, the other m - edges_hot
                                   gathers do */
    int64_t edges_hot_f64;      /* the same for fp64 runs (20,480 vertices) */
    int32_t thread_max;         /* the class thresholds the handle was built with */
    int32_t warp_max;
    float build_ms;             /* device time of pr_graph_create's work (CUDA events on
                                   its stream, from the first to the last launch); with a
                                   host col_idx it includes waiting for that array's copy,
                                   which runs beside the stages that read only row_ptr */
    float build_stage_ms[PR_BUILD_STAGES];   /* device time of each stage, if the
                                   handle was built with stage_timing; else 0 */
} pr_graph_info;

/* Statistics of the most recent pr_run on a handle (filled by pr_graph_last_run). */
typedef struct pr_run_stats {
    int32_t iterations;         /* updates performed */
    int32_t converged;          /* 1 if the last update had L1 < tol (tol > 0) */
    double l1;                  /* L1 distance of the last update */
    double dangling_mass;       /* D of the final vector */
    float loop_ms;              /* device time of the iteration loop alone (CUDA events
                                   recorded on the run's stream around the graph launch) */
    float total_ms;             /* device time from the first to the last kernel of pr_run */
    int32_t launches;           /* kernels pr_run launched: init, the update launches
                                   (two per trip of the graph's loop; when the loop ends
                                   on a trip's first update, its second launch returns
                                   at once), output */
} pr_run_stats;

/*
 * Builds the device-side graph from an out-edge CSR.
 *   n        number of vertices (1 <= n <= 2^31 - 2)
 *   m        number of edges (0 <= m <= 2^31 - 1), and in addition
 *            m + 3 min(n, m) + PR_LAYOUT_SLACK <= 2^31 - 1: the work layout
 *            pads every row with in-edges to a multiple of 4 entries and keeps
 *            int32 offsets; larger graphs get PR_ERR_TOO_LARGE
 *   row_ptr  int64[n + 1], row_ptr[0] = 0, non-decreasing, row_ptr[n] = m;
 *            the out-edges of u are col_idx[row_ptr[u] .. row_ptr[u+1])
 *   col_idx  int32[m], targets in [0, n); duplicates and self-loops are kept
 *            and count with their multiplicity; may be NULL when m = 0
 *   out      receives the handle on success (untouched on failure)
 * Inputs are borrowed for the duration of the call only: the caller may free
 * or overwrite them once it returns (the call synchronises `stream`).
 * The handle also holds the state and the iteration graph of fp32 runs
 * (about 12 bytes per vertex, in device_bytes), built while the last build
 * step runs on the device; those of fp64 runs are made by the first fp64
 * pr_run.
 * Returns PR_OK, PR_ERR_INVALID_ARG, PR_ERR_INVALID_GRAPH, PR_ERR_TOO_LARGE,
 * PR_ERR_OOM, PR_ERR_TIMEOUT or PR_ERR_CUDA.
 */
pr_status pr_graph_create(int64_t n, int64_t m, const int64_t *row_ptr,
                          const int32_t *col_idx, void *stream, pr_graph **out);

/*
 * pr_graph_create with options: the in-degree class thresholds (gpu-graph-
 * study, "PageRank T4 - degree-bucketed load balancing", uses 32 and 1024,
 * the defaults) and per-stage timing of the build. The thresholds decide
 * only which kernel path each row takes: the ranks agree with every
 * setting within the rounding of the row sums. opts may be NULL. Options
 * outside the ranges of pr_options give PR_ERR_INVALID_ARG before any work;
 * otherwise the same arguments, results and errors as pr_graph_create.
 */
pr_status pr_graph_create_ex(int64_t n, int64_t m, const int64_t *row_ptr,
                             const int32_t *col_idx, const pr_options *opts, void *stream,
                             pr_graph **out);

/*
 * Runs the power iteration on a graph.
 *   d          damping factor, 0 <= d <= 1
 *   tol        L1 tolerance; the run stops after the first update with
 *              L1 < tol. tol <= 0 runs exactly max_iter updates.
 *   max_iter   cap on the number of updates, >= 1
 *   dtype      PR_F32 or PR_F64: the precision of the iteration and of
 *              ranks_out and x_init
 *   ranks_out  n values of dtype, written with the final ranks
 *              (caller-owned, host or device)
 *   x_init     NULL for the uniform start 1/n, else n values of dtype used
 *              as the start vector (warm start); not renormalised. It must be
 *              a probability vector (every value >= 0, sum 1 up to rounding):
 *              the L1 and dangling-mass totals are exact fixed-point sums
 *              sized for totals of at most 2
 *   iters_out  optional (NULL): number of updates performed
 *   l1_out     optional (NULL): L1 distance of the last update
 * The whole loop runs on the device; the call synchronises `stream` once,
 * at the end. The first PR_F64 run on a handle allocates that precision's
 * state (PR_ERR_OOM if it cannot; the handle stays usable). Returns PR_OK,
 * PR_NOT_CONVERGED, or an error.
 */
pr_status pr_run(pr_graph *g, double d, double tol, int32_t max_iter,
                 pr_dtype dtype, void *ranks_out, const void *x_init,
                 int32_t *iters_out, double *l1_out, void *stream);

/*
 * Copies the in-edge CSR out of the handle (for verification).
 *   in_ptr  int32[n + 1]: the in-edges of v are in_col[in_ptr[v] .. in_ptr[v+1])
 *   in_col  int32[m]: the sources, ascending within each row (the order of
 *           a stable counting sort by destination); may be NULL when m = 0
 * Buffers are caller-owned, host or device. Synchronises `stream`.
 */
pr_status pr_get_in_csr(const pr_graph *g, int32_t *in_ptr, int32_t *in_col,
                        void *stream);

/* Fills *info with the sizes of the preprocessed graph. */
pr_status pr_graph_get_info(const pr_graph *g, pr_graph_info *info);

/* Fills *stats with the statistics of the handle's most recent pr_run. */
pr_status pr_graph_last_run(const pr_graph *g, pr_run_stats *stats);

/* Padding slack of the work layout in pr_graph_create's size limit. */
#define PR_LAYOUT_SLACK 8192

/* Largest `count` that pr_exclusive_scan_noalloc accepts (2^26). */
#define PR_SCAN_NOALLOC_MAX (1LL << 26)

/*
 * Exclusive prefix sum of int32 counts into int32 offsets that allocates no
 * device memory: offsets[i] = counts[0] + ... + counts[i-1] for i in
 * [0, count], so offsets[count] is the total (the CSR offsets of a degree
 * array). The pages have no counterpart: this is the library's own
 * single-pass look-back scan (the one pr_graph_create uses for in_ptr)
 * offered to callers that must not call cudaMalloc, such as code running
 * inside a framework that owns all device memory through its own pool and
 * hands the library only buffers it has already carved out.
 *   counts   device pointer (memory of the current device), `count` int32
 *            values, each >= 0, whose total must fit int32
 *   offsets  device pointer (memory of the current device), `count + 1`
 *            int32 values (caller-owned)
 *   count    0 <= count <= PR_SCAN_NOALLOC_MAX; larger counts are rejected
 *            with PR_ERR_TOO_LARGE and a message
 * Scratch: the look-back descriptors live in one fixed file-scope device
 * array sized for PR_SCAN_NOALLOC_MAX elements (about 64 KB), which every
 * device that loads the library holds until the process exits. The first
 * call on a device looks up that array's device address
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture. Every call shares the array and clears the
 * part it uses, so calls that overlap on the GPU (from two host threads, or
 * on two streams without ordering) race and give wrong results: serialize
 * them. The call synchronizes `stream` and returns PR_OK,
 * PR_ERR_INVALID_ARG (NULL pointers, pointers that are not memory of the
 * current device, count < 0, or a negative entry in counts, which the kernel
 * detects), PR_ERR_TOO_LARGE (count beyond the scratch, or a total above
 * INT32_MAX, which the kernel detects), PR_ERR_TIMEOUT or PR_ERR_CUDA. After
 * an error that the kernel detected, the contents of offsets are not
 * meaningful. It makes no cudaMalloc or cudaFree call.
 */
pr_status pr_exclusive_scan_noalloc(const int32_t *counts, int32_t *offsets, int64_t count,
                                    void *stream);

/* The path a random gather takes (pr_measure_gather_rate). */
typedef enum pr_gather_path {
    PR_GATHER_LOAD = 0,         /* ld.global.cg from the warps: the path the update uses */
    PR_GATHER_TMA = 1,          /* the tensor memory accelerator: cp.async.bulk.tensor
                                   tile::gather4 copies of four 16-byte rows into shared
                                   memory, issued by the lanes, completed on mbarriers */
    PR_GATHER_BOTH = 2          /* both at once, the gathers split between them in the
                                   ratio of their rates measured alone */
} pr_gather_path;

/*
 * Measures the current GPU's rate of random gathers: loads of single dtype
 * elements from uniformly random positions of an n-element state vector,
 * each of which misses L1 and costs one L2 request. This is the bound of the
 * update's gathers that the shared-memory copy of the state's head does not
 * serve (those are m - edges_hot per update, see pr_graph_info), so a run's
 * rate of such gathers can be reported as a fraction of it. The pages have
 * no counterpart: it is the denominator of the update kernel's gather
 * roofline, and, with `path`, the measurement of whether a second request
 * path (the TMA's tile::gather4, which fetches a 16-byte row per gathered
 * element) adds to the rate of the warps' loads. The indices are drawn on
 * the device (SplitMix64 of the position, reduced mod n) and streamed as
 * int32; the time is that of three passes after a warm-up, taken with CUDA
 * events on `stream`. PR_GATHER_BOTH also measures the two paths alone first.
 *   n             elements of the state vector, 1 <= n <= 2^31 - 2 (pass the
 *                 graph's n to measure at the run's working-set size)
 *   dtype         PR_F32 or PR_F64: the element type gathered
 *   gathers       gathers per pass, 1 <= gathers <= 2^30 (about 2^27 gives a
 *                 pass of a few tenths of a millisecond)
 *   path          PR_GATHER_LOAD, PR_GATHER_TMA or PR_GATHER_BOTH
 *   gathers_per_s receives the measured rate
 * Allocates about n * sizeof(dtype) + 4 * gathers bytes from the library's
 * pool for the duration of the call and synchronizes `stream`. Every wait on
 * a copy is bounded; one that gives up makes the call return PR_ERR_TIMEOUT
 * (the context stays usable). Returns PR_OK, PR_ERR_INVALID_ARG, PR_ERR_OOM,
 * PR_ERR_TIMEOUT or PR_ERR_CUDA.
 */
pr_status pr_measure_gather_rate(int64_t n, pr_dtype dtype, int64_t gathers, pr_gather_path path,
                                 double *gathers_per_s, void *stream);

/* Frees the handle and returns all device memory it owns to the library's
 * pool (see the handle's description). NULL is ignored. The
 * caller must make sure no work using the handle is still in flight on a
 * stream other than the ones its calls already synchronised. */
void pr_graph_destroy(pr_graph *g);

/* Message for the last error returned on the calling thread ("" if none). */
const char *pr_last_error(void);

/* Library version string. */
const char *pr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGERANK_GB300_H */
