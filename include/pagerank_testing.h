/*
 * pagerank_testing.h - test hooks of the GB300 PageRank library.
 *
 * These entry points exist so that the library's failure paths can be
 * exercised without faulting a GPU: an allocation failure is made on the
 * host, and a device-side wait is made to run out by giving it a flag that
 * nothing sets. They are exported from the same shared library as the calls
 * of pagerank.h, change no result of those calls while unused, and are not
 * meant for production code. The pages have no counterpart; the failure
 * behaviour they exercise follows "Day 40 - PageRank on a real graph in
 * CUDA", section "Validate before timing" (the program checks itself and
 * reports a failure instead of producing numbers).
 */
#ifndef PAGERANK_GB300_TESTING_H
#define PAGERANK_GB300_TESTING_H

#include <stdint.h>

#include "pagerank.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Makes the k-th device allocation from the library's memory pool, counted
 * from this call, fail as if the device were out of memory: the entry point
 * that made it returns PR_ERR_OOM. k = 0 switches the hook off; k < 0 is
 * treated as 0. Process-wide (every thread, every device); the hook switches
 * itself off once it has fired.
 */
void pr_test_fail_alloc_after(int64_t k);

/*
 * Bytes of the current device's library pool that are allocated to the
 * caller's handles and calls right now (cudaMemPoolAttrUsedMemCurrent), after
 * a cudaDeviceSynchronize so that stream-ordered frees have landed; 0 if the
 * pool has not been created on this device. Returns PR_OK,
 * PR_ERR_INVALID_ARG (used is NULL) or PR_ERR_CUDA.
 */
pr_status pr_test_pool_used_bytes(int64_t *used);

/*
 * Runs the look-back exclusive scan that pr_graph_create uses on `count`
 * zero counts held in pool memory of its own, with the first tile withheld:
 * its descriptor is never published, so every tile that walks back to it
 * waits until `spin_limit` polls have passed, then sets the timeout bit of
 * the error word and finishes. Every CTA reads and writes only inside the
 * call's own buffers. Returns PR_ERR_TIMEOUT when a wait ran out (the
 * expected outcome), PR_OK if none did, PR_ERR_INVALID_ARG for count outside
 * (8192, 2^24] (more than one 8,192-element tile) or spin_limit outside
 * [1, 2^20], PR_ERR_OOM or PR_ERR_CUDA.
 * Synchronises `stream`; the CUDA context stays usable.
 */
pr_status pr_test_scan_timeout(int64_t count, int32_t spin_limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGERANK_GB300_TESTING_H */
