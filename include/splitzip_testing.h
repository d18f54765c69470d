/*
 * splitzip_testing.h -- test controls of the SplitZip library (not for
 * production callers).
 *
 * The single-launch encode pipeline (the engine of splitzip_encode_noalloc)
 * computes the exclusive prefix of escape counts across 8192-element tiles
 * with a decoupled look-back: a tile waits until its predecessors have
 * published their counts.  Every such wait is bounded; when the bound runs
 * out the kernel records SPLITZIP_ERR_TIMEOUT in the workspace, publishes a
 * (wrong) prefix so that later tiles are not held up, keeps every write in
 * bounds and returns, leaving the CUDA context usable.  This entry point lets
 * a test make that wait run out on purpose, with a flag that keeps tile 0
 * from ever publishing, and a small poll limit so the test ends quickly.  (The
 * default three-launch encode has no spin-waits: its tile offsets come from
 * counters the first launch completes before the second reads them; the stall
 * flag has no effect on it.)  The method's pages have no counterpart: this entry point
 * exists only to exercise the error path.
 */
#ifndef SPLITZIP_TESTING_H
#define SPLITZIP_TESTING_H

#include "splitzip.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Tile 0 never publishes its prefix: every later tile's wait runs out
 * (single-launch pipeline only). */
#define SPLITZIP_TEST_STALL_FIRST_TILE 0x1u
/* Encode with the single-launch pipeline (the engine of
 * splitzip_encode_noalloc) instead of the three-launch encode. */
#define SPLITZIP_TEST_PIPELINED 0x2u

typedef struct splitzip_encode_test_opts {
    uint32_t spin_limit;  /* polls (about 100 ns apart) before a wait gives up; 0 = default */
    uint32_t flags;       /* SPLITZIP_TEST_* bits */
} splitzip_encode_test_opts;

/* splitzip_encode / splitzip_encode_e5m2 (is_e5m2 != 0) with test controls.
 * Same arguments, ownership and errors as splitzip_encode. */
splitzip_status splitzip_encode_test(const void *d_x, uint64_t n, uint32_t chunk_size,
                                     const splitzip_codebook *cb, const splitzip_streams *out,
                                     void *d_workspace, splitzip_stream_t s, int is_e5m2,
                                     const splitzip_encode_test_opts *opts);

#ifdef __cplusplus
}
#endif

#endif /* SPLITZIP_TESTING_H */
