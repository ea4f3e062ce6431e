/*
 * gk_testing.h -- test hooks of the GB300 decode-attention library.  Not part
 * of the decode path; no counterpart on the pages.
 */
#ifndef GK_TESTING_H
#define GK_TESTING_H

#include "gk.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gk_selftest_wait_timeout -- exercise the bounded shared-memory barrier wait
 * that every pipeline stage of the attention kernel uses: one warp waits on a
 * barrier phase that nothing completes, gives up after limit_ns nanoseconds of
 * device wall time (1 us .. 1 s), sets GK_DEVERR_TIMEOUT and returns.  Nothing
 * faults or hangs; the context stays usable.  Synchronises `stream` and
 * returns the error word in *bits (cleared afterwards), with
 * GK_ERR_DEVICE_BOUNDS when a bit is set.
 */
gk_status gk_selftest_wait_timeout(uint64_t limit_ns, void *stream, uint32_t *bits);

#ifdef __cplusplus
}
#endif

#endif /* GK_TESTING_H */
