/*
 * qmm_testing.h -- test hooks of the qmm library (not part of the product
 * interface; the library's tests use them to exercise its failure paths
 * without faulting or hanging a GPU).  The paper pages have no counterpart.
 */
#ifndef QMM_TESTING_H
#define QMM_TESTING_H

#include <stdint.h>

#include "qmm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bound, in nanoseconds, of every device-side wait of later calls on this
 * handle (default 2 s).  0 is rejected with QMM_ERR_INVALID_ARG. */
int qmm_testing_set_wait_limit_ns(qmm_handle h, uint64_t limit_ns);

/* When enable != 0, later tensor-core qmm_gemm calls on this handle skip the
 * copy of their first k stage, so the MMA issuer's wait on it runs out: the
 * kernel latches the timeout bit, waits for its own copies and MMAs in
 * flight, frees its tensor memory and returns; qmm_sync_status then reports
 * QMM_ERR_TIMEOUT and dst holds no result.  Pass 0 to restore normal calls. */
int qmm_testing_skip_first_stage_load(qmm_handle h, int enable);

#ifdef __cplusplus
}
#endif

#endif /* QMM_TESTING_H */
