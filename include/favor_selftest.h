/*
 * favor_selftest.h — test hooks of the FAVOR+ library (not part of the
 * attention calls).  C ABI, plain pointers; the caller owns every buffer.
 */
#ifndef FAVOR_SELFTEST_H
#define FAVOR_SELFTEST_H

#include <stdint.h>

#include "favor.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * favor_selftest_wait_timeout — exercises the bounded waits every tensor-core
 * kernel uses, on `stream`, with no fault: one CTA of two warps waits on two
 * mbarriers that nothing ever completes.  Warp 0 starts at once; its wait
 * gives up after the library's wait limit (1 s of %globaltimer), stores
 * FAVOR_ERR_TIMEOUT into *status (if it is still 0) and raises the CTA's
 * shared abort flag.  Warp 1 starts its wait 0.5 s later and returns as soon
 * as it sees the flag.  Device outputs: returned[w] = 1 if warp w's wait
 * completed, 2 if it gave up; times_ns[0] = start, times_ns[1 + w] = return
 * time of warp w (%globaltimer, ns).  All three pointers are device memory
 * (int32 status, int32[2], int64[3]).
 *
 * Errors: FAVOR_ERR_INVALID_ARG for a NULL pointer; FAVOR_ERR_CUDA if the
 * launch fails.  The context stays usable after the call.
 */
favor_status favor_selftest_wait_timeout(int32_t* status, int32_t* returned, int64_t* times_ns,
                                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FAVOR_SELFTEST_H */
