/* medusa_test_hooks.h: entry points of libmedusa_gb300 that exist only for its
 * own failure-detection tests.  They are NOT part of the library's API: a
 * program that computes with the library never calls them, and they may
 * change or disappear without notice.  The paper has no counterpart.
 *
 * Same conventions as medusa.h (caller-owned device pointers, stream-ordered,
 * host validation before any launch, device errors in d_status).
 */
#ifndef MEDUSA_TEST_HOOKS_H
#define MEDUSA_TEST_HOOKS_H

#include "medusa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* medusa_linear_test_stall: runs medusa_linear (bf16) with the loads of its
 * first pipeline stage withheld, so the kernel's bounded barrier waits (1 s)
 * run out on purpose: the kernel stops every role, waits (bounded) for its
 * copies and MMAs in flight, frees its tensor memory and sets
 * MEDUSA_DEV_TIMEOUT in d_status; y is not meaningful.  The context stays
 * usable (no fault, no trap), so a test can check the status and then make an
 * ordinary call.  Same arguments and validation as medusa_linear. */
medusa_status medusa_linear_test_stall(const void* x, const void* w, void* y, int T, int K, int Nout, void* ws,
                                       size_t ws_bytes, int32_t* d_status, medusa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_TEST_HOOKS_H */
