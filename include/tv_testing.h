/*
 * tv_testing.h -- hooks that libtv's own tests use to reach code paths that ordinary
 * inputs never take.  They are not part of the stable interface of tv.h: a program that
 * serves requests has no reason to call them.
 */
#ifndef TV_TESTING_H_
#define TV_TESTING_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * tv_testing_set_wait_fault -- make the bounded waits of the tensor-core attention kernel
 * run out, so that a test can check that the kernel gives up cleanly.
 *
 * The pages describe no such hook.  The tensor-core kernel waits on mbarriers for data
 * that other warps, the other CTA of its cluster, the TMA engine or the tensor cores
 * deliver; every wait has a wall-clock deadline after which the kernel records
 * TV_ERR_TIMEOUT in the call's status word, tells the peer CTA to stop, waits for its own
 * copies and MMAs in flight, frees its tensor memory and returns.  This hook exercises
 * that path without any fault:
 *   skip_key_loads : 1 = the S-side producer of every cluster issues no TMA loads at all,
 *                    so the first wait on a key stage can only end at its deadline;
 *                    0 = normal operation.
 *   deadline_ns    : deadline of every wait in nanoseconds; 0 restores the default (2 s).
 *   exit_counts    : device int32[2] or NULL.  When set, every CTA of the kernel adds 1 to
 *                    exit_counts[0] as it leaves, and 1 to exit_counts[1] if it left through
 *                    the abort path (after freeing its tensor memory).
 * The setting is process-wide and applies to every later tv_verify_attn call on the
 * tensor-core path until it is reset with (0, 0, NULL); calls made while it is on produce
 * no valid output.  Returns TV_OK, or TV_ERR_INVALID_ARG for skip_key_loads outside {0, 1}.
 */
int tv_testing_set_wait_fault(int skip_key_loads, uint64_t deadline_ns, int32_t* exit_counts);

#ifdef __cplusplus
}
#endif

#endif /* TV_TESTING_H_ */
