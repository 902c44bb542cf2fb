/*
 * verify_attn_testing.h -- test hooks of libverify_attn.so (not part of the
 * compute API).
 */
#ifndef VERIFY_ATTN_TESTING_H
#define VERIFY_ATTN_TESTING_H

#include "verify_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Exercise the bounded-wait error path without hanging anything: launches one
 * kernel that waits on an mbarrier no one ever arrives on, for at most wait_ns
 * nanoseconds (0 < wait_ns <= 1e8), after which the kernel records
 * VA_ERR_TIMEOUT in the status word of `workspace` and exits.  A following
 * verify_attn_check_status() on the same stream returns VA_ERR_TIMEOUT.
 * The library has no counterpart in the method: it tests the error path that
 * every pipeline wait of the attention kernel relies on.
 */
va_status verify_attn_selftest_wait_timeout(void *workspace, unsigned long long wait_ns, va_stream stream);

/*
 * Fault injection on the host side of the attention calls, for the recovery
 * tests.  Until called again, every later attention launch of the process
 * (a) uses wait_ns (0 < wait_ns <= 1e8) as the limit of each bounded device
 * wait instead of the default (wait_ns = 0 restores the default), and (b) if
 * drop_part >= 0, lets CTA number drop_part of the tcgen05 attention kernels
 * (the ones that merge split segments themselves) skip announcing the
 * segment parts it computed, as if that message were lost:
 * the other parts of those segments then wait for it until the limit runs
 * out, record VA_ERR_TIMEOUT and finish without merging (drop_part < 0: off).
 * Nothing on the GPU faults or hangs; the call's outputs are undefined.
 */
va_status verify_attn_test_inject(unsigned long long wait_ns, int drop_part);

/*
 * Path of verify_build_index for the tests.  mode 0 (the default): each
 * top-k selection first tries the one-pass sampled-threshold select and falls
 * back to the radix select over all keys when the sample cannot decide;
 * mode 1: the radix select over all keys only.  Both give the same sets; the
 * tests compare each with the oracle.  Applies to every later launch of the
 * process until called again.  Returns VA_ERR_INVALID_ARG for another mode.
 */
va_status verify_attn_test_index_path(int mode);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_TESTING_H */
