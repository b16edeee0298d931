/*
 * bit_moe_expert_gb300 -- per-kernel timing for benchmarks.
 *
 * Not part of the layer itself (the pages define no such call): while enabled,
 * every kernel launch of moe_route / moe_forward is bracketed by two CUDA events
 * recorded on the launch's own stream, so a kernel's device time can be read
 * back per kernel kind.  Events between kernels remove the overlap that
 * programmatic dependent launch gives, so enable it only for a separate timing
 * pass, never inside stream capture.  Disabled by default.  Host-side state is
 * process-wide and not thread-safe.
 */
#ifndef BIT_MOE_EXPERT_GB300_MOE_PROFILE_H
#define BIT_MOE_EXPERT_GB300_MOE_PROFILE_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Turns timing on (1) or off (0); returns the previous setting. */
int moe_profile_enable(int on);

/* Number of kernel kinds the library launches, and the name of kind `id`
 * (NULL for an id out of range). */
int moe_profile_kernel_count(void);
const char* moe_profile_kernel_name(int id);

/* Synchronises on the recorded events and returns, for kernel kind `id`, the
 * summed device time in milliseconds and the number of timed launches since
 * the last reset.  MOE_ERR_INVALID_ARG for a bad id or null pointers,
 * MOE_ERR_CUDA if an event query fails. */
moe_status moe_profile_read(int id, double* total_ms, long long* launches);

/* Forgets all recorded times (synchronises on pending events first). */
void moe_profile_reset(void);

/* Test hook of the decode kernel (moe_forward and moe_layer with T <= 4), for
 * tests of failure detection only; no counterpart on the source pages.  The
 * kernel's CTAs meet once at a barrier over the grid (every h value of the
 * call written) with a bounded wait.
 *   wait_limit_cycles  limit of that wait, in SM clock cycles (<= 0 restores
 *                      the default, about 2 s at the maximum clock); a wait
 *                      that runs out records MOE_ERR_TIMEOUT in the workspace
 *                      status word and the kernel carries on to its end
 *   drop_cta           a CTA of the launch whose arrival at the barrier is
 *                      skipped, so that every CTA's wait runs out; -1 for none
 *                      (the default)
 * Applies to the current device, to launches made after it returns.  A call
 * whose wait ran out leaves its outputs meaningless; the next call on the same
 * workspace is unaffected.  Synchronous (a copy to device memory); not for
 * use during stream capture. */
moe_status moe_debug_decode(long long wait_limit_cycles, int drop_cta);

#ifdef __cplusplus
}
#endif
#endif
