/*
 * zero_debug.h -- test hooks of the GB300 ZeRO shard-step library.  Not part
 * of the method: they exist so that tests can exercise failure paths without
 * a GPU fault, and check host-side planning without a GPU.
 */
#ifndef ZERO_GB300_DEBUG_H
#define ZERO_GB300_DEBUG_H

#include <stdint.h>

#include "zero.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Make the staged reduce's bounded waits run out: every stage of its bulk
 * copies then expects `bytes` more than its copies deliver, so the copies
 * land but the stage's mbarrier phase never completes.  Each block gives up
 * after one second of waiting, sets the device error word, counts as an
 * overflow (the step is skipped and, with a dynamic loss scale, the scale is
 * halved) and returns; the step's result read reports ZERO_ERR_TIMEOUT.
 * Applies to launches made after the call, process-wide; 0 (the default)
 * restores normal operation.  Errors: none. */
zero_status zero_debug_set_stage_tx_pad(uint32_t bytes);

/* The reduce planner's choice for n_rows rows (one stepped rank's shard of a
 * FlatParameter each), as a step (mode 0) or a micro-step accumulation (1:
 * the first, 2: a later one) would make it: *staged = 1 for the staged
 * (bulk-copy) reduce, 0 for the plain one.  Row j: in_addr[j], the address of
 * its first contribution's first element; ld[j], the contributor row stride
 * in elements; shard[j], its element count; acc_addr[j] (modes 1 and 2), its
 * fp32 accumulator.  Host logic only: no address is dereferenced and no GPU
 * is needed.  Errors: INVALID_ARG (NULL arrays or output, n_rows < 1,
 * n_contrib < 1, unknown dtype or mode, mode 1/2 without acc_addr). */
zero_status zero_debug_reduce_form(zero_dtype grad_dtype, int32_t n_contrib, int32_t n_rows,
                                   const uint64_t *in_addr, const int64_t *ld,
                                   const int64_t *shard, const uint64_t *acc_addr,
                                   int32_t mode, int32_t *staged);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_DEBUG_H */
