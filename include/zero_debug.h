/*
 * zero_debug.h -- test hooks of the GB300 ZeRO shard-step library.  Not part
 * of the method: they exist so that tests can exercise failure paths without
 * a GPU fault.
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

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_DEBUG_H */
