/*
 * sink_attn_testing.h - test hooks of libsinkattn. Not for production use:
 * they make calls fail on purpose so that tests can exercise the error paths
 * that sink_attn.h documents, without faulting or hanging the GPU.
 */
#ifndef SINK_ATTN_TESTING_H
#define SINK_ATTN_TESTING_H

#include "sink_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* When on (process-wide, for calls made after this one), the TMA producer of
 * the 64-wide tensor-core forward (causal layers without a window of 256 or
 * less) and of the 64-wide tensor-core backward stops issuing loads after its
 * first stage: the kernel's consumers then wait for data that never comes,
 * their bounded waits run out (sink_attn_set_wait_limit_ns), the kernel sets
 * SINK_FLAG_TIMEOUT and returns, every copy and product it did issue having
 * completed. The outputs of such a call are invalid. Off by default; pass 0
 * to turn it off. */
SINK_API void sink_attn_testing_withhold_load(int on);

#ifdef __cplusplus
}
#endif
#endif /* SINK_ATTN_TESTING_H */
