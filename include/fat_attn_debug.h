/*
 * fat_attn_debug.h -- test hooks of the fused relative-position attention library.
 * Not needed for normal use; the test-suite uses them to check the device-side bucket mapping
 * and the bounded pipeline waits without faulting the GPU.
 */
#ifndef FAT_ATTN_DEBUG_H
#define FAT_ATTN_DEBUG_H
#include <stdint.h>
#include "fat_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Writes, for delta = delta_lo .. delta_lo + n - 1, the T5 bucket id the attention kernels use
 * (same device functions and host thresholds) into out_dev[0 .. n-1] (device int32): the kernels
 * compute it two ways (a binary search over thresholds staged in shared memory for their bias
 * tables, a direct count elsewhere); an entry where the two disagree is -1. Asynchronous on
 * `stream`. Errors as in fat_attn.h (FAT_EINVAL_BUCKETS for bad bucket arguments).
 */
int fat_attn_debug_buckets(long long delta_lo, int n, int num_buckets, int max_distance,
                           int bidirectional, int32_t *out_dev, void *stream);

/*
 * Process-wide knobs for the watchdog test. timeout_ns: time limit of every pipeline wait
 * (<= 0 restores the default of 4 s). flags bit 0: the forward producer warp issues no copies,
 * so the consumers' waits run out, the kernel records FAT_DEVERR_TIMEOUT_FWD and exits cleanly;
 * bit 1: likewise for the backward's first copies (FAT_DEVERR_TIMEOUT_BWD). The forward over
 * short documents at head_dim 64 runs as persistent CTAs when there are enough 128-row blocks,
 * else as a grid of one-tile CTAs (both compute the same results): bit 2 takes the grid, bit 3
 * the persistent CTAs, whatever the size (the tests compare them).
 */
void fat_attn_debug_set_watchdog(long long timeout_ns, int flags);

#ifdef __cplusplus
}
#endif
#endif
