/*
 * tma_intensity.h -- the TMA load-mode x compute-intensity experiment of
 * "B-08. Hopper TMA：从单线程 Bulk Copy 到吞吐墙" (www.lqnn.cn), sections 3 and 5
 * (modes sync / bulk1d / tensor2d / pipe2, the fma_iters sweep), as a kernel of
 * libgemm_gb300.so, so the page's measurement can be repeated on GB300.
 *
 * Every element of `in` passes through `fma_iters` fused multiply-adds
 * y <- fma(y, a, b) (starting from y = x) and is written to the same index of
 * `out`; the mode only changes how each 4 KiB tile reaches shared memory:
 *   0 sync     : the block's 256 threads copy the tile with plain loads;
 *   1 bulk1d   : one thread issues a 1-D cp.async.bulk of 1024 consecutive
 *                floats, all threads wait on its mbarrier immediately;
 *   2 tensor2d : a 2-D tensor-map copy of a 32 x 32 tile of the rows x cols
 *                matrix view of `in` (rows = n / cols), immediate wait;
 *   3 pipe2    : 1-D bulk copies, double-buffered (next tile in flight while the
 *                current one is computed).
 * Grid: one 256-thread block per 64 tiles.  n must be a multiple of 65536;
 * mode 2 also needs cols and n / cols multiples of 32.  in, out: device
 * pointers, 16-byte aligned, caller-owned.  error_word: device int32 or NULL;
 * a mode whose barrier wait runs out (1 s) writes 1 there.  Asynchronous on
 * `stream`.  Returns GEMM_ERR_INVALID_ARG / GEMM_ERR_ALIGNMENT /
 * GEMM_ERR_TENSORMAP / GEMM_ERR_LAUNCH on failure.
 */
#ifndef GB300_TMA_INTENSITY_H
#define GB300_TMA_INTENSITY_H

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

gemm_status_t tma_intensity_run(int32_t mode, int32_t fma_iters, float a, float b,
                                const float *in, float *out, int64_t n, int32_t cols,
                                int32_t *error_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_TMA_INTENSITY_H */
