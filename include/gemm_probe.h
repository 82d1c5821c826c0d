/*
 * gemm_probe.h -- measurement aid of libgemm_gb300.so: the issue rate of the
 * tensor-core instruction the GEMM kernels are built on.
 *
 * The GEMM's compute-bound roofline needs a dense tensor peak.  Besides a
 * library GEMM's measured throughput, the theoretical figure is
 *     SM count x SM clock x (dense FLOP per clock per SM),
 * and the last factor is taken from this probe rather than a data sheet: each
 * CTA (one per SM) issues `iters` tcgen05.mma.cta_group::1.kind::f16 (M = 128,
 * N = 256, K = 16, fp16 operands from shared memory, fp32 accumulation in one
 * TMEM accumulator) back to back from one thread, with no loads, and times
 * first issue to completion of the last with the SM cycle counter.  Each MMA is
 * 2 * 128 * 256 * 16 = 1,048,576 FLOP, so
 *     FLOP per clock per SM = iters * 1048576 / cycles[cta].
 * (The GEMM's own operands are K-contiguous fp16/bf16, the same instruction.)
 *
 * grid   : CTAs, 1 .. number of SMs (one per SM: each holds 49 KiB of shared
 *          memory and 256 TMEM columns, launched one per SM);
 * iters  : MMAs per CTA, 1 .. 1 << 24;
 * cycles : device array of `grid` int64: SM clock cycles (clock64) of CTA i;
 * ns     : device array of `grid` int64: the same interval in %globaltimer ns;
 * error_word : device int32; set to 1 if the completion wait ran out (2 s),
 *          in which case the CTA's entries are -1;
 * All device pointers are caller-owned and 8-byte (error_word 4-byte) aligned.
 * Asynchronous on `stream`.  Returns GEMM_ERR_INVALID_ARG for a bad argument,
 * GEMM_ERR_LAUNCH if the launch failed.
 */
#ifndef GB300_GEMM_PROBE_H
#define GB300_GEMM_PROBE_H

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

gemm_status_t gemm_probe_mma_rate(int32_t grid, int32_t iters, int64_t *cycles, int64_t *ns,
                                  int32_t *error_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_PROBE_H */
