/*
 * mxa_testing.h -- test hooks of libmxa.so: run the device functions the
 * attention kernels use to quantize P and dS on caller data, so that tests
 * can check them bit for bit against an independent codec.  Not part of the
 * attention API (include/mxa.h).
 *
 *   P quantization: E4M3 round-to-nearest-even with saturation to +-448
 *   (FLAMIA notes sec. 5, the P cap 2^(c+tau) <= 448: larger values saturate
 *   silently).
 *   dS quantization: one UE8M0 scale per 32 x 32 block from the block
 *   max-abs, e = ceil(log2(amax / 448)), taken with a warp-wide max over the
 *   register layout the kernels hold (one warp = 32 rows of 32 values) (FA4
 *   write-up, "Квантование dS без транспонирования").
 */
#ifndef MXA_TESTING_H
#define MXA_TESTING_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#include "mxa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* codes[i] = E4M3 code of x[i] (device pointers, n % 4 == 0, x 16-byte and
 * codes 4-byte aligned), through the kernels' packed conversion.  The caller
 * owns both buffers.  Status: MXA_OK, MXA_ERR_ARG, MXA_ERR_ALIGN,
 * MXA_ERR_CUDA (launch failure; asynchronous faults surface at the next
 * synchronization). */
mxa_status mxa_test_e4m3(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream);

/* Quantize nblocks blocks of 32 x 32 fp32 values (row-major, device) with the
 * kernels' dS block routine: codes [nblocks][32][32], scale bytes
 * [nblocks].  `shift` is the power-of-two boost the values carry (0, or 8 as
 * in the dK/dV kernel, whose dS inherits the 2^8 P boost); the returned
 * scale is that of the unboosted block.  codes must be 4-byte aligned; the
 * caller owns all buffers.  Status: MXA_OK, MXA_ERR_ARG (shift outside
 * [0, 16], negative count, null pointer), MXA_ERR_ALIGN, MXA_ERR_CUDA. */
mxa_status mxa_test_ds_blocks(const float* x, int nblocks, int shift, uint8_t* codes, uint8_t* scales,
                              cudaStream_t stream);

/* Run the attention kernels' bounded wait (the one every warp role uses) in
 * a one-warp kernel, on a barrier that nothing arrives on, with a spin budget
 * of budget_cycles SM clocks instead of the kernels' two seconds.  Nothing
 * asynchronous is in flight, so the wait runs out, records the device error
 * word and the kernel returns: the next mxa_get_error() reports
 * MXA_ERR_TIMEOUT and clears the word.  This exercises the timeout report of
 * mxa.h's error contract without stalling any real work.  Status: MXA_OK,
 * MXA_ERR_ARG (budget outside [0, 2^31]), MXA_ERR_CUDA. */
mxa_status mxa_test_wait_timeout(long long budget_cycles, cudaStream_t stream);

/* Block-scaled MMA rate probe: `ctas` CTAs (one per SM; launch at most the
 * SM count) each issue `iters` groups of four tcgen05.mma kind::mxf8f6f4
 * block_scale instructions of the attention forward's S shape (M = 128,
 * N = 256, K = 32 each, E4M3 operands in 128-byte-swizzled shared memory,
 * UE8M0 scales in tensor memory) from one thread, back to back, then wait for
 * them.  cycles (device, int64 [ctas], 8-byte aligned, caller-owned)
 * receives each CTA's SM clocks from its first issue to completion, or -1 if
 * its bounded wait ran out (then mxa_get_error() reports MXA_ERR_TIMEOUT).
 * FLOP per CTA = iters * 4 * 2 * 128 * 256 * 32.  The attention kernels'
 * tensor-core roofline is measured with it.  Status: MXA_OK, MXA_ERR_ARG
 * (iters outside [1, 2^24], ctas outside [1, 4096], null cycles),
 * MXA_ERR_ALIGN, MXA_ERR_CUDA. */
mxa_status mxa_test_mma_rate(int iters, int ctas, long long* cycles, cudaStream_t stream);

/* Exponential-unit rate probe: `ctas` CTAs (one per SM; launch at most the
 * SM count) of 512 threads, each thread running eight independent chains of
 * `iters` ex2.approx.ftz.f32 (the attention kernels' exponential, FLAMIA
 * notes sec. 7: the exponential unit is the co-bound of the tensor cores).
 * cycles (device, int64 [ctas], 8-byte aligned, caller-owned) receives each
 * CTA's SM clocks for its loop.  Exponentials per CTA = iters * 8 * 512.
 * The attention kernels' exponential-unit utilisation is measured against
 * it.  Status: MXA_OK, MXA_ERR_ARG (iters outside [1, 2^24], ctas outside
 * [1, 4096], null cycles), MXA_ERR_ALIGN, MXA_ERR_CUDA. */
mxa_status mxa_test_ex2_rate(int iters, int ctas, long long* cycles, cudaStream_t stream);

/* The attention forward's row maximum on fully visible key tiles, read with
 * the scores themselves (tcgen05.ld.red .max, sm_103a; FLAMIA notes sec. 7:
 * on B300 the TMEM read is merged with the row-max reduction).  x (device,
 * fp32 [128, 64], caller-owned): row r is stored to TMEM lane r, then read
 * back as two 32-column loads with their maxima.  out (device, fp32
 * [128, 3]): the maxima of columns [0, 32) and [32, 64) of each row, and the
 * number of the row's values that did not read back bit for bit.  One CTA,
 * 64 TMEM columns.  Status: MXA_OK, MXA_ERR_ARG (null pointer), MXA_ERR_ALIGN
 * (not 4-byte aligned), MXA_ERR_CUDA. */
mxa_status mxa_test_tmem_max(const float* x, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MXA_TESTING_H */
