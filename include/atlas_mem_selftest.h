/*
 * atlas_mem_selftest.h -- self-test of the library's tensor-core building
 * blocks.  No counterpart in the pages: it exists so that tests can check,
 * on the GPU, the shared-memory operand layout, the tcgen05.mma instruction
 * descriptor and the TMEM accumulator layout that every tensor-core kernel
 * of the library relies on.
 */
#ifndef ATLAS_MEM_SELFTEST_H
#define ATLAS_MEM_SELFTEST_H
#ifdef __cplusplus
extern "C" {
#endif

/* D = A * B^T with one CTA: M in {64, 128}, 16 <= N <= 256, 16 <= K <= 128
 * (multiples of 16).  A: device 16-bit (bf16 if bf16 != 0 else fp16), [M][K]
 * (a_mn_major == 0, K-major operand) or [K][M] (a_mn_major != 0, MN-major);
 * B: device [N][K] (b_mn_major == 0) or [K][N] (b_mn_major != 0).
 * raw_out: device [128][N] fp32, the raw accumulator of all 128 TMEM lanes.
 * status: device int, set to 1 if the kernel's bounded wait gave up.
 * Asynchronous on `stream`; returns ATLAS_OK (0), ATLAS_ERR_INVALID_ARG (1)
 * or ATLAS_ERR_CUDA (3). */
int atlas_mem_selftest_mma(int M, int N, int K, int a_mn_major, int b_mn_major, int bf16, const void* A,
                           const void* B, float* raw_out, int* status, void* stream);

/* Layout check of the 16x32bx2 TMEM load used on M = 64 accumulators.
 * Runs D = A * B^T (M = 64, A: device bf16 [64][K], B: device bf16 [N][K],
 * 64 <= N <= 256, 16 <= K <= 128, multiples of 16) and has every warp w of 4
 * load columns [col, col + 32) of its 32-lane sub-partition with that shape.
 * raw_out: device fp32 [128][16]: row w * 32 + t = the 16 registers of
 * thread t of warp w.  Before the MMA, lanes 16-31 of every sub-partition
 * are marked over the accumulator's columns; status: device int, 1 if the
 * bounded wait gave up, 2 if the MMA changed a mark. */
int atlas_mem_selftest_ld16x2(int N, int K, const void* A, const void* B, float* raw_out, int col, int* status,
                              void* stream);

/* Failure detection without a fault: one CTA waits, with the library's
 * bounded mbarrier wait limited to max_cycles (1 .. 2^31 SM clock cycles),
 * on a barrier that nothing arrives at.  The wait gives up, the kernel stores
 * ATLAS_ERR_TIMEOUT (5) into *status (device int) and the cycles it waited
 * into *waited_cycles (device), and returns; the context stays usable.
 * Asynchronous on `stream`; returns ATLAS_OK, ATLAS_ERR_INVALID_ARG or
 * ATLAS_ERR_CUDA. */
int atlas_mem_selftest_wait_timeout(long long max_cycles, int* status, long long* waited_cycles, void* stream);

#ifdef __cplusplus
}
#endif
#endif
