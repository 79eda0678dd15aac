/*
 * fa_selftest.h -- test hooks of the GB300 attention-backward library.
 *
 * Not part of the attention API: these entry points let the test suite check
 * the tcgen05 building blocks on their own.  The pages have no counterpart.
 */
#ifndef FA_GB300_SELFTEST_H
#define FA_GB300_SELFTEST_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One-CTA tcgen05.mma GEMM, C fp32 [128 x N] (row-major, device), in one of
 * the operand forms of the backward kernel (16-bit inputs, device, row-major):
 *   mode 0: C = A B^T,    A [128 x K], B [N x K]   (both K-major, shared memory)
 *   mode 1: C = A B,      A [128 x K] held in tensor memory, B [K x N] MN-major
 *   mode 2: C = A^T B,    A [K x 128], B [K x N]   (both MN-major, shared memory)
 * N, K in {64, 128}; bf16 != 0 selects bf16, else fp16.  err: device int that
 * receives a non-zero bit if the completion wait ran out (bounded at 2 s).
 * Returns 0, 1 (bad argument) or 3 (CUDA error). */
int fa_selftest_umma(int mode, int N, int K, int bf16, const void *A, const void *B, float *C,
                     int *err, cudaStream_t stream);

/* Deterministic-order semaphore wait in isolation: one CTA waits until
 * sem[0] >= target with a budget of budget_ns nanoseconds, then adds 1.
 * On expiry it sets *err (device) and returns without adding.  Used to test
 * that a wait that can never succeed ends with an error instead of a hang. */
int fa_selftest_semaphore(int *sem, int target, long long budget_ns, int *err,
                          cudaStream_t stream);

/* Register layout of the 16-lane tensor-memory access shapes: one CTA of 128
 * threads, 32 allocated columns, out = device uint32 [128 x 32].
 *   which 0: thread r writes (r << 8 | c) into column c of lane r with the
 *            32-lane shape, then every thread reads 2 x 16 registers with the
 *            16x256b.x4 shape at lane offsets 0 and 16 of its warp's quarter
 *            into out[r * 32 + 16 h + reg].
 *   which 1: every thread writes 0x80000000 | r << 8 | h << 4 | reg with the
 *            16x128b.x4 shape at lane offsets h = 0, 1 over zeros; out[lane *
 *            32 + column] is what the 32-lane shape then reads.
 * Returns 0, 1 (bad argument) or 3 (CUDA error). */
int fa_selftest_tmem_layout(int which, unsigned int *out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
