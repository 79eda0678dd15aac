// fa_selftest.cu -- one-CTA tcgen05 GEMMs in the three operand forms the
// backward kernel uses, so the shared-memory / instruction descriptors and
// the TMEM data layout can be checked against a plain matmul:
//   mode 0: C = A * B^T, A [128 x K] and B [N x K] both K-major in swizzled
//           shared memory (the S = K Q^T and dP = V dO^T form)
//   mode 1: C = A * Bt, A [128 x K] in TMEM (bf16/fp16 pairs written by
//           tcgen05.st), Bt [K x N] MN-major in shared memory (the
//           dV += P^T dO and dK += dS^T Q form)
//   mode 2: C = At^T * Bt, At [K x 128] and Bt [K x N] both MN-major in shared
//           memory (the dQ form)
// C is fp32 [128 x N].  K in {64, 128}, N in {64, 128}.
// A second kernel writes and reads tensor memory through the 16-lane access
// shapes the softmax warps use, so their register <-> (lane, column) mapping
// can be checked against the plain 32-lane shape.
#include "fa_device.cuh"
#include "../../include/fa_selftest.h"

namespace fa {
namespace {

constexpr int kThreads = 128;

// element (r, c) of a [rows x 64] half-tile in the 128B-swizzled layout
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return (uint32_t)(r * 128 + (((c >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// Copies a row-major [rows x cols] 16-bit matrix into shared memory as
// cols/64 swizzled halves of [rows x 64] each (half stride rows*128 bytes).
__device__ void fill_swizzled(uint8_t *dst, const uint16_t *src, int rows, int cols) {
    for (int idx = threadIdx.x; idx < rows * cols; idx += blockDim.x) {
        int r = idx / cols, c = idx % cols;
        int half = c / 64;
        *reinterpret_cast<uint16_t *>(dst + half * rows * 128 + sw_off(r, c % 64)) = src[idx];
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) selftest_kernel(int mode, int N, int K,
                                                            const uint16_t *A, const uint16_t *B,
                                                            float *C, int *err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;              // up to 128 x 128 x 2 = 32 KB
    uint8_t *sB = smem + 32768;      // up to 128 x 128 x 2 = 32 KB
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), 256);
        tmem_relinquish();
    }
    // operands into shared memory
    if (mode == 0) {
        fill_swizzled(sA, A, 128, K);  // rows M, K-major
        fill_swizzled(sB, B, N, K);    // rows N, K-major
    } else if (mode == 1) {
        fill_swizzled(sB, B, K, N);    // rows K, MN-major
    } else {
        fill_swizzled(sA, A, K, 128);  // rows K, M-major
        fill_swizzled(sB, B, K, N);    // rows K, N-major
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (mode == 1) {
        // thread m owns row m of A; columns 128.. hold K/2 packed pairs
        const int m = threadIdx.x;
        for (int k0 = 0; k0 < K; k0 += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
                pk[t] = (uint32_t)A[m * K + k0 + 2 * t] | ((uint32_t)A[m * K + k0 + 2 * t + 1] << 16);
            tmem_st16(tmem + lane_base + 128 + k0 / 2, pk);
        }
        tmem_wait_st();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        for (int kk = 0; kk < K / 16; ++kk) {
            uint32_t acc = kk > 0;
            if (mode == 0) {
                const uint32_t off = (kk % 4) * 32;  // K step inside a 64-wide half
                uint64_t ad = sw128_desc(a_base + (kk / 4) * 128 * 128 + off, 16, 1024);
                uint64_t bd = sw128_desc(b_base + (kk / 4) * N * 128 + off, 16, 1024);
                mma_ss(tmem, ad, bd, make_idesc(128, N, kBf16, false, false), acc);
            } else if (mode == 1) {
                uint64_t bd = sw128_desc(b_base + kk * 2048, K * 128, 1024);
                mma_ts(tmem, tmem + 128 + kk * 8, bd, make_idesc(128, N, kBf16, false, true), acc);
            } else {
                uint64_t ad = sw128_desc(a_base + kk * 2048, K * 128, 1024);
                uint64_t bd = sw128_desc(b_base + kk * 2048, K * 128, 1024);
                mma_ss(tmem, ad, bd, make_idesc(128, N, kBf16, true, true), acc);
            }
        }
        mma_commit(smem_u32(&bar));
    }
    WaitCtl w{&abort_flag, err, 2000000000LL};
    bool ok = mbar_wait(smem_u32(&bar), 0, w);
    tc_fence_after();
    if (ok) {
        for (int n0 = 0; n0 < N; n0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + n0, r);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) C[threadIdx.x * N + n0 + t] = __uint_as_float(r[t]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    (void)lane;
}

// which 0: each thread writes (row << 8 | column) into columns 0..31 of its
//          own lane with the 32-lane shape, then reads them back with
//          tmem_ld16x256 at lane offsets 0 and 16 of its warp's quarter:
//          out[thread * 32 + 16 * h + reg].
// which 1: zeros with the 32-lane shape, then tmem_st16x128 of the values
//          0x80000000 | thread << 8 | h << 4 | reg at lane offsets h = 0, 1,
//          read back with the 32-lane shape: out[row * 32 + column].
__global__ void __launch_bounds__(128) tmem_layout_kernel(int which, uint32_t *out) {
    __shared__ uint32_t tmem_base_s;
    const int warp = threadIdx.x / 32;
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    const uint32_t row = threadIdx.x;
    uint32_t a[16], b[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        a[c] = which == 0 ? (row << 8 | (uint32_t)c) : 0u;
        b[c] = which == 0 ? (row << 8 | (uint32_t)(16 + c)) : 0u;
    }
    tmem_st16(tmem + lb, a);
    tmem_st16(tmem + lb + 16, b);
    tmem_wait_st();
    __syncwarp();
    if (which == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t r[16];
            tmem_ld16x256(tmem + lb + ((uint32_t)(16 * h) << 16), r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) out[threadIdx.x * 32 + 16 * h + k] = r[k];
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t r[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                r[k] = 0x80000000u | (uint32_t)threadIdx.x << 8 | (uint32_t)h << 4 | (uint32_t)k;
            tmem_st16x128(tmem + lb + ((uint32_t)(16 * h) << 16), r);
        }
        tmem_wait_st();
        __syncwarp();
        uint32_t r[32];
        tmem_ld32(tmem + lb, r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) out[row * 32 + c] = r[c];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 32);
}

__global__ void semaphore_kernel(int *sem, int target, long long budget_ns, int *err) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncwarp();
    if (threadIdx.x == 0) {
        WaitCtl w{&abort_flag, err, budget_ns};
        if (sem_wait_geq(sem, target, w)) red_release_add_gpu(sem, 1);
    }
}

}  // namespace
}  // namespace fa

extern "C" int fa_selftest_umma(int mode, int N, int K, int bf16, const void *A, const void *B,
                                float *C, int *err, cudaStream_t stream) {
    if (mode < 0 || mode > 2 || (N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
    if (!A || !B || !C || !err) return 1;
    const int smem = 65536 + 1024;
    auto kern = bf16 ? fa::selftest_kernel<true> : fa::selftest_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 3;
    kern<<<1, fa::kThreads, smem, stream>>>(mode, N, K, (const uint16_t *)A, (const uint16_t *)B,
                                            C, err);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int fa_selftest_semaphore(int *sem, int target, long long budget_ns, int *err,
                                     cudaStream_t stream) {
    if (!sem || !err || budget_ns <= 0) return 1;
    fa::semaphore_kernel<<<1, 32, 0, stream>>>(sem, target, budget_ns, err);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int fa_selftest_tmem_layout(int which, unsigned int *out, cudaStream_t stream) {
    if ((which != 0 && which != 1) || !out) return 1;
    fa::tmem_layout_kernel<<<1, 128, 0, stream>>>(which, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
