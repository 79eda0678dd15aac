// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass without any device
// allocation, for callers that cannot allocate device memory when they call
// the library (see include/fa.h).
//
// The scratch the backward kernels need (Dv, LSE2, the fp32 dQ accumulator,
// the work-unit list and the error word) lives in one file-scope device array
// of FA_NOALLOC_SCRATCH_BYTES.  The array exists on every GPU that loads this
// library, for the life of the process.  Host code only ever sees a stand-in
// for its name, so the device address is looked up once per device, with that
// device current, and handed to the kernels as an ordinary pointer.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device; looked up on the first
// call for that device (lookup = false: only what an earlier call found,
// possibly null).
fa_status scratch_address(void **out, bool lookup = true) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_setup_mutex);
    if (!g_scratch_addr[dev] && lookup) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_scratch_bytes(void) { return (size_t)FA_NOALLOC_SCRATCH_BYTES; }

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                         const int *cu_seqlens_q, const int *cu_seqlens_k, int deterministic,
                         fa_dtype dtype, cudaStream_t stream) {
    const size_t need = fa_bwd_workspace_bytes(B, Sq, Sk, Hq, Hkv, D, cu_seqlens_q != nullptr,
                                               deterministic);
    if (need == 0) {
        // sizes the planner refuses: let the regular validation name the problem
        return fa_bwd_with_workspace(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D,
                                     softmax_scale, causal, cu_seqlens_q, cu_seqlens_k,
                                     deterministic, dtype, nullptr, 0, stream);
    }
    if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    fa_status st = scratch_address(&scratch);
    if (st != FA_OK) return st;
    return fa_bwd_with_workspace(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D,
                                 softmax_scale, causal, cu_seqlens_q, cu_seqlens_k, deterministic,
                                 dtype, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}

fa_status fa_bwd_noalloc_status(cudaStream_t stream) {
    void *scratch = nullptr;
    fa_status st = scratch_address(&scratch, false);
    if (st != FA_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    if (!scratch) return FA_OK;   // no call has used the array on this device
    // the error word sits at the start of the backward's workspace layout
    size_t err_off = 0;
    int h = 0;
    if (cudaMemcpy(&h, static_cast<unsigned char *>(scratch) + err_off, sizeof(int),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (h != 0 && cudaMemset(static_cast<unsigned char *>(scratch) + err_off, 0, sizeof(int)) !=
                      cudaSuccess)
        return FA_ERR_CUDA;
    if (h & 4) return FA_ERR_INVALID_ARG;   // a varlen length out of bounds
    return h ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
