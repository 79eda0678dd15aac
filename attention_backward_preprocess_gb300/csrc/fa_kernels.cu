// fa_kernels.cu -- the bandwidth-bound kernels around the main backward kernel:
//   schedule_kernel     builds the list of work units (sequence, K/V block, kv head)
//   preprocess_kernel   Dv = rowsum(dO o O), LSE2 = LSE * log2(e), zero dQaccum
//   postprocess_kernel  dQ = cast(dQaccum * scale)
#include "fa_device.cuh"
#include "fa_params.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// lengths the attention uses (seqused, when given, else the stored ones)
__device__ __forceinline__ int seq_len_q(const BwdParams &p, int b) { return used_len_q(p, b); }
__device__ __forceinline__ int seq_len_k(const BwdParams &p, int b) { return used_len_k(p, b); }

// ------------------------------------------------------------------ schedule
// Work units in the order (n_block, sequence, kv head): every unit of a given
// (sequence, kv head) comes after the units with smaller n_block, which the
// deterministic dQ order relies on, and under a causal mask the units with the
// most query blocks (small n_block) come first.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) schedule_kernel(BwdParams p) {
    __shared__ int warp_sums[32];
    __shared__ int total_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int max_nb = (p.Sk + kBlockN - 1) / kBlockN;
    int base = 0;
    for (int n = 0; n < max_nb; ++n) {
        for (int b0 = 0; b0 < p.B; b0 += 1024) {
            const int b = b0 + tid;
            int flag = 0;
            if (b < p.B) flag = seq_len_k(p, b) > n * kBlockN;
            // block-wide exclusive scan of flag
            int x = flag;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) warp_sums[wid] = x;
            __syncthreads();
            if (wid == 0) {
                int s = warp_sums[lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    int y = __shfl_up_sync(0xffffffffu, s, o);
                    if (lane >= o) s += y;
                }
                warp_sums[lane] = s;   // inclusive
                if (lane == 31) total_s = s;
            }
            __syncthreads();
            const int pos = x - flag + (wid > 0 ? warp_sums[wid - 1] : 0);
            if (flag) {
                for (int hk = 0; hk < p.Hkv; ++hk) {
                    const long long idx = (long long)(base + pos) * p.Hkv + hk;
                    if (idx < p.max_tiles) p.tiles[idx] = make_int4(b, n, hk, 0);
                }
            }
            base += total_s;
            __syncthreads();
        }
    }
    if (tid == 0) *p.ntiles = min(base * p.Hkv, p.max_tiles);
}

// ---------------------------------------------------------------- preprocess
// grid (row chunks, sequences); D/8 threads per (position, head) row, each
// reading 16 bytes of O and of dO.  Padding rows up to the next multiple of
// 128 get Dv = 0 and LSE2 = +inf (so P = 0 there).  Every workspace row of
// the sequence has its dQ accumulator zeroed, and in deterministic mode its
// semaphores as well.
template <int D, typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(BwdParams p) {
    constexpr int TPR = D / 8;   // threads per row
    const int b = blockIdx.y;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long rid = gid / TPR;
    const int part = (int)(gid % TPR);
    const int lq = seq_len_q(p, b);
    const int lq_round = (lq + kRowTile - 1) / kRowTile * kRowTile;
    const int s = (int)(rid / p.Hq), h = (int)(rid % p.Hq);
    // no early return: the row sum below is a full-warp shuffle
    const bool active = s < lq_round;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        *p.err = 0;            // per-call error word
        p.unit_counter[0] = 0;   // the main kernel's dynamic work-unit counter ...
        p.unit_counter[1] = 0;   // ... and its count of CTAs that ran out of units
    }
    const long long wr = active ? ws_row(p, b, h, s) : 0;
    float acc = 0.f;
    // O / dO rows hold Dh <= D columns (a multiple of 8): parts past Dh add 0
    if (active && s < lq && part * 8 < p.Dh) {
        const long long trow = p.varlen ? (long long)p.cu_q[b] + s : (long long)b * p.Sq + s;
        const long long off = (trow * p.Hq + h) * p.Dh + part * 8;
        const uint4 ov = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.o) + off);
        const uint4 dv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.dout) + off);
        const uint32_t oa[4] = {ov.x, ov.y, ov.z, ov.w}, da[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 of = Cvt<T>::unpack(oa[t]), df = Cvt<T>::unpack(da[t]);
            acc = fmaf(of.x, df.x, acc);
            acc = fmaf(of.y, df.y, acc);
        }
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
    if (!active) return;
    if (part == 0) {
        float l2 = __int_as_float(0x7f800000);   // +inf on padding rows
        if (s < lq) {
            const long long li = p.varlen ? (long long)h * p.cu_q[p.B] + p.cu_q[b] + s
                                          : ((long long)b * p.Hq + h) * p.Sq + s;
            float l = p.lse[li];
            if (l == -__int_as_float(0x7f800000)) l = 0.f;   // get_validated_lse
            l2 = l * kLog2e;
        }
        p.dvec[wr] = (s < lq) ? acc : 0.f;
        p.lse2[wr] = l2;
        if (p.deterministic && (s % 64) == 0) p.sem[wr / 64] = 0;
    }
    float4 *z = reinterpret_cast<float4 *>(p.dqacc + wr * D) + part * 2;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// --------------------------------------------------------------- postprocess
// dQ[row, h, :] = cast(dQaccum[ws_row(b, h, s), :] * scale) for s < Lq
// (FlashAttentionBackwardPostprocess: acc.load() * scale, then a predicated
// store clipped to the sequence length).
template <int D, typename T>
__global__ void __launch_bounds__(256) postprocess_kernel(BwdParams p) {
    constexpr int TPR = D / 8;
    const int b = blockIdx.y;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long rid = gid / TPR;
    const int part = (int)(gid % TPR);
    const int lq = seq_len_q(p, b);
    const int s = (int)(rid / p.Hq), h = (int)(rid % p.Hq);
    if (s >= lq || part * 8 >= p.Dh) return;   // dQ rows hold Dh <= D columns
    const long long wr = ws_row(p, b, h, s);
    const float4 *src = reinterpret_cast<const float4 *>(p.dqacc + wr * D) + part * 2;
    const float4 a = src[0], c = src[1];
    const float sc = p.scale;
    uint4 o;
    o.x = Cvt<T>::pack(a.x * sc, a.y * sc);
    o.y = Cvt<T>::pack(a.z * sc, a.w * sc);
    o.z = Cvt<T>::pack(c.x * sc, c.y * sc);
    o.w = Cvt<T>::pack(c.z * sc, c.w * sc);
    const long long trow = p.varlen ? (long long)p.cu_q[b] + s : (long long)b * p.Sq + s;
    *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dq) + (trow * p.Hq + h) * p.Dh + part * 8) = o;
}

}  // namespace

cudaError_t launch_schedule(const BwdParams &p, cudaStream_t stream) {
    schedule_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

static dim3 row_grid(const BwdParams &p, int lanes_per_row, int rows_per_seq) {
    const long long threads = (long long)rows_per_seq * p.Hq * lanes_per_row;
    return dim3((unsigned)((threads + 255) / 256), (unsigned)p.B, 1);
}

cudaError_t launch_preprocess(const BwdParams &p, int bf16, cudaStream_t stream) {
    const dim3 grid = row_grid(p, p.D / 8, p.sq_round);
    if (p.D == 128) {
        if (bf16) preprocess_kernel<128, __nv_bfloat16><<<grid, 256, 0, stream>>>(p);
        else preprocess_kernel<128, __half><<<grid, 256, 0, stream>>>(p);
    } else {
        if (bf16) preprocess_kernel<64, __nv_bfloat16><<<grid, 256, 0, stream>>>(p);
        else preprocess_kernel<64, __half><<<grid, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_postprocess(const BwdParams &p, int bf16, cudaStream_t stream) {
    const dim3 grid = row_grid(p, p.D / 8, p.Sq);
    if (p.D == 128) {
        if (bf16) postprocess_kernel<128, __nv_bfloat16><<<grid, 256, 0, stream>>>(p);
        else postprocess_kernel<128, __half><<<grid, 256, 0, stream>>>(p);
    } else {
        if (bf16) postprocess_kernel<64, __nv_bfloat16><<<grid, 256, 0, stream>>>(p);
        else postprocess_kernel<64, __half><<<grid, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace fa
