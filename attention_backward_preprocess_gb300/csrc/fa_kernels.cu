// fa_kernels.cu -- the bandwidth-bound kernels around the main backward kernel:
//   schedule_kernel     builds the list of work units (sequence, K/V block, kv head)
//   preprocess_kernel   Dv = rowsum(dO o O), LSE2 = LSE * log2(e), zero dQaccum
//   postprocess_kernel  dQ = cast(dQaccum * scale)
//   dbias_zero_kernel   0 in the dBias entries the main kernel does not write
#include "fa_bwd_units.cuh"
#include "fa_device.cuh"
#include "fa_params.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// lengths the attention uses (seqused, when given, else the stored ones)
__device__ __forceinline__ int seq_len_q(const BwdParams &p, int b) { return used_len_q(p, b); }
__device__ __forceinline__ int seq_len_k(const BwdParams &p, int b) { return used_len_k(p, b); }

// ------------------------------------------------------------------ schedule
// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// exclusive prefix and leaves the block total in *total.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;   // inclusive
        if (lane == 31) *total = s;
    }
    __syncthreads();
    const int r = x - v + (wid > 0 ? warp_sums[wid - 1] : 0);
    __syncthreads();
    return r;
}

// Work units of a varlen problem.  Consecutive sequences form a group once
// their units reach p.unit_group (about 1.5 grids of the main kernel), and
// inside a group the units go in the order (n_block, sequence, kv head): the
// units that run at the same time then sweep the rows of a few sequences,
// whose Q, dO and dQ-accumulator rows stay in L2 (over all sequences at once
// they did not: the varlen workload's main kernel moved 1.07 GB of DRAM
// traffic against about 0.4 GB algorithmic).  Every unit of a (sequence, kv
// head) still comes after those with a smaller n_block, which the
// deterministic dQ order relies on, and under a causal mask a group's units
// with the most query blocks come first.  One block of 1024 threads; more
// than kSchedSeqs sequences, and the deterministic order (unit_group 0: few
// units of one ordering chain should run at once), take the ungrouped order.
constexpr int kSchedSeqs = 4096;
__global__ void __launch_bounds__(1024) schedule_kernel(BwdParams p) {
    __shared__ int s_nb[kSchedSeqs];    // key blocks of sequence b (0: none)
    __shared__ int s_off[kSchedSeqs];   // units of the sequences before b
    __shared__ int warp_sums[32];
    __shared__ int chunk_total;
    const int tid = threadIdx.x;
    const int max_nb = (p.Sk + kBlockN - 1) / kBlockN;
    if (p.unit_group > 0 && p.B <= kSchedSeqs) {
        for (int b = tid; b < p.B; b += 1024) {
            int nb = 0;
            // a sequence whose lengths break the planned layout gets no unit
            // (and the call reports the error)
            if (!varlen_seq_ok(p, b)) atomicOr(p.err, kErrBadLength);
            else nb = (seq_len_k(p, b) + kBlockN - 1) / kBlockN;
            s_nb[b] = nb;
        }
        __syncthreads();
        int carry = 0;
        for (int b0 = 0; b0 < p.B; b0 += 1024) {
            const int b = b0 + tid;
            const int c = b < p.B ? s_nb[b] * p.Hkv : 0;
            const int e = block_excl_scan(c, warp_sums, &chunk_total);
            if (b < p.B) s_off[b] = carry + e;
            carry += chunk_total;
            __syncthreads();
        }
        const int T = max(p.unit_group, 1);
        for (int b = tid; b < p.B; b += 1024) {
            const int nb = s_nb[b];
            if (nb == 0) continue;
            const int g = s_off[b] / T;
            int bs = b, be = b + 1;   // the group: sequences [bs, be)
            while (bs > 0 && s_off[bs - 1] / T == g) --bs;
            while (be < p.B && s_off[be] / T == g) ++be;
            long long idx0 = s_off[bs];   // the group's first unit, then past smaller n blocks
            for (int n = 0; n < nb; ++n) {
                int rank = 0, act = 0;    // group sequences with block n: before b, in all
                for (int b2 = bs; b2 < be; ++b2)
                    if (s_nb[b2] > n) {
                        ++act;
                        if (b2 < b) ++rank;
                    }
                for (int hk = 0; hk < p.Hkv; ++hk) {
                    const long long idx = idx0 + (long long)rank * p.Hkv + hk;
                    if (idx < p.max_tiles) p.tiles[idx] = make_int4(b, n, hk, 0);
                }
                idx0 += (long long)act * p.Hkv;
            }
        }
        if (tid == 0) *p.ntiles = min(carry, p.max_tiles);
        return;
    }
    // ungrouped: (n_block, sequence, kv head)
    int base = 0;
    for (int n = 0; n < max_nb; ++n) {
        for (int b0 = 0; b0 < p.B; b0 += 1024) {
            const int b = b0 + tid;
            int flag = 0;
            if (b < p.B) {
                if (!varlen_seq_ok(p, b)) {
                    if (n == 0) atomicOr(p.err, kErrBadLength);
                } else {
                    flag = seq_len_k(p, b) > n * kBlockN;
                }
            }
            const int pos = block_excl_scan(flag, warp_sums, &chunk_total);
            if (flag) {
                for (int hk = 0; hk < p.Hkv; ++hk) {
                    const long long idx = (long long)(base + pos) * p.Hkv + hk;
                    if (idx < p.max_tiles) p.tiles[idx] = make_int4(b, n, hk, 0);
                }
            }
            base += chunk_total;
            __syncthreads();
        }
    }
    if (tid == 0) *p.ntiles = min(base * p.Hkv, p.max_tiles);
}

// ---------------------------------------------------------------- preprocess
// grid (row chunks, sequences); D/8 threads per (position, head) row, each
// reading 16 bytes of O and of dO.  With varlen each thread takes RPT = 4 rows
// whose loads are in flight together (the sequence offsets are read first; one
// row per thread ran at a third of the HBM bandwidth there); dense problems
// keep one row per thread (4 was slower there).
// Padding rows up to the next multiple of 128 get Dv = 0 and LSE2 = +inf (so
// P = 0 there).  Every workspace row of the sequence has its dQ accumulator
// zeroed, and in deterministic mode its semaphores as well.  DV is the tile
// width of O / dO (the value side), DQ that of the accumulator (the query /
// key side); each of the DV / 8 threads of a row zeroes DQ / (DV / 8) floats.
template <int DQ, int DV, typename T, int RPT>
__global__ void __launch_bounds__(256) preprocess_kernel(BwdParams p) {
    constexpr int TPR = DV / 8;   // threads per row
    constexpr int ZF = DQ / TPR;  // accumulator floats each thread zeroes
    static_assert(ZF % 4 == 0, "whole float4 stores");
    const int b = blockIdx.y;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        *p.err = 0;            // per-call error word
        p.unit_counter[0] = 0;   // the main kernel's dynamic work-unit counter ...
        p.unit_counter[1] = 0;   // ... and its count of CTAs that ran out of units
    }
    // varlen lengths outside the planned layout: nothing of this sequence is
    // touched (the scheduler reports the error)
    if (p.varlen && !varlen_seq_ok(p, b)) return;
    const int lq = seq_len_q(p, b);
    const int lq_round = (lq + kRowTile - 1) / kRowTile * kRowTile;
    const long long nrows = (long long)lq_round * p.Hq;   // (position, head) rows, padded
    // block-uniform exit: no row of this block belongs to the sequence
    if ((long long)blockIdx.x * (blockDim.x / TPR) * RPT >= nrows) return;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long r0 = gid / TPR * RPT;
    const int part = (int)(gid % TPR);
    const long long qbase = p.varlen ? (long long)p.cu_q[b] : (long long)b * p.Sq;
    const long long ltot = p.varlen ? (long long)p.cu_q[p.B] : 0;   // varlen LSE row length
    float acc[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        acc[k] = 0.f;
        const long long row = r0 + k;
        const int s = (int)(row / p.Hq), h = (int)(row % p.Hq);
        // O / dO rows hold Dhv <= DV columns (a multiple of 8): parts past Dhv add 0
        if (row < nrows && s < lq && part * 8 < p.Dhv) {
            const long long off = ((qbase + s) * p.Hq + h) * p.Dhv + part * 8;
            const uint4 ov = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.o) + off);
            const uint4 dv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.dout) + off);
            const uint32_t oa[4] = {ov.x, ov.y, ov.z, ov.w}, da[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 of = Cvt<T>::unpack(oa[t]), df = Cvt<T>::unpack(da[t]);
                acc[k] = fmaf(of.x, df.x, acc[k]);
                acc[k] = fmaf(of.y, df.y, acc[k]);
            }
        }
    }
    // the row sums: full-warp shuffles (every lane of a live warp takes part)
#pragma unroll
    for (int k = 0; k < RPT; ++k)
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o, TPR);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const long long row = r0 + k;
        if (row >= nrows) break;
        const int s = (int)(row / p.Hq), h = (int)(row % p.Hq);
        const long long wr = ws_row(p, b, h, s);
        if (part == 0) {
            float l2 = __int_as_float(0x7f800000);   // +inf on padding rows
            if (s < lq) {
                const long long li = p.varlen ? (long long)h * ltot + qbase + s
                                              : ((long long)b * p.Hq + h) * p.Sq + s;
                float l = p.lse[li];
                if (l == -__int_as_float(0x7f800000)) l = 0.f;   // get_validated_lse
                l2 = l * kLog2e;
            }
            p.dvec[wr] = (s < lq) ? acc[k] : 0.f;
            p.lse2[wr] = l2;
            if (p.deterministic && (s % 64) == 0) p.sem[wr / 64] = 0;
        }
        float4 *z = reinterpret_cast<float4 *>(p.dqacc + wr * DQ + part * ZF);
#pragma unroll
        for (int c = 0; c < ZF / 4; ++c) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// --------------------------------------------------------------- postprocess
// dQ[row, h, :] = cast(dQaccum[ws_row(b, h, s), :] * scale) for s < Lq
// (FlashAttentionBackwardPostprocess: acc.load() * scale, then a predicated
// store clipped to the sequence length); RPT rows per thread, as above.
template <int D, typename T, int RPT>
__global__ void __launch_bounds__(256) postprocess_kernel(BwdParams p) {
    constexpr int TPR = D / 8;
    const int b = blockIdx.y;
    if (p.varlen && !varlen_seq_ok(p, b)) return;
    const int lq = seq_len_q(p, b);
    const long long nrows = (long long)lq * p.Hq;
    if ((long long)blockIdx.x * (blockDim.x / TPR) * RPT >= nrows) return;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long r0 = gid / TPR * RPT;
    const int part = (int)(gid % TPR);
    if (part * 8 >= p.Dh) return;   // dQ rows hold Dh <= D columns
    const long long qbase = p.varlen ? (long long)p.cu_q[b] : (long long)b * p.Sq;
    const float sc = p.scale;
    float4 a[RPT], c[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const long long row = r0 + k;
        if (row < nrows) {
            const int s = (int)(row / p.Hq), h = (int)(row % p.Hq);
            const float4 *src = reinterpret_cast<const float4 *>(p.dqacc + ws_row(p, b, h, s) * D) + part * 2;
            a[k] = src[0];
            c[k] = src[1];
        }
    }
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const long long row = r0 + k;
        if (row >= nrows) break;
        const int s = (int)(row / p.Hq), h = (int)(row % p.Hq);
        uint4 o;
        o.x = Cvt<T>::pack(a[k].x * sc, a[k].y * sc);
        o.y = Cvt<T>::pack(a[k].z * sc, a[k].w * sc);
        o.z = Cvt<T>::pack(c[k].x * sc, c[k].y * sc);
        o.w = Cvt<T>::pack(c[k].z * sc, c[k].w * sc);
        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dq) + ((qbase + s) * p.Hq + h) * p.Dh + part * 8) = o;
    }
}

// ------------------------------------------------------------- dBias zeros
// dBias (dense problems) is the whole [B, Hq, Sq, Sk] tensor dS.  The main
// kernel writes the entries of the row blocks its work units visit, inside
// the used lengths; this kernel writes 0 to every other entry (tiles the mask
// leaves out, rows and keys past the used lengths), before the main kernel
// runs.  One block per (batch, query head, key block); the visited rows come
// from the main kernel's own unit decoding (BM: its query rows per step), so
// the two cover the tensor exactly once.  16-byte stores, 16 threads per
// 128-key row segment: the tensor must start on a 16-byte boundary and Sk be
// a multiple of 8 (the host zeroes the whole tensor otherwise).
template <int BM>
__global__ void __launch_bounds__(256) dbias_zero_kernel(BwdParams p) {
    const int nblk = (p.Sk + kBlockN - 1) / kBlockN;
    const int n = (int)(blockIdx.x % (unsigned)nblk);
    const int bh = (int)(blockIdx.x / (unsigned)nblk);   // b * Hq + query head
    const int b = bh / p.Hq, hq = bh - b * p.Hq;
    // the dense unit order: groups of unit_group (batch, kv head) pairs (a
    // divisor of B * Hkv), n-block-major inside a group
    const int pair = b * p.Hkv + hq / p.G, gs = p.unit_group;
    const Unit u = decode_unit<BM>(p, (pair / gs) * gs * nblk + n * gs + pair % gs);
    const int n0 = n * kBlockN, c_end = min(n0 + kBlockN, p.Sk);
    // rows [r0, r1) get dS from the main kernel in the keys [n0, ck)
    const int r0 = u.nm > 0 ? u.m_begin * BM : 0;
    const int r1 = u.nm > 0 ? max(r0, min((u.m_begin + u.nm) * BM, u.lq)) : 0;
    const int ck = min(max(u.lk, n0), c_end);
    uint16_t *base = reinterpret_cast<uint16_t *>(p.dbias) + (long long)bh * p.Sq * p.Sk;
    const int seg = threadIdx.x & 15, sub = threadIdx.x >> 4;   // 8 keys, one of 16 rows
    const int col = n0 + 8 * seg;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    // whole rows: [0, r0) and [r1, Sq)
    const int nfull = r0 + (p.Sq - r1);
    if (col < c_end) {
        for (int v = sub; v < nfull; v += 16) {
            const int row = v < r0 ? v : v - r0 + r1;
            *reinterpret_cast<uint4 *>(base + (long long)row * p.Sk + col) = z;
        }
    }
    // rows [r0, r1) past the used keys: [ck, c_end)
    if (ck < c_end) {
        for (int row = r0 + sub; row < r1; row += 16) {
            uint16_t *dst = base + (long long)row * p.Sk;
            if (col >= ck) {
                if (col < c_end) *reinterpret_cast<uint4 *>(dst + col) = z;
            } else if (col + 8 > ck) {
                for (int c = ck; c < col + 8; ++c) dst[c] = 0;
            }
        }
    }
}

}  // namespace

cudaError_t launch_dbias_zero(const BwdParams &p, int bm, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.Hq * ((p.Sk + kBlockN - 1) / kBlockN);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (bm == 64) dbias_zero_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else dbias_zero_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_schedule(const BwdParams &p, cudaStream_t stream) {
    schedule_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

static dim3 row_grid(const BwdParams &p, int lanes_per_row, int rows_per_seq, int rpt) {
    const long long threads = ((long long)rows_per_seq * p.Hq + rpt - 1) / rpt * lanes_per_row;
    return dim3((unsigned)((threads + 255) / 256), (unsigned)p.B, 1);
}

template <int DQ, int DV, typename T>
static void launch_pre_t(const BwdParams &p, cudaStream_t stream) {
    if (p.varlen)
        preprocess_kernel<DQ, DV, T, 4><<<row_grid(p, DV / 8, p.sq_round, 4), 256, 0, stream>>>(p);
    else
        preprocess_kernel<DQ, DV, T, 1><<<row_grid(p, DV / 8, p.sq_round, 1), 256, 0, stream>>>(p);
}
template <typename T>
static cudaError_t launch_pre_dt(const BwdParams &p, cudaStream_t stream) {
    // (accumulator, value) tile widths: one head dim of 64 or 128, or the
    // wide kernel's 128 / 256 on either side
    if (p.D == 64 && p.Dv == 64) launch_pre_t<64, 64, T>(p, stream);
    else if (p.D == 128 && p.Dv == 128) launch_pre_t<128, 128, T>(p, stream);
    else if (p.D == 256 && p.Dv == 256) launch_pre_t<256, 256, T>(p, stream);
    else if (p.D == 256 && p.Dv == 128) launch_pre_t<256, 128, T>(p, stream);
    else if (p.D == 128 && p.Dv == 256) launch_pre_t<128, 256, T>(p, stream);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}
template <int D, typename T>
static void launch_post_t(const BwdParams &p, cudaStream_t stream) {
    if (p.varlen)
        postprocess_kernel<D, T, 4><<<row_grid(p, D / 8, p.Sq, 4), 256, 0, stream>>>(p);
    else
        postprocess_kernel<D, T, 1><<<row_grid(p, D / 8, p.Sq, 1), 256, 0, stream>>>(p);
}

cudaError_t launch_preprocess(const BwdParams &p, int bf16, cudaStream_t stream) {
    return bf16 ? launch_pre_dt<__nv_bfloat16>(p, stream) : launch_pre_dt<__half>(p, stream);
}

cudaError_t launch_postprocess(const BwdParams &p, int bf16, cudaStream_t stream) {
    if (p.D == 256) {
        if (bf16) launch_post_t<256, __nv_bfloat16>(p, stream);
        else launch_post_t<256, __half>(p, stream);
    } else if (p.D == 128) {
        if (bf16) launch_post_t<128, __nv_bfloat16>(p, stream);
        else launch_post_t<128, __half>(p, stream);
    } else {
        if (bf16) launch_post_t<64, __nv_bfloat16>(p, stream);
        else launch_post_t<64, __half>(p, stream);
    }
    return cudaGetLastError();
}

}  // namespace fa
