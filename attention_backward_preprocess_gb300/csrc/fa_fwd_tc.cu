// fa_fwd_tc.cu -- forward pass O = softmax(Q K^T * c + mask) V and the
// per-row log-sum-exp LSE, on the 5th-generation tensor cores.  It supplies
// the O and LSE the backward pass consumes (same layouts, same bottom-right
// causal mask, -inf LSE / zero O for a query row that sees no key).
//
// One CTA per (128-query tile, sequence, query head); the tiles of the longest
// causal rows are launched first.  Per block of 128 keys:
//   S = Q K^T           tcgen05 SS, M = 128 queries, N = 128 keys, fp32 in TMEM
//   P = exp2(S c log2e - m), row sums, P written back to TMEM as bf16/fp16 pairs
//   O += P V            tcgen05 TS (P from TMEM), N = D
// S is double buffered, so S of block n+1 runs while the softmax warps turn
// block n into P, and O += P V of block n-1 runs meanwhile too.  The running
// row maximum m is raised only when a block's maximum exceeds it by more than
// 2^8 (then O and the row sum are rescaled); otherwise P is taken against the
// older, smaller m, which keeps P <= 2^8 and the result exact up to rounding.
// The epilogue divides O by the row sum and writes O and LSE = (m + log2 l) ln 2.
//
// Warps: 0 TMA producer (Q once, K/V blocks through a stage ring), 1 MMA
// issuer, 4-7 softmax (thread = query row of its TMEM lane quarter), 2-3 idle.
//
// This kernel serves the instances with one softmax warp per query row (D =
// 128 without the bias or dropout); the others run in fa_fwd_split.cu.
#include <type_traits>

#include "fa_device.cuh"
#include "fa_fwd_common.h"
#include "fa_params.h"

namespace fa {
namespace {

// kDQ / kDV: tile widths of the query / key side and of the value side (128
// or 256; 128 and 128 for one head dim of at most 128), kBN keys per block
// (128; 64 when a side is 256 wide, so that the K / V ring still has two or
// three slots next to the 64 KB Q tile).
template <int kDQ, int kDV, int kBN, typename T>
struct FwdCfg {
    static constexpr int DQ = kDQ, DV = kDV;
    static constexpr int BM = 128;                 // queries per CTA
    static constexpr int BN = kBN;                 // keys per block
    static constexpr int kThreads = 8 * 32;
    static constexpr int W_SM = 4;                 // first softmax warp
    // TMEM: S buffer x2 (BN columns each; P overwrites the first BN/2) | O (DV)
    static constexpr int TM_S = 0;
    static constexpr int TM_O = 2 * BN;
    static constexpr int TM_COLS = 512;
    static_assert(TM_O + DV <= TM_COLS, "TMEM overflow");
    // shared memory
    static constexpr int Q_BYTES = BM * DQ * 2;
    static constexpr int K_BYTES = BN * DQ * 2;
    static constexpr int V_BYTES = BN * DV * 2;
    // ring slots: as many as fit next to the barriers, the misc words and the
    // alignment slack, at most four
    static constexpr int kFixed = 16 * 8 + 32 + 1024;
    static constexpr int kStages = (Q_BYTES + 4 * (K_BYTES + V_BYTES) + kFixed <= 232448) ? 4
                                   : (Q_BYTES + 3 * (K_BYTES + V_BYTES) + kFixed <= 232448) ? 3 : 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + kStages * K_BYTES;
    static constexpr int OFF_BAR = OFF_V + kStages * V_BYTES;
    static constexpr int NUM_BARS = 16;
    static constexpr int kv_empty(int st) { return 8 + kStages + st; }
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM slot, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;   // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
    static_assert(8 + 2 * kStages <= NUM_BARS, "barrier slots");
    // one CTA per SM: the CTA takes all 512 TMEM columns
    static_assert(2 * (SMEM_BYTES + 1024) > 233472, "two CTAs would share an SM");
    static constexpr uint32_t IDESC_S = make_idesc(128, BN, Cvt<T>::is_bf16, false, false);
    static constexpr uint32_t IDESC_PV = make_idesc(128, DV, Cvt<T>::is_bf16, false, true);
};

enum {
    F_Q_FULL = 0,
    F_S_FULL = 1,     // +b: S of the block in S buffer b complete
    F_P_FULL = 3,     // +b: P written back (and O rescaled) by the 4 softmax warps
    F_PV_DONE = 5,    // +b: O += P V of the block in S buffer b complete
    F_O_FINAL = 7,
    F_KV_FULL = 8,    // +stage; the KV_EMPTY barriers follow them (kv_empty)
};

// Lazy rescaling threshold (log2 units): P is taken against a running maximum
// that may lag the true one by up to this much.
constexpr float kRescaleLog2 = 8.f;

template <int kDQ, int kDV, int kBN, typename T, int kFlags>
__global__ void __launch_bounds__(FwdCfg<kDQ, kDV, kBN, T>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap map_q,
                  const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  void *o_out, float *lse_out, int nmb) {
    using C = FwdCfg<kDQ, kDV, kBN, T>;
    constexpr int DQ = C::DQ, DV = C::DV, BM = C::BM, BN = C::BN, S = C::kStages;
    static_assert((kFlags & (kFwdBias | kFwdDrop)) == 0,
                  "the bias and dropout instances run in fa_fwd_split.cu");
    constexpr bool kAlibi = (kFlags & kFwdAlibi) != 0;
    constexpr bool kExt = kAlibi;   // scores other than the plain scaled ones
    // ---- tile of this CTA: longest causal rows first
    const int bh = blockIdx.x % (p.B * p.Hq);
    const int m = nmb - 1 - blockIdx.x / (p.B * p.Hq);
    const int b = bh / p.Hq, h = bh - b * p.Hq, hk = h / p.G;
    // varlen lengths outside the planned maps: the sequence is left alone and
    // the call reports the error (uniform: the whole CTA leaves)
    if (p.varlen && !varlen_seq_ok(p, b)) {
        if (threadIdx.x == 0 && h == 0 && m == nmb - 1) atomicOr(p.err, kErrBadLength);
        return;
    }
    const int q0 = p.varlen ? p.cu_q[b] : 0, k0 = p.varlen ? p.cu_k[b] : 0;
    const int lq = used_len_q(p, b), lk = used_len_k(p, b);
    if (m * BM >= lq) return;                       // uniform: the whole CTA leaves
    // key j is visible to query i iff -win_lo <= j - i - diag <= win_hi, j < lk
    const int diag = lk - lq;
    const long long first_key = max(0LL, (long long)m * BM + diag - p.win_lo);
    const long long last_key = min((long long)lk - 1, (long long)m * BM + BM - 1 + diag + p.win_hi);
    // key blocks [n_begin, n_begin + nblk) hold every key some row of the tile sees
    const int n_begin = (int)(first_key / BN);
    const int nblk = last_key < first_key ? 0 : (int)(last_key / BN) + 1 - n_begin;
    const int bidx = p.varlen ? 0 : b;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 16);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar(F_Q_FULL), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(F_S_FULL + i), 1);
            mbar_init(bar(F_P_FULL + i), 4);
            mbar_init(bar(F_PV_DONE + i), 1);
        }
        mbar_init(bar(F_O_FINAL), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(F_KV_FULL + s), 1);
            mbar_init(bar(C::kv_empty(s)), 1);
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_q);
        prefetch_tmap(&map_k);
        prefetch_tmap(&map_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl w{abort_flag, p.err, p.budget_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && nblk > 0) {
            mbar_arrive_expect_tx(bar(F_Q_FULL), C::Q_BYTES);
#pragma unroll
            for (int hh = 0; hh < DQ / 64; ++hh)
                tma_load_4d(sbase + C::OFF_Q + hh * BM * 128, &map_q, bar(F_Q_FULL), hh * 64, h,
                            q0 + m * BM, bidx);
            uint32_t empty_ph = 0;
            int armed = -1;   // the last block whose K/V load was issued
            for (int n = 0; n < nblk; ++n) {
                const int st = n % S;
                if (n >= S) {
                    if (!mbar_wait(bar(C::kv_empty(st)), empty_ph >> st & 1u, w)) break;
                    empty_ph ^= 1u << st;
                }
                const uint32_t full = bar(F_KV_FULL + st);
                mbar_arrive_expect_tx(full, C::K_BYTES + C::V_BYTES);
                armed = n;
#pragma unroll
                for (int hh = 0; hh < DQ / 64; ++hh)
                    tma_load_4d(sbase + C::OFF_K + st * C::K_BYTES + hh * BN * 128, &map_k, full,
                                hh * 64, hk, k0 + (n_begin + n) * BN, bidx);
#pragma unroll
                for (int hh = 0; hh < DV / 64; ++hh)
                    tma_load_4d(sbase + C::OFF_V + st * C::V_BYTES + hh * BN * 128, &map_v, full,
                                hh * 64, hk, k0 + (n_begin + n) * BN, bidx);
            }
            // wind-down: no K/V load may land after the CTA exits (after an
            // abort its consumers may not have waited for it).  The Q load needs
            // no wait here: it is issued first, and the MMA warp waits for it
            // with the whole budget before any wait can run out.
            for (int st = 0; st < S && st <= armed; ++st) {
                const int nl = armed - ((armed - st) % S);   // last block loaded into slot st
                mbar_wait_drain(bar(F_KV_FULL + st), (uint32_t)(nl / S) & 1u, p.err, p.budget_ns);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        // S of block n is issued before O += P V of block n-1, so it runs while
        // the softmax warps work on block n-1 (n counts the tile's blocks from 0).
        if (nblk > 0) {
            bool ok = mbar_wait_warp(bar(F_Q_FULL), 0, w);
            uint32_t full_ph = 0;
            const uint64_t dQ_k = sw128_desc(sbase + C::OFF_Q, 16, 1024);
            auto issue_pv = [&](int n) -> bool {
                const int bb = n & 1, st = n % S;
                if (!mbar_wait_warp(bar(F_P_FULL + bb), (uint32_t)(n >> 1) & 1u, w)) return false;
                tc_fence_after();
                // O += P V: P (queries x keys) from TMEM, V (keys x d) MN-major,
                // K step = 16 keys = 2048 bytes of the swizzled tile
                const uint64_t dV_mn = sw128_desc(sbase + C::OFF_V + st * C::V_BYTES, BN * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_warp(tmem + C::TM_O, tmem + C::TM_S + bb * BN + 8 * kk,
                                desc_add(dV_mn, kk * 2048), C::IDESC_PV, (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(bar(F_PV_DONE + bb));
                mma_commit_warp(bar(C::kv_empty(st)));
                return true;
            };
            for (int n = 0; ok && n < nblk; ++n) {
                const int bb = n & 1, st = n % S;
                if (!(ok = mbar_wait_warp(bar(F_KV_FULL + st), full_ph >> st & 1u, w))) break;
                full_ph ^= 1u << st;
                // S buffer bb last held P of block n-2
                if (n >= 2 && !(ok = mbar_wait_warp(bar(F_PV_DONE + bb), (uint32_t)((n - 2) >> 1) & 1u, w)))
                    break;
                tc_fence_after();
                const uint64_t dK_k = sw128_desc(sbase + C::OFF_K + st * C::K_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DQ / 16; ++kk) {
                    const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
                    const uint32_t qo = (kk / 4) * (BM * 128) + (kk % 4) * 32;
                    mma_ss_warp(tmem + C::TM_S + bb * BN, desc_add(dQ_k, qo), desc_add(dK_k, ko),
                                C::IDESC_S, kk > 0);
                }
                mma_commit_warp(bar(F_S_FULL + bb));
                if (n >= 1 && !(ok = issue_pv(n - 1))) break;
            }
            if (ok && issue_pv(nblk - 1)) mma_commit_warp(bar(F_O_FINAL));
            // make sure no MMA is still running before tensor memory is freed
            mma_commit_warp(bar(F_Q_FULL));
            mbar_wait_drain_warp(bar(F_Q_FULL), 1, p.err, p.budget_ns);
        }
    } else if (warp >= C::W_SM) {
        // ------------------------------------------------------------- softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;          // query row of the tile
        const int qi = m * BM + r;                  // query index within the sequence
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        // keys [kmin, kmax] are visible to this row (none if kmax < kmin)
        const int kmin = (int)max(0LL, (long long)qi + diag - p.win_lo);
        const int kmax = (int)min((long long)lk - 1, (long long)qi + diag + p.win_hi);
        // ALiBi slope of this head, log2 units
        const float slope2 = (kAlibi && p.alibi)
                                 ? __ldg(p.alibi + (long long)b * p.alibi_bstride + h) * 1.4426950408889634f
                                 : 0.f;
        // ALiBi in raw-score units, and whether it is linear over every
        // visible key (no key right of the diagonal)
        const float slope_u = slope2 / p.scale_log2;
        const bool lin = p.win_hi <= 0;
        float m_run = -INFINITY, l_run = 0.f;       // running max (log2 units), row sum
        bool ok = true;
        for (int n = 0; n < nblk; ++n) {
            const int bb = n & 1;
            const int kb = (n_begin + n) * BN;
            if (!(ok = mbar_wait_warp(bar(F_S_FULL + bb), (uint32_t)(n >> 1) & 1u, w))) break;
            tc_fence_after();
            const uint32_t scol = lane_addr + C::TM_S + bb * BN;
            // element e of the block (key kb + e) is visible iff lo <= e <= hi
            const int lo = kmin - kb, hi = kmax - kb;
            // ALiBi: key kb + e lies (kb + e) - (qi + diag) = fbase + e from the diagonal
            const float fbase = (float)(kb - qi - diag);
            // scaled score of element e with its ALiBi term, log2 units
            auto score2 = [&](uint32_t raw, int e) __attribute__((always_inline)) -> float {
                const float x = fmaf(-slope2, fabsf(fbase + (float)e), 0.f);
                return fmaf(__uint_as_float(raw), p.scale_log2, x);
            };
            // Blocks inside every row's band (all but the edge blocks) take the
            // pass without per-element tests.
            const bool edge = __any_sync(0xffffffffu, lo > 0 || hi < BN - 1);
            float alpha = 1.f, sum = 0.f, m_use = m_run;
            float sumv[4] = {0.f, 0.f, 0.f, 0.f};   // row sum in four independent chains
            // kLin: ALiBi with no visible key right of the diagonal (win_hi <= 0,
            // e.g. causal), where -slope |fbase + e| = slope (fbase + e) is linear
            // in e: pass 1 takes the maximum of raw + (slope / scale) e (one FMA
            // per score, scaled once), pass 2 adds slope e to a per-block
            // constant (two FMAs per score instead of an add, an abs-FMA and an
            // FMA, and one subtraction fewer)
            auto block_pass = [&](auto mask_tag, auto lin_tag) __attribute__((always_inline)) {
                constexpr bool kMask = decltype(mask_tag)::value;
                constexpr bool kLin = decltype(lin_tag)::value;
                // the row's 128 scores, held in registers: four loads in
                // flight and one wait, one round trip to tensor memory per
                // block instead of eight (the softmax is latency bound)
                uint32_t srr[BN / 32][32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(scol + 32 * c, srr[c]);
                tmem_wait_ld();
                auto chunk = [&](int c, uint32_t (&dst)[32]) __attribute__((always_inline)) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[i] = srr[c][i];
                };
                // pass 1: row maximum of the block (without ALiBi the maximum of
                // the raw scores, scaled once: the scale is positive), in eight
                // independent chains
                float mxv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxv[i] = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t sr[32];
                    chunk(c, sr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = 32 * c + i;
                        const float x = kLin   ? fmaf(slope_u, (float)e, __uint_as_float(sr[i]))
                                        : kExt ? score2(sr[i], e)
                                               : __uint_as_float(sr[i]);
                        mxv[i & 7] = (!kMask || (e >= lo && e <= hi)) ? fmaxf(mxv[i & 7], x) : mxv[i & 7];
                    }
                }
                float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                                 fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
                if (!kExt || kLin) mx *= p.scale_log2;
                if (kLin) mx += slope2 * fbase;
                const float m_new = fmaxf(m_run, mx);
                m_use = (m_run == -INFINITY || m_new > m_run + kRescaleLog2) ? m_new : m_run;
                alpha = (m_use == m_run) ? 1.f : ex2(m_run - m_use);
                const float mref = (m_use == -INFINITY) ? 0.f : m_use;
                const float cl = kLin ? fmaf(slope2, fbase, -mref) : 0.f;
                // pass 2: P = exp2(s2 - m) into the first BN/2 columns as pairs;
                // column j/2 of the buffer holds keys j, j+1 (with the scores
                // read chunk by chunk, each S column is read before a P pair
                // lands on it)
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t sr[32];
                    chunk(c, sr);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * c + 2 * i;
                        float p0, p1;
                        if (kLin) {
                            p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), p.scale_log2, fmaf(slope2, (float)e, cl)));
                            p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), p.scale_log2,
                                          fmaf(slope2, (float)(e + 1), cl)));
                        } else if (kExt) {
                            p0 = ex2(score2(sr[2 * i], e) - mref);
                            p1 = ex2(score2(sr[2 * i + 1], e + 1) - mref);
                        } else {
                            p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), p.scale_log2, -mref));
                            p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), p.scale_log2, -mref));
                        }
                        if (kMask) {
                            p0 = (e >= lo && e <= hi) ? p0 : 0.f;
                            p1 = (e + 1 >= lo && e + 1 <= hi) ? p1 : 0.f;
                        }
                        sumv[i & 3] += p0 + p1;
                        pk[i] = Cvt<T>::pack(p0, p1);
                    }
                    tmem_st16(scol + 16 * c, pk);
                }
            };
            auto run = [&](auto mask_tag) __attribute__((always_inline)) {
                if constexpr (kAlibi) {
                    if (lin) block_pass(mask_tag, std::true_type{});
                    else block_pass(mask_tag, std::false_type{});
                } else {
                    block_pass(mask_tag, std::false_type{});
                }
            };
            if (edge) run(std::true_type{});
            else run(std::false_type{});
            sum = (sumv[0] + sumv[1]) + (sumv[2] + sumv[3]);
            l_run = l_run * alpha + sum;
            m_run = m_use;
            // O holds blocks < n: rescale it when a row's maximum moved
            if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                if (!(ok = mbar_wait_warp(bar(F_PV_DONE + ((n - 1) & 1)), (uint32_t)((n - 1) >> 1) & 1u, w)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(lane_addr + C::TM_O + 32 * c, orr);
                    tmem_wait_ld();
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        lo[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                        hi[i] = __float_as_uint(__uint_as_float(orr[16 + i]) * alpha);
                    }
                    tmem_st16(lane_addr + C::TM_O + 32 * c, lo);
                    tmem_st16(lane_addr + C::TM_O + 32 * c + 16, hi);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(F_P_FULL + bb));
        }
        // ---------------------------------------------------------- epilogue
        // O = acc / l, LSE = (m + log2 l) ln 2; a row that sees no key gets
        // O = 0 and LSE = -inf
        if (ok && nblk > 0) {
            ok = mbar_wait_warp(bar(F_O_FINAL), 0, w);
            tc_fence_after();
        }
        if (ok) {
            const bool live = qi < lq;
            const long long row = p.varlen ? (long long)q0 + qi : (long long)b * p.Sq + qi;
            if (live) {
                float *lse_dst = p.varlen ? lse_out + (long long)h * p.cu_q[p.B] + q0 + qi
                                          : lse_out + ((long long)b * p.Hq + h) * p.Sq + qi;
                *lse_dst = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            T *dst = reinterpret_cast<T *>(o_out) + (row * p.Hq + h) * p.Dhv;   // Dhv <= DV columns
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) {
                uint32_t orr[32];
                if (nblk > 0) {
                    tmem_ld32(lane_addr + C::TM_O + 32 * c, orr);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) orr[i] = 0u;
                }
                if (live) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = Cvt<T>::pack(__uint_as_float(orr[2 * i]) * inv,
                                             __uint_as_float(orr[2 * i + 1]) * inv);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (32 * c + 8 * i < p.Dhv)
                            reinterpret_cast<uint4 *>(dst + 32 * c)[i] =
                                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

using FwdKernel = void (*)(BwdParams, CUtensorMap, CUtensorMap, CUtensorMap, void *, float *, int);

template <int kD, typename T, int kI = 0>
FwdKernel fwd_kernel_for(int need) {
    // the first instance built that has every flag needed (null: it is one of
    // fa_fwd_split.cu's)
    constexpr int f = kFwdFlagSets[kI];
    if constexpr (kI + 1 < kNumFwdFlagSets) {
        if ((need & f) != need) return fwd_kernel_for<kD, T, kI + 1>(need);
    }
    if constexpr (fwd_split(kD, f))
        return nullptr;
    else
        return fwd_tc_kernel<kD, kD, 128, T, f>;
}

template <int kDQ, int kDV, int kBN, typename T>
cudaError_t launch_fwd_cfg(FwdKernel kern, const BwdParams &p, const CUtensorMap &mq,
                           const CUtensorMap &mk, const CUtensorMap &mv, void *o, float *lse,
                           int max_lq, cudaStream_t stream) {
    using C = FwdCfg<kDQ, kDV, kBN, T>;
    if (kern == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int nmb = (max_lq + C::BM - 1) / C::BM;
    const long long grid = (long long)nmb * p.B * p.Hq;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, C::kThreads, C::SMEM_BYTES, stream>>>(p, mq, mk, mv, o, lse, nmb);
    return cudaGetLastError();
}

template <int kD, typename T>
cudaError_t launch_fwd_tc_t(const BwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                            const CUtensorMap &mv, void *o, float *lse, int max_lq, int need,
                            cudaStream_t stream) {
    return launch_fwd_cfg<kD, kD, 128, T>(fwd_kernel_for<kD, T>(need), p, mq, mk, mv, o, lse,
                                          max_lq, stream);
}

// Wide or unequal head dims (plain mask only): 64 keys per block when a side
// is 256 wide, else the 128-key block of the plain D = 128 instance.
template <typename T>
cudaError_t launch_fwd_wide_t(const BwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                              const CUtensorMap &mv, void *o, float *lse, int max_lq,
                              cudaStream_t stream) {
    if (p.D == 256 && p.Dv == 256)
        return launch_fwd_cfg<256, 256, 64, T>(fwd_tc_kernel<256, 256, 64, T, 0>, p, mq, mk, mv, o, lse,
                                               max_lq, stream);
    if (p.D == 256 && p.Dv == 128)
        return launch_fwd_cfg<256, 128, 64, T>(fwd_tc_kernel<256, 128, 64, T, 0>, p, mq, mk, mv, o, lse,
                                               max_lq, stream);
    if (p.D == 128 && p.Dv == 256)
        return launch_fwd_cfg<128, 256, 64, T>(fwd_tc_kernel<128, 256, 64, T, 0>, p, mq, mk, mv, o, lse,
                                               max_lq, stream);
    if (p.D == 128 && p.Dv == 128)
        return launch_fwd_cfg<128, 128, 128, T>(fwd_tc_kernel<128, 128, 128, T, 0>, p, mq, mk, mv, o,
                                                lse, max_lq, stream);
    return cudaErrorInvalidValue;
}

// Error word of the forward pass (its bounded waits record timeouts here).
__device__ int g_fwd_err;

}  // namespace

int *fwd_error_word() {
    void *ptr = nullptr;
    return cudaGetSymbolAddress(&ptr, g_fwd_err) == cudaSuccess ? static_cast<int *>(ptr) : nullptr;
}

// Query rows of one TMA box for Q in the forward pass, and key rows of one box
// for K / V (tile widths of the two sides).
int fwd_block_m() { return FwdCfg<128, 128, 128, __nv_bfloat16>::BM; }
int fwd_block_n(int Dq_tile, int Dv_tile) { return (Dq_tile > 128 || Dv_tile > 128) ? 64 : 128; }

cudaError_t launch_fwd_tc(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                          const CUtensorMap &v, void *o, float *lse, int max_lq, int bf16,
                          cudaStream_t stream) {
    if (p.D != p.Dv || p.D > 128 || p.Dh != p.Dhv)   // wide or unequal head dims
        return bf16 ? launch_fwd_wide_t<__nv_bfloat16>(p, q, k, v, o, lse, max_lq, stream)
                    : launch_fwd_wide_t<__half>(p, q, k, v, o, lse, max_lq, stream);
    const int need = (p.alibi ? kFwdAlibi : 0) | (p.bias ? kFwdBias : 0) | (p.drop_t > 0 ? kFwdDrop : 0);
    const int f = fwd_instance_flags(need);
    if (fwd_split(p.D, f)) return launch_fwd_split(p, q, k, v, o, lse, max_lq, bf16, f, stream);
    if (p.D != 128) return cudaErrorInvalidValue;
    return bf16 ? launch_fwd_tc_t<128, __nv_bfloat16>(p, q, k, v, o, lse, max_lq, need, stream)
                : launch_fwd_tc_t<128, __half>(p, q, k, v, o, lse, max_lq, need, stream);
}

}  // namespace fa
