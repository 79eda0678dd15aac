// fa_fwd_split.cu -- the forward pass (O and LSE, as in fa_fwd_tc.cu) with
// two softmax warps per query row, for the instances fwd_split() selects: the
// bias and dropout instances and every instance at D = 64.
//
// One CTA per (128-query tile, sequence, query head); per block of 128 keys
//   S = Q K^T           tcgen05 SS, M = 128 queries, N = 128 keys, fp32 in TMEM
//   P = exp2(S c log2e - m), row sums, P written back to TMEM as bf16/fp16 pairs
//   O += P V            tcgen05 TS (P from TMEM), N = D
// with the lazily raised running maximum of fa_fwd_tc.cu (O and the row sums
// rescaled only when a block's maximum exceeds m by more than 2^8).
//
// What differs from the one-warp-per-row kernel:
// * the two warps of a TMEM lane quarter (w and w + 4) take 64 keys of each
//   block apiece and exchange their partial row maxima once per block (and
//   their row sums at the end) through tensor memory, so both reach the same
//   running maximum; each rescales and stores half of the row's O;
// * K and V blocks go through rings of their own (a K slot is free once its
//   S is computed, a V slot once O += P V has read it);
// * without the bias or dropout (D = 64 plain and ALiBi) the scores stay in
//   registers and three S buffers fit tensor memory.
//
// Warps: 0 TMA producer, 1 MMA issuer, 4-11 softmax, 2-3 idle.
#include <type_traits>

#include "fa_device.cuh"
#include "fa_fwd_common.h"
#include "fa_params.h"

namespace fa {
namespace {

// One TMEM column: thread t of the warp writes / reads column col of lane
// (lane_base + t); the load waits for its own completion.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t tmem_ld1_wait(uint32_t taddr) {
    uint32_t v;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v)
        : "r"(taddr)
        : "memory");
    return v;
}

template <int kD, typename T>
struct SplitCfg {
    static constexpr int D = kD;
    static constexpr int BM = 128;                 // queries per CTA
    static constexpr int BN = 128;                 // keys per block
    static constexpr int kStages = (kD == 128) ? 3 : 4;   // slots of the K ring and of the V ring
    static constexpr int kThreads = 12 * 32;
    static constexpr int W_SM = 4;                 // first softmax warp (8 of them)
    // TMEM: NB S buffers (BN columns each; the P pairs of each half of the
    // keys overwrite the first half of that half's S) | O (D) | with two S
    // buffers, 4 columns where the two softmax warps of a row exchange their
    // maxima and sums (with three, the last S columns of each half serve)
    static constexpr int TM_S = 0;
    static constexpr int TM_COLS = 512;
    static constexpr int tm_o(int nb) { return nb * BN; }
    static constexpr int tm_x(int nb) { return nb * BN + D; }
    static_assert(tm_x(2) + 4 <= TM_COLS, "TMEM overflow");
    // shared memory
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + kStages * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + kStages * KV_BYTES;
    // barriers: Q | S full, P full, PV done (one per S buffer) | O final |
    // K full, K empty, V full, V empty (one per ring slot) | exchange (one per
    // lane quarter)
    static constexpr int s_full(int b) { return 1 + b; }
    static constexpr int p_full(int b) { return 4 + b; }
    static constexpr int pv_done(int b) { return 7 + b; }
    static constexpr int O_FINAL = 10;
    static constexpr int k_full(int st) { return 11 + st; }
    static constexpr int k_empty(int st) { return 11 + kStages + st; }
    static constexpr int v_full(int st) { return 11 + 2 * kStages + st; }
    static constexpr int v_empty(int st) { return 11 + 3 * kStages + st; }
    static constexpr int xch(int quarter) { return 11 + 4 * kStages + quarter; }
    static constexpr int NUM_BARS = 32;
    static_assert(11 + 4 * kStages + 4 <= NUM_BARS, "barrier slots");
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM slot, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;   // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
    // one CTA per SM: the CTA takes all 512 TMEM columns
    static_assert(2 * (SMEM_BYTES + 1024) > 233472, "two CTAs would share an SM");
    static constexpr uint32_t IDESC_S = make_idesc(128, BN, Cvt<T>::is_bf16, false, false);
    static constexpr uint32_t IDESC_PV = make_idesc(128, D, Cvt<T>::is_bf16, false, true);
};

constexpr int F_Q_FULL = 0;

// Lazy rescaling threshold (log2 units): P is taken against a running maximum
// that may lag the true one by up to this much.
constexpr float kRescaleLog2 = 8.f;

template <int kD, typename T, int kFlags>
__global__ void __launch_bounds__(SplitCfg<kD, T>::kThreads, 1)
    fwd_split_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap map_q,
                  const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  void *o_out, float *lse_out, int nmb) {
    using C = SplitCfg<kD, T>;
    constexpr int D = C::D, BM = C::BM, BN = C::BN, S = C::kStages;
    constexpr bool kAlibi = (kFlags & kFwdAlibi) != 0, kBias = (kFlags & kFwdBias) != 0,
                   kDrop = (kFlags & kFwdDrop) != 0;
    constexpr bool kExt = kAlibi || kBias;   // scores other than the plain scaled ones
    // Without the bias or dropout the softmax holds a block's scores in
    // registers, and three S buffers fit tensor memory (with D = 128 exactly):
    // S of block n + 2 is then issued before O += P V of block n, and the
    // chain softmax -> P V -> next S into the freed buffer spans three blocks
    // instead of two.
    constexpr bool kResident = !kBias && !kDrop;
    // two softmax warps per row, each taking HK keys of a block and DW columns of O
    constexpr int HK = BN / 2, DW = D / 2;
    static_assert(DW % 32 == 0, "a softmax warp rescales and stores whole 32-column chunks of O");
    constexpr int NB = (kResident && 3 * BN + D <= C::TM_COLS) ? 3 : 2;
    constexpr int TM_O = C::tm_o(NB);
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
        for (int i = 0; i < NB; ++i) {
            mbar_init(bar(C::s_full(i)), 1);
            mbar_init(bar(C::p_full(i)), 8);
            mbar_init(bar(C::pv_done(i)), 1);
        }
        mbar_init(bar(C::O_FINAL), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(C::k_full(s)), 1);
            mbar_init(bar(C::k_empty(s)), 1);
            mbar_init(bar(C::v_full(s)), 1);
            mbar_init(bar(C::v_empty(s)), 1);
        }
        for (int qq = 0; qq < 4; ++qq) mbar_init(bar(C::xch(qq)), 2);
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
        // K and V blocks go through rings of their own: K of block j is
        // needed when S of block j is issued (NB - 1 blocks ahead of O += P V
        // of block j) and its slot is free once that S completes; V of block j is needed by
        // and freed after O += P V of block j.  Loads follow the MMA order:
        // K of block j, then V of block j - (NB - 1).
        if (lane == 0 && nblk > 0) {
            mbar_arrive_expect_tx(bar(F_Q_FULL), C::Q_BYTES);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
                tma_load_4d(sbase + C::OFF_Q + hh * BM * 128, &map_q, bar(F_Q_FULL), hh * 64, h,
                            q0 + m * BM, bidx);
            uint32_t k_ph = 0, v_ph = 0;   // empty-barrier phase bit of each slot
            int k_armed = -1, v_armed = -1;  // the last block whose K / V load was issued
            auto load = [&](int j, bool is_k) -> bool {
                const int st = j % S;
                if (j >= S) {
                    uint32_t &ph = is_k ? k_ph : v_ph;
                    if (!mbar_wait(bar(is_k ? C::k_empty(st) : C::v_empty(st)), ph >> st & 1u, w))
                        return false;
                    ph ^= 1u << st;
                }
                const uint32_t full = bar(is_k ? C::k_full(st) : C::v_full(st));
                mbar_arrive_expect_tx(full, C::KV_BYTES);
                (is_k ? k_armed : v_armed) = j;
                const uint32_t dst = sbase + (is_k ? C::OFF_K : C::OFF_V) + st * C::KV_BYTES;
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh)
                    tma_load_4d(dst + hh * BN * 128, is_k ? &map_k : &map_v, full, hh * 64, hk,
                                k0 + (n_begin + j) * BN, bidx);
                return true;
            };
            for (int j = 0; j < nblk + NB - 1; ++j) {
                if (j < nblk && !load(j, true)) break;
                if (j >= NB - 1 && !load(j - (NB - 1), false)) break;
            }
            // wind-down: no K/V load may land after the CTA exits (after an
            // abort its consumers may not have waited for it).  The Q load needs
            // no wait here: it is issued first, and the MMA warp waits for it
            // with the whole budget before any wait can run out.
            for (int st = 0; st < S; ++st) {
                if (st <= k_armed) {
                    const int jl = k_armed - ((k_armed - st) % S);   // last K block in slot st
                    mbar_wait_drain(bar(C::k_full(st)), (uint32_t)(jl / S) & 1u, p.err, p.budget_ns);
                }
                if (st <= v_armed) {
                    const int jl = v_armed - ((v_armed - st) % S);
                    mbar_wait_drain(bar(C::v_full(st)), (uint32_t)(jl / S) & 1u, p.err, p.budget_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        // Order: S of blocks 0 .. NB-2, then per n: S of block n + NB - 1 (into
        // the buffer O += P V of block n - 1 has just read), O += P V of block n.
        if (nblk > 0) {
            bool ok = mbar_wait_warp(bar(F_Q_FULL), 0, w);
            uint32_t k_ph = 0, v_ph = 0;   // full-barrier phase bit of each slot
            const uint64_t dQ_k = sw128_desc(sbase + C::OFF_Q, 16, 1024);
            auto issue_s = [&](int j) -> bool {
                const int bb = j % NB, st = j % S;
                if (!mbar_wait_warp(bar(C::k_full(st)), k_ph >> st & 1u, w)) return false;
                k_ph ^= 1u << st;
                // S buffer bb last held P of block j - NB
                if (j >= NB && !mbar_wait_warp(bar(C::pv_done(bb)), (uint32_t)((j - NB) / NB) & 1u, w))
                    return false;
                tc_fence_after();
                const uint64_t dK_k = sw128_desc(sbase + C::OFF_K + st * C::KV_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
                    const uint32_t qo = (kk / 4) * (BM * 128) + (kk % 4) * 32;
                    mma_ss_warp(tmem + C::TM_S + bb * BN, desc_add(dQ_k, qo), desc_add(dK_k, ko),
                                C::IDESC_S, kk > 0);
                }
                mma_commit_warp(bar(C::s_full(bb)));
                mma_commit_warp(bar(C::k_empty(st)));
                return true;
            };
            auto issue_pv = [&](int n) -> bool {
                const int bb = n % NB, st = n % S;
                if (!mbar_wait_warp(bar(C::p_full(bb)), (uint32_t)(n / NB) & 1u, w)) return false;
                if (!mbar_wait_warp(bar(C::v_full(st)), v_ph >> st & 1u, w)) return false;
                v_ph ^= 1u << st;
                tc_fence_after();
                // O += P V: P (queries x keys) from TMEM, V (keys x d) MN-major,
                // K step = 16 keys = 2048 bytes of the swizzled tile; the pairs
                // of keys 16 kk .. 16 kk + 15 sit at column HK * part + 8 * (kk
                // within the part) of the S buffer
                const uint64_t dV_mn = sw128_desc(sbase + C::OFF_V + st * C::KV_BYTES, BN * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_warp(tmem + TM_O,
                                tmem + C::TM_S + bb * BN + HK * (16 * kk / HK) + 8 * kk % (HK / 2),
                                desc_add(dV_mn, kk * 2048), C::IDESC_PV, (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(bar(C::pv_done(bb)));
                mma_commit_warp(bar(C::v_empty(st)));
                return true;
            };
            for (int j = 0; ok && j < NB - 1 && j < nblk; ++j) ok = issue_s(j);
            for (int n = 0; ok && n < nblk; ++n) {
                if (n + NB - 1 < nblk && !(ok = issue_s(n + NB - 1))) break;
                ok = issue_pv(n);
            }
            if (ok) mma_commit_warp(bar(C::O_FINAL));
            // make sure no MMA is still running before tensor memory is freed
            mma_commit_warp(bar(F_Q_FULL));
            mbar_wait_drain_warp(bar(F_Q_FULL), 1, p.err, p.budget_ns);
        }
    } else if (warp >= C::W_SM) {
        // ------------------------------------------------------------- softmax
        // One query row per lane of a TMEM lane quarter, two warps per
        // quarter: warp half hf takes keys [HK hf, HK hf + HK) of every block
        // and O columns [DW hf, DW hf + DW).  The two exchange their partial
        // row maxima once per block (and their row sums at the end) through
        // tensor memory, so both take the same running maximum.
        const int quarter = warp & 3;
        const int hf = (warp - C::W_SM) >> 2;
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
        // elementwise bias row of this query (null: none, or a padding row)
        const T *brow = nullptr;
        if (kBias && p.bias && qi < lq)
            brow = reinterpret_cast<const T *>(p.bias) + (long long)b * p.bias_bs +
                   (long long)h * p.bias_hs + (long long)qi * p.bias_rs;
        // the bias of this half's HK keys k0 .. k0 + HK - 1 of a block as
        // packed pairs (0 past lk), fetched before the block's S is waited for
        // so the loads' latency hides behind it; 16-byte loads when all HK are
        // in range (k0 is a multiple of 64, the row start 16-byte aligned)
        auto fetch_bias = [&](uint32_t (&bw)[HK / 2], int k0) __attribute__((always_inline)) {
            if (brow && k0 + HK <= lk) {
#pragma unroll
                for (int t = 0; t < HK / 8; ++t) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(brow + k0) + t);
                    bw[4 * t] = v.x;
                    bw[4 * t + 1] = v.y;
                    bw[4 * t + 2] = v.z;
                    bw[4 * t + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < HK / 2; ++i) {
                    const float f0 = (brow && k0 + 2 * i < lk) ? static_cast<float>(brow[k0 + 2 * i]) : 0.f;
                    const float f1 =
                        (brow && k0 + 2 * i + 1 < lk) ? static_cast<float>(brow[k0 + 2 * i + 1]) : 0.f;
                    bw[i] = Cvt<T>::pack(f0, f1);
                }
            }
        };
        // bias of keys 32c .. 32c + 31 of the half in log2 units
        auto load_bias = [&](float (&bl)[32], const uint32_t (&bw)[HK / 2], int c) __attribute__((always_inline)) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float2 f = Cvt<T>::unpack(bw[16 * c + u]);
                bl[2 * u] = f.x * 1.4426950408889634f;
                bl[2 * u + 1] = f.y * 1.4426950408889634f;
            }
        };
        // Exchange of one value per row with the other warp of the quarter, at
        // phase k of the quarter's barrier: the maxima of block k (k < nblk),
        // then the row sums (k = nblk).  The value of half hf goes to column
        // xcol(k, hf): with three S buffers, the last S column of that half in
        // the buffer of block k (already read into registers; P and the next
        // S of the buffer come after both warps have read it), or the next to
        // last of the final block's buffer for the sums; with two, slot k % 2
        // of the exchange columns (a warp cannot reuse a slot before its
        // partner has read it: it would first have to pass the partner's next
        // arrival).
        const uint32_t xbar = bar(C::xch(quarter));
        auto xcol = [&](int k, int half) __attribute__((always_inline)) -> uint32_t {
            if (NB == 3) {
                const int blk = k < nblk ? k : nblk - 1;
                return (uint32_t)(C::TM_S + (blk % NB) * BN + HK * half + HK - (k < nblk ? 1 : 2));
            }
            return (uint32_t)(C::tm_x(2) + 2 * (k & 1) + half);
        };
        auto exchange = [&](float v, int k, float &other) __attribute__((always_inline)) -> bool {
            tmem_st1(lane_addr + xcol(k, hf), __float_as_uint(v));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar);
            if (!mbar_wait_warp(xbar, (uint32_t)k & 1u, w)) return false;
            tc_fence_after();
            other = __uint_as_float(tmem_ld1_wait(lane_addr + xcol(k, hf ^ 1)));
            return true;
        };
        float m_run = -INFINITY, l_run = 0.f;       // running max (log2 units), this half's row sum
        bool ok = true;
        for (int n = 0; n < nblk; ++n) {
            const int bb = n % NB;
            const int kh = (n_begin + n) * BN + HK * hf;   // first key of this warp's half
            // dropout keep flags of this row's HK keys (bit l of kw[c]: key
            // kh + 32c + l), drawn before S is ready (the wait hides them)
            uint32_t kw[HK / 32];
            if (kDrop) {
                const uint32_t tt4 = (uint32_t)p.drop_t * 0x01010101u;
#pragma unroll
                for (int g = 0; g < HK / 16; ++g) {
                    const uint4 R = philox4x32_10(make_uint4((uint32_t)(kh >> 4) + g, (uint32_t)qi,
                                                             (uint32_t)(b * p.Hq + h), p.drop_offset),
                                                  p.drop_key0, p.drop_key1);
                    const uint32_t wd[4] = {R.x, R.y, R.z, R.w};
                    uint32_t bits = 0u;
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        // bytes >= t -> 0xFF; the low bits of the 4 bytes gathered
                        // into bits 28-31 by one product
                        const uint32_t ge = __vcmpgeu4(wd[wi], tt4) & 0x01010101u;
                        bits |= ((ge * 0x10204080u) >> 28) << (4 * wi);
                    }
                    if (g & 1) kw[g >> 1] |= bits << 16;
                    else kw[g >> 1] = bits;
                }
                if (p.drop_mask && qi < lq) {
                    // the flags for the backward: word (kh + 32c) / 32 of this
                    // query row, for the words that hold a key below lk
                    const long long mrow = p.varlen ? (long long)h * p.cu_q[p.B] + q0 + qi
                                                    : ((long long)b * p.Hq + h) * p.Sq + qi;
                    uint32_t *mdst = p.drop_mask + mrow * p.drop_mask_w;
#pragma unroll
                    for (int c = 0; c < HK / 32; ++c) {
                        const int wi = (kh >> 5) + c;
                        if (kh + 32 * c < lk && wi < p.drop_mask_w) mdst[wi] = kw[c];
                    }
                }
            }
            uint32_t bw[kBias ? HK / 2 : 1];
            if constexpr (kBias) fetch_bias(bw, kh);
            if (!(ok = mbar_wait_warp(bar(C::s_full(bb)), (uint32_t)(n / NB) & 1u, w))) break;
            tc_fence_after();
            const uint32_t scol = lane_addr + C::TM_S + bb * BN + HK * hf;
            // element e of the half (key kh + e) is visible iff lo <= e <= hi
            const int lo = kmin - kh, hi = kmax - kh;
            // ALiBi: key kh + e lies (kh + e) - (qi + diag) = fbase + e from the diagonal
            const float fbase = (float)(kh - qi - diag);
            // scaled score of element e with its bias (bl: bias * log2e), log2 units
            auto score2 = [&](uint32_t raw, int e, float bl) __attribute__((always_inline)) -> float {
                float x = kBias ? bl : 0.f;
                if (kAlibi) x = fmaf(-slope2, fabsf(fbase + (float)e), x);
                return fmaf(__uint_as_float(raw), p.scale_log2, x);
            };
            // Halves inside every row's band (all but the edge blocks) take the
            // passes without per-element tests.
            const bool edge = __any_sync(0xffffffffu, lo > 0 || hi < HK - 1);
            // the row's HK scores: without the bias or dropout, held in
            // registers (one round trip to tensor memory per block); with them
            // (more registers live), loaded chunk by chunk in each pass
            uint32_t srr[kResident ? HK / 32 : 1][32];
            if (kResident) {
#pragma unroll
                for (int c = 0; c < HK / 32; ++c) tmem_ld32(scol + 32 * c, srr[kResident ? c : 0]);
                tmem_wait_ld();
            }
            auto chunk = [&](int c, uint32_t (&dst)[32]) __attribute__((always_inline)) {
                if (kResident) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[i] = srr[kResident ? c : 0][i];
                } else {
                    tmem_ld32(scol + 32 * c, dst);
                    tmem_wait_ld();
                }
            };
            // pass 1: maximum of the half (without ALiBi or bias the maximum of
            // the raw scores, scaled once: the scale is positive), in eight
            // independent chains
            auto half_max = [&](auto mask_tag) __attribute__((always_inline)) -> float {
                constexpr bool kMask = decltype(mask_tag)::value;
                float mxv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxv[i] = -INFINITY;
#pragma unroll
                for (int c = 0; c < HK / 32; ++c) {
                    uint32_t sr[32];
                    chunk(c, sr);
                    float bl[32];
                    if constexpr (kBias) load_bias(bl, bw, c);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = 32 * c + i;
                        const float x = kExt ? score2(sr[i], e, bl[i]) : __uint_as_float(sr[i]);
                        mxv[i & 7] = (!kMask || (e >= lo && e <= hi)) ? fmaxf(mxv[i & 7], x) : mxv[i & 7];
                    }
                }
                const float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                                       fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
                return kExt ? mx : mx * p.scale_log2;
            };
            float mx = edge ? half_max(std::true_type{}) : half_max(std::false_type{});
            float mx_other;
            if (!(ok = exchange(mx, n, mx_other))) break;
            mx = fmaxf(mx, mx_other);   // both warps of the row reach the same running maximum
            const float m_new = fmaxf(m_run, mx);
            const float m_use = (m_run == -INFINITY || m_new > m_run + kRescaleLog2) ? m_new : m_run;
            const float alpha = (m_use == m_run) ? 1.f : ex2(m_run - m_use);
            const float mref = (m_use == -INFINITY) ? 0.f : m_use;
            float sumv[4] = {0.f, 0.f, 0.f, 0.f};   // row sum in four independent chains
            // pass 2: P = exp2(s2 - m) as pairs into the first HK/2 columns of
            // the half; column j/2 holds keys j, j+1 (with the scores read
            // chunk by chunk, each S column is read before a P pair lands on it)
            auto half_p = [&](auto mask_tag) __attribute__((always_inline)) {
                constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
                for (int c = 0; c < HK / 32; ++c) {
                    uint32_t sr[32];
                    chunk(c, sr);
                    float bl[32];
                    if constexpr (kBias) load_bias(bl, bw, c);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * c + 2 * i;
                        float p0, p1;
                        if (kExt) {
                            p0 = ex2(score2(sr[2 * i], e, bl[2 * i]) - mref);
                            p1 = ex2(score2(sr[2 * i + 1], e + 1, bl[2 * i + 1]) - mref);
                        } else {
                            p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), p.scale_log2, -mref));
                            p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), p.scale_log2, -mref));
                        }
                        if (kMask) {
                            p0 = (e >= lo && e <= hi) ? p0 : 0.f;
                            p1 = (e + 1 >= lo && e + 1 <= hi) ? p1 : 0.f;
                        }
                        sumv[i & 3] += p0 + p1;   // the row sum is taken before dropout
                        if (kDrop) {   // keys 2i, 2i + 1 of the chunk
                            p0 = ((kw[c] >> (2 * i)) & 1u) ? p0 * p.drop_scale : 0.f;
                            p1 = ((kw[c] >> (2 * i + 1)) & 1u) ? p1 * p.drop_scale : 0.f;
                        }
                        pk[i] = Cvt<T>::pack(p0, p1);
                    }
                    tmem_st16(scol + 16 * c, pk);
                }
            };
            if (edge) half_p(std::true_type{});
            else half_p(std::false_type{});
            l_run = l_run * alpha + ((sumv[0] + sumv[1]) + (sumv[2] + sumv[3]));
            m_run = m_use;
            // O holds blocks < n: rescale this warp's columns when a row's maximum moved
            if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                if (!(ok = mbar_wait_warp(bar(C::pv_done((n - 1) % NB)), (uint32_t)((n - 1) / NB) & 1u, w)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < DW / 32; ++c) {
                    const uint32_t ocol = lane_addr + TM_O + DW * hf + 32 * c;
                    uint32_t orr[32];
                    tmem_ld32(ocol, orr);
                    tmem_wait_ld();
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        lo[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                        hi[i] = __float_as_uint(__uint_as_float(orr[16 + i]) * alpha);
                    }
                    tmem_st16(ocol, lo);
                    tmem_st16(ocol + 16, hi);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::p_full(bb)));
        }
        // ---------------------------------------------------------- epilogue
        // O = acc / l, LSE = (m + log2 l) ln 2 with l the two halves' sums; a
        // row that sees no key gets O = 0 and LSE = -inf
        if (ok && nblk > 0) {
            float l_other = 0.f;
            ok = exchange(l_run, nblk, l_other);
            l_run += l_other;
            if (ok) ok = mbar_wait_warp(bar(C::O_FINAL), 0, w);
            tc_fence_after();
        }
        if (ok) {
            const bool live = qi < lq;
            const long long row = p.varlen ? (long long)q0 + qi : (long long)b * p.Sq + qi;
            if (live && hf == 0) {
                float *lse_dst = p.varlen ? lse_out + (long long)h * p.cu_q[p.B] + q0 + qi
                                          : lse_out + ((long long)b * p.Hq + h) * p.Sq + qi;
                *lse_dst = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            // this warp's DW columns; Dh <= D columns are stored
            T *dst = reinterpret_cast<T *>(o_out) + (row * p.Hq + h) * p.Dh + DW * hf;
            const int dh_left = p.Dh - DW * hf;
#pragma unroll
            for (int c = 0; c < DW / 32; ++c) {
                uint32_t orr[32];
                if (nblk > 0) {
                    tmem_ld32(lane_addr + TM_O + DW * hf + 32 * c, orr);
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
                        if (32 * c + 8 * i < dh_left)
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

template <int kD, typename T, int kFlags>
cudaError_t launch_split_t(const BwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                           const CUtensorMap &mv, void *o, float *lse, int max_lq, cudaStream_t stream) {
    using C = SplitCfg<kD, T>;
    auto kern = fwd_split_kernel<kD, T, kFlags>;
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

// the instance with exactly these flags, if it is a two-warps-per-row one
template <int kD, typename T, int kI = 0>
cudaError_t launch_split_flags(const BwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                               const CUtensorMap &mv, void *o, float *lse, int max_lq, int flags,
                               cudaStream_t stream) {
    constexpr int f = kFwdFlagSets[kI];
    if (flags == f) {
        if constexpr (fwd_split(kD, f))
            return launch_split_t<kD, T, f>(p, mq, mk, mv, o, lse, max_lq, stream);
        else
            return cudaErrorInvalidValue;
    }
    if constexpr (kI + 1 < kNumFwdFlagSets)
        return launch_split_flags<kD, T, kI + 1>(p, mq, mk, mv, o, lse, max_lq, flags, stream);
    else
        return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_fwd_split(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                             const CUtensorMap &v, void *o, float *lse, int max_lq, int bf16,
                             int flags, cudaStream_t stream) {
    if (p.D == 128)
        return bf16 ? launch_split_flags<128, __nv_bfloat16>(p, q, k, v, o, lse, max_lq, flags, stream)
                    : launch_split_flags<128, __half>(p, q, k, v, o, lse, max_lq, flags, stream);
    return bf16 ? launch_split_flags<64, __nv_bfloat16>(p, q, k, v, o, lse, max_lq, flags, stream)
                : launch_split_flags<64, __half>(p, q, k, v, o, lse, max_lq, flags, stream);
}

}  // namespace fa
