// fa_bwd_wide.cu -- the attention-backward main kernel for wide or unequal
// head dims: a query / key dim Dqk and a value dim Dv of up to 256 each, equal
// or not (the Composable Kernel page "block_fmha_bwd_dq_dk_dv_pipeline_trload_
// kr_ktr_vr.hpp" carries the two as kQKHeaddim and kVHeaddim in its problem
// traits).  It computes what the main kernel computes (STAGE 1-7 of that
// page), with the tiling changed so that 256-wide tiles fit one SM:
//
// * A work unit is (sequence b, K/V block of 128 keys, kv head hk, column half
//   c).  The half selects which 128 columns of dK, dQ (Dqk side) and of dV
//   (Dv side) the unit produces; both halves recompute S^T and dP^T over the
//   full head dims.  Tensor memory then holds dK and dV of one half (128 + 128
//   columns) next to the pipelined S buffers, as for D = 128.
// * 32 queries per step (64 would not leave room for full-width K, V and two
//   Q / dO stages in shared memory): S^T = K Q^T and dP^T = V dO^T run as
//   M = 128, N = 32 tcgen05 MMAs over Dqk / Dv; dV += P^T dO and dK += dS^T Q
//   (TS, the half's 128 columns of dO / Q), dQ^T = K^T dS (SS, the half's 128
//   columns of K, M = 128 rows of d).
// * dS is staged in shared memory query-major (stmatrix.trans), the K-major
//   B operand of dQ^T.  The dQ reducers add dQ^T straight out of tensor
//   memory into the fp32 accumulator with coalesced red.global.add (lane = d,
//   one 128-byte request per query row).
//
// Tile widths DQ, DV are 128 or 256; the tensor maps fill the columns past
// Dqk / Dv with zeros, which adds nothing to the products.  The masks, causal
// skipping, varlen units and used lengths are those of the main kernel, the
// band with a lower edge (a left window) in an instance of its own (kBand);
// ALiBi, the bias, dropout and the deterministic order are not built for these
// head dims (the host refuses them).
//
// Warp roles (12 warps): 0 TMA producer | 1 MMA warp A (S^T, dP^T; allocates
// tensor memory) | 2 MMA warp B (dV, dK, dQ^T) | 3 idle | 4-7 dQ reducers |
// 8-11 softmax / elementwise (one TMEM lane quarter each; they also write dK
// and dV at the end of a unit).  Every wait is bounded, and a CTA that gives
// up still waits for the MMAs and loads it issued before it frees tensor
// memory.
#include "fa_bwd_units.cuh"
#include "fa_device.cuh"
#include "fa_params.h"

namespace fa {
namespace {

template <int kDQ, int kDV, typename T>
struct WideCfg {
    static constexpr int DQ = kDQ, DV = kDV;   // tile widths of the two sides
    static constexpr int BN = kBlockN;         // keys per unit
    static constexpr int BM = 32;              // queries per step
    static constexpr int NH = (kDQ > kDV ? kDQ : kDV) / 128;   // column halves
    static constexpr int kSBuf = 3;
    // TMEM: dK half 128 | dV half 128 | S buffer x3 (32 each: S^T, then P^T
    // and dS^T as 16-bit pairs in its two halves, then the step's dQ^T) | X 32
    static constexpr int TM_DK = 0, TM_DV = 128, TM_S = 256;
    static constexpr int TM_X = TM_S + kSBuf * BM;
    static constexpr int TM_COLS = 512;
    static_assert(TM_X + BM <= TM_COLS, "TMEM overflow");
    static __device__ __forceinline__ int s_col(int b) { return TM_S + b * BM; }
    static __device__ __forceinline__ int p_col(int b) { return TM_S + b * BM; }
    static __device__ __forceinline__ int ds_col(int b) { return TM_S + b * BM + 16; }
    // shared memory (byte offsets from a 1024-aligned base); K, V, Q, dO in
    // 64-column panels of 128-byte swizzled rows
    static constexpr int K_BYTES = BN * DQ * 2, V_BYTES = BN * DV * 2;
    static constexpr int Q_BYTES = BM * DQ * 2, DO_BYTES = BM * DV * 2;
    static constexpr int DS_BYTES = BM * BN * 2;   // dS, query-major, two 64-key panels
    static constexpr int OFF_K = 0, OFF_V = K_BYTES, OFF_Q = OFF_V + V_BYTES;
    static constexpr int kStages =
        (OFF_Q + 3 * (Q_BYTES + DO_BYTES) + 2 * DS_BYTES + 6 * BM * 4 + 2048 <= 232448 - 1024) ? 3 : 2;
    static constexpr int OFF_DO = OFF_Q + kStages * Q_BYTES;
    static constexpr int OFF_DS = OFF_DO + kStages * DO_BYTES;
    static constexpr int OFF_LSE = OFF_DS + 2 * DS_BYTES;
    static constexpr int OFF_DVEC = OFF_LSE + kStages * BM * 4;
    static constexpr int OFF_BAR = OFF_DVEC + kStages * BM * 4;
    static constexpr int NUM_BARS = 40;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM slot, abort flag, unit ring
    static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;   // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
    static constexpr int kRing = 4;
    static constexpr int kThreads = 12 * 32;
    static constexpr int W_MMA_B = 2, W_RED = 4, W_SM = 8;
    static constexpr int kSmWarps = 4;
    static constexpr int kConsumerWarps = 2 + 4 + kSmWarps;
    static constexpr uint32_t IDESC_S = make_idesc(128, BM, Cvt<T>::is_bf16, false, false);
    static constexpr uint32_t IDESC_KV = make_idesc(128, 128, Cvt<T>::is_bf16, false, true);
    static constexpr uint32_t IDESC_DQ = make_idesc(128, BM, Cvt<T>::is_bf16, true, false);
};

enum {
    W_KV_FULL = 0, W_KV_EMPTY = 1,
    W_S_FULL = 2,      // +b
    W_P_FULL = 5,      // +b
    W_DS_FULL = 8,     // +b
    W_DQ_FULL = 11,    // +b
    W_S_FREE = 14,     // +b
    W_DP_FULL = 17, W_X_FREE = 18,
    W_DSB_FREE = 19,   // +d: dQ^T MMA done reading dS tile d
    W_KDONE = 21, W_ACC_FULL = 22, W_ACC_EMPTY = 23, W_DRAIN = 24,
    W_UNIT_FULL = 25,  // +k
    W_UNIT_EMPTY = 29, // +k
    W_STAGE0 = 33      // full[kStages], then empty[kStages]
};

struct WideMaps {
    CUtensorMap q, k, v, dout;
};

template <int kDQ, int kDV, typename T, bool kBand>
__global__ void __launch_bounds__(WideCfg<kDQ, kDV, T>::kThreads, 1)
    bwd_wide_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ WideMaps maps) {
    using C = WideCfg<kDQ, kDV, T>;
    constexpr int DQ = C::DQ, DV = C::DV, BM = C::BM, BN = C::BN, S = C::kStages, NH = C::NH;
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
        mbar_init(bar(W_KV_FULL), 1);
        mbar_init(bar(W_KV_EMPTY), 2);   // one commit per MMA warp
        for (int b = 0; b < 3; ++b) {
            mbar_init(bar(W_S_FULL + b), 1);
            mbar_init(bar(W_P_FULL + b), C::kSmWarps);
            mbar_init(bar(W_DS_FULL + b), C::kSmWarps);
            mbar_init(bar(W_DQ_FULL + b), 1);
            mbar_init(bar(W_S_FREE + b), 4);
        }
        mbar_init(bar(W_DP_FULL), 1);
        mbar_init(bar(W_X_FREE), C::kSmWarps);
        for (int d = 0; d < 2; ++d) mbar_init(bar(W_DSB_FREE + d), 1);
        mbar_init(bar(W_KDONE), 1);
        mbar_init(bar(W_ACC_FULL), 1);
        mbar_init(bar(W_ACC_EMPTY), C::kSmWarps);
        mbar_init(bar(W_DRAIN), 2);
        for (int k = 0; k < C::kRing; ++k) {
            mbar_init(bar(W_UNIT_FULL + k), 1);
            mbar_init(bar(W_UNIT_EMPTY + k), C::kConsumerWarps);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(W_STAGE0 + s), 1);                    // full: producer expect_tx
            mbar_init(bar(W_STAGE0 + S + s), 2 + C::kSmWarps);  // empty: MMA warps + softmax
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&maps.q);
        prefetch_tmap(&maps.k);
        prefetch_tmap(&maps.v);
        prefetch_tmap(&maps.dout);
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
    const int ntiles = (p.varlen ? *p.ntiles : p.num_units) * NH;
    UnitRing ring;
    ring.slot = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 32);
    ring.full0 = bar(W_UNIT_FULL);
    ring.empty0 = bar(W_UNIT_EMPTY);
    auto next_unit = [&]() -> int {
        int t = -1;
        if (lane == 0) {
            if (mbar_wait(ring.full0 + 8u * ring.k, ring.ph, w)) {
                t = ring.slot[ring.k];
                mbar_arrive(ring.empty0 + 8u * ring.k);
            }
        }
        t = __shfl_sync(0xffffffffu, t, 0);
        ring.advance(C::kRing);
        return t;
    };
    // unit t: column half t % NH of the key-block unit t / NH (the two halves
    // of a key block run next to each other and share its rows in L2)
    auto has_dk = [](int half) { return 128 * half < DQ; };
    auto has_dv = [](int half) { return 128 * half < DV; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_ph = 0, st_ph = 0;
            int stage = 0, kv_armed = 0;
            uint32_t st_armed = 0, st_last = 0;
            bool ok = true;
            while (ok) {
                if (!(ok = mbar_wait(ring.empty0 + 8u * ring.k, ring.ph ^ 1, w))) break;
                int t = atomicAdd(p.unit_counter, 1);
                if (t >= ntiles) {
                    t = -1;
                    __threadfence();
                    if (atomicAdd(p.unit_counter + 1, 1) == (int)gridDim.x - 1) {
                        atomicExch(p.unit_counter, 0);
                        atomicExch(p.unit_counter + 1, 0);
                    }
                }
                ring.slot[ring.k] = t;
                mbar_arrive(ring.full0 + 8u * ring.k);
                ring.advance(C::kRing);
                if (t < 0) break;
                const Unit u = decode_unit<BM>(p, t / NH);
                if (u.iters == 0) continue;
                if (!(ok = mbar_wait(bar(W_KV_EMPTY), kv_ph ^ 1, w))) break;
                kv_ph ^= 1;
                mbar_arrive_expect_tx(bar(W_KV_FULL), C::K_BYTES + C::V_BYTES);
                ++kv_armed;
                const int krow = u.k_row0 + u.n_block * BN;
#pragma unroll
                for (int hh = 0; hh < DQ / 64; ++hh)
                    tma_load_4d(sbase + C::OFF_K + hh * BN * 128, &maps.k, bar(W_KV_FULL), hh * 64,
                                u.hk, krow, u.bidx);
#pragma unroll
                for (int hh = 0; hh < DV / 64; ++hh)
                    tma_load_4d(sbase + C::OFF_V + hh * BN * 128, &maps.v, bar(W_KV_FULL), hh * 64,
                                u.hk, krow, u.bidx);
                for (int it = 0; it < u.iters; ++it) {
                    const int g = u.g_of(it, p.G), m = u.m_of(it, p.G);
                    const int h = u.hk * p.G + g;
                    if (!(ok = mbar_wait(bar(W_STAGE0 + S + stage), st_ph ^ 1, w))) break;
                    const uint32_t full = bar(W_STAGE0 + stage);
                    mbar_arrive_expect_tx(full, C::Q_BYTES + C::DO_BYTES + 2 * BM * 4);
                    st_armed |= 1u << stage;
                    st_last = (st_last & ~(1u << stage)) | (st_ph << stage);
                    const int qrow = u.q_row0 + m * BM;
#pragma unroll
                    for (int hh = 0; hh < DQ / 64; ++hh)
                        tma_load_4d(sbase + C::OFF_Q + stage * C::Q_BYTES + hh * BM * 128, &maps.q, full,
                                    hh * 64, h, qrow, u.bidx);
#pragma unroll
                    for (int hh = 0; hh < DV / 64; ++hh)
                        tma_load_4d(sbase + C::OFF_DO + stage * C::DO_BYTES + hh * BM * 128, &maps.dout,
                                    full, hh * 64, h, qrow, u.bidx);
                    const long long r0 = ws_row(p, u.b, h, m * BM);
                    bulk_load(sbase + C::OFF_LSE + stage * BM * 4, p.lse2 + r0, BM * 4, full);
                    bulk_load(sbase + C::OFF_DVEC + stage * BM * 4, p.dvec + r0, BM * 4, full);
                    if (++stage == S) { stage = 0; st_ph ^= 1; }
                }
            }
            // wind-down: no load may land after the CTA exits
            if (kv_armed > 0)
                mbar_wait_drain(bar(W_KV_FULL), (uint32_t)(kv_armed - 1) & 1u, p.err, p.budget_ns);
            for (int s2 = 0; s2 < S; ++s2)
                if (bit(st_armed, s2)) mbar_wait_drain(bar(W_STAGE0 + s2), bit(st_last, s2), p.err, p.budget_ns);
        }
    } else if (warp == 1) {
        // ---------------------------------------------- MMA warp A: S^T, dP^T
        uint32_t kv_ph = 0, sfree_ph = 0, xfree_ph = 0, s_ph = 0;
        int s_stage = 0, nb = 0;
        bool ok = true;
        const uint64_t dK_k = sw128_desc(sbase + C::OFF_K, 16, 1024);
        const uint64_t dV_k = sw128_desc(sbase + C::OFF_V, 16, 1024);
        while (ok) {
            const int t = next_unit();
            if (t < 0) break;
            const Unit u = decode_unit<BM>(p, t / NH);
            if (u.iters == 0) continue;
            if (!(ok = mbar_wait_warp(bar(W_KV_FULL), kv_ph, w))) break;
            kv_ph ^= 1;
            for (int j = 0; j < u.iters; ++j) {
                if (!(ok = mbar_wait_warp(bar(W_STAGE0 + s_stage), s_ph, w))) break;
                if (!(ok = mbar_wait_warp(bar(W_S_FREE + nb), bit(sfree_ph, nb) ^ 1u, w))) break;
                sfree_ph ^= 1u << nb;
                tc_fence_after();
                const uint64_t dQ_k = sw128_desc(sbase + C::OFF_Q + s_stage * C::Q_BYTES, 16, 1024);
                const uint64_t dDO_k = sw128_desc(sbase + C::OFF_DO + s_stage * C::DO_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DQ / 16; ++kk)
                    mma_ss_warp(tmem + C::s_col(nb), desc_add(dK_k, (kk / 4) * (BN * 128) + (kk % 4) * 32),
                                desc_add(dQ_k, (kk / 4) * (BM * 128) + (kk % 4) * 32), C::IDESC_S, kk > 0);
                mma_commit_warp(bar(W_S_FULL + nb));
                if (!(ok = mbar_wait_warp(bar(W_X_FREE), xfree_ph ^ 1u, w))) break;
                xfree_ph ^= 1u;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DV / 16; ++kk)
                    mma_ss_warp(tmem + C::TM_X, desc_add(dV_k, (kk / 4) * (BN * 128) + (kk % 4) * 32),
                                desc_add(dDO_k, (kk / 4) * (BM * 128) + (kk % 4) * 32), C::IDESC_S, kk > 0);
                mma_commit_warp(bar(W_DP_FULL));
                mma_commit_warp(bar(W_STAGE0 + S + s_stage));
                if (++s_stage == S) { s_stage = 0; s_ph ^= 1; }
                if (++nb == C::kSBuf) nb = 0;
            }
            if (!ok) break;
            mma_commit_warp(bar(W_KV_EMPTY));
        }
        mma_commit_warp(bar(W_DRAIN));
        mbar_wait_drain_warp(bar(W_DRAIN), 0, p.err, p.budget_ns);
    } else if (warp == C::W_MMA_B) {
        // --------------------------------------- MMA warp B: dV, dK, dQ^T
        uint32_t kv_ph = 0, acc_ph = 0, p_ph = 0, ds_ph = 0, kd_ph = 0;
        int c_stage = 0, cb = 0, db = 0;
        bool ok = true;
        while (ok) {
            const int t = next_unit();
            if (t < 0) break;
            const int half = t % NH;
            const Unit u = decode_unit<BM>(p, t / NH);
            if (u.iters == 0) continue;
            const bool dk_on = has_dk(half), dv_on = has_dv(half);
            if (!(ok = mbar_wait_warp(bar(W_KV_FULL), kv_ph, w))) break;
            kv_ph ^= 1;
            // the half's 128 columns of K (A of dQ^T, MN-major: M = d)
            const uint64_t dKT_mn = sw128_desc(sbase + C::OFF_K + 2 * half * (BN * 128), BN * 128, 1024);
            for (int it = 0; it < u.iters; ++it) {
                if (it == 0) {
                    if (!(ok = mbar_wait_warp(bar(W_ACC_EMPTY), acc_ph ^ 1, w))) break;
                    acc_ph ^= 1;
                }
                if (!(ok = mbar_wait_warp(bar(W_P_FULL + cb), bit(p_ph, cb), w))) break;
                p_ph ^= 1u << cb;
                tc_fence_after();
                if (dv_on) {
                    // dV += P^T dO (the half's 128 columns of dO, MN-major, K step = 16 rows)
                    const uint64_t dDO_mn = sw128_desc(
                        sbase + C::OFF_DO + c_stage * C::DO_BYTES + 2 * half * (BM * 128), BM * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts_warp(tmem + C::TM_DV, tmem + C::p_col(cb) + 8 * kk, desc_add(dDO_mn, kk * 2048),
                                    C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
                }
                if (!(ok = mbar_wait_warp(bar(W_DS_FULL + cb), bit(ds_ph, cb), w))) break;
                ds_ph ^= 1u << cb;
                tc_fence_after();
                if (dk_on) {
                    // dK += dS^T Q (the half's 128 columns of Q)
                    const uint64_t dQ_mn = sw128_desc(
                        sbase + C::OFF_Q + c_stage * C::Q_BYTES + 2 * half * (BM * 128), BM * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts_warp(tmem + C::TM_DK, tmem + C::ds_col(cb) + 8 * kk, desc_add(dQ_mn, kk * 2048),
                                    C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_warp(bar(W_STAGE0 + S + c_stage));
                if (it == u.iters - 1) mma_commit_warp(bar(W_ACC_FULL));
                // dQ^T overwrites the P^T / dS^T that dV and dK read
                mma_commit_warp(bar(W_KDONE));
                if (!(ok = mbar_wait_warp(bar(W_KDONE), kd_ph, w))) break;
                kd_ph ^= 1u;
                tc_fence_after();
                if (dk_on) {
                    // dQ^T = K^T dS: B = dS query-major (K-major: 16 keys = 32 bytes,
                    // two 64-key panels of BM rows)
                    const uint64_t dDS_k = sw128_desc(sbase + C::OFF_DS + db * C::DS_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ss_warp(tmem + C::s_col(cb), desc_add(dKT_mn, kk * 2048),
                                    desc_add(dDS_k, (kk / 4) * (BM * 128) + (kk % 4) * 32), C::IDESC_DQ,
                                    kk > 0);
                }
                mma_commit_warp(bar(W_DQ_FULL + cb));
                mma_commit_warp(bar(W_DSB_FREE + db));
                if (++c_stage == S) c_stage = 0;
                if (++cb == C::kSBuf) cb = 0;
                db ^= 1;
            }
            if (!ok) break;
            mma_commit_warp(bar(W_KV_EMPTY));
        }
        mma_commit_warp(bar(W_DRAIN));
        mbar_wait_drain_warp(bar(W_DRAIN), 0, p.err, p.budget_ns);
    } else if (warp >= C::W_RED && warp < C::W_SM) {
        // ------------------------------------------------------ dQ reducers
        // Lane r = d of the half (TMEM lane quarter warp & 3): the step's 32
        // query rows out of tensor memory, the S buffer released, then one
        // coalesced red.global.add per query row (32 lanes = 32 consecutive d).
        const int quarter = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t dq_ph = 0;
        int cb = 0;
        bool ok = true;
        while (ok) {
            const int t = next_unit();
            if (t < 0) break;
            const int half = t % NH;
            const Unit u = decode_unit<BM>(p, t / NH);
            const bool dk_on = has_dk(half);
            const int d = 128 * half + 32 * quarter + lane;   // accumulator column
            for (int it = 0; it < u.iters; ++it) {
                const int g = u.g_of(it, p.G), m = u.m_of(it, p.G);
                if (!(ok = mbar_wait_warp(bar(W_DQ_FULL + cb), bit(dq_ph, cb), w))) break;
                dq_ph ^= 1u << cb;
                tc_fence_after();
                uint32_t v[32];
                if (dk_on) {
                    tmem_ld32(lane_addr + C::s_col(cb), v);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(W_S_FREE + cb));
                if (++cb == C::kSBuf) cb = 0;
                if (dk_on && d < p.Dh) {   // columns past Dqk stay 0
                    const long long row0 = ws_row(p, u.b, u.hk * p.G + g, m * BM);
                    const int rows_left = u.lq - m * BM;
                    float *dst = p.dqacc + row0 * DQ + d;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < rows_left) red_add_f32(dst + (long long)i * DQ, __uint_as_float(v[i]));
                }
            }
        }
    } else if (warp >= C::W_SM) {
        // ------------------------------------------------ softmax / elementwise
        const int quarter = warp & 3;
        const int j = quarter * 32 + lane;          // key row within the block
        const int g4 = lane >> 2, q4 = lane & 3;    // 16-lane access shapes
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t s_ph = 0, dp_ph = 0, st_ph = 0, acc_ph = 0, dsb_ph = 0;
        int stage = 0, cb = 0, db = 0;
        bool ok = true;
        while (ok) {
            const int t = next_unit();
            if (t < 0) break;
            const int half = t % NH;
            const Unit u = decode_unit<BM>(p, t / NH);
            const int n0 = u.n_block * BN;
            const int kj = n0 + j;
            const bool key_ok = kj < u.lk;
            const int kb = n0 + quarter * 32 + g4;  // first key of this thread's 16-lane rows
            const int diag = u.lk - u.lq;
            const int whi = p.win_hi, wlo = p.win_lo;
            for (int it = 0; it < u.iters; ++it) {
                const int m0 = u.m_of(it, p.G) * BM;
                const bool masked_hi = n0 + BN - 1 - (m0 + diag) > whi;
                // kBand: some element of the tile lies below the band's lower edge
                const bool masked_lo = kBand && n0 - (m0 + BM - 1 + diag) < -wlo;
                if (!(ok = mbar_wait(bar(W_STAGE0 + stage), st_ph, w))) break;
                if (!(ok = mbar_wait(bar(W_S_FULL + cb), bit(s_ph, cb), w))) break;
                s_ph ^= 1u << cb;
                tc_fence_after();
                const uint32_t lse2 = sbase + C::OFF_LSE + stage * BM * 4;
                const uint32_t dvv = sbase + C::OFF_DVEC + stage * BM * 4;
                // element (h, k, r, e): key kb + 16h + 8r, query 8k + 2 q4 + e
                float P[32];
                __syncwarp();
                {
                    uint32_t sr[2][16];
                    tmem_ld16x256(lane_addr + C::s_col(cb), sr[0]);
                    tmem_ld16x256(lane_addr + (16u << 16) + C::s_col(cb), sr[1]);
                    uint64_t nl2[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 l = ld_shared_f32x2(lse2 + 4 * (8 * k + 2 * q4));
                        nl2[k] = f2_pack(-l.x, -l.y);
                    }
                    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
                    tmem_wait_ld();
                    const int lim_hi = kb - (m0 + diag) - 2 * q4 - whi;
                    const int lim_lo = kb - (m0 + diag) - 2 * q4 + wlo;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int kr = 16 * h + 8 * r;
                                const float2 x = f2_unpack(f2_fma(
                                    f2_pack(__uint_as_float(sr[h][4 * k + 2 * r]),
                                            __uint_as_float(sr[h][4 * k + 2 * r + 1])),
                                    sc2, nl2[k]));
                                float pv0 = ex2(x.x), pv1 = ex2(x.y);
                                if (masked_hi) {   // key - query - diag > whi
                                    if (lim_hi + kr > 8 * k) pv0 = 0.f;
                                    if (lim_hi + kr > 8 * k + 1) pv1 = 0.f;
                                }
                                if (kBand && masked_lo) {   // key - query - diag < -wlo
                                    if (lim_lo + kr < 8 * k) pv0 = 0.f;
                                    if (lim_lo + kr < 8 * k + 1) pv1 = 0.f;
                                }
                                if (kb + kr >= u.lk) { pv0 = 0.f; pv1 = 0.f; }
                                P[16 * h + 4 * k + 2 * r] = pv0;
                                P[16 * h + 4 * k + 2 * r + 1] = pv1;
                                pk[2 * k + r] = Cvt<T>::pack(pv0, pv1);
                            }
                        }
                        tmem_st16x128(lane_addr + ((uint32_t)(16 * h) << 16) + C::p_col(cb), pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(W_P_FULL + cb));
                if (!(ok = mbar_wait(bar(W_DP_FULL), dp_ph, w))) break;
                dp_ph ^= 1u;
                tc_fence_after();
                const uint32_t sds = sbase + C::OFF_DS + db * C::DS_BYTES;
                __syncwarp();
                {
                    uint32_t dr[2][16];
                    tmem_ld16x256(lane_addr + C::TM_X, dr[0]);
                    tmem_ld16x256(lane_addr + (16u << 16) + C::TM_X, dr[1]);
                    uint64_t dd[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 v = ld_shared_f32x2(dvv + 4 * (8 * k + 2 * q4));
                        dd[k] = f2_pack(v.x, v.y);
                    }
                    tmem_wait_ld();
                    // dP^T read: X is free; the dS tile db may still be read by
                    // the dQ^T MMA of step j - 2
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(W_X_FREE));
                    if (!(ok = mbar_wait(bar(W_DSB_FREE + db), bit(dsb_ph, db) ^ 1u, w))) break;
                    dsb_ph ^= 1u << db;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int e0 = 16 * h + 4 * k + 2 * r;
                                const uint64_t dpv = f2_pack(__uint_as_float(dr[h][4 * k + 2 * r]),
                                                             __uint_as_float(dr[h][4 * k + 2 * r + 1]));
                                const float2 ds = f2_unpack(f2_mul(f2_pack(P[e0], P[e0 + 1]), f2_sub(dpv, dd[k])));
                                pk[2 * k + r] = Cvt<T>::pack(ds.x, ds.y);
                            }
                        }
                        tmem_st16x128(lane_addr + ((uint32_t)(16 * h) << 16) + C::ds_col(cb), pk);
                        // dS into shared memory query-major: the registers of keys
                        // 8r.. and queries 8k.. form an 8x8 tile that stmatrix.trans
                        // stores with the queries as rows.  Thread t addresses
                        // query row 8 (t / 8) + t % 8, the 16-byte chunk of keys
                        // quarter 32 + 16 h + 8 r .. + 7 of its 128-byte row.
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int keycol = quarter * 32 + 16 * h + 8 * r;
                            const int qrow = 8 * (lane >> 3) + (lane & 7);
                            const int panel = keycol >> 6, chunk = (keycol & 63) >> 3;
                            const uint32_t addr =
                                sds + panel * (BM * 128) + qrow * 128 + ((chunk ^ (qrow & 7)) << 4);
                            stmatrix_x4_trans(addr, pk[r], pk[2 + r], pk[4 + r], pk[6 + r]);
                        }
                    }
                }
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(W_DS_FULL + cb));
                    mbar_arrive(bar(W_STAGE0 + S + stage));
                }
                if (++stage == S) { stage = 0; st_ph ^= 1; }
                if (++cb == C::kSBuf) cb = 0;
                db ^= 1;
            }
            if (!ok) break;
            // ---------------------------------------------- dK / dV of the half out
            const long long orow = (long long)(p.varlen ? u.k_row0 + kj : u.b * p.Sk + kj);
            T *dk_dst = reinterpret_cast<T *>(p.dk) + (orow * p.Hkv + u.hk) * p.Dh + 128 * half;
            T *dv_dst = reinterpret_cast<T *>(p.dv) + (orow * p.Hkv + u.hk) * p.Dhv + 128 * half;
            const int dk_cols = has_dk(half) ? min(128, p.Dh - 128 * half) : 0;
            const int dv_cols = has_dv(half) ? min(128, p.Dhv - 128 * half) : 0;
            if (u.iters == 0) {
                if (key_ok && n0 < u.lk) {
                    for (int c = 0; 8 * c < dk_cols; ++c) reinterpret_cast<uint4 *>(dk_dst)[c] = make_uint4(0, 0, 0, 0);
                    for (int c = 0; 8 * c < dv_cols; ++c) reinterpret_cast<uint4 *>(dv_dst)[c] = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            if (!(ok = mbar_wait(bar(W_ACC_FULL), acc_ph, w))) break;
            acc_ph ^= 1;
            tc_fence_after();
            __syncwarp();
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const int ncols = which == 0 ? dk_cols : dv_cols;
                if (ncols <= 0) continue;   // uniform across the CTA
                const float mul = which == 0 ? p.scale : 1.f;
                T *dst = which == 0 ? dk_dst : dv_dst;
                const int col0 = which == 0 ? C::TM_DK : C::TM_DV;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t a[32];
                    tmem_ld32(lane_addr + col0 + 32 * ch, a);
                    tmem_wait_ld();
                    if (key_ok) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            pk[c] = Cvt<T>::pack(__uint_as_float(a[2 * c]) * mul, __uint_as_float(a[2 * c + 1]) * mul);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (32 * ch + 8 * c < ncols)
                                reinterpret_cast<uint4 *>(dst + 32 * ch)[c] =
                                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(W_ACC_EMPTY));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

template <int kDQ, int kDV, typename T>
static cudaError_t launch_wide_t(const BwdParams &p, const WideMaps &maps, int grid, cudaStream_t stream) {
    using C = WideCfg<kDQ, kDV, T>;
    // a lower band edge has an instance of its own: its per-element test slows
    // the plain kernel even when skipped
    auto kern = p.win_lo < kNoWindow ? bwd_wide_kernel<kDQ, kDV, T, true> : bwd_wide_kernel<kDQ, kDV, T, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::kThreads, C::SMEM_BYTES, stream>>>(p, maps);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_wide_dt(const BwdParams &p, const WideMaps &maps, int grid, cudaStream_t stream) {
    if (p.D == 256 && p.Dv == 256) return launch_wide_t<256, 256, T>(p, maps, grid, stream);
    if (p.D == 256 && p.Dv == 128) return launch_wide_t<256, 128, T>(p, maps, grid, stream);
    if (p.D == 128 && p.Dv == 256) return launch_wide_t<128, 256, T>(p, maps, grid, stream);
    if (p.D == 128 && p.Dv == 128) return launch_wide_t<128, 128, T>(p, maps, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

// Rows of one TMA box for Q / dO in the wide kernel, and its column halves.
int wide_block_m() { return WideCfg<256, 256, __nv_bfloat16>::BM; }
int wide_halves(int Dq_tile, int Dv_tile) { return (Dq_tile > Dv_tile ? Dq_tile : Dv_tile) / 128; }

cudaError_t launch_bwd_wide(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dout, int bf16, int grid,
                            cudaStream_t stream) {
    WideMaps maps{q, k, v, dout};
    return bf16 ? launch_wide_dt<__nv_bfloat16>(p, maps, grid, stream)
                : launch_wide_dt<__half>(p, maps, grid, stream);
}

}  // namespace fa
