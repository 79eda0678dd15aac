// fa_bwd_main.cu -- the fused attention-backward main kernel for sm_103a.
//
// One work unit = (sequence b, K/V column block of 128 keys, kv head hk).  The
// unit keeps K and V resident in shared memory and its dK, dV accumulators in
// tensor memory, and streams the query-row blocks of every query head of the
// GQA group (the K/V-stationary loop of the Composable Kernel page
// "block_fmha_bwd_dq_dk_dv_pipeline_trload_kr_ktr_vr.hpp", whose hot loop runs
// over the Q row blocks of one K/V tile).  Per row block of BM queries:
//
//   S^T  = K Q^T          tcgen05.mma SS, M=128 keys, N=BM      (STAGE 1)
//   P^T  = exp2(S^T c log2e - LSE2)  softmax warps, mask on diagonal tiles
//                                                                (STAGE 2)
//   dP^T = V dO^T         tcgen05.mma SS                          (STAGE 4)
//   dV  += P^T dO         tcgen05.mma TS (P^T bf16 in TMEM)       (STAGE 3)
//   dS^T = P^T o (dP^T - Dv)  softmax warps                       (STAGE 5)
//   dK  += dS^T Q         tcgen05.mma TS (dS^T bf16 in TMEM)      (STAGE 6)
//   dQ^T = K^T dS^T       tcgen05.mma SS (dS^T staged in shared memory;
//                         D = 64: dQ = dS K), added into the fp32
//                         accumulator in the workspace (STAGE 7): at D = 128
//                         each 32-row chunk goes through shared memory and
//                         one TMA bulk reduce-add (cp.reduce.async.bulk), at
//                         D = 64 through red.global.add.v4.f32 (the atomic
//                         "update_tile" path); in deterministic mode in a
//                         fixed n-block order through per-row-block
//                         semaphores (the wait_eq / arrive_inc pattern of
//                         CollectiveEpilogueBwdGQA in
//                         "flash-attention/hopper/epilogue_bwd.hpp")
//
// and at the end dK * c, dV are written out (CollectiveEpilogueBwd::store:
// registers -> shared memory, staged in the dS^T tiles, -> TMA tensor store;
// plain stores for a block that ends past the used key length; zeros for a
// unit with no visible query, store_zero).
//
// Persistent CTAs (one per SM) take units from a global counter.  Warp roles
// (16 warps, 512 threads):
//   warp 0        TMA producer: K and V once per unit (they swap shared-memory
//                 slots from one unit to the next, so the next unit's K loads
//                 while this unit's last dQ still reads its K), Q / dO / LSE2
//                 / Dv per step through a 3-stage ring; takes the units and
//                 passes them on through a ring in shared memory
//   warp 1        MMA warp A: S^T and dP^T of every step; also allocates and
//                 frees tensor memory
//   warp 2        MMA warp B: dV, dK, then dQ^T of every step
//   warp 3        bulk-reduce issuer (D = 128): adds each staged dQ chunk to
//                 the accumulator and, in deterministic mode, counts the
//                 completed adds on the row blocks' semaphores
//   warps 4-7     dQ reducers: dQ^T out of tensor memory into the staging
//                 buffers (one TMEM lane quarter each); in deterministic mode
//                 the first of them waits for the row block's semaphore before
//                 a step's chunks are handed to the issuer
//   warps 8-15    softmax / elementwise, two groups of four; group g handles
//                 query columns [g BM/2, (g+1) BM/2) of every key row, and
//                 in the epilogue group 0 writes dK, group 1 writes dV
// Every wait is bounded (see fa_device.cuh); a wait that gives up sets the
// CTA abort flag and the device error word, and the CTA winds down: every
// MMA and TMA load it issued completes before tensor memory is freed.
#include "fa_bwd_units.cuh"
#include "fa_device.cuh"
#include "fa_params.h"

namespace fa {
namespace {

template <int kD, typename T>
struct MainCfg {
    static constexpr int D = kD;
    static constexpr int BN = kBlockN;                 // keys per unit
    static constexpr int BM = (kD == 128) ? 64 : 128;  // queries per step
    static constexpr int HALF = BM / 2;                // query columns per softmax group
    static constexpr int NCH = HALF / 32;              // 32-column chunks per group
    // dQ GEMM orientation: the MMA's M (=128) is d when D = 128 (dQ^T = K^T dS^T,
    // TMEM lanes = d) and the query row when D = 64 (dQ = dS K, lanes = query).
    static constexpr bool kDqT = (kD == 128);
    // Software pipeline.  TMEM (512 columns):
    //   D = 128 (BM = 64):  dK 128 | dV 128 | S buffer x3 (64 each) | X 64
    //   D = 64 (BM = 128):  dK 64 | dV 64 | S buffer x2 (128 each) | X 128
    // An S buffer carries one step through its life: S^T, then P^T and dS^T
    // as bf16 pairs, then -- once dV and dK have read those -- that step's dQ
    // (dQ^T for D = 128), until the reducers take it out.  X holds dP^T,
    // which the softmax warps read as soon as it is complete.  S^T of step j
    // thus waits only for the dQ of step j - kSBuf to be drained, and dP^T of
    // step j only for the softmax warps to have read dP^T of step j-1.
    static constexpr int kSBuf = (kD == 128) ? 3 : 2;
    static constexpr int kStages = 3;
    // Warp roles: 0 producer | 1 MMA warp A (S, dP) | 2 MMA warp B (dV, dK,
    // dQ) | 3 bulk-reduce issuer (D = 128) | 4-7 dQ reducers | 8-15 softmax
    // (two groups of four, one per TMEM lane quarter).  Warp 3 idles when
    // D = 64.
    static constexpr int W_MMA_B = 2, W_ISSUE = 3, W_RED = 4, W_SM = 8;
    static constexpr int kThreads = 16 * 32;
    static constexpr int TM_DK = 0;
    static constexpr int TM_DV = D;
    static constexpr int TM_S = 2 * D;
    static constexpr int TM_X = TM_S + kSBuf * BM;         // dP^T
    static constexpr int TM_COLS = 512;
    static_assert(TM_X + BM <= TM_COLS, "TMEM overflow");
    // Columns (S buffer b, softmax group g, 32-query chunk ch).  In the HALF
    // columns of group g, the bf16 pairs of P^T fill the first HALF/2 and
    // those of dS^T the second: chunk ch's P^T lands on S^T columns this group
    // has already read, and dS^T is written after all of them were read.
    static __device__ __forceinline__ int s_col(int b, int g, int ch) {
        return TM_S + b * BM + g * HALF + 32 * ch;
    }
    static __device__ __forceinline__ int p_col(int b, int g, int ch) {   // P^T bf16 pairs
        return TM_S + b * BM + g * HALF + 16 * ch;
    }
    static __device__ __forceinline__ int dp_col(int g, int ch) { return TM_X + g * HALF + 32 * ch; }
    static __device__ __forceinline__ int ds_col(int b, int g, int ch) {  // dS^T bf16 pairs
        return TM_S + b * BM + g * HALF + 16 * NCH + 16 * ch;
    }
    // dQ^T (D = 128: 64 query columns) or dQ (D = 64: 64 d columns)
    static __device__ __forceinline__ int dq_col(int b) { return TM_S + b * BM; }
    // A-operand column of MMA K step kk (queries 16kk .. 16kk+15) of P^T / dS^T
    static __device__ __forceinline__ int p_op(int b, int kk) {
        const int g = (16 * kk) / HALF;
        return p_col(b, g, 0) + (16 * kk - g * HALF) / 2;
    }
    static __device__ __forceinline__ int ds_op(int b, int kk) {
        const int g = (16 * kk) / HALF;
        return ds_col(b, g, 0) + (16 * kk - g * HALF) / 2;
    }
    // shared memory (byte offsets from a 1024-aligned base)
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int QO_BYTES = BM * D * 2;
    static constexpr int DS_BYTES = BN * BM * 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_Q = OFF_V + KV_BYTES;
    static constexpr int OFF_DO = OFF_Q + kStages * QO_BYTES;
    static constexpr int OFF_DS = OFF_DO + kStages * QO_BYTES;
    // D = 128 (non-deterministic mode): the reducers pass each dQ^T tile (64
    // query rows x 128 d, fp32) to the accumulator in two chunks of 32 rows,
    // each staged in shared memory in the workspace's row-major layout and
    // added by one TMA bulk reduce; two staging buffers let a chunk be
    // written while the previous one is still being read.
    static constexpr bool kBulk = kDqT;
    static constexpr int CHUNK_ROWS = 32;
    static constexpr int CHUNK_BYTES = CHUNK_ROWS * D * 4;
    static constexpr int STG_BYTES = kBulk ? 2 * CHUNK_BYTES : 0;
    static_assert(!kBulk || CHUNK_BYTES == DS_BYTES, "a dQ chunk is parked in a dS^T tile");
    static constexpr int kDsBuf = 2;                       // dS^T tiles in shared memory
    static constexpr int OFF_STG = OFF_DS + kDsBuf * DS_BYTES;
    static constexpr int OFF_LSE = OFF_STG + STG_BYTES;
    static constexpr int OFF_DV = OFF_LSE + kStages * BM * 4;
    static constexpr int OFF_BAR = OFF_DV + kStages * BM * 4;
    static constexpr int NUM_BARS = 54;
    static_assert(40 + 2 * kStages <= 46, "barrier slots");
    // TMEM slot (+0), abort flag (+16), unit ring (+32), chunk rows (+48)
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory overflow");
    static constexpr int kRing = 4;             // work-unit hand-off ring depth
    // ring consumers: MMA warp(s) + 4 reducers + 8 softmax warps
    static constexpr int kConsumerWarps = 14;
    static constexpr uint32_t IDESC_S = make_idesc(128, BM, Cvt<T>::is_bf16, false, false);
    static constexpr uint32_t IDESC_KV = make_idesc(128, D, Cvt<T>::is_bf16, false, true);
    static constexpr uint32_t IDESC_DQ = make_idesc(128, 64, Cvt<T>::is_bf16, true, true);
};

// Barrier indices.  Hand-offs that can be committed before their waiter has
// looked at the previous phase come one per buffer, so that no barrier ever
// runs two phases ahead of a waiter.
enum {
    // K and V swap shared-memory slots from one unit to the next: unit u (u-th
    // unit of the CTA) keeps K in slot u % 2 and V in the other, so the next
    // unit's K can land in the slot whose V only warp A's dP^T reads, while
    // warp B still reads this unit's K for its last dQ.
    B_K_FULL = 0,       // +s: a K tile landed in slot s
    B_V_FULL = 46,      // +s: a V tile landed in slot s
    B_S_FULL = 2,       // +b, S buffer b: S^T complete
    B_P_FULL = 5,       // +b: P^T written back
    B_DS_FULL = 8,      // +b: dS^T written back (TMEM and shared memory)
    B_DQ_FULL = 11,     // +b: dQ^T complete
    B_S_FREE = 14,      // +b (D = 128): the reducers took dQ^T out of S buffer b
    B_DP_FULL = 17,     // dP^T complete
    B_X_FREE = 18,      // (D = 128) the softmax warps read dP^T
    B_RED_DONE = 19,    // (D = 128) each reducer warp made its last chunk arrivals
    B_DSB_FREE = 20,    // +d (D = 128): dQ^T MMA done reading dS^T tile d
    B_KDONE = 22,       // (D = 128) dV and dK of the step complete
    B_ACC_FULL = 23, B_ACC_EMPTY = 24, B_DRAIN = 25,
    B_UNIT_FULL = 26,   // +k, k < kRing: unit index k of the ring written
    B_UNIT_EMPTY = 30,  // +k: every consumer warp has read it
    B_STG_FULL = 34,    // +b: the 4 reducer warps wrote dQ staging buffer b
    B_STG_FREE = 36,    // +b: the bulk reduce has read staging buffer b
    B_TILE_FULL = 38,   // +d: the reducers wrote a dQ chunk into dS^T tile d
    B_STAGE0 = 40,      // full[kStages], then empty[kStages]
    B_FREE_A = 48,      // warp A's MMAs of a unit completed (its reads of both slots)
    B_FREE_B = 49,      // warp B's MMAs of a unit completed (its reads of the K slot)
    B_EPI_FULL = 50,    // +g: softmax group g wrote a dK / dV slice into its staging tile
    B_EPI_FREE = 52     // +g: the tensor store of group g has read its staging tile
};

struct MainMaps {
    CUtensorMap q, k, v, dout;
    CUtensorMap dk, dv;   // outputs, the geometry of k and v
};

// Extension flags of an instance: a band with a lower edge (a left window),
// ALiBi, the elementwise bias / dBias, dropout.  Without flags: the plain
// kernel (no mask, or a band with an upper edge only, e.g. causal).  Each
// extension gets compiled in only where asked for: its code slows the softmax
// warps even when skipped at run time (measured: the bias code made a
// windowed run 1.8x slower, the ALiBi arithmetic 11 %).  kFAbs: ALiBi where a
// visible key may lie right of the diagonal (a band with an upper edge above
// it), which needs -slope |i + diag - j|; without it (e.g. causal) the bias is
// linear in the key, slope (j - i - diag), and costs one add per pair.
enum : int { kFBand = 1, kFAlibi = 2, kFBias = 4, kFDrop = 8, kFAbs = 16 };
// the instances built, each a superset of the flags before it in its chain
constexpr int kMainFlagSets[] = {0,
                                 kFBand,
                                 kFBand | kFAlibi,
                                 kFBand | kFAlibi | kFAbs,
                                 kFBand | kFAlibi | kFAbs | kFBias,
                                 kFBand | kFDrop,
                                 kFBand | kFAlibi | kFAbs | kFBias | kFDrop};

// The elementwise bias of one 32-query chunk (from query qc) x a softmax
// warp's 32 keys (from key kw), 8 queries (k) at a time: one 16-byte load per
// lane (lane L: query 8k + 2(L%4) + (L/4)%2, keys 8(L/8) .. +7), all 32 lanes
// together 8 rows of 64 contiguous bytes.  0 past the used lengths lq / lk.
// Rows start on 16-byte boundaries (base and row stride are checked on the
// host); the ragged end of the used keys is read element by element.
template <typename T>
__device__ __forceinline__ void load_bias_chunk(uint32_t (&bw)[4][4], const T *bias_h, long long rs, int qc,
                                                int kw, int lq, int lk, int lane) {
    const int bq = ((lane & 3) << 1) | ((lane >> 2) & 1);
    const int bk = kw + 8 * (lane >> 3);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int qi = qc + 8 * k + bq;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qi < lq && bk < lk) {
            const T *src = bias_h + (long long)qi * rs + bk;
            if (bk + 8 <= lk) {
                v = __ldg(reinterpret_cast<const uint4 *>(src));
            } else {
                const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src);
                uint32_t e[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) e[i] = bk + i < lk ? (uint32_t)__ldg(s16 + i) : 0u;
                v = make_uint4(e[0] | e[1] << 16, e[2] | e[3] << 16, e[4] | e[5] << 16, e[6] | e[7] << 16);
            }
        }
        bw[k][0] = v.x;
        bw[k][1] = v.y;
        bw[k][2] = v.z;
        bw[k][3] = v.w;
    }
}

// Dropout: a softmax thread's 32 keep flags of a chunk from the lanes' words
// (lane L: query c0 + L, bit l = key kb - g4 + l): bit 4 (2k + e) + 2h + r =
// (key kb + 16h + 8r, query c0 + 8k + 2q4 + e) kept.
__device__ __forceinline__ uint32_t thread_keep_flags(uint32_t kmask, int q4, int g4) {
    uint32_t f = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            // bits 0, 8, 16, 24 after the shift: (h, r) = (0, 0), (0, 1), (1, 0),
            // (1, 1); gathered to 4 bits
            const uint32_t x = (__shfl_sync(0xffffffffu, kmask, 8 * k + 2 * q4 + e) >> g4) & 0x01010101u;
            f |= ((x * 0x10204080u) >> 28) << (4 * (2 * k + e));
        }
    return f;
}

// load_bias_chunk's words into the order of the S^T registers: bw[k][2h + r]
// = the (query 8k + 2q4, 8k + 2q4 + 1) pair of key g4 + 16h + 8r (lane = 4 g4
// + q4).  As loaded, the lane bits (from the top) hold key bits 4, 3, query
// bit 0 and query bits 2, 1, the register bits key bits 2, 1 and the half
// key bit 0; key bits 4 and 3 trade places with the register bits, query bit
// 0 with the half.
__device__ __forceinline__ void bias_to_st_order(uint32_t (&bw)[4][4], int lane) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        xchg_lane_reg(bw[k][0], bw[k][2], 16, lane & 16);
        xchg_lane_reg(bw[k][1], bw[k][3], 16, lane & 16);
        xchg_lane_reg(bw[k][0], bw[k][1], 8, lane & 8);
        xchg_lane_reg(bw[k][2], bw[k][3], 8, lane & 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) bw[k][i] = xchg_lane_half(bw[k][i], 4, lane & 4);
    }
}

template <int kD, typename T, int kFlags>
__global__ void __launch_bounds__(MainCfg<kD, T>::kThreads, 1)
    bwd_main_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ MainMaps maps) {
    using C = MainCfg<kD, T>;
    constexpr int D = C::D, BM = C::BM, BN = C::BN, S = C::kStages, HALF = C::HALF, NCH = C::NCH;
    constexpr bool kExt = (kFlags & kFBand) != 0, kAlibi = (kFlags & kFAlibi) != 0,
                   kBias = (kFlags & kFBias) != 0, kDrop = (kFlags & kFDrop) != 0;
    // ALiBi with no visible key right of the diagonal: -slope |d| = slope d
    constexpr bool kAlibiLin = kAlibi && (kFlags & kFAbs) == 0;
    // D = 64, or an elementwise bias, without dropout: the dS pass reads P^T
    // back from tensor memory (the rounded operand of dV) instead of keeping
    // the step's fp32 values of P per thread in registers between the passes
    // (with a bias the registers hold the bias chunk meanwhile)
    constexpr bool kPFromTmem = (NCH == 2 || kBias) && !kDrop;
    // two 32-query chunks per softmax warp (D = 64) with P kept in registers:
    // the two 16-lane halves of a TMEM tile are loaded one after the other
    // (register pressure)
    constexpr bool kSplitH = NCH == 2 && !kPFromTmem;
    // dropout with the forward's stored flags: the lanes' words gathered into
    // each thread's flags after the S wait (else right after their loads)
    constexpr bool kLateKeep = kDrop && NCH == 2;
    // the bias chunk loaded at the top of the step (else at the chunk's start)
    constexpr bool kEarlyBias = kBias && NCH == 1 && kPFromTmem;
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
        for (int sl = 0; sl < 2; ++sl) {
            mbar_init(bar(B_K_FULL + sl), 1);
            mbar_init(bar(B_V_FULL + sl), 1);
        }
        mbar_init(bar(B_FREE_A), 1);
        mbar_init(bar(B_FREE_B), 1);
        mbar_init(bar(B_RED_DONE), 4);
        for (int g = 0; g < 2; ++g) {
            mbar_init(bar(B_EPI_FULL + g), 4);
            mbar_init(bar(B_EPI_FREE + g), 1);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_FULL + b), 8);
            mbar_init(bar(B_DS_FULL + b), 8);
            mbar_init(bar(B_DQ_FULL + b), 1);
            mbar_init(bar(B_S_FREE + b), 4);
        }
        mbar_init(bar(B_DP_FULL), 1);
        mbar_init(bar(B_X_FREE), 8);
        // dS^T tile d is free once the dQ^T MMA read it and -- bulk mode --
        // once the dQ chunk the reducers parked in it has been read
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar(B_DSB_FREE + d), C::kBulk ? 2 : 1);
            mbar_init(bar(B_TILE_FULL + d), 4);
        }
        mbar_init(bar(B_KDONE), 1);
        mbar_init(bar(B_ACC_FULL), 1);
        mbar_init(bar(B_ACC_EMPTY), 8);
        mbar_init(bar(B_DRAIN), 2);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_STG_FULL + b), 4);
            mbar_init(bar(B_STG_FREE + b), 1);
        }
        for (int k = 0; k < C::kRing; ++k) {
            mbar_init(bar(B_UNIT_FULL + k), 1);
            mbar_init(bar(B_UNIT_EMPTY + k), C::kConsumerWarps);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(B_STAGE0 + s), 1);          // full: producer expect_tx
            // empty: a commit per MMA warp + 8 softmax warps
            mbar_init(bar(B_STAGE0 + S + s), 2 + 8);
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
    const int ntiles = p.varlen ? *p.ntiles : p.num_units;
    UnitRing ring;
    ring.slot = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 32);
    ring.full0 = bar(B_UNIT_FULL);
    ring.empty0 = bar(B_UNIT_EMPTY);
    // consumer side: next unit index (whole warp, converged), -1 at the end or on abort
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

    if (warp < C::W_RED) {
        // warpgroup 0: producer, MMA issue, bulk-reduce issue
        if (warp == 0) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                uint32_t st_ph = 0;
                int stage = 0;
                bool ok = true;
                // K / V tiles issued so far: unit v (the v-th unit with work) has its
                // K in slot v % 2 and its V in the other, as phase v / 2 of the
                // slot's K / V barrier
                int kn = 0, vn = 0;
                // the phase parity of the last load armed on each barrier, so that
                // every load still in flight can be waited for before the CTA exits
                uint32_t st_armed = 0, st_last = 0;   // bit s: stage s armed / its parity
                // one Q / dO / LSE2 / Dv stage of step it of unit u
                auto load_stage = [&](const Unit &u, int it) __attribute__((always_inline)) -> bool {
                    const int g = u.g_of(it, p.G), m = u.m_of(it, p.G);
                    const int h = u.hk * p.G + g;
                    if (!mbar_wait(bar(B_STAGE0 + S + stage), st_ph ^ 1, w)) return false;
                    const uint32_t full = bar(B_STAGE0 + stage);
                    mbar_arrive_expect_tx(full, 2 * C::QO_BYTES + 2 * BM * 4);
                    st_armed |= 1u << stage;
                    st_last = (st_last & ~(1u << stage)) | (st_ph << stage);
                    const int qrow = u.q_row0 + m * BM;
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh) {
                        tma_load_4d(sbase + C::OFF_Q + stage * C::QO_BYTES + hh * BM * 128, &maps.q,
                                    full, hh * 64, h, qrow, u.bidx);
                        tma_load_4d(sbase + C::OFF_DO + stage * C::QO_BYTES + hh * BM * 128,
                                    &maps.dout, full, hh * 64, h, qrow, u.bidx);
                    }
                    const long long r0 = ws_row(p, u.b, h, m * BM);
                    bulk_load(sbase + C::OFF_LSE + stage * BM * 4, p.lse2 + r0, BM * 4, full);
                    bulk_load(sbase + C::OFF_DV + stage * BM * 4, p.dvec + r0, BM * 4, full);
                    if (++stage == S) { stage = 0; st_ph ^= 1; }
                    return true;
                };
                // a K or V tile of 128 keys into slot sl
                auto load_kv = [&](const Unit &u, const CUtensorMap *map, uint32_t full, int sl)
                    __attribute__((always_inline)) {
                    mbar_arrive_expect_tx(full, C::KV_BYTES);
                    const int krow = u.k_row0 + u.n_block * BN;
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh)
                        tma_load_4d(sbase + C::OFF_K + sl * C::KV_BYTES + hh * BN * 128, map, full,
                                    hh * 64, u.hk, krow, u.bidx);
                };
                while (ok) {
                    // take the next unit and publish it to the other warps
                    if (!(ok = mbar_wait(ring.empty0 + 8u * ring.k, ring.ph ^ 1, w))) break;
                    int t = atomicAdd(p.unit_counter, 1);
                    if (t >= ntiles) {
                        t = -1;
                        // the last CTA to run out resets the counters for the next launch
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
                    const Unit u = decode_unit<BM>(p, t);
                    if (u.iters == 0) continue;
                    const int nu = kn, ks = nu & 1;         // K slot; V goes to the other
                    // K into the slot that held the previous unit's V, once warp
                    // A's MMAs of that unit completed
                    if (nu > 0 && !(ok = mbar_wait(bar(B_FREE_A), (uint32_t)(nu - 1) & 1u, w))) break;
                    load_kv(u, &maps.k, bar(B_K_FULL + ks), ks);
                    ++kn;
                    // the first step's Q / dO, so that S^T of the unit can start
                    if (!(ok = load_stage(u, 0))) break;
                    // V into the slot of the previous unit's K, once warp B's dQ^T
                    // read it too
                    if (nu > 0 && !(ok = mbar_wait(bar(B_FREE_B), (uint32_t)(nu - 1) & 1u, w))) break;
                    load_kv(u, &maps.v, bar(B_V_FULL + (ks ^ 1)), ks ^ 1);
                    ++vn;
                    for (int it = 1; it < u.iters; ++it)
                        if (!(ok = load_stage(u, it))) break;
                }
                // wind-down (after an abort some loads may not have been waited
                // for by their consumers): none may land after the CTA exits
                for (int v = max(kn - 2, 0); v < kn; ++v)
                    mbar_wait_drain(bar(B_K_FULL + (v & 1)), (uint32_t)(v >> 1) & 1u, p.err, p.budget_ns);
                for (int v = max(vn - 2, 0); v < vn; ++v)
                    mbar_wait_drain(bar(B_V_FULL + ((v & 1) ^ 1)), (uint32_t)(v >> 1) & 1u, p.err,
                                    p.budget_ns);
                for (int s2 = 0; s2 < S; ++s2)
                    if (bit(st_armed, s2)) mbar_wait_drain(bar(B_STAGE0 + s2), bit(st_last, s2), p.err, p.budget_ns);
            }
        } else if (warp == 1) {
            // ------------------------------------------- MMA warp A: S and dP
            // Issues S^T_j = K Q_j^T into S buffer j%3 and dP^T_j = V dO_j^T into
            // X for every step j, ahead of warp B.  Before S_j it waits until the
            // reducers took the dQ^T of step j-3 out of that S buffer, before dP_j
            // until the softmax warps read dP^T of step j-1.
            uint32_t sfree_ph = 0, xfree_ph = 0, s_ph = 0;   // sfree: bit per buffer
            int s_stage = 0, nb = 0;
            bool ok = true;
            int nu = 0;   // units with work so far: K in slot nu % 2, V in the other
            while (ok) {
                const int t = next_unit();
                if (t < 0) break;
                const Unit u = decode_unit<BM>(p, t);
                if (u.iters == 0) continue;
                const int ks = nu & 1;
                const uint32_t uph = (uint32_t)(nu >> 1) & 1u;
                const uint64_t dK_k = sw128_desc(sbase + C::OFF_K + ks * C::KV_BYTES, 16, 1024);
                const uint64_t dV_k = sw128_desc(sbase + C::OFF_K + (ks ^ 1) * C::KV_BYTES, 16, 1024);
                if (!(ok = mbar_wait_warp(bar(B_K_FULL + ks), uph, w))) break;
                for (int j = 0; j < u.iters; ++j) {
                    if (!(ok = mbar_wait_warp(bar(B_STAGE0 + s_stage), s_ph, w))) break;
                    if (!(ok = mbar_wait_warp(bar(B_S_FREE + nb), bit(sfree_ph, nb) ^ 1u, w))) break;
                    sfree_ph ^= 1u << nb;
                    tc_fence_after();
                    const uint64_t dQ_k = sw128_desc(sbase + C::OFF_Q + s_stage * C::QO_BYTES, 16, 1024);
                    const uint64_t dDO_k = sw128_desc(sbase + C::OFF_DO + s_stage * C::QO_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
                        const uint32_t qo = (kk / 4) * (BM * 128) + (kk % 4) * 32;
                        mma_ss_warp(tmem + C::s_col(nb, 0, 0), desc_add(dK_k, ko), desc_add(dQ_k, qo),
                                    C::IDESC_S, kk > 0);
                    }
                    mma_commit_warp(bar(B_S_FULL + nb));
                    if (!(ok = mbar_wait_warp(bar(B_X_FREE), xfree_ph ^ 1u, w))) break;
                    xfree_ph ^= 1u;
                    // V of the unit lands after K (its slot frees later)
                    if (j == 0 && !(ok = mbar_wait_warp(bar(B_V_FULL + (ks ^ 1)), uph, w))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
                        const uint32_t qo = (kk / 4) * (BM * 128) + (kk % 4) * 32;
                        mma_ss_warp(tmem + C::TM_X, desc_add(dV_k, ko), desc_add(dDO_k, qo),
                                    C::IDESC_S, kk > 0);
                    }
                    mma_commit_warp(bar(B_DP_FULL));
                    mma_commit_warp(bar(B_STAGE0 + S + s_stage));   // warp A's share of the stage
                    if (++s_stage == S) { s_stage = 0; s_ph ^= 1; }
                    if (++nb == C::kSBuf) nb = 0;
                }
                if (!ok) break;
                mma_commit_warp(bar(B_FREE_A));   // both slots' reads by this warp done
                ++nu;
            }
            // every MMA this warp issued completes before tensor memory is freed
            // (also after an abort)
            mma_commit_warp(bar(B_DRAIN));
            mbar_wait_drain_warp(bar(B_DRAIN), 0, p.err, p.budget_ns);
        } else if (warp == C::W_MMA_B) {
            // ---------------------------------------- MMA warp B: dV, dK and dQ
            // For step j (S buffer j%3, dS^T tile j%2): dV += P^T dO once P^T is
            // written back, dK += dS^T Q once dS^T is; then, after dV and dK have
            // finished reading the S buffer, dQ^T = K^T dS^T into that same buffer.
            uint32_t acc_ph = 0, p_ph = 0, ds_ph = 0, kd_ph = 0;   // p / ds: bit per buffer
            int c_stage = 0, cb = 0, db = 0;
            bool ok = true;
            int nu = 0;   // units with work so far: K in slot nu % 2
            while (ok) {
                const int t = next_unit();
                if (t < 0) break;
                const Unit u = decode_unit<BM>(p, t);
                if (u.iters == 0) continue;
                const int ks = nu & 1;
                const uint64_t dK_mn = sw128_desc(sbase + C::OFF_K + ks * C::KV_BYTES, BN * 128, 1024);
                // K for dQ
                if (!(ok = mbar_wait_warp(bar(B_K_FULL + ks), (uint32_t)(nu >> 1) & 1u, w))) break;
                for (int it = 0; it < u.iters; ++it) {
                    if (it == 0) {
                        if (!(ok = mbar_wait_warp(bar(B_ACC_EMPTY), acc_ph ^ 1, w))) break;
                        acc_ph ^= 1;
                    }
                    const uint32_t sQ = sbase + C::OFF_Q + c_stage * C::QO_BYTES;
                    const uint32_t sDO = sbase + C::OFF_DO + c_stage * C::QO_BYTES;
                    if (!(ok = mbar_wait_warp(bar(B_P_FULL + cb), bit(p_ph, cb), w))) break;
                    p_ph ^= 1u << cb;
                    tc_fence_after();
                    // dV += P^T dO  (P^T bf16 in TMEM; dO MN-major: K step = 16 rows = 2048 B)
                    const uint64_t dDO_mn = sw128_desc(sDO, BM * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts_warp(tmem + C::TM_DV, tmem + C::p_op(cb, kk), desc_add(dDO_mn, kk * 2048),
                                    C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
                    if (!(ok = mbar_wait_warp(bar(B_DS_FULL + cb), bit(ds_ph, cb), w))) break;
                    ds_ph ^= 1u << cb;
                    tc_fence_after();
                    // dK += dS^T Q
                    const uint64_t dQ_mn = sw128_desc(sQ, BM * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts_warp(tmem + C::TM_DK, tmem + C::ds_op(cb, kk), desc_add(dQ_mn, kk * 2048),
                                    C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_warp(bar(B_STAGE0 + S + c_stage));   // warp B's share of the stage
                    // after the unit's last dK the accumulators are final: the
                    // softmax warps write them out while dQ^T of the step runs
                    if (it == u.iters - 1) mma_commit_warp(bar(B_ACC_FULL));
                    // dQ^T overwrites the P^T / dS^T that dV and dK read: wait for them
                    mma_commit_warp(bar(B_KDONE));
                    if (!(ok = mbar_wait_warp(bar(B_KDONE), kd_ph, w))) break;
                    kd_ph ^= 1u;
                    tc_fence_after();
                    // D = 128: dQ^T = K^T dS^T (M = d); D = 64: dQ = dS K (M = query);
                    // both operands MN-major, K step = 16 keys = 2048 B
                    const uint64_t dDS_mn =
                        sw128_desc(sbase + C::OFF_DS + db * C::DS_BYTES, BN * 128, 1024);
                    const uint64_t dq_a = C::kDqT ? dK_mn : dDS_mn;
                    const uint64_t dq_b = C::kDqT ? dDS_mn : dK_mn;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ss_warp(tmem + C::dq_col(cb), desc_add(dq_a, kk * 2048),
                                    desc_add(dq_b, kk * 2048), C::IDESC_DQ, kk > 0);
                    mma_commit_warp(bar(B_DQ_FULL + cb));
                    mma_commit_warp(bar(B_DSB_FREE + db));   // dS^T tile db read
                    if (++c_stage == S) c_stage = 0;
                    if (++cb == C::kSBuf) cb = 0;
                    db ^= 1;
                }
                if (!ok) break;
                mma_commit_warp(bar(B_FREE_B));   // the K slot's reads by this warp done
                ++nu;
            }
            mma_commit_warp(bar(B_DRAIN));
            mbar_wait_drain_warp(bar(B_DRAIN), 0, p.err, p.budget_ns);
        } else if (warp == C::W_ISSUE && C::kBulk) {
            // ------------------------------------------------ bulk-reduce issuer
            // One thread adds every dQ chunk to the fp32 accumulator.  Step j's
            // first chunk (query rows 0-31) waits in dS^T tile j%2, whose dS^T
            // the dQ^T MMA has consumed by then; its second chunk (rows 32-63)
            // in staging buffer j%2.  The reducers put the step's first
            // workspace row next to the buffers (row -1 after the last step).  At most two chunks are in flight: after issuing
            // one the issuer waits until the one before it has been read, then
            // frees its buffer.
            // Deterministic mode: the contributions to a 64-row block of the
            // accumulator are added in n-block order -- a step's first chunk is
            // marked parked only once the row block's semaphore counts every
            // earlier n block (the reducers wait), and the issuer counts its
            // own steps once their chunks have completed, two steps at a time:
            // the completed bulk groups, the async-proxy fence and release
            // adds, as the GQA epilogue of the FlashAttention pages orders its
            // bulk reduce and arrive_inc.
            if (lane == 0) {
                volatile long long *stg_row = reinterpret_cast<volatile long long *>(smem + C::OFF_MISC + 48);
                const bool det = p.deterministic;
                uint32_t tile_ph = 0, stg_ph = 0;   // bit d: parity of buffer d
                // deterministic mode: the counts of kRelBatch steps are released
                // together, after one wait for all their adds to complete, and so
                // are those of a unit's last steps.  A release waits for every
                // bulk reduce still in flight (about 2200 cycles, an L2 reduce),
                // so it goes out with nothing in flight, once per batch; longer
                // batches lengthen the ordering chains between units.  Measured
                // on B = 1, 16 heads, 32768 keys, D = 128 (median main ms): 21.4
                // (batches of 2, no flush at a unit's end), 21.9 / 21.7 / 21.0 /
                // 21.4 / 20.2-21.0 / 27.3 / 28.9 (batches of 2 / 3 / 4 / 6 / 8 /
                // 12 / 16 with the flush).
                constexpr int kRelBatch = 8;
                int *pend[kRelBatch] = {};          // semaphores of the steps not yet counted
                int npend = 0;
                bool done = false;
                if (!det) {
                    // the plain loop: no semaphores
                    for (int j = 0;; ++j) {
                        const int d = j & 1;
                        if (!mbar_wait(bar(B_TILE_FULL + d), bit(tile_ph, d), w)) break;
                        tile_ph ^= 1u << d;
                        const long long row = stg_row[d];
                        if (row < 0) { done = true; break; }
                        bulk_reduce_add_f32(p.dqacc + row * D, sbase + C::OFF_DS + d * C::DS_BYTES,
                                            C::CHUNK_BYTES);
                        bulk_commit_group();
                        bulk_wait_read_all_but_one();   // second chunk of step j-1 read
                        if (j > 0) mbar_arrive(bar(B_STG_FREE + (d ^ 1)));
                        if (!mbar_wait(bar(B_STG_FULL + d), bit(stg_ph, d), w)) break;
                        stg_ph ^= 1u << d;
                        bulk_reduce_add_f32(p.dqacc + (row + 32) * D, sbase + C::OFF_STG + d * C::CHUNK_BYTES,
                                            C::CHUNK_BYTES);
                        bulk_commit_group();
                        bulk_wait_read_all_but_one();   // first chunk of step j read
                        mbar_arrive(bar(B_DSB_FREE + d));
                    }
                } else {
                    for (int j = 0;; ++j) {
                        const int d = j & 1;
                        if (!mbar_wait(bar(B_TILE_FULL + d), bit(tile_ph, d), w)) break;
                        tile_ph ^= 1u << d;
                        long long row = stg_row[d];
                        if (row < 0) { done = true; break; }
                        const bool unit_end = (row >> 62) & 1;
                        row &= ~(1ll << 62);
                        // the reducer that parked the chunk saw the row block's
                        // semaphore count every earlier n block (acquire), and
                        // TILE_FULL passed that on to this thread
                        int *sem = p.sem + row / 64;
                        fence_async_global();
                        bulk_reduce_add_f32(p.dqacc + row * D, sbase + C::OFF_DS + d * C::DS_BYTES,
                                            C::CHUNK_BYTES);
                        bulk_commit_group();
                        bulk_wait_read_all_but_one();   // second chunk of step j-1 read
                        if (j > 0) mbar_arrive(bar(B_STG_FREE + (d ^ 1)));
                        if (!mbar_wait(bar(B_STG_FULL + d), bit(stg_ph, d), w)) break;
                        stg_ph ^= 1u << d;
                        bulk_reduce_add_f32(p.dqacc + (row + 32) * D, sbase + C::OFF_STG + d * C::CHUNK_BYTES,
                                            C::CHUNK_BYTES);
                        bulk_commit_group();
                        if (kRelBatch == 1) {
                            // one step late: step j-1's adds complete, count them
                            if (npend) {
                                bulk_wait_all_but<2>();
                                fence_async_global();
                                red_release_add_gpu(pend[0], 1);
                            }
                            pend[0] = sem;
                            npend = 1;
                        } else {
                            pend[npend++] = sem;
                            // all adds of the batch complete (or of a unit's last
                            // steps: the next unit's steps would delay them): count them
                            if (npend == kRelBatch || unit_end) {
                                bulk_wait_all();
                                fence_async_global();
                                fence_acq_rel_gpu();     // one release fence for the batch
#pragma unroll
                                for (int i = 0; i < kRelBatch; ++i)
                                    if (i < npend) red_relaxed_add_gpu(pend[i], 1);
                                npend = 0;
                            }
                        }
                        bulk_wait_read_all_but_one();   // first chunk of step j read
                        mbar_arrive(bar(B_DSB_FREE + d));
                    }
                }
                bulk_wait_all();
                if (done && det) {
                    fence_async_global();
#pragma unroll
                    for (int i = 0; i < kRelBatch; ++i)
                        if (i < npend) red_release_add_gpu(pend[i], 1);
                }
            }
        }
    } else if (warp < C::W_SM) {
        // warpgroup 1: dQ reducers
        if (C::kBulk) {
            // -------------------------------------------- dQ reducers (bulk mode)
            // Lane r = d of the dQ^T tile (64 query rows x 128 d, fp32) in S
            // buffer cb.  A step is read out as two chunks of 32 rows and the S
            // buffer released at once; each chunk is then written, column r of a
            // [32 rows x 128 d] block, to shared memory -- rows 0-31 into the
            // step's dS^T tile, rows 32-63 into a staging buffer -- and the
            // issuer warp adds it to the accumulator.
            const int quarter = warp & 3;
            const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
            const int r = quarter * 32 + lane;
            volatile long long *stg_row = reinterpret_cast<volatile long long *>(smem + C::OFF_MISC + 48);
            uint32_t dq_ph = 0, stg_free_ph = 0;   // bit b: parity of buffer b
            int cb = 0;                            // TMEM X buffer of the next step
            bool ok = true;
            // step iterator over the units of the ring: row of (head g, row block
            // m) = head0 + g * hstride + m * BM, heads innermost, row blocks
            // from the last one down (the MMA warps' order)
            long long head0 = 0, hstride = 0;
            int g_it = 0, m_it = -1, m_first = 0, n_cur = 0, diag_cur = 0;
            bool units_done = false;
            auto next_row = [&](long long &row0, int &nb) __attribute__((always_inline)) -> bool {
                while (m_it < m_first) {
                    if (units_done) return false;
                    const int t = next_unit();
                    if (t < 0) { units_done = true; return false; }
                    const Unit u = decode_unit<BM>(p, t);
                    if (u.nm == 0) continue;
                    n_cur = u.n_block;
                    diag_cur = u.lk - u.lq;
                    head0 = ws_row(p, u.b, u.hk * p.G, 0);
                    hstride = ws_row(p, u.b, u.hk * p.G + 1, 0) - head0;
                    m_first = u.m_begin;
                    m_it = u.m_begin + u.nm - 1;
                    g_it = 0;
                }
                row0 = head0 + g_it * hstride + (long long)m_it * BM;
                // deterministic order: contributions counted from the row block's
                // first key block (block 0 unless the band has a lower edge)
                nb = kExt ? n_cur - first_key_block(p, m_it * BM, diag_cur) : n_cur;
                if (++g_it == p.G) { g_it = 0; --m_it; }
                return true;
            };
            // dQ^T of the step in S buffer b -> (X, Y); releases the buffer
            auto load_step = [&](uint32_t (&X)[32], uint32_t (&Y)[32], int b) __attribute__((always_inline)) {
                tc_fence_after();
                __syncwarp();
                tmem_ld32(lane_addr + C::dq_col(b), X);
                tmem_ld32(lane_addr + C::dq_col(b) + 32, Y);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S_FREE + b));
            };
            auto wait_dq = [&](int b) __attribute__((always_inline)) -> bool {
                if (!mbar_wait_warp(bar(B_DQ_FULL + b), bit(dq_ph, b), w)) return false;
                dq_ph ^= 1u << b;
                return true;
            };
            auto wait_stg = [&](int sb) __attribute__((always_inline)) -> bool {
                if (!mbar_wait_warp(bar(B_STG_FREE + sb), bit(stg_free_ph, sb) ^ 1u, w)) return false;
                stg_free_ph ^= 1u << sb;
                return true;
            };
            // column r of a [32 rows x 128 d] fp32 block at buf; then tell the issuer
            auto write_chunk = [&](const uint32_t (&X)[32], uint32_t buf, uint32_t full_bar) __attribute__((always_inline)) {
                const uint32_t dst = buf + 4 * r;
#pragma unroll
                for (int i = 0; i < 32; ++i) st_shared_b32(dst + 4 * D * i, X[i]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar);
            };
            uint32_t R0[32], R1[32];
            long long row0 = 0;
            int nb = 0;   // earlier contributions to the step's row block
            int db = 0;   // dS^T tile / staging buffer of the step
            // deterministic mode: lane 0 of the first reducer warp waits until
            // the step's row block counts nb earlier contributions before it
            // marks the first chunk parked; the issuer acquires that through
            // TILE_FULL.  The first read goes out before the dQ^T wait, so its
            // round trip falls in time this warp spends waiting anyway.
            const bool det_w = p.deterministic && warp == C::W_RED;
            int sem_v = 0;
            while (ok && next_row(row0, nb)) {
                if (det_w && lane == 0) sem_v = ld_acquire_gpu(p.sem + row0 / 64);
                if (!(ok = wait_dq(cb))) break;
                load_step(R0, R1, cb);
                if (++cb == C::kSBuf) cb = 0;
                // rows 0-31 into the dS^T tile the dQ^T MMA has just consumed (its
                // previous chunk was read before the softmax wrote this step's dS^T)
                // deterministic mode: bit 62 marks a unit's last step, whose
                // count the issuer then releases at once
                if (lane == 0 && warp == C::W_RED)
                    stg_row[db] = row0 | (det_w && m_it < m_first ? (1ll << 62) : 0ll);
                if (det_w) {
                    int got = 1;
                    if (lane == 0 && sem_v < nb) got = sem_wait_geq(p.sem + row0 / 64, nb, w) ? 1 : 0;
                    if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
                }
                write_chunk(R0, sbase + C::OFF_DS + db * C::DS_BYTES, bar(B_TILE_FULL + db));
                // rows 32-63 into staging buffer db
                if (!(ok = wait_stg(db))) break;
                write_chunk(R1, sbase + C::OFF_STG + db * C::CHUNK_BYTES, bar(B_STG_FULL + db));
                db ^= 1;
            }
            // End marker for the issuer, sent by the first reducer warp for
            // all four once each of them has made its last chunk arrivals: a
            // warp that finished early must not arrive on a TILE_FULL phase
            // that a slower warp (one waiting on a semaphore) has yet to
            // arrive on for a real step.
            if (ok) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_RED_DONE));
                if (warp == C::W_RED && mbar_wait_warp(bar(B_RED_DONE), 0, w) && lane == 0) {
                    stg_row[db] = -1;
                    mbar_arrive_cnt(bar(B_TILE_FULL + db), 4);
                }
            }
        } else {
            // ------------------------------ dQ reducers (deterministic mode, D = 64)
            const int quarter = warp & 3;
            const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
            const int r = quarter * 32 + lane;   // TMEM lane: d (kDqT) or query row
            uint32_t dq_ph = 0;
            int cb = 0;
            bool ok = true;
            float *const dqacc = p.dqacc;
            while (ok) {
                const int t = next_unit();
                if (t < 0) break;
                const Unit u = decode_unit<BM>(p, t);
                for (int it = 0; it < u.iters; ++it) {
                    const int g = u.g_of(it, p.G), m = u.m_of(it, p.G);
                    const int h = u.hk * p.G + g;
                    if (!(ok = mbar_wait(bar(B_DQ_FULL + cb), bit(dq_ph, cb), w))) break;
                    dq_ph ^= 1u << cb;
                    tc_fence_after();
                    uint32_t v0[32], v1[32];
                    __syncwarp();
                    tmem_ld32(lane_addr + C::dq_col(cb), v0);
                    tmem_ld32(lane_addr + C::dq_col(cb) + 32, v1);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_S_FREE + cb));
                    if (++cb == C::kSBuf) cb = 0;
                    const long long row0 = ws_row(p, u.b, h, m * BM);
                    int *sem = p.sem + row0 / 64;
                    if (p.deterministic) {
                        // contributions to this row block arrive in n-block order:
                        // wait until the 4 reducer warps of every earlier n block added
                        bool got = true;
                        const int nb = kExt ? u.n_block - first_key_block(p, m * BM, u.lk - u.lq)
                                            : u.n_block;
                        if (lane == 0) got = sem_wait_geq(sem, 4 * nb, w);
                        got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                        if (!got) { ok = false; break; }
                        __threadfence();
                    }
                    const int rows_left = u.lq - m * BM;
                    if (C::kDqT) {
                        // lane r = d; columns = BM (=64) query rows; a warp adds 32
                        // consecutive d of one row: one 128-byte request
                        float *dst = dqacc + row0 * D + r;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < rows_left) red_add_f32(dst + (long long)i * D, __uint_as_float(v0[i]));
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (32 + i < rows_left)
                                red_add_f32(dst + (long long)(32 + i) * D, __uint_as_float(v1[i]));
                    } else {
                        // lane r = query row; columns = the 64 d of that row
                        if (r < rows_left) {
                            float *dst = dqacc + (row0 + r) * D;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(
                                                 dst + 4 * c),
                                             "f"(__uint_as_float(v0[4 * c])),
                                             "f"(__uint_as_float(v0[4 * c + 1])),
                                             "f"(__uint_as_float(v0[4 * c + 2])),
                                             "f"(__uint_as_float(v0[4 * c + 3]))
                                             : "memory");
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(
                                                 dst + 32 + 4 * c),
                                             "f"(__uint_as_float(v1[4 * c])),
                                             "f"(__uint_as_float(v1[4 * c + 1])),
                                             "f"(__uint_as_float(v1[4 * c + 2])),
                                             "f"(__uint_as_float(v1[4 * c + 3]))
                                             : "memory");
                        }
                    }
                    if (p.deterministic) {
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) red_release_add_gpu(sem, 1);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ softmax / elementwise
        const int grp = (warp - C::W_SM) / 4;      // query-column group
        const int quarter = warp & 3;
        const int j = quarter * 32 + lane;          // key row within the block
        const int g4 = lane >> 2, q4 = lane & 3;     // 16-lane access shapes
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t s_ph = 0, dp_ph = 0, st_ph = 0, acc_ph = 0, dsb_ph = 0;   // s_ph, dsb_ph: bit per buffer
        uint32_t epi_ph = 0;             // parity of this group's staging-tile barriers
        int stage = 0, cb = 0, db = 0;   // stage, S buffer, dS^T tile of the step
        bool ok = true;
        // dBias rows take 16-byte stores when every row starts on a 16-byte boundary
        const bool dbias_v4 = kBias && (reinterpret_cast<uintptr_t>(p.dbias) & 15u) == 0 && (p.Sk & 7) == 0;
        // Taking the next unit from the ring and decoding it before the dK / dV
        // epilogue, rather than after it (about 1300 cycles per unit), was
        // measured and is off: 1 % faster on the 2k causal workload, but the
        // build that had it ran the deterministic order 25 % slower (24.6-24.9
        // against 19.2-20.0 ms on B = 1, 16 heads, 32768 keys), even with the
        // early fetch switched off at run time there -- register allocation at
        // the 128-register cap, not the order of the fetch.
        constexpr bool kEarlyFetch = false;
        int t = -1;
        Unit un;
        auto fetch = [&]() __attribute__((always_inline)) {
            t = next_unit();
            if (t >= 0) un = decode_unit<BM>(p, t);
        };
        if (kEarlyFetch) fetch();
        while (ok) {
            if (!kEarlyFetch) fetch();
            if (t < 0) break;
            const Unit u = un;
            const int n0 = u.n_block * BN;
            const int kj = n0 + j;                   // key index within the sequence
            const bool key_ok = kj < u.lk;
            const int kb = n0 + quarter * 32 + g4;   // first key of this thread's 16-lane rows
            // key kj is visible to query qi iff -win_lo <= kj - qi - diag <= win_hi
            const int diag = u.lk - u.lq;
            const int whi = p.win_hi, wlo = p.win_lo;
            for (int it = 0; it < u.iters; ++it) {
                const int m = u.m_of(it, p.G);
                const int m0 = m * BM;
                // the tile crosses the upper / lower edge of the band: mask
                // element by element (one compare per edge and element)
                const bool masked_hi = n0 + BN - 1 - (m0 + diag) > whi;
                const bool masked_lo = kExt && n0 - (m0 + BM - 1 + diag) < -wlo;
                // ALiBi slope of the step's query head, in log2 units (0: none)
                float slope2 = 0.f;
                if (kAlibi && p.alibi)
                    slope2 = __ldg(p.alibi + (long long)u.b * p.alibi_bstride + u.hk * p.G + u.g_of(it, p.G)) *
                             1.4426950408889634f;
                // elementwise bias / dBias of the step's (sequence, query head)
                // (dense problems): element (query qi, key kj) at qi * stride + kj
                const T *bias_h = nullptr;
                uint16_t *dbias_h = nullptr;
                uint32_t bw[4][4];   // bias of one 32-query chunk (load_bias_chunk)
                if constexpr (kBias) {
                    const int hq = u.hk * p.G + u.g_of(it, p.G);
                    if (p.bias) {
                        bias_h = reinterpret_cast<const T *>(p.bias) + (long long)u.b * p.bias_bs +
                                 (long long)hq * p.bias_hs;
                        // one chunk per warp (D = 128) and P not held in
                        // registers: loaded before S is ready, so that the
                        // wait covers the loads' latency
                        if (kEarlyBias)
                            load_bias_chunk(bw, bias_h, p.bias_rs, m0 + grp * HALF, n0 + quarter * 32, u.lq,
                                            u.lk, lane);
                    }
                    if (p.dbias)
                        dbias_h = reinterpret_cast<uint16_t *>(p.dbias) +
                                  ((long long)u.b * p.Hq + hq) * p.Sq * p.Sk;
                }
                // dropout: drawn before S is ready (the wait hides it).  Lane L
                // draws the random bytes of query c0 + L of each chunk for the
                // warp's 32 keys (two Philox outputs of 16 keys) and packs the
                // keep flags into one word (bit l: key n0 + 32 quarter + l); a
                // thread then takes the words of its 8 queries by shuffles and
                // keeps the 32 flags of its own elements in one word:
                // kb32[ch] bit 4 (2k + e) + 2h + r = (key kb + 16h + 8r, query
                // c0 + 8k + 2q4 + e) kept.
                uint32_t kb32[NCH], kraw[NCH];
                if (kDrop) {
                    const uint32_t hq = (uint32_t)(u.hk * p.G + u.g_of(it, p.G));
                    const uint32_t tt4 = (uint32_t)p.drop_t * 0x01010101u;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        const int c0 = grp * HALF + 32 * ch;
                        uint32_t kmask = 0u;
                        if (p.drop_mask) {
                            // the forward's flags: word (n0 + 32 quarter) / 32 of
                            // query m0 + c0 + lane (0 past the used lengths)
                            const int qi = m0 + c0 + lane, kw0 = (n0 + 32 * quarter) >> 5;
                            if (qi < u.lq && n0 + 32 * quarter < u.lk && kw0 < p.drop_mask_w) {
                                const long long mrow =
                                    p.varlen ? (long long)hq * p.cu_q[p.B] + u.q_row0 + qi
                                             : ((long long)u.b * p.Hq + hq) * p.Sq + qi;
                                kmask = __ldg(p.drop_mask + mrow * p.drop_mask_w + kw0);
                            }
                        } else {
#pragma unroll
                            for (int g = 0; g < 2; ++g) {
                                const uint4 R = philox4x32_10(
                                    make_uint4((uint32_t)((n0 + 32 * quarter) >> 4) + g,
                                               (uint32_t)(m0 + c0 + lane), (uint32_t)u.b * p.Hq + hq,
                                               p.drop_offset),
                                    p.drop_key0, p.drop_key1);
                                const uint32_t wd[4] = {R.x, R.y, R.z, R.w};
#pragma unroll
                                for (int wi = 0; wi < 4; ++wi) {
                                    // bytes >= t -> 0xFF; the low bits of the 4 bytes
                                    // gathered into bits 28-31 by one product
                                    const uint32_t ge = __vcmpgeu4(wd[wi], tt4) & 0x01010101u;
                                    kmask |= ((ge * 0x10204080u) >> 28) << (16 * g + 4 * wi);
                                }
                            }
                        }
                        // loaded flags at D = 64: gathered after the S wait, which
                        // then covers the load (0.357 -> 0.313 ms on B = 4, H =
                        // 16, 2048 keys, causal; at D = 128 the same order cost
                        // 3-6 %)
                        kraw[ch] = kmask;
                        if (!(kLateKeep && p.drop_mask)) kb32[ch] = thread_keep_flags(kmask, q4, g4);
                    }
                }
                if (!(ok = mbar_wait(bar(B_STAGE0 + stage), st_ph, w))) break;
                if (!(ok = mbar_wait(bar(B_S_FULL + cb), bit(s_ph, cb), w))) break;
                if (kDrop && kLateKeep && p.drop_mask) {
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) kb32[ch] = thread_keep_flags(kraw[ch], q4, g4);
                }
                s_ph ^= 1u << cb;
                tc_fence_after();
                const uint32_t lse2 = sbase + C::OFF_LSE + stage * BM * 4;   // fp32 [BM]
                const uint32_t dv = sbase + C::OFF_DV + stage * BM * 4;
                // Element (h, k, r, e) of a 32-query chunk -- register 4k + 2r + e
                // of the lane-offset-h load -- is key kb + 16h + 8r, query
                // column 8k + 2*q4 + e of the chunk.  A thread thus needs 8
                // LSE2 / Dv values per chunk (4 eight-byte loads) instead of 32.
                float P[HALF];
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    // Two 32-query chunks per warp (D = 64, kSplitH): each 16-lane
                    // half of S^T is loaded when it is processed, so that the
                    // registers of one half are free again for the other (the
                    // chunk's P stays live into the dS pass next to them).
                    uint32_t sr[2][16];
                    tmem_ld16x256(lane_addr + C::s_col(cb, grp, ch), sr[0]);
                    if (!kSplitH) tmem_ld16x256(lane_addr + (16u << 16) + C::s_col(cb, grp, ch), sr[1]);
                    const int c0 = grp * HALF + 32 * ch;     // first query of the chunk
                    uint64_t nl2[4];   // (-LSE2, -LSE2) of the thread's query pairs
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 l = ld_shared_f32x2(lse2 + 4 * (c0 + 8 * k + 2 * q4));
                        nl2[k] = f2_pack(-l.x, -l.y);
                    }
                    if constexpr (kBias) {
                        if (!kEarlyBias && bias_h)
                            load_bias_chunk(bw, bias_h, p.bias_rs, m0 + c0, n0 + quarter * 32, u.lq, u.lk, lane);
                    }
                    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
                    tmem_wait_ld();
                    if constexpr (kBias) {
                        if (bias_h) bias_to_st_order(bw, lane);
                    }
                    // element (key kb + kr, query column 8k + e) has
                    // kj - qi - diag = lim + kr - 8k - e
                    const int lim = kb - (m0 + c0 + diag) - 2 * q4;
                    const int lim_hi = lim - whi, lim_lo = lim + wlo;
                    const float flim = (float)lim;
                    if (kAlibiLin) {
                        // linear ALiBi: slope (lim - 8k - e) joins -LSE2 here and
                        // slope kr is added per key offset below
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float a0 = slope2 * (flim - (float)(8 * k));
                            nl2[k] = f2_add(nl2[k], f2_pack(a0, a0 - slope2));
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (kSplitH && h == 1) {
                            tmem_ld16x256(lane_addr + (16u << 16) + C::s_col(cb, grp, ch), sr[1]);
                            tmem_wait_ld();
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int kr = 16 * h + 8 * r;    // key offset from kb
                                uint64_t addend = nl2[k];
                                if (kAlibiLin && kr > 0)
                                    addend = f2_add(addend, f2_pack(slope2 * (float)kr, slope2 * (float)kr));
                                const float2 x = f2_unpack(f2_fma(
                                    f2_pack(__uint_as_float(sr[h][4 * k + 2 * r]),
                                            __uint_as_float(sr[h][4 * k + 2 * r + 1])),
                                    sc2, addend));
                                float x0 = x.x, x1 = x.y;
                                if (kAlibi && !kAlibiLin) {
                                    // -slope * |qi + diag - kj|
                                    const float fd = flim + (float)(kr - 8 * k);
                                    x0 = fmaf(-slope2, fabsf(fd), x0);
                                    x1 = fmaf(-slope2, fabsf(fd - 1.f), x1);
                                }
                                if (kBias && bias_h) {   // + bias * log2e (0 past the used lengths)
                                    const float2 bb = Cvt<T>::unpack(bw[k][2 * h + r]);
                                    x0 = fmaf(bb.x, 1.4426950408889634f, x0);
                                    x1 = fmaf(bb.y, 1.4426950408889634f, x1);
                                }
                                float pv0 = ex2(x0);
                                float pv1 = ex2(x1);
                                bool keep0 = true, keep1 = true;
                                if (kDrop) {
                                    keep0 = (kb32[ch] >> (4 * (2 * k) + 2 * h + r)) & 1u;
                                    keep1 = (kb32[ch] >> (4 * (2 * k + 1) + 2 * h + r)) & 1u;
                                }
                                if (masked_hi) {   // lim + kr - 8k - e > whi
                                    if (lim_hi + kr > 8 * k) pv0 = 0.f;
                                    if (lim_hi + kr > 8 * k + 1) pv1 = 0.f;
                                }
                                if (kExt && masked_lo) {   // lim + kr - 8k - e < -wlo
                                    if (lim_lo + kr < 8 * k) pv0 = 0.f;
                                    if (lim_lo + kr < 8 * k + 1) pv1 = 0.f;
                                }
                                if (kb + kr >= u.lk) { pv0 = 0.f; pv1 = 0.f; }
                                if (!kPFromTmem) {
                                    P[32 * ch + 16 * h + 4 * k + 2 * r] = pv0;
                                    P[32 * ch + 16 * h + 4 * k + 2 * r + 1] = pv1;
                                }
                                if (kDrop) {
                                    // dV takes the dropped-out, rescaled P
                                    pk[2 * k + r] = Cvt<T>::pack(keep0 ? pv0 * p.drop_scale : 0.f,
                                                                 keep1 ? pv1 * p.drop_scale : 0.f);
                                } else {
                                    pk[2 * k + r] = Cvt<T>::pack(pv0, pv1);
                                }
                            }
                        }
                        tmem_st16x128(lane_addr + ((uint32_t)(16 * h) << 16) + C::p_col(cb, grp, ch), pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + cb));
                if (!(ok = mbar_wait(bar(B_DP_FULL), dp_ph, w))) break;
                dp_ph ^= 1u;
                tc_fence_after();
                const uint32_t sds = sbase + C::OFF_DS + db * C::DS_BYTES;
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint32_t dr[2][16];
                    uint32_t pt[2][8];   // kPFromTmem: P^T pairs of the chunk, per 16-lane half
                    tmem_ld16x256(lane_addr + C::dp_col(grp, ch), dr[0]);
                    if (kPFromTmem) tmem_ld16x128(lane_addr + C::p_col(cb, grp, ch), pt[0]);
                    if (!kSplitH) tmem_ld16x256(lane_addr + (16u << 16) + C::dp_col(grp, ch), dr[1]);
                    if (kPFromTmem && !kSplitH)
                        tmem_ld16x128(lane_addr + (16u << 16) + C::p_col(cb, grp, ch), pt[1]);
                    const int c0 = grp * HALF + 32 * ch;
                    uint64_t dd[4];   // Dv of the thread's query pairs
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 v = ld_shared_f32x2(dv + 4 * (c0 + 8 * k + 2 * q4));
                        dd[k] = f2_pack(v.x, v.y);
                    }
                    tmem_wait_ld();
                    if (!kSplitH && ch == NCH - 1) {
                        // dP^T read: X is free for the next step's dP^T
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_X_FREE));
                    }
                    if (ch == 0) {
                        // the dS^T tile db may still be read by the dQ MMA of step
                        // j-2: wait before the first write into it
                        if (!(ok = mbar_wait(bar(B_DSB_FREE + db), bit(dsb_ph, db) ^ 1u, w))) break;
                        dsb_ph ^= 1u << db;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (kSplitH && h == 1) {
                            tmem_ld16x256(lane_addr + (16u << 16) + C::dp_col(grp, ch), dr[1]);
                            if (kPFromTmem) tmem_ld16x128(lane_addr + (16u << 16) + C::p_col(cb, grp, ch), pt[1]);
                            tmem_wait_ld();
                            if (ch == NCH - 1) {
                                // the last half of dP^T read: X is free again
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(bar(B_X_FREE));
                            }
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int e0 = 32 * ch + 16 * h + 4 * k + 2 * r;
                                uint64_t dpv = f2_pack(__uint_as_float(dr[h][4 * k + 2 * r]),
                                                       __uint_as_float(dr[h][4 * k + 2 * r + 1]));
                                if (kDrop) {   // dS = P (M s dP - Dv)
                                    const uint32_t k0b = (kb32[ch] >> (4 * (2 * k) + 2 * h + r)) & 1u;
                                    const uint32_t k1b = (kb32[ch] >> (4 * (2 * k + 1) + 2 * h + r)) & 1u;
                                    dpv = f2_mul(dpv, f2_pack(k0b ? p.drop_scale : 0.f, k1b ? p.drop_scale : 0.f));
                                }
                                float2 pp;
                                if (kPFromTmem) pp = Cvt<T>::unpack(pt[h][2 * k + r]);
                                else pp = make_float2(P[e0], P[e0 + 1]);
                                const float2 ds = f2_unpack(f2_mul(f2_pack(pp.x, pp.y), f2_sub(dpv, dd[k])));
                                pk[2 * k + r] = Cvt<T>::pack(ds.x, ds.y);
                            }
                        }
                        tmem_st16x128(lane_addr + ((uint32_t)(16 * h) << 16) + C::ds_col(cb, grp, ch), pk);
                        // dS^T rows into shared memory (128B-swizzled halves of 64
                        // queries): the registers of keys 8r.. and queries 8k.. form
                        // an 8x8 tile in stmatrix's fragment layout.  Thread t
                        // addresses row t%8 (key jr) of tile k = t/8, a 16-byte
                        // chunk of the key's 128-byte row.
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int jr = quarter * 32 + 16 * h + 8 * r + (lane & 7);
                            const int i0 = c0 + 8 * (lane >> 3);
                            const int half = i0 / 64, cidx = (i0 % 64) / 8;
                            const uint32_t row = sds + half * (BN * 128) + jr * 128 + ((cidx ^ (lane & 7)) << 4);
                            stmatrix_x4(row, pk[r], pk[2 + r], pk[4 + r], pk[6 + r]);
                        }
                    }
                    if (kBias && dbias_h) {
                        // dBias = dS, inside the used lengths: the warp's 32 keys x
                        // the chunk's queries, read back transposed from its own
                        // part of the dS^T tile (before the MMAs are told it is
                        // full; nothing else writes that part meanwhile), 8
                        // queries at a time.  Thread t supplies key row t of the
                        // warp (matrix t/8) and gets query 8k + t/4, keys 8i +
                        // 2(t%4) (+1) in register i; two exchanges give it keys
                        // 8(t%4) .. +7 instead: one 16-byte store, 8 rows of 64
                        // contiguous bytes per warp.
                        __syncwarp();
                        const int jr = quarter * 32 + lane;
                        const int kj = n0 + quarter * 32 + 8 * (lane & 3);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int i0 = c0 + 8 * k;
                            const int half = i0 / 64, cidx = (i0 % 64) / 8;
                            uint32_t d[4];
                            ldmatrix_x4_trans(sds + half * (BN * 128) + jr * 128 + ((cidx ^ (lane & 7)) << 4), d[0],
                                              d[1], d[2], d[3]);
                            xchg_lane_reg(d[0], d[2], 2, lane & 2);
                            xchg_lane_reg(d[1], d[3], 2, lane & 2);
                            xchg_lane_reg(d[0], d[1], 1, lane & 1);
                            xchg_lane_reg(d[2], d[3], 1, lane & 1);
                            const int qi = m0 + i0 + (lane >> 2);
                            if (qi < u.lq && kj < u.lk) {
                                uint16_t *dst = dbias_h + (long long)qi * p.Sk + kj;
                                if (dbias_v4 && kj + 8 <= u.lk) {
                                    *reinterpret_cast<uint4 *>(dst) = make_uint4(d[0], d[1], d[2], d[3]);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 8; ++i)
                                        if (kj + i < u.lk) dst[i] = (uint16_t)(d[i >> 1] >> (16 * (i & 1)));
                                }
                            }
                        }
                    }
                }
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_DS_FULL + cb));
                    mbar_arrive(bar(B_STAGE0 + S + stage));
                }
                if (++stage == S) { stage = 0; st_ph ^= 1; }
                if (++cb == C::kSBuf) cb = 0;
                db ^= 1;
            }
            if (!ok) break;
            if (kEarlyFetch) fetch();
            // ---------------------------------------------------- dK / dV out
            T *out = reinterpret_cast<T *>(grp == 0 ? p.dk : p.dv);
            const long long orow = (long long)(p.varlen ? u.k_row0 + kj : u.b * p.Sk + kj);
            // the tensors' rows hold Dh <= D columns (a multiple of 8)
            T *dst = out + (orow * p.Hkv + u.hk) * p.Dh;
            if (u.iters == 0) {
                if (key_ok && n0 < u.lk) {
#pragma unroll
                    for (int c = 0; c < D / 8; ++c)
                        if (8 * c < p.Dh) reinterpret_cast<uint4 *>(dst)[c] = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            if (!(ok = mbar_wait(bar(B_ACC_FULL), acc_ph, w))) break;
            acc_ph ^= 1;
            tc_fence_after();
            __syncwarp();
            const float mul = grp == 0 ? p.scale : 1.f;
            const int col0 = grp == 0 ? C::TM_DK : C::TM_DV;
            if (n0 + BN <= u.lk) {
                // Every key row of the block is inside the used length: the
                // tile leaves by tensor stores.  Group g stages 64-column slices
                // of its [128 keys x D] tile in dS^T tile g (free once the last
                // dQ^T MMA -- and, D = 128, the issuer -- finished with both
                // tiles) in the store's 128-byte swizzle; the group's first
                // lane issues the store and waits until it has read the tile.
                bool free_ok = true;
                for (int d = 0; d < 2; ++d)
                    free_ok = free_ok && mbar_wait(bar(B_DSB_FREE + d), bit(dsb_ph, d) ^ 1u, w);
                if (!(ok = free_ok)) break;
                const uint32_t tile = sbase + C::OFF_DS + grp * C::DS_BYTES;
                const CUtensorMap *omap = grp == 0 ? &maps.dk : &maps.dv;
#pragma unroll 1
                for (int sl = 0; sl < D / 64; ++sl) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        uint32_t a[32];
                        tmem_ld32(lane_addr + col0 + 64 * sl + 32 * h2, a);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            pk[c] = Cvt<T>::pack(__uint_as_float(a[2 * c]) * mul,
                                                 __uint_as_float(a[2 * c + 1]) * mul);
                        // key row j: 16-byte chunk c of its 128-byte row at c ^ (j % 8)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            st_shared_v4(tile + j * 128 + (((4 * h2 + c) ^ (j & 7)) << 4), pk[4 * c],
                                         pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                    if (sl == D / 64 - 1) {
                        // the accumulators are read: the next unit may use them
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY));
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_EPI_FULL + grp));
                    if (quarter == 0) {
                        if (!(ok = mbar_wait_warp(bar(B_EPI_FULL + grp), epi_ph, w))) break;
                        if (lane == 0) {
                            tma_store_4d(omap, tile, 64 * sl, u.hk, u.k_row0 + n0, u.bidx);
                            bulk_commit_group();
                            bulk_wait_read_all();
                            mbar_arrive(bar(B_EPI_FREE + grp));
                        }
                        __syncwarp();
                    }
                    if (!(ok = mbar_wait_warp(bar(B_EPI_FREE + grp), epi_ph, w))) break;
                    epi_ph ^= 1;
                }
                if (!ok) break;
                // the other group's store has read its tile too before the next
                // unit's dS^T may land in either tile
                if (!(ok = mbar_wait_warp(bar(B_EPI_FREE + (grp ^ 1)), epi_ph ^ 1u, w))) break;
                continue;
            }
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t a[32];
                tmem_ld32(lane_addr + col0 + 32 * ch, a);
                tmem_wait_ld();
                if (key_ok) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        pk[c] = Cvt<T>::pack(__uint_as_float(a[2 * c]) * mul,
                                             __uint_as_float(a[2 * c + 1]) * mul);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (32 * ch + 8 * c < p.Dh)
                            reinterpret_cast<uint4 *>(dst + 32 * ch)[c] =
                                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace

template <int kD, typename T, int kI = 0>
static auto main_kernel_for(int need) {
    // the first instance built that has every flag needed
    constexpr int f = kMainFlagSets[kI];
    if constexpr (kI + 1 < (int)(sizeof(kMainFlagSets) / sizeof(int))) {
        if ((need & f) != need) return main_kernel_for<kD, T, kI + 1>(need);
    }
    return bwd_main_kernel<kD, T, f>;
}

template <int kD, typename T>
static cudaError_t launch_main_t(const BwdParams &p, const MainMaps &maps, int grid,
                                 cudaStream_t stream) {
    using C = MainCfg<kD, T>;
    const int need = (p.win_lo < kNoWindow ? kFBand : 0) |
                     (p.alibi ? kFAlibi | (p.win_hi > 0 ? kFAbs : 0) : 0) |
                     ((p.bias || p.dbias) ? kFBias : 0) | (p.drop_t > 0 ? kFDrop : 0);
    auto kern = main_kernel_for<kD, T>(need);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;

    kern<<<grid, C::kThreads, C::SMEM_BYTES, stream>>>(p, maps);
    return cudaGetLastError();
}

// Rows of one TMA box for Q / dO (the main kernel's BM).
int main_block_m(int D) { return D == 128 ? MainCfg<128, __nv_bfloat16>::BM : MainCfg<64, __nv_bfloat16>::BM; }

cudaError_t launch_bwd_main(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dout, const CUtensorMap &dk,
                            const CUtensorMap &dv, int bf16, int grid, cudaStream_t stream) {
    MainMaps maps{q, k, v, dout, dk, dv};
    if (p.D == 128)
        return bf16 ? launch_main_t<128, __nv_bfloat16>(p, maps, grid, stream)
                    : launch_main_t<128, __half>(p, maps, grid, stream);
    return bf16 ? launch_main_t<64, __nv_bfloat16>(p, maps, grid, stream)
                : launch_main_t<64, __half>(p, maps, grid, stream);
}

}  // namespace fa
