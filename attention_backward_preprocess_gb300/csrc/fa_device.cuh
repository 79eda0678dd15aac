// fa_device.cuh -- sm_103a device primitives written as inline PTX:
// mbarriers with bounded waits, TMA (tensor and plain bulk copies), tcgen05
// tensor-memory allocation, MMA issue, commit, and TMEM loads / stores, and the
// shared-memory matrix / instruction descriptors of tcgen05.mma.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ------------------------------------------------------------------ errors
// Device error word bits (the host reports kErrBadLength as FA_ERR_INVALID_ARG,
// any other non-zero value as FA_ERR_TIMEOUT).
enum : int {
    kErrWaitTimeout = 1,       // an mbarrier wait ran out
    kErrSemaphoreTimeout = 2,  // a deterministic-order semaphore wait ran out
    kErrBadLength = 4,         // a varlen sequence longer than the maximum given, or
                               // cu_seqlens[B] different from the packed total given
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared state every warp consults while it waits: a CTA-wide abort flag in
// shared memory (set by whichever warp gives up first, so the others stop
// waiting for it), the global error word and the wait budget.
struct WaitCtl {
    volatile int *abort_flag;  // shared memory
    int *err;                  // global
    long long budget_ns;
};

__device__ __forceinline__ void raise_error(const WaitCtl &w, int bit) {
    *w.abort_flag = 1;
    atomicOr(w.err, bit);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
// count arrivals at once
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            bar),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Packed fp32 pairs (two lanes of one 64-bit register): the f32x2 forms of
// fma / sub / mul issue one instruction per pair, each lane rounded as the
// scalar instruction would be.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Four 8x8 16-bit matrices into shared memory: register i of thread t is
// row t/4, elements 2(t%4), 2(t%4)+1 of matrix i; thread t supplies the
// address of row t%8 of matrix t/8.
__device__ __forceinline__ void stmatrix_x4(uint32_t row_addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                            uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(row_addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// The same four 8x8 matrices stored transposed: element (row t/4, column
// 2(t%4) + e) of matrix i lands in row 2(t%4) + e, column t/4 of it; thread
// t supplies the address of (transposed) row t%8 of matrix t/8.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t row_addr, uint32_t r0, uint32_t r1,
                                                  uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(
                     row_addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// Four 8x8 16-bit matrices from shared memory, transposed: register i of
// thread t holds elements (row 2(t%4) + e, column t/4), e = 0 (low half) and
// 1, of matrix i; thread t supplies the address of row t%8 of matrix t/8.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t row_addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(row_addr)
                 : "memory");
}

// Warp-wide exchanges that move one bit of an element's position between the
// lane index and its place in the thread's registers (transposes across
// lanes).  Lane bit `mask` trades places with the register bit that selects
// x1 over x0: afterwards a lane whose bit is 0 holds, in x0 / x1, what lanes
// without / with the bit held in x0, and a lane whose bit is set what they
// held in x1.  `set` is (lane & mask) != 0.
__device__ __forceinline__ void xchg_lane_reg(uint32_t &x0, uint32_t &x1, int mask, bool set) {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, set ? x0 : x1, mask);
    if (set) x0 = r;
    else x1 = r;
}
// The same with the 16-bit half of a word: afterwards a lane whose bit is 0
// holds the low halves of itself and its partner (low: the lane without the
// bit), a lane whose bit is set their high halves.
__device__ __forceinline__ uint32_t xchg_lane_half(uint32_t w, int mask, bool set) {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, w, mask);
    return set ? __byte_perm(w, r, 0x3276) : __byte_perm(w, r, 0x5410);
}

// Shared-memory accesses by 32-bit shared-window address (base + immediate
// offsets; no generic-address conversion).
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ float2 ld_shared_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// Bounded slow path of mbar_wait, kept out of line so the common case (the
// phase has already completed) costs one try_wait and a branch.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            int *err, long long budget_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((long long)(globaltimer_ns() - t0) > budget_ns) {
            *abort_flag = 1;
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}
// Wind-down wait: the phase with the given parity of a barrier that tracks
// this CTA's own asynchronous work (MMAs, TMA loads) already issued.  Unlike
// mbar_wait it does not give up when the CTA aborts -- that work must finish
// before tensor memory is freed or the CTA exits -- but it is still bounded
// by the budget (then it raises the error and returns false).
static __device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int *err,
                                                    long long budget_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if ((long long)(globaltimer_ns() - t0) > budget_ns) {
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}
// Waits until the phase with the given parity has completed.  Bounded: gives
// up (returns false) when another warp has aborted or the budget runs out
// (then raises the error itself).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &w) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w.abort_flag, w.err, w.budget_ns);
}

// ------------------------------------------------- global-memory semaphores
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A release fence at GPU scope followed by relaxed adds: each add is then a
// release of everything before the fence (the fence-then-strong-write release
// pattern of the PTX memory model), and several adds share one fence.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void red_relaxed_add_gpu(int *p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Fire-and-forget fp32 add in global memory (no value returned).
__device__ __forceinline__ void red_add_f32(float *p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
// Single-thread bounded wait until *sem >= target (acquire).  Returns false
// if another warp aborted or the budget ran out (then raises the error).
__device__ __forceinline__ bool sem_wait_geq(const int *sem, int target, const WaitCtl &w) {
    if (ld_acquire_gpu(sem) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(32);
        if (ld_acquire_gpu(sem) >= target) return true;
        if (*w.abort_flag) return false;
        if ((long long)(globaltimer_ns() - t0) > w.budget_ns) {
            raise_error(w, kErrSemaphoreTimeout);
            return false;
        }
    }
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}
// 4-D tiled load (coordinates innermost first) completing on an mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(m), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
// 4-D tiled store shared -> global (coordinates innermost first) in this
// thread's bulk group; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     m),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Bulk reduce-add of a contiguous shared-memory block into global memory (fp32
// add performed by the TMA unit; both addresses 16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_reduce_add_f32(float *dst, uint32_t src, uint32_t bytes) {
    asm volatile(
        "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
        "r"(src), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk operation of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Same, but allow the most recent committed group to still be reading.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until every committed bulk operation of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Same, but allow the N most recent committed groups to be still in progress.
template <int N>
__device__ __forceinline__ void bulk_wait_all_but() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's async-proxy (TMA) global accesses with its generic ones.
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma, TMA).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05
// TMEM addresses: bits 31..16 lane, bits 15..0 column.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Warp-wide forms: the whole warp executes them in converged control flow and
// elect.sync picks one lane (always the same, the lowest active) to issue, so
// the operands stay warp-uniform.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            bar)
        : "memory");
}
// Bounded wait of a whole converged warp: every lane probes once (one
// instruction, one barrier state); only if that fails does lane 0 wait and
// broadcast the outcome, so the warp stays converged.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtl &w) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait_slow(bar, parity, w.abort_flag, w.err, w.budget_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// mbar_wait_drain for a whole converged warp (lane 0 waits, the outcome is
// broadcast).
__device__ __forceinline__ bool mbar_wait_drain_warp(uint32_t bar, uint32_t parity, int *err,
                                                     long long budget_ns) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_drain(bar, parity, err, budget_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Arrive on an mbarrier once every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32 bits: thread t of the warp gets columns
// [col, col+32) of lane (lane_base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// 16 lanes x 256 bits (8 columns), 4 repetitions along the columns: with
// g = t / 4 and q = t % 4, register 4k + e of thread t holds lane
// lane_base + g + 8 * (e / 2), column col + 8k + 2q + (e % 2) -- the
// accumulator fragment of a 16x8 mma tile, so a thread sees 8 columns of 2
// lanes instead of 32 columns of 1.
__device__ __forceinline__ void tmem_ld16x256(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 16 lanes x 128 bits (4 columns), 4 repetitions: register 2k + e of thread t
// goes to lane lane_base + t / 4 + 8e, column col + 4k + t % 4.  With 16-bit
// pairs packed per column this is the same (lane, element) set as
// tmem_ld16x256 reads from a 32-bit matrix.
// The 16x128b shape read back: the registers tmem_st16x128 wrote.
__device__ __forceinline__ void tmem_ld16x128(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.16x128b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_st16x128(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// Shared-memory matrix descriptor of tcgen05.mma for a 128-byte-swizzled
// operand (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B: rows of 128
// bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8), 8-row atoms of
// 1024 bytes).  Fields: start address >> 4 (bits 0-13), leading byte offset
// >> 4 (16-29), stride byte offset >> 4 (32-45), descriptor version 1
// (46-47), base offset 0 (49-51, atoms are 1024-byte aligned), swizzle mode
// 2 = 128B (61-63).
//  K-major operand : rows are M/N, 64 K-elements per row; SBO = 1024 (next 8
//                    rows); LBO unused; a K step of 16 elements adds 32 bytes.
//  MN-major operand: rows are K, 64 M/N-elements per row; SBO = 1024 (next
//                    8 K-rows); LBO = byte distance to the next 64 M/N
//                    elements; a K step of 16 adds 2048 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// The descriptor of (base address + bytes): the start address sits in the low
// 14 bits as address >> 4 and shared-memory addresses stay below 256 KB, so
// an offset is one add with no carry into the other fields.  Lets the MMA
// issuer build a descriptor per operand tile once and step through K with
// compile-time offsets.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
    return desc + (uint64_t)(bytes >> 4);
}

// Instruction descriptor of tcgen05.mma.kind::f16 with an fp32 accumulator:
// D format f32 (bits 4-5 = 1), A / B format (7-9 / 10-12: 0 fp16, 1 bf16),
// A / B major (15 / 16: 0 K-major, 1 MN-major), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool bf16, bool a_mn, bool b_mn) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------ conversions
template <typename T> struct Cvt;
template <> struct Cvt<__nv_bfloat16> {
    // two fp32 -> packed pair, lo in the low half (round to nearest even)
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    }
    static constexpr bool is_bf16 = true;
};
template <> struct Cvt<__half> {
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ float2 unpack(uint32_t u) {
        __half2 h = *reinterpret_cast<__half2 *>(&u);
        return __half22float2(h);
    }
    static constexpr bool is_bf16 = false;
};

// Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011): ten rounds of the S-box (two 32x32 -> 64-bit products of
// counter words 0 and 2, the high halves xor-ed into words 1 and 3 with the
// round key), the key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace fa
