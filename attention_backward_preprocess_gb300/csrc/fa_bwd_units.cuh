// fa_bwd_units.cuh -- the work units of the backward main kernels and the
// shared-memory ring that hands them from the producer warp to the others.
#pragma once

#include "fa_device.cuh"
#include "fa_params.h"

namespace fa {

// Work units are handed out dynamically: the producer warp takes the next
// index from a global counter and passes it to the other warps of the CTA
// through a small ring in shared memory.  Dense units leave the counter group
// by group of (sequence, kv head) pairs, n_block-major inside a group, so the
// units that run at the same time sweep the same rows of Q, dO and the dQ
// accumulator in L2; idle CTAs take the next unit, which balances the uneven
// causal work.  -1 ends the sequence.
struct UnitRing {
    volatile int *slot;   // kRing ints in shared memory
    uint32_t full0, empty0;
    int k = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void advance(int ring) {
        if (++k == ring) { k = 0; ph ^= 1; }
    }
};

__device__ __forceinline__ uint32_t bit(uint32_t mask, int b) { return (mask >> b) & 1u; }

struct Unit {
    int b, n_block, hk;
    int lq, lk;
    int q_row0, k_row0, bidx;   // TMA row offset and batch coordinate
    int m_begin, nm, iters;     // row blocks [m_begin, m_begin + nm) per head; iters = G * nm
    // Iteration order: row blocks from the last to the first, the G query
    // heads of the group innermost.  Under a causal mask every unit of a
    // (sequence, kv head) starts at the same last row block, so the units
    // that run side by side sweep the same Q / dO / dQ-accumulator rows
    // together and share them in L2.
    __device__ __forceinline__ int g_of(int it, int G) const { return it % G; }
    __device__ __forceinline__ int m_of(int it, int G) const { return m_begin + nm - 1 - it / G; }
};

// Work unit t: dense problems enumerate groups of (batch, kv head) pairs,
// then n_block, then the pair inside the group; varlen problems read the list
// the scheduler kernel wrote.
template <int BM>
__device__ __forceinline__ Unit decode_unit(const BwdParams &p, int t) {
    Unit u;
    if (p.varlen) {
        const int4 e = p.tiles[t];
        u.b = e.x;
        u.n_block = e.y;
        u.hk = e.z;
        u.q_row0 = p.cu_q[u.b];
        u.k_row0 = p.cu_k[u.b];
        u.lq = used_len_q(p, u.b);
        u.lk = used_len_k(p, u.b);
        u.bidx = 0;
    } else {
        // groups of unit_group (batch, kv head) pairs, one after the other;
        // inside a group the n blocks in increasing order (longest causal
        // units first), the pairs of the group interleaved.  Units that run at
        // the same time then share their dQ / Q / dO rows in L2.
        const int gs = p.unit_group;
        const int nblk = p.num_units / (p.B * p.Hkv);
        const int grp = t / (gs * nblk);
        const int r = t - grp * gs * nblk;
        u.n_block = r / gs;
        const int bh = grp * gs + (r - u.n_block * gs);
        u.b = bh / p.Hkv;
        u.hk = bh - u.b * p.Hkv;
        u.q_row0 = 0;
        u.k_row0 = 0;
        u.lq = used_len_q(p, u.b);
        u.lk = used_len_k(p, u.b);
        u.bidx = u.b;
    }
    // queries that see a key of [n0, n0 + kBlockN): i >= n0 - diag - win_hi
    // (the first key against the upper edge of the band) and
    // i <= n0 + kBlockN - 1 - diag + win_lo (the last key against the lower edge)
    const int n0 = u.n_block * kBlockN;
    const long long diag = u.lk - u.lq;
    const long long first_row = max(0LL, (long long)n0 - diag - p.win_hi);
    const long long last_row = min((long long)u.lq - 1, (long long)n0 + kBlockN - 1 - diag + p.win_lo);
    u.m_begin = (int)min(first_row / BM, (long long)(u.lq + BM - 1) / BM);
    u.nm = last_row < first_row ? 0 : (int)(last_row / BM + 1 - u.m_begin);
    if (n0 >= u.lk) u.nm = 0;
    u.iters = p.G * u.nm;
    return u;
}

// First key block with a key that some query of the rows [m0, ...) of a
// sequence can see: the block holding key m0 + diag - win_lo.  A row block
// receives dQ contributions from the key blocks n_first, n_first + 1, ... in
// turn, so in deterministic mode the unit of key block n waits until its row
// block's semaphore counts n - n_first earlier contributions.
__device__ __forceinline__ int first_key_block(const BwdParams &p, int m0, int diag) {
    const long long j = (long long)m0 + diag - p.win_lo;
    return j <= 0 ? 0 : (int)(j / kBlockN);
}

}  // namespace fa
