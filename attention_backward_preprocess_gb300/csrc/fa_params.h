// fa_params.h -- host/device parameter block of the backward kernels and the
// workspace row mapping they share.
#pragma once

#include <cstdint>

namespace fa {

constexpr int kRowTile = 128;   // workspace rows are padded per (sequence, head) to this
constexpr int kBlockN = 128;    // keys per work unit of the main kernel
constexpr int kNoWindow = 1 << 30;   // an unbounded side of the visible band

struct BwdParams {
    // tensors (public layouts, see fa.h)
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int B, Sq, Sk, Hq, Hkv, D, G;
    int Dh;             // head dim of the tensors; D is the tile width it is padded to
                        // (64, 128 or 256: columns past Dh are zero in shared memory)
    int Dv, Dhv;        // the value side (v, o, dout, dv): tile width and head dim
                        // (equal to D / Dh unless the value head dim differs)
    float scale;        // c
    float scale_log2;   // c * log2(e)
    int causal, deterministic, varlen;
    const int *cu_q, *cu_k;
    // varlen: the packed row counts the tensor maps were built for; the
    // kernels check them against cu_q[B] / cu_k[B] before touching a row
    long long total_q, total_k;
    // Visible band: key j is visible to query i iff j < Lk and
    // -win_lo <= j - i - (Lk - Lq) <= win_hi (kNoWindow: unbounded; a causal
    // mask makes win_hi <= 0).
    int win_lo, win_hi;
    // ALiBi: slope alibi[b * alibi_bstride + h] (natural-log units), the score
    // gets -slope * |i + (Lk - Lq) - j|; null: none
    const float *alibi;
    int alibi_bstride;
    // used lengths per sequence (null: the stored lengths); clamped to
    // [0, stored length]
    const int *seqused_q, *seqused_k;
    // elementwise bias (dense problems; input dtype), natural-log units:
    // bias[b * bias_bs + h * bias_hs + i * bias_rs + j]; null: none
    const void *bias;
    long long bias_bs, bias_hs, bias_rs;
    // backward: dBias = dS written as [B, Hq, Sq, Sk] (input dtype); null: not
    void *dbias;
    // dropout: entry (b, h, i, j) kept iff byte j % 4 of word (j / 4) % 4 of
    // Philox4x32-10(counter (j / 16, i, b * Hq + h, drop_offset), key
    // (drop_key0, drop_key1)) is >= drop_t; kept entries scaled by drop_scale
    // = 256 / (256 - drop_t).  drop_t = 0: no dropout
    int drop_t;
    uint32_t drop_key0, drop_key1, drop_offset;
    float drop_scale;
    // optional keep flags as bits (null: none): word w of query row r (the
    // LSE row order: (b * Hq + h) * Sq + i, varlen h * total_q + cu_q[b] + i)
    // at drop_mask[r * drop_mask_w + w], bit l = key 32 w + l kept.  The
    // forward writes the words of the key blocks it visits; the backward reads
    // them instead of drawing the mask again.
    uint32_t *drop_mask;
    int drop_mask_w;
    // workspace
    int *err;           // device error word
    int4 *tiles;        // work units (b, n_block, hk, 0)
    int *ntiles;        // varlen: number of work units written by the scheduler
    int num_units;      // dense: B * ceil(Sk / 128) * Hkv work units
    int unit_group;     // dense: (batch, kv head) pairs per group of the unit order,
                        // divides B * Hkv; varlen: units per group of sequences
                        // (0: no groups)
    int *unit_counter;  // [0] next work unit to hand out, [1] CTAs that ran out;
                        // reset by the last CTA of each launch (and by the preprocess)
    int max_tiles;
    float *dvec;        // Dv per workspace row
    float *lse2;        // LSE * log2(e) per workspace row (+inf on padding rows)
    float *dqacc;       // fp32 dQ accumulator [rows, D]
    int *sem;           // deterministic-order semaphores, one per 64 workspace rows
    long long rows;     // workspace rows
    long long rows_per_head;  // varlen: rows of one head; dense: round_up(Sq, 128)
    int sq_round;       // round_up(Sq, 128)
    long long budget_ns;      // bound of every device-side wait
};

// Varlen: cu_seqlens agree with the packed totals and with the maximum
// lengths the workspace was planned for (Sq / Sk), for sequence b.  A call
// where this fails reports kErrBadLength, and no kernel touches the
// sequence's rows.
__device__ __forceinline__ bool varlen_seq_ok(const BwdParams &p, int b) {
    if (p.cu_q[p.B] != p.total_q || p.cu_k[p.B] != p.total_k) return false;
    const int lq = p.cu_q[b + 1] - p.cu_q[b], lk = p.cu_k[b + 1] - p.cu_k[b];
    return lq >= 0 && lk >= 0 && lq <= p.Sq && lk <= p.Sk;
}

// Rows of sequence b the attention uses (query / key side).
__device__ __forceinline__ int used_len_q(const BwdParams &p, int b) {
    const int stored = p.varlen ? p.cu_q[b + 1] - p.cu_q[b] : p.Sq;
    return p.seqused_q ? min(max(p.seqused_q[b], 0), stored) : stored;
}
__device__ __forceinline__ int used_len_k(const BwdParams &p, int b) {
    const int stored = p.varlen ? p.cu_k[b + 1] - p.cu_k[b] : p.Sk;
    return p.seqused_k ? min(max(p.seqused_k[b], 0), stored) : stored;
}

// Workspace row of (sequence b, query head h, position s).
__device__ __forceinline__ long long ws_row(const BwdParams &p, int b, int h, int s) {
    if (p.varlen) {
        long long pad = ((long long)p.cu_q[b] + (long long)b * kRowTile) / kRowTile * kRowTile;
        return (long long)h * p.rows_per_head + pad + s;
    }
    return ((long long)b * p.Hq + h) * p.sq_round + s;
}

}  // namespace fa
