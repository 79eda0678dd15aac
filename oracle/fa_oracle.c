/*
 * fa_oracle.c -- fp64 CPU oracle for exact-softmax attention and its analytic
 * backward pass (dQ, dK, dV).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, per sequence b and query head h (kv head hk = h / G,
 * G = Hq / Hkv, the head-group mapping of CollectiveEpilogueBwdGQA in
 * "flash-attention/hopper/epilogue_bwd.hpp", to_underlying_arguments):
 *
 *   s_ij   = scale * <q_i, k_j>                         (STAGE 1, Q@K Gemm0 of
 *                                                        the Composable Kernel
 *                                                        page)
 *   mask   : key j is visible to query i iff j < Lk and, when causal,
 *            j <= i + (Lk - Lq)   (bottom-right alignment; the pages do not
 *            define the mask, this is the reading taken).  Optional local
 *            window (window_left wl, window_right wr, -1 = unbounded on that
 *            side): additionally i + (Lk - Lq) - wl <= j <= i + (Lk - Lq) + wr.
 *            The Composable Kernel page masks with a generic
 *            mask.IsOutOfBound(row, col) it does not print; this band, aligned
 *            like the causal mask, is the reading taken for it.
 *   ALiBi  : optional per-head slope m_h (the ALIBI bias kind of the
 *            Composable Kernel page, STAGE 2, added after the scale; the
 *            page does not print the encoding): s_ij -= m_h |i + (Lk - Lq) - j|
 *   bias   : optional elementwise bias (the ELEMENTWISE_BIAS kind of the
 *            Composable Kernel page, STAGE 2: added to the scaled score in
 *            natural-log units): s_ij += bias[b, h, i, j]; its gradient is
 *            dBias_ij = dS_ij (STAGE 5, the dbias tile is the cast ds tile)
 *   dropout: optional, with drop probability t / 256 (t = the threshold byte)
 *            and keep scale 256 / (256 - t): entry (i, j) is kept iff its
 *            random byte is >= t (the Composable Kernel page's FmhaDropout:
 *            dropped entries carry a negative P, kept ones are scaled by
 *            rp_undrop).  O_i = sum_j P_ij M_ij s v_j, dV_j = sum_i P_ij M_ij s
 *            dO_i, dS_ij = P_ij (M_ij s dP_ij - Dv_i).  The random byte of
 *            (sequence b, query head h, query i, key j) is byte j % 4 of word
 *            (j / 4) % 4 of Philox4x32-10 (Salmon et al., "Parallel random
 *            numbers: as easy as 1, 2, 3", SC 2011) with counter
 *            (j / 16, i, b * Hq + h, offset) and key (seed low, seed high);
 *            the pages print no generator, this one is the reading taken.
 *   seqused: optional per-sequence used lengths (seqused of SeqlenInfo in the
 *            FlashAttention pages): Lq = seqused_q[b], Lk = seqused_k[b]; the
 *            rows keep their places, rows past the used length are neither
 *            read nor written.
 *   LSE_i  = log sum_{visible j} exp(s_ij)   (natural log; -inf if no key is
 *            visible)
 *   P_ij   = exp(s_ij - LSE_i) on visible entries, 0 elsewhere.  A row whose
 *            LSE is -inf uses 0 instead (get_validated_lse of the Composable
 *            Kernel page); such a row has no visible entry, so P stays 0.
 *   O_i    = sum_j P_ij v_j
 *   dP_ij  = <dO_i, v_j>                                 (STAGE 4, Gemm2)
 *   Dv_i   = <dO_i, O_i>      (the preprocess quantity; derived from
 *            Dv_i = sum_j P_ij dP_ij because sum_j P_ij v_j = O_i)
 *   dS_ij  = P_ij (dP_ij - Dv_i)                         (STAGE 5)
 *   dV_j   = sum_{g in group} sum_i P_ij dO_i            (STAGE 3, Gemm1)
 *   dK_j   = scale * sum_{g in group} sum_i dS_ij q_i    (STAGE 6, Gemm3 and
 *                                                        the final dK scale)
 *   dQ_i   = scale * sum_j dS_ij k_j                     (STAGE 7, Gemm4 and
 *                                                        the QGrad scale)
 *
 * The backward takes O and LSE either from the caller (the forward's stored,
 * rounded values, as the GPU sees them) or, when those pointers are NULL,
 * computes them itself in fp64 ("fully fp64" variant).
 *
 * Head dims: D for the query / key side (q, k, dq, dk) and Dv for the value
 * side (v, o, dout, dv); Dv = D unless given (the Composable Kernel page's
 * problem traits carry the two as kQKHeaddim and kVHeaddim).  Every dot
 * product above runs over its own side's dim: <q_i, k_j> over D, <dO_i, v_j>
 * and <dO_i, O_i> over Dv.
 *
 * Layouts (row-major, d innermost, like the GPU path's public layout):
 *   dense : q, dq [B, Sq, Hq, D];  o, dout [B, Sq, Hq, Dv];
 *           k, dk [B, Sk, Hkv, D];  v, dv [B, Sk, Hkv, Dv];  lse [B, Hq, Sq]
 *   varlen: cu_q / cu_k give prefix sums of nseq = B lengths;
 *           q [total_q, Hq, D]; k [total_k, Hkv, D] (v, o, dout likewise with
 *           Dv); lse [Hq, total_q]
 *
 * Everything is a plain loop over the definition above.  Parallelism is over
 * independent output rows only (no reductions across threads), so results do
 * not depend on the thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Optional extensions; a NULL pointer means none of them. */
typedef struct {
    int window_left, window_right;  /* -1: unbounded on that side */
    const double *alibi;            /* slopes, alibi[b * alibi_bstride + h]; NULL: none */
    int alibi_bstride;
    const int *seqused_q, *seqused_k;  /* [B]; NULL: the full lengths */
    const double *bias;             /* bias[b * bias_bs + h * bias_hs + i * bias_rs + j]; NULL: none */
    long bias_bs, bias_hs, bias_rs;
    int dropout_t;                  /* threshold byte t in [0, 255]; 0: no dropout */
    unsigned long long dropout_seed;
    unsigned int dropout_offset;
    int head_dim_v;                 /* Dv, the value-side head dim; 0: equal to D */
} oracle_ext_t;

typedef struct {
    const double *q, *k, *v, *o, *dout, *lse;
    int B, Sq, Sk, Hq, Hkv, D, Dv, G;
    double scale;
    int causal;
    const int *cu_q, *cu_k;
    long total_q, total_k;
    oracle_ext_t ext;
} prob_t;

/* rows the layout reserves for sequence b */
static int stored_len_q(const prob_t *p, int b) {
    return p->cu_q ? p->cu_q[b + 1] - p->cu_q[b] : p->Sq;
}
static int stored_len_k(const prob_t *p, int b) {
    return p->cu_k ? p->cu_k[b + 1] - p->cu_k[b] : p->Sk;
}
/* rows the attention uses */
static int seq_len_q(const prob_t *p, int b) {
    return p->ext.seqused_q ? p->ext.seqused_q[b] : stored_len_q(p, b);
}
static int seq_len_k(const prob_t *p, int b) {
    return p->ext.seqused_k ? p->ext.seqused_k[b] : stored_len_k(p, b);
}
/* index of the (b, s, head) row in a [.., S, H, D] or packed [total, H, D]
 * tensor: q / dq (row_q), k / dk (row_k), o / dout (row_o, Dv wide), v / dv
 * (row_v, Dv wide) */
static long row_q(const prob_t *p, int b, int s, int h) {
    long base = p->cu_q ? (long)p->cu_q[b] + s : (long)b * p->Sq + s;
    return (base * p->Hq + h) * p->D;
}
static long row_k(const prob_t *p, int b, int s, int hk) {
    long base = p->cu_k ? (long)p->cu_k[b] + s : (long)b * p->Sk + s;
    return (base * p->Hkv + hk) * p->D;
}
static long row_o(const prob_t *p, int b, int s, int h) {
    long base = p->cu_q ? (long)p->cu_q[b] + s : (long)b * p->Sq + s;
    return (base * p->Hq + h) * p->Dv;
}
static long row_v(const prob_t *p, int b, int s, int hk) {
    long base = p->cu_k ? (long)p->cu_k[b] + s : (long)b * p->Sk + s;
    return (base * p->Hkv + hk) * p->Dv;
}
static long lse_index(const prob_t *p, int b, int s, int h) {
    if (p->cu_q) return (long)h * p->total_q + p->cu_q[b] + s;
    return ((long)b * p->Hq + h) * p->Sq + s;
}
static int visible(const prob_t *p, int b, int i, int j) {
    int lq = seq_len_q(p, b), lk = seq_len_k(p, b);
    int diag = lk - lq;
    if (j < 0 || j >= lk || i < 0 || i >= lq) return 0;
    if (p->causal && j > i + diag) return 0;
    if (p->ext.window_left >= 0 && j < i + diag - p->ext.window_left) return 0;
    if (p->ext.window_right >= 0 && j > i + diag + p->ext.window_right) return 0;
    return 1;
}
/* Philox4x32-10: ten rounds of the Philox S-box on a 128-bit counter with a
 * 64-bit key, the key bumped by the Weyl constants between rounds (Salmon et
 * al., SC 2011, section 3 and table 2). */
static void philox4x32_10(const unsigned int ctr_in[4], const unsigned int key_in[2],
                          unsigned int out[4]) {
    unsigned int c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    unsigned int k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        unsigned long long p0 = (unsigned long long)0xD2511F53u * c[0];
        unsigned long long p1 = (unsigned long long)0xCD9E8D57u * c[2];
        unsigned int hi0 = (unsigned int)(p0 >> 32), lo0 = (unsigned int)p0;
        unsigned int hi1 = (unsigned int)(p1 >> 32), lo1 = (unsigned int)p1;
        unsigned int n0 = hi1 ^ c[1] ^ k0, n1 = lo1, n2 = hi0 ^ c[3] ^ k1, n3 = lo0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

/* Dropout factor M_ij s of entry (b, h, i, j): 0 when dropped, the keep scale
 * 256 / (256 - t) when kept; 1 without dropout. */
static double dropout_factor(const prob_t *p, int b, int h, int i, int j) {
    if (p->ext.dropout_t <= 0) return 1.0;
    unsigned int ctr[4] = {(unsigned int)j >> 4, (unsigned int)i, (unsigned int)(b * p->Hq + h),
                           p->ext.dropout_offset};
    unsigned int key[2] = {(unsigned int)p->ext.dropout_seed,
                           (unsigned int)(p->ext.dropout_seed >> 32)};
    unsigned int out[4];
    philox4x32_10(ctr, key, out);
    unsigned int byte = (out[(j >> 2) & 3] >> (8 * (j & 3))) & 0xFFu;
    if ((int)byte < p->ext.dropout_t) return 0.0;
    return 256.0 / (256.0 - p->ext.dropout_t);
}

static double dot(const double *a, const double *b, int n) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += a[t] * b[t];
    return acc;
}
static double score(const prob_t *p, int b, int h, int i, int j) {
    int hk = h / p->G;
    double s = p->scale * dot(p->q + row_q(p, b, i, h), p->k + row_k(p, b, j, hk), p->D);
    if (p->ext.alibi) {
        double slope = p->ext.alibi[(long)b * p->ext.alibi_bstride + h];
        int dist = i + (seq_len_k(p, b) - seq_len_q(p, b)) - j;
        s -= slope * (double)(dist < 0 ? -dist : dist);
    }
    if (p->ext.bias)
        s += p->ext.bias[(long)b * p->ext.bias_bs + (long)h * p->ext.bias_hs +
                         (long)i * p->ext.bias_rs + j];
    return s;
}

/* Forward statistics of one query row: LSE_i (natural log) and, if o_out is
 * not NULL, O_i = sum_j P_ij v_j.  The row's scores are computed once into a
 * scratch row; the max shift is for range safety only. */
static double row_forward(const prob_t *p, int b, int h, int i, double *o_out) {
    int lk = seq_len_k(p, b), hk = h / p->G, Dv = p->Dv;
    double *s = (double *)malloc(sizeof(double) * (lk > 0 ? lk : 1));
    double m = -INFINITY;
    for (int j = 0; j < lk; ++j) {
        s[j] = visible(p, b, i, j) ? score(p, b, h, i, j) : -INFINITY;
        if (s[j] > m) m = s[j];
    }
    if (o_out) for (int d = 0; d < Dv; ++d) o_out[d] = 0.0;
    if (m == -INFINITY) { /* no visible key */
        free(s);
        return -INFINITY;
    }
    double sum = 0.0;
    for (int j = 0; j < lk; ++j)
        if (s[j] != -INFINITY) sum += exp(s[j] - m);
    double lse = m + log(sum);
    if (o_out) {
        for (int j = 0; j < lk; ++j)
            if (s[j] != -INFINITY) {
                double pij = exp(s[j] - lse);
                const double *vj = p->v + row_v(p, b, j, hk);
                double f = dropout_factor(p, b, h, i, j);
                for (int d = 0; d < Dv; ++d) o_out[d] += pij * f * vj[d];
            }
    }
    free(s);
    return lse;
}

/* The LSE the backward uses for row i (given or own), with the -inf guard. */
static double row_lse_for_backward(const prob_t *p, int b, int h, int i, double *o_scratch) {
    double lse = p->lse ? p->lse[lse_index(p, b, i, h)] : row_forward(p, b, h, i, o_scratch);
    if (lse == -INFINITY) lse = 0.0; /* get_validated_lse */
    return lse;
}

/* Dv_i = <dO_i, O_i>, O given or recomputed in fp64. */
static double row_dvec(const prob_t *p, int b, int h, int i, double *o_scratch) {
    const double *doi = p->dout + row_o(p, b, i, h);
    if (p->o) return dot(doi, p->o + row_o(p, b, i, h), p->Dv);
    row_forward(p, b, h, i, o_scratch);
    return dot(doi, o_scratch, p->Dv);
}

static double prob(const prob_t *p, int b, int h, int i, int j, double lse_i) {
    if (!visible(p, b, i, j)) return 0.0;
    return exp(score(p, b, h, i, j) - lse_i);
}
static double dprob(const prob_t *p, int b, int h, int i, int j) {
    int hk = h / p->G;
    return dot(p->dout + row_o(p, b, i, h), p->v + row_v(p, b, j, hk), p->Dv);
}

/* dQ_i = scale * sum_j P_ij (dP_ij - Dv_i) k_j */
static void row_dq(const prob_t *p, int b, int h, int i, double *dq_out, double *scratch) {
    int lk = seq_len_k(p, b), hk = h / p->G, D = p->D;
    double lse = row_lse_for_backward(p, b, h, i, scratch);
    double dv = row_dvec(p, b, h, i, scratch);
    for (int d = 0; d < D; ++d) dq_out[d] = 0.0;
    for (int j = 0; j < lk; ++j) {
        double pij = prob(p, b, h, i, j, lse);
        if (pij == 0.0) continue;
        double ds = pij * (dropout_factor(p, b, h, i, j) * dprob(p, b, h, i, j) - dv);
        const double *kj = p->k + row_k(p, b, j, hk);
        for (int d = 0; d < D; ++d) dq_out[d] += ds * kj[d];
    }
    for (int d = 0; d < D; ++d) dq_out[d] *= p->scale;
}

/* dK_j, dV_j for key row j of kv head hk, summed over the G query heads of the
 * group.  lse_g / dvec_g hold, for each head g of the group, the per-row LSE
 * (already guarded) and Dv of sequence b. */
static void col_dkdv(const prob_t *p, int b, int hk, int j, double *const *lse_g,
                     double *const *dvec_g, double *dk_out, double *dv_out) {
    int lq = seq_len_q(p, b), D = p->D, Dv = p->Dv;
    for (int d = 0; d < D; ++d) dk_out[d] = 0.0;
    for (int d = 0; d < Dv; ++d) dv_out[d] = 0.0;
    for (int g = 0; g < p->G; ++g) {
        int h = hk * p->G + g;
        for (int i = 0; i < lq; ++i) {
            double pij = prob(p, b, h, i, j, lse_g[g][i]);
            if (pij == 0.0) continue;
            const double *doi = p->dout + row_o(p, b, i, h);
            const double *qi = p->q + row_q(p, b, i, h);
            double f = dropout_factor(p, b, h, i, j);
            double ds = pij * (f * dprob(p, b, h, i, j) - dvec_g[g][i]);
            for (int d = 0; d < Dv; ++d) dv_out[d] += pij * f * doi[d];
            for (int d = 0; d < D; ++d) dk_out[d] += ds * qi[d];
        }
    }
    for (int d = 0; d < D; ++d) dk_out[d] *= p->scale;
}

/* Per-row LSE (guarded) and Dv for every query row of the G heads of (b, hk). */
static void group_row_stats(const prob_t *p, int b, int hk, double **lse_g, double **dvec_g,
                            int nthreads) {
    int lq = seq_len_q(p, b);
    for (int g = 0; g < p->G; ++g) {
        int h = hk * p->G + g;
        double *lse = lse_g[g], *dvec = dvec_g[g];
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
        for (int i = 0; i < lq; ++i) {
            double *scratch = (double *)malloc(sizeof(double) * p->Dv);
            if (!p->lse && !p->o) {
                /* own forward: LSE and O of the row from one pass */
                double l = row_forward(p, b, h, i, scratch);
                lse[i] = (l == -INFINITY) ? 0.0 : l; /* get_validated_lse */
                dvec[i] = dot(p->dout + row_o(p, b, i, h), scratch, p->Dv);
            } else {
                lse[i] = row_lse_for_backward(p, b, h, i, scratch);
                dvec[i] = row_dvec(p, b, h, i, scratch);
            }
            free(scratch);
        }
    }
}

static int make_prob(prob_t *p, const double *q, const double *k, const double *v,
                     const double *o, const double *lse, const double *dout, int B, int Sq,
                     int Sk, int Hq, int Hkv, int D, double scale, int causal, const int *cu_q,
                     const int *cu_k, const oracle_ext_t *ext) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    if ((cu_q == NULL) != (cu_k == NULL)) return 1;
    p->q = q; p->k = k; p->v = v; p->o = o; p->lse = lse; p->dout = dout;
    p->B = B; p->Sq = Sq; p->Sk = Sk; p->Hq = Hq; p->Hkv = Hkv; p->D = D; p->G = Hq / Hkv;
    p->scale = scale; p->causal = causal; p->cu_q = cu_q; p->cu_k = cu_k;
    p->total_q = cu_q ? cu_q[B] : (long)B * Sq;
    p->total_k = cu_k ? cu_k[B] : (long)B * Sk;
    memset(&p->ext, 0, sizeof(p->ext));
    p->ext.window_left = p->ext.window_right = -1;
    if (ext) p->ext = *ext;
    if (p->ext.window_left < -1 || p->ext.window_right < -1) return 1;
    if (p->ext.dropout_t < 0 || p->ext.dropout_t > 255) return 1;
    if (p->ext.head_dim_v < 0) return 1;
    p->Dv = p->ext.head_dim_v > 0 ? p->ext.head_dim_v : D;
    for (int b = 0; b < B; ++b) {
        if (p->ext.seqused_q &&
            (p->ext.seqused_q[b] < 0 || p->ext.seqused_q[b] > stored_len_q(p, b)))
            return 1;
        if (p->ext.seqused_k &&
            (p->ext.seqused_k[b] < 0 || p->ext.seqused_k[b] > stored_len_k(p, b)))
            return 1;
    }
    return 0;
}

/* ---------------------------------------------------------------- public */

int oracle_forward(const double *q, const double *k, const double *v, int B, int Sq, int Sk,
                   int Hq, int Hkv, int D, double scale, int causal, const int *cu_q,
                   const int *cu_k, double *o, double *lse, int nthreads,
                   const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, q, k, v, NULL, NULL, NULL, B, Sq, Sk, Hq, Hkv, D, scale, causal, cu_q,
                  cu_k, ext))
        return 1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            int lq = seq_len_q(&p, b);
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
            for (int i = 0; i < lq; ++i)
                lse[lse_index(&p, b, i, h)] = row_forward(&p, b, h, i, o + row_o(&p, b, i, h));
        }
    return 0;
}

/* Full backward.  o / lse may be NULL (then the oracle's own fp64 forward is
 * used).  dq has q's layout, dk k's, dv v's. */
int oracle_backward(const double *q, const double *k, const double *v, const double *o,
                    const double *lse, const double *dout, int B, int Sq, int Sk, int Hq,
                    int Hkv, int D, double scale, int causal, const int *cu_q, const int *cu_k,
                    double *dq, double *dk, double *dv, int nthreads,
                    const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, q, k, v, o, lse, dout, B, Sq, Sk, Hq, Hkv, D, scale, causal, cu_q, cu_k,
                  ext))
        return 1;
    double **lse_g = (double **)malloc(sizeof(double *) * p.G);
    double **dvec_g = (double **)malloc(sizeof(double *) * p.G);
    for (int b = 0; b < B; ++b) {
        int lq = seq_len_q(&p, b), lk = seq_len_k(&p, b);
        for (int g = 0; g < p.G; ++g) {
            lse_g[g] = (double *)malloc(sizeof(double) * (lq > 0 ? lq : 1));
            dvec_g[g] = (double *)malloc(sizeof(double) * (lq > 0 ? lq : 1));
        }
        for (int h = 0; h < Hq; ++h) {
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
            for (int i = 0; i < lq; ++i) {
                double *scratch = (double *)malloc(sizeof(double) * p.Dv);
                row_dq(&p, b, h, i, dq + row_q(&p, b, i, h), scratch);
                free(scratch);
            }
        }
        for (int hk = 0; hk < Hkv; ++hk) {
            group_row_stats(&p, b, hk, lse_g, dvec_g, nthreads);
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
            for (int j = 0; j < lk; ++j)
                col_dkdv(&p, b, hk, j, lse_g, dvec_g, dk + row_k(&p, b, j, hk),
                         dv + row_v(&p, b, j, hk));
        }
        for (int g = 0; g < p.G; ++g) { free(lse_g[g]); free(dvec_g[g]); }
    }
    free(lse_g);
    free(dvec_g);
    return 0;
}

/* Sampled backward: dQ for n_qrows query rows given as (b, s, h) triples, and
 * dK / dV for n_krows key rows given as (b, s, hk) triples.  Outputs are
 * packed [n, D] (dV rows [n, Dv]).  Each requested row is computed exactly as
 * in the full backward. */
int oracle_backward_sampled(const double *q, const double *k, const double *v, const double *o,
                            const double *lse, const double *dout, int B, int Sq, int Sk, int Hq,
                            int Hkv, int D, double scale, int causal, const int *cu_q,
                            const int *cu_k, int n_qrows, const int *qrows, double *dq_rows,
                            int n_krows, const int *krows, double *dk_rows, double *dv_rows,
                            int nthreads, const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, q, k, v, o, lse, dout, B, Sq, Sk, Hq, Hkv, D, scale, causal, cu_q, cu_k,
                  ext))
        return 1;
    for (int r = 0; r < n_qrows; ++r) {
        int b = qrows[3 * r], s = qrows[3 * r + 1], h = qrows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || s < 0 || s >= seq_len_q(&p, b)) return 2;
    }
    for (int r = 0; r < n_krows; ++r) {
        int b = krows[3 * r], s = krows[3 * r + 1], hk = krows[3 * r + 2];
        if (b < 0 || b >= B || hk < 0 || hk >= Hkv || s < 0 || s >= seq_len_k(&p, b)) return 2;
    }
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int r = 0; r < n_qrows; ++r) {
        double *scratch = (double *)malloc(sizeof(double) * p.Dv);
        row_dq(&p, qrows[3 * r], qrows[3 * r + 2], qrows[3 * r + 1], dq_rows + (long)r * D,
               scratch);
        free(scratch);
    }
    /* key rows: group by (b, hk) so that the per-row statistics of each group
     * are computed once */
    char *done = (char *)calloc(n_krows > 0 ? n_krows : 1, 1);
    double **lse_g = (double **)malloc(sizeof(double *) * p.G);
    double **dvec_g = (double **)malloc(sizeof(double *) * p.G);
    for (int r0 = 0; r0 < n_krows; ++r0) {
        if (done[r0]) continue;
        int b = krows[3 * r0], hk = krows[3 * r0 + 2], lq = seq_len_q(&p, b);
        for (int g = 0; g < p.G; ++g) {
            lse_g[g] = (double *)malloc(sizeof(double) * (lq > 0 ? lq : 1));
            dvec_g[g] = (double *)malloc(sizeof(double) * (lq > 0 ? lq : 1));
        }
        group_row_stats(&p, b, hk, lse_g, dvec_g, nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
        for (int r = r0; r < n_krows; ++r) {
            if (krows[3 * r] != b || krows[3 * r + 2] != hk) continue;
            col_dkdv(&p, b, hk, krows[3 * r + 1], lse_g, dvec_g, dk_rows + (long)r * D,
                     dv_rows + (long)r * p.Dv);
            done[r] = 1;
        }
        for (int g = 0; g < p.G; ++g) { free(lse_g[g]); free(dvec_g[g]); }
    }
    free(done);
    free(lse_g);
    free(dvec_g);
    return 0;
}

/* The preprocess quantities of every query row: Dv_i = <dO_i, O_i> (O given,
 * or the oracle's own when NULL) and the guarded natural-log LSE the
 * backward uses.  Outputs have lse's layout. */
int oracle_preprocess(const double *q, const double *k, const double *v, const double *o,
                      const double *lse, const double *dout, int B, int Sq, int Sk, int Hq,
                      int Hkv, int D, double scale, int causal, const int *cu_q, const int *cu_k,
                      double *dvec_out, double *lse_out, int nthreads,
                      const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, q, k, v, o, lse, dout, B, Sq, Sk, Hq, Hkv, D, scale, causal, cu_q, cu_k,
                  ext))
        return 1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            int lq = seq_len_q(&p, b);
#pragma omp parallel for schedule(dynamic, 8) num_threads(nthreads)
            for (int i = 0; i < lq; ++i) {
                double *scratch = (double *)malloc(sizeof(double) * p.Dv);
                long li = lse_index(&p, b, i, h);
                lse_out[li] = row_lse_for_backward(&p, b, h, i, scratch);
                dvec_out[li] = row_dvec(&p, b, h, i, scratch);
                free(scratch);
            }
        }
    return 0;
}

/* Dense P and dS of one (b, h) head problem, row-major [Lq, Lk] -- for the
 * invariant checks on tiny inputs. */
int oracle_head_matrices(const double *q, const double *k, const double *v, const double *o,
                         const double *lse, const double *dout, int B, int Sq, int Sk, int Hq,
                         int Hkv, int D, double scale, int causal, const int *cu_q,
                         const int *cu_k, int b, int h, double *P, double *dS,
                         const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, q, k, v, o, lse, dout, B, Sq, Sk, Hq, Hkv, D, scale, causal, cu_q, cu_k,
                  ext))
        return 1;
    int lq = seq_len_q(&p, b), lk = seq_len_k(&p, b);
    double *scratch = (double *)malloc(sizeof(double) * p.Dv);
    for (int i = 0; i < lq; ++i) {
        double l = row_lse_for_backward(&p, b, h, i, scratch);
        double dvec = row_dvec(&p, b, h, i, scratch);
        for (int j = 0; j < lk; ++j) {
            double pij = prob(&p, b, h, i, j, l);
            P[(long)i * lk + j] = pij;
            dS[(long)i * lk + j] = pij * (dropout_factor(&p, b, h, i, j) * dprob(&p, b, h, i, j) - dvec);
        }
    }
    free(scratch);
    return 0;
}

/* Philox4x32-10 of one counter and key, for the known-answer pins. */
void oracle_philox4x32_10(const unsigned int *ctr, const unsigned int *key, unsigned int *out) {
    philox4x32_10(ctr, key, out);
}

/* The dropout factor M s of every (i, j) of one head problem, [Lq, Lk]. */
int oracle_dropout_factors(int B, int Sq, int Sk, int Hq, int Hkv, int D, const int *cu_q,
                           const int *cu_k, int b, int h, double *F, const oracle_ext_t *ext) {
    prob_t p;
    if (make_prob(&p, NULL, NULL, NULL, NULL, NULL, NULL, B, Sq, Sk, Hq, Hkv, D, 1.0, 0, cu_q, cu_k,
                  ext))
        return 1;
    int lq = seq_len_q(&p, b), lk = seq_len_k(&p, b);
    for (int i = 0; i < lq; ++i)
        for (int j = 0; j < lk; ++j) F[(long)i * lk + j] = dropout_factor(&p, b, h, i, j);
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
