/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused exact-softmax attention backward.
 *
 * The backward of O = softmax(Q K^T * scale + mask) V, given the forward's O
 * and per-row log-sum-exp LSE, produces dQ, dK, dV without materialising the
 * S x S probability matrix.  It runs as three kernels in stream order:
 *
 *   1. preprocess   Dv_i = sum_d dO_id * O_id (fp32), LSE2_i = LSE_i * log2(e)
 *                   (LSE = -inf replaced by 0, the get_validated_lse guard of
 *                   the Composable Kernel page
 *                   "block_fmha_bwd_dq_dk_dv_pipeline_trload_kr_ktr_vr.hpp"),
 *                   zero the fp32 dQ accumulator (CollectiveEpilogueBwdGQA's
 *                   "already zero-initialized" precondition in
 *                   "flash-attention/hopper/epilogue_bwd.hpp").
 *   2. main         one work unit per (K/V column block of 128 keys, batch,
 *                   kv head): recompute S and P = exp2(S*scale*log2e - LSE2)
 *                   (STAGE 1-2 of the Composable Kernel page), dV += P^T dO
 *                   (STAGE 3), dP = dO V^T (STAGE 4), dS = P o (dP - Dv)
 *                   (STAGE 5), dK += dS^T Q (STAGE 6, scaled at the end),
 *                   dQ += dS K (STAGE 7) into the fp32 accumulator; dK / dV
 *                   summed over the query heads of a GQA group.
 *   3. postprocess  dQ = cast(dQaccum * scale) (FlashAttentionBackwardPostprocess
 *                   of "flash_bwd_postprocess.py").
 *
 * Layouts (all contiguous, d innermost, CollectiveEpilogueBwd's
 * (seqlen, d, head, batch) shape with stride (int64, 1, int64, int64)):
 *   dense : q, o, dout, dq : [B, Sq, Hq, D];  k, v, dk, dv : [B, Sk, Hkv, D]
 *           lse : fp32 [B, Hq, Sq], natural log
 *   D is a multiple of 8 in [64, 256]; it runs at the tile width 64 (D = 64),
 *   128 (D <= 128) or 256, the tensor-map loads filling the columns past D
 *   with zeros (the FlashAttention postprocess page pads the head dim
 *   likewise).  Head dims up to 128 run in the main kernel (64 queries x 128
 *   keys per step); above 128, and for a value head dim different from D
 *   (fa_ext head_dim_v: v, o, dout, dv then have Dv columns), in a second
 *   kernel that produces dK / dV / dQ in 128-column halves (32 queries x 128
 *   keys per step, S and dP recomputed per half).  That kernel has the causal
 *   mask, both band edges of a local window, varlen and used lengths, but
 *   not ALiBi, the bias, dropout or the deterministic order
 *   (FA_ERR_UNSUPPORTED); fa_fwd / fa_fwd_ext run these head dims with the
 *   same masks.
 *   varlen: cu_seqlens_q / cu_seqlens_k != NULL (both or neither): int32
 *           device arrays of B+1 prefix sums; tensors packed [total, H, D];
 *           lse fp32 [Hq, total_q]; Sq / Sk are the MAXIMUM lengths.  A
 *           sequence longer than Sq / Sk, or packed totals above B * Sq /
 *           B * Sk, make the call fail with FA_ERR_INVALID_ARG: the totals
 *           are checked on the host before any launch, each sequence on the
 *           device (no row of an offending sequence is read or written, and
 *           the error is reported through the device error word).
 * Causal masking is bottom-right aligned: key j is visible to query i iff
 * j <= i + (Lk - Lq).
 *
 * Ownership: the caller owns every tensor and the stream.  All tensor
 * pointers are device pointers aligned to 16 bytes.  dq, dk, dv are fully
 * overwritten (key rows no query sees get zeros).  fa_bwd uses a per-device
 * workspace owned by the library (grown on demand); calls that overlap on
 * different streams of one device must use fa_bwd_with_workspace with their
 * own workspaces.
 *
 * Errors: arguments are validated before any launch (FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED); a failed launch returns FA_ERR_CUDA.  Otherwise the
 * call is asynchronous, except that deterministic calls, and varlen calls
 * whose packed totals are not given (fa_ext total_q / total_k), synchronise
 * `stream` before returning.  Every wait inside the kernels is bounded; a
 * wait that runs out records FA_ERR_TIMEOUT in a device word that
 * fa_device_status() reads (deterministic mode reads it before returning),
 * and so does a varlen length the device finds out of bounds
 * (FA_ERR_INVALID_ARG).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, bad scale */
    FA_ERR_UNSUPPORTED = 2,  /* head dims without a kernel (see the layouts above),
                                dtype, or GPU not sm_103 */
    FA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    FA_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out */
    FA_ERR_SCRATCH_LIMIT = 5 /* fa_bwd_noalloc: the problem needs more scratch than
                                FA_NOALLOC_SCRATCH_BYTES */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/* Backward pass.  softmax_scale is the plain scale c (S = c Q K^T); dK and dQ
 * carry the factor c, dV does not.  deterministic != 0 accumulates dQ in a
 * fixed order (ordered per-block semaphores) so repeated calls are
 * bit-identical; it then also synchronises `stream` and returns
 * FA_ERR_TIMEOUT if a semaphore wait ran out. */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, void *dq, void *dk, void *dv, int B, int Sq, int Sk, int Hq,
                 int Hkv, int D, float softmax_scale, int causal, const int *cu_seqlens_q,
                 const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                 cudaStream_t stream);

/* Bytes of device workspace fa_bwd_with_workspace needs for these sizes
 * (varlen = cu_seqlens given).  0 means the sizes are invalid. */
size_t fa_bwd_workspace_bytes(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                              int deterministic);

/* fa_bwd on a caller-owned device workspace of at least
 * fa_bwd_workspace_bytes(...) bytes, 256-byte aligned.  The workspace needs
 * no initialisation; it must not be used by another call in flight. */
fa_status fa_bwd_with_workspace(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                int B, int Sq, int Sk, int Hq, int Hkv, int D,
                                float softmax_scale, int causal, const int *cu_seqlens_q,
                                const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* The three stages of fa_bwd_with_workspace as separate calls (same
 * arguments, same workspace), for timing and testing each kernel.  They must
 * run in this order on one stream. */
fa_status fa_bwd_preprocess(const void *o, const void *dout, const float *lse, int B, int Sq,
                            int Sk, int Hq, int Hkv, int D, const int *cu_seqlens_q,
                            const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status fa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dk,
                      void *dv, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                      float softmax_scale, int causal,
                      const int *cu_seqlens_q, const int *cu_seqlens_k, int deterministic,
                      fa_dtype dtype, void *workspace, size_t workspace_bytes,
                      cudaStream_t stream);
fa_status fa_bwd_postprocess(void *dq, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                             float softmax_scale, const int *cu_seqlens_q,
                             const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Where the preprocess outputs live inside a workspace, in fp32 elements
 * from the workspace base: Dv at *dvec_off, LSE2 at *lse2_off, each indexed
 * by workspace row; the fp32 dQ accumulator at *dqacc_off, [rows, Dt], where
 * Dt is the tile width the head dim runs at (64 for D = 64, except 128 for
 * dense problems of at least 4096 keys; 128 for D up to 128; 256 above; the
 * columns past D stay 0).
 * Workspace row of (sequence b, query head h, position s):
 *   dense : (b * Hq + h) * round_up(Sq, 128) + s
 *   varlen: h * rows_per_head + pad(b) + s, pad(b) = (cu_q[b] + 128 b) / 128 * 128,
 *           rows_per_head = round_up(B * (Sq + 128), 128)
 * (the padded varlen offset of FlashAttentionBackwardPostprocess).  *rows is
 * the total row count. */
fa_status fa_bwd_workspace_layout(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                                  int deterministic, size_t *dvec_off, size_t *lse2_off,
                                  size_t *dqacc_off, size_t *rows);

/* Where a workspace keeps its synchronisation state, in bytes from the
 * workspace base: the device error word (*err_off; int32, 0 while no error
 * was recorded), and in deterministic mode the ordering semaphores (*sem_off,
 * *n_sem int32 entries, one per 64 workspace rows: the row block at
 * workspace rows [64 i, 64 i + 64) has entry i, which counts the key blocks
 * whose dQ contributions to that row block have been added -- the
 * arrive_inc / wait_eq counters of CollectiveEpilogueBwdGQA on the
 * FlashAttention page "flash-attention/hopper/epilogue_bwd.hpp").  Without
 * deterministic mode *sem_off and *n_sem are 0.  The preprocess stage
 * zeroes both; this call exists for tests and tools that inspect them. */
fa_status fa_bwd_workspace_sync_layout(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                                       int deterministic, size_t *err_off, size_t *sem_off,
                                       size_t *n_sem);

/* Forward pass O = softmax(Q K^T * scale + mask) V with LSE (natural log,
 * -inf for a query row that sees no key; such rows get O = 0): the inputs
 * fa_bwd consumes, same layouts and masking.  One tcgen05 kernel per call
 * (S = Q K^T and O += P V on the tensor cores, fp32 accumulation, online
 * softmax in the log2 domain).  Varlen calls read cu_seqlens_q[B] /
 * cu_seqlens_k[B] back to the host (one stream synchronisation).  Timeouts
 * of its bounded waits are reported by fa_device_status(NULL, ...). */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Sq,
                 int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                 const int *cu_seqlens_q, const int *cu_seqlens_k, fa_dtype dtype,
                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Extensions: a local window, ALiBi and used lengths.  They do not appear in
 * the five benchmark workloads; fa_fwd_ext / fa_bwd_ext take them through one
 * struct (NULL = none, which equals fa_fwd / fa_bwd).
 *
 * window_left / window_right (-1 = unbounded on that side): key j stays
 *   visible to query i only if i + (Lk - Lq) - window_left <= j <= i + (Lk -
 *   Lq) + window_right, a band around the same bottom-right diagonal as the
 *   causal mask (the Composable Kernel page masks with a generic
 *   mask.IsOutOfBound(row, col); this band is the reading taken).  causal
 *   != 0 intersects it with j <= i + (Lk - Lq).
 * alibi_slopes: device fp32, [Hq] (alibi_batch_stride 0) or [B, Hq]
 *   (alibi_batch_stride Hq); the score of (i, j) in head h of sequence b
 *   becomes scale * <q_i, k_j> - slope * |i + (Lk - Lq) - j| (the ALIBI bias
 *   kind of the Composable Kernel page, added after the scale).  LSE includes
 *   the bias; fa_bwd_ext must get the same slopes as the forward.
 * seqused_q / seqused_k: device int32 [B] (SeqlenInfo's seqused on the
 *   FlashAttention pages): sequence b uses its first seqused_q[b] query rows
 *   and seqused_k[b] key rows (values are clamped to [0, stored length]);
 *   Lq / Lk above are these used lengths.  Rows past them are neither read
 *   nor written (o, lse, dq, dk, dv keep what they held).
 * ------------------------------------------------------------------------- */
/* bias (dense problems only; FA_ERR_UNSUPPORTED with cu_seqlens): an
 *   elementwise additive bias in the input dtype, natural-log units, added
 *   after the scale (the ELEMENTWISE_BIAS kind of the Composable Kernel page,
 *   STAGE 2): element (b, h, i, j) at bias[b * bias_batch_stride + h *
 *   bias_head_stride + i * bias_row_stride + j]; a stride of 0 broadcasts.
 *   The pointer must be 16-byte aligned and the strides multiples of 8.
 * dbias (fa_bwd_ext, optional, also without bias): dBias = dS = P o (dP - D)
 *   (the page's dbias tile, STAGE 5), written as a contiguous
 *   [B, Hq, Sq, Sk] tensor in the input dtype, fully overwritten: 0 wherever
 *   dS is 0 (masked entries, tiles no work unit visits, rows and columns past
 *   the used lengths). */
/* dropout_p in [0, 1): dropout on P, as on the Composable Kernel page
 *   (FmhaDropout: dropped entries drop out of dV and of dP, kept ones are
 *   scaled by 1 / (1 - p)).  The drop probability is quantised to t / 256,
 *   t = round(256 p) (at most 255), and the keep scale is 256 / (256 - t).
 *   The mask is a pure function of (dropout_seed, dropout_offset, sequence,
 *   query head, i, j): entry (b, h, i, j) is dropped iff byte j % 4 of word
 *   (j / 4) % 4 of Philox4x32-10 (Salmon et al., SC 2011) with counter
 *   (j / 16, i, b * Hq + h, dropout_offset) and key (low, high 32 bits of
 *   dropout_seed) is below t.  fa_bwd_ext must get the forward's seed and
 *   offset.  The pages print no generator; this one is the reading taken.
 * dropout_mask (optional, device, 4-byte aligned; used only when t > 0): the
 *   keep flags as bits, W = ceil(Sk / 32) uint32 words per query row, rows in
 *   the order of lse ([B, Hq, Sq], or [Hq, total_q] with cu_seqlens; Sk is
 *   then the max_seqlen_k given).  Bit l of word w of row (b, h, i) is 1 iff
 *   key 32 w + l is kept.  fa_fwd_ext writes the words of the key blocks it
 *   visits (others are left as they were); fa_bwd_ext given the same buffer
 *   reads them instead of running Philox again (in deterministic mode the
 *   results are bit-identical to drawing the mask).  The buffer must hold
 *   B * Hq * Sq * W words (Hq * total_q * W with cu_seqlens). */
/* head_dim_v (0 = equal to D): the value head dim Dv of v, o, dout and dv
 *   (kVHeaddim next to kQKHeaddim in the Composable Kernel page's problem
 *   traits); a multiple of 8 in [8, 256], with D > 64 when it differs from D.
 * total_q / total_k (varlen only; both 0 = not given): the packed row counts
 *   cu_seqlens_q[B] and cu_seqlens_k[B], which the tensor maps are built
 *   for.  Given, the call needs no read-back of cu_seqlens and does not
 *   synchronise the stream.  They must equal cu_seqlens[B] and be at most
 *   B * Sq / B * Sk; the device checks the first and reports a mismatch as
 *   FA_ERR_INVALID_ARG through the error word, without reading or writing
 *   any row of the offending sequences.  The tensors must hold at least
 *   that many rows: a count larger than the rows allocated lets the tiled
 *   loads of the last rows run past the end of the tensors. */
typedef struct {
    int window_left;
    int window_right;
    const float *alibi_slopes;
    int alibi_batch_stride;
    const int *seqused_q;
    const int *seqused_k;
    const void *bias;
    long long bias_batch_stride;
    long long bias_head_stride;
    long long bias_row_stride;
    void *dbias;
    float dropout_p;
    unsigned long long dropout_seed;
    unsigned int dropout_offset;
    unsigned int *dropout_mask;
    long long total_q;
    long long total_k;
    int head_dim_v;
} fa_ext;

/* fa_fwd with extensions.  Errors as fa_fwd, plus FA_ERR_INVALID_ARG for a
 * window side below -1, an ALiBi stride other than 0 / Hq, or a slope or
 * seqused pointer not 4-byte aligned. */
fa_status fa_fwd_ext(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                     const int *cu_seqlens_q, const int *cu_seqlens_k, const fa_ext *ext,
                     fa_dtype dtype, cudaStream_t stream);

/* fa_bwd with extensions.  workspace NULL: the library's own (as fa_bwd);
 * otherwise a caller workspace as for fa_bwd_with_workspace (the extensions
 * do not change its size). */
fa_status fa_bwd_ext(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                     int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                     const int *cu_seqlens_q, const int *cu_seqlens_k, const fa_ext *ext,
                     int deterministic, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* CUDA graphs.  A backward call that issues only launches and memsets on
 * `stream` can be captured into a CUDA graph and replayed: fa_bwd_ext /
 * fa_bwd_with_workspace with a caller workspace for dense problems, and for
 * varlen problems when ext gives the packed totals; fa_bwd_stages_ext (or
 * the three stage calls, dense) in every mode.  A deterministic fa_bwd /
 * fa_bwd_ext reads its device status back before returning (a host wait) and
 * cannot be captured; capture its stages instead and read the status with
 * fa_device_status after the replay.  Make one uncaptured call with the same
 * sizes first (it loads the kernels).  Each replay reads the buffers that
 * were captured, so new inputs are written into them. */

/* The stages of fa_bwd_ext as separate calls on a caller-owned workspace:
 * `stages` is a bit mask of FA_STAGE_PRE (the preprocess), FA_STAGE_MAIN (the
 * work-unit scheduler for varlen, and the main kernel; with ext->dbias also
 * the zeroing of dBias before it) and FA_STAGE_POST (the dQ postprocess), run
 * in that order; the other arguments as fa_bwd_ext, where ext may be NULL and
 * workspace may not.  Across calls the stages must run in this order, on one
 * stream and one workspace, with the same arguments.  Pointers a chosen
 * stage does not read may be NULL (preprocess: o, dout, lse; main: q, k, v,
 * dout, dk, dv; postprocess: dq).  The call never waits for the device when
 * varlen totals are given in ext (or the problem is dense): a deterministic
 * call's device status is then read afterwards with fa_device_status on the
 * same workspace.  Errors as fa_bwd_ext, plus FA_ERR_INVALID_ARG for an
 * empty or unknown stage mask.  Defined by the same passages as fa_bwd. */
#define FA_STAGE_PRE 1
#define FA_STAGE_MAIN 2
#define FA_STAGE_POST 4
fa_status fa_bwd_stages_ext(int stages, const void *q, const void *k, const void *v,
                            const void *o, const void *dout, const float *lse, void *dq,
                            void *dk, void *dv, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                            float softmax_scale, int causal, const int *cu_seqlens_q,
                            const int *cu_seqlens_k, const fa_ext *ext, int deterministic,
                            fa_dtype dtype, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the device error word of
 * this device's library workspace (FA_OK or FA_ERR_TIMEOUT).  For a caller
 * workspace, pass it; NULL means the library's own. */
fa_status fa_device_status(void *workspace, cudaStream_t stream);

/* Upper limit, in nanoseconds, of every device-side wait (default 2e9).
 * Returns the previous value; 0 leaves it unchanged. */
long long fa_set_wait_timeout_ns(long long ns);

const char *fa_status_string(fa_status s);

/* ---------------------------------------------------------------------------
 * Allocation-free backward.  The attention-backward pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate device
 * memory when they call the library: an inference-engine plugin whose enqueue
 * step must not allocate, a framework that owns all device memory through its
 * own pool and allows no other allocation, or a latency-critical loop that
 * must not enter the driver's allocator (which can synchronise the device).
 *
 * fa_bwd_noalloc takes the same arguments as fa_bwd and computes the same
 * result, but its scratch (Dv, LSE2, the fp32 dQ accumulator, the work-unit
 * list, the error word) is a fixed device array of FA_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library holds
 * until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   - Problems whose scratch (fa_bwd_workspace_bytes of the same sizes) is
 *     larger than FA_NOALLOC_SCRATCH_BYTES are rejected with
 *     FA_ERR_SCRATCH_LIMIT before anything runs.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and remembers it for the life of the process;
 *     make that first call before any stream capture.  The remembered
 *     address does not survive cudaDeviceReset: do not call fa_bwd_noalloc
 *     again on a device after resetting it.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call re-initialises what must start at zero, so no clearing is needed
 *     between calls, but calls that overlap on the GPU (other streams, other
 *     host threads) race on the array and must be serialised by the caller.
 *   - Deterministic calls, and varlen calls (their packed totals are read
 *     back from cu_seqlens), synchronise `stream` before returning, as
 *     fa_bwd does.
 *   - Device-side errors (a bounded wait that ran out, a varlen length out
 *     of bounds) are recorded in the array's own error word, which
 *     fa_bwd_noalloc_status reads; fa_device_status does not see it.
 * ------------------------------------------------------------------------- */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* FA_NOALLOC_SCRATCH_BYTES, for callers that load the library dynamically. */
size_t fa_bwd_noalloc_scratch_bytes(void);

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                         const int *cu_seqlens_q, const int *cu_seqlens_k, int deterministic,
                         fa_dtype dtype, cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the device error word of
 * the fixed scratch array on the current device: FA_OK, FA_ERR_TIMEOUT (a
 * bounded wait ran out) or FA_ERR_INVALID_ARG (a varlen sequence longer than
 * the maximum given).  Allocates nothing either; before the first
 * fa_bwd_noalloc on the device it returns FA_OK. */
fa_status fa_bwd_noalloc_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
