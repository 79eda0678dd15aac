// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// workspace planning, TMA tensor-map encoding and the kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_params.h"

namespace fa {
cudaError_t launch_schedule(const BwdParams &p, cudaStream_t stream);
cudaError_t launch_preprocess(const BwdParams &p, int bf16, cudaStream_t stream);
cudaError_t launch_postprocess(const BwdParams &p, int bf16, cudaStream_t stream);
cudaError_t launch_dbias_zero(const BwdParams &p, int bm, cudaStream_t stream);
cudaError_t launch_fwd_tc(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                          const CUtensorMap &v, void *o, float *lse, int max_lq, int bf16,
                          cudaStream_t stream);
int fwd_block_m();
int fwd_block_n(int Dq_tile, int Dv_tile);
int *fwd_error_word();
cudaError_t launch_bwd_main(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dout, const CUtensorMap &dk,
                            const CUtensorMap &dv, int bf16, int grid, cudaStream_t stream);
int main_block_m(int D);
cudaError_t launch_bwd_wide(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dout, int bf16, int grid,
                            cudaStream_t stream);
int wide_block_m();
int wide_halves(int Dq_tile, int Dv_tile);
}  // namespace fa

namespace {

std::atomic<long long> g_budget_ns{2000000000LL};

constexpr float kLog2e = 1.4426950408889634f;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tile width a head dim runs at: 64, 128 or 256 (the columns past D are
// zero-filled by the TMA loads; the FlashAttention postprocess page likewise
// pads the head dim to a multiple of its block size).
int pad_d(int D) { return D <= 64 ? 64 : D <= 128 ? 128 : 256; }

// Backward tile width of a query / key head dim.  D = 64 runs in the 128-wide
// tile (its upper 64 columns zero) for dense problems of at least 4096 keys:
// its softmax, not the tensor core, sets the step time, and the wider tile's
// 64-query steps carry half the elementwise work per step (B = 2, 32 / 8
// heads, 8192 keys, causal: main kernel 2.204 -> 1.911 ms).  Shorter and
// varlen problems keep the 64-wide tile, whose 128-query steps halve the unit
// transitions (16 sequences of 256..2048 keys: 0.378 against 0.435 ms).
int bwd_pad_d(int D, int Sk, bool varlen) {
    if (D <= 64 && !varlen && Sk >= 4096) return 128;
    return pad_d(D);
}

// Head dims with a kernel: a query / key dim D that is a multiple of 8 in
// [64, 256]; a value dim Dv (0: equal to D) that is a multiple of 8 in
// [8, 256].  One head dim of at most 128 runs in the main kernel; a head dim
// above 128, or Dv != D (then D > 64), runs in the wide kernel.
bool head_dims_ok(int D, int Dv) {
    if (D < 64 || D > 256 || D % 8 != 0) return false;
    if (Dv == 0 || Dv == D) return true;
    return Dv >= 8 && Dv <= 256 && Dv % 8 == 0 && D > 64;
}
bool wide_dims(int D, int Dv) { return D > 128 || (Dv != 0 && Dv != D); }
int value_tile(int D, int Dv) {   // tile width of the value side
    return wide_dims(D, Dv) ? ((Dv == 0 ? D : Dv) <= 128 ? 128 : 256) : pad_d(D);
}

struct Layout {
    size_t err, ntiles, tiles, dvec, lse2, dqacc, sem, total;  // byte offsets / size
    long long rows, rows_per_head;
    int sq_round, max_tiles;
};

bool plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen, int deterministic,
          Layout *L) {
    if (B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return false;
    const long long T = fa::kRowTile;
    L->sq_round = (int)round_up((size_t)Sq, T);
    if (varlen) {
        L->rows_per_head = (long long)round_up((size_t)B * ((size_t)Sq + T), T);
        L->rows = (long long)Hq * L->rows_per_head;
    } else {
        L->rows_per_head = L->sq_round;
        L->rows = (long long)B * Hq * L->sq_round;
    }
    const long long tiles = (long long)B * ((Sk + fa::kBlockN - 1) / fa::kBlockN) * Hkv;
    if (tiles > (1LL << 30)) return false;
    L->max_tiles = (int)tiles;
    size_t off = 0;
    L->err = off;       off += 256;
    L->ntiles = off;    off += 256;
    L->tiles = off;     off = round_up(off + (size_t)tiles * 16, 256);
    L->dvec = off;      off = round_up(off + (size_t)L->rows * 4, 256);
    L->lse2 = off;      off = round_up(off + (size_t)L->rows * 4, 256);
    L->dqacc = off;     off = round_up(off + (size_t)L->rows * bwd_pad_d(D, Sk, varlen) * 4, 256);
    L->sem = off;       off = round_up(off + (deterministic ? (size_t)(L->rows / 64) * 4 : 0), 256);
    L->total = off;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return FA_ERR_CUDA;
    if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status check_shape(int B, int Sq, int Sk, int Hq, int Hkv, int D, fa_dtype dtype,
                      const int *cu_q, const int *cu_k) {
    if (B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if ((cu_q == nullptr) != (cu_k == nullptr)) return FA_ERR_INVALID_ARG;
    if (!head_dims_ok(D, 0)) return FA_ERR_UNSUPPORTED;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
    // TMA coordinates are 32-bit
    if ((long long)B * Sq > (1LL << 31) - 1 || (long long)B * Sk > (1LL << 31) - 1)
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// ----------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 4-D map over a [batch, rows, heads, D] 16-bit tensor (d innermost), box of
// 64 d x 1 head x box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool encode_rows_map(CUtensorMap *m, const void *base, int D, int H, long long rows, int batch,
                     int box_rows, int bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)rows * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------- library-owned workspace
struct DeviceWs {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
std::vector<DeviceWs> g_ws;

fa_status library_workspace(size_t need, cudaStream_t stream, void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
    DeviceWs &w = g_ws[dev];
    if (w.bytes < need) {
        if (w.ptr) {
            if (cudaFreeAsync(w.ptr, stream) != cudaSuccess) return FA_ERR_CUDA;
            w.ptr = nullptr;
            w.bytes = 0;
        }
        size_t grow = round_up(need + need / 8, 1 << 21);
        if (cudaMallocAsync(&w.ptr, grow, stream) != cudaSuccess) return FA_ERR_CUDA;
        w.bytes = grow;
    }
    *out = w.ptr;
    return FA_OK;
}

void *library_workspace_peek() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    if ((int)g_ws.size() <= dev) return nullptr;
    return g_ws[dev].ptr;
}

// Totals of the packed varlen tensors (cu[B]); read back from the device.
fa_status varlen_totals(const int *cu_q, const int *cu_k, int B, cudaStream_t stream,
                        long long *tq, long long *tk) {
    int h[2] = {0, 0};
    if (cudaMemcpyAsync(&h[0], cu_q + B, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(&h[1], cu_k + B, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return FA_ERR_CUDA;
    if (h[0] < 0 || h[1] < 0) return FA_ERR_INVALID_ARG;
    *tq = h[0];
    *tk = h[1];
    return FA_OK;
}

// The packed row counts of a varlen call: the caller's (fa_ext total_q /
// total_k, both > 0), which need no host synchronisation, else cu[B] read
// back from the device.  Every sequence fits the planned layout only if the
// totals are at most B times the maximum lengths; the kernels check
// cu_seqlens against the totals and the maximum lengths (kErrBadLength).
fa_status packed_totals(const fa_ext *ext, const int *cu_q, const int *cu_k, int B, int Sq,
                        int Sk, cudaStream_t stream, long long *tq, long long *tk) {
    if (ext && (ext->total_q != 0 || ext->total_k != 0)) {
        *tq = ext->total_q;
        *tk = ext->total_k;
    } else {
        fa_status st = varlen_totals(cu_q, cu_k, B, stream, tq, tk);
        if (st != FA_OK) return st;
    }
    if (*tq > (long long)B * Sq || *tk > (long long)B * Sk) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Host check of the caller's packed totals (before the device is touched):
// varlen only, both positive, at most B times the maximum lengths.
fa_status check_ext_totals(const fa_ext *ext, bool varlen, int B, int Sq, int Sk) {
    if (!ext || (ext->total_q == 0 && ext->total_k == 0)) return FA_OK;
    if (!varlen || ext->total_q <= 0 || ext->total_k <= 0) return FA_ERR_INVALID_ARG;
    if (ext->total_q > (long long)B * Sq || ext->total_k > (long long)B * Sk) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

struct Prepared {
    fa::BwdParams p;
    Layout L;
    long long total_q, total_k;
};

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// The visible band, ALiBi slopes and used lengths of the parameter block
// (ext NULL: none, only the causal mask).
fa_status apply_ext(fa::BwdParams &p, int causal, const fa_ext *ext) {
    int wl = -1, wr = -1;
    p.alibi = nullptr;
    p.alibi_bstride = 0;
    p.seqused_q = p.seqused_k = nullptr;
    p.bias = nullptr;
    p.bias_bs = p.bias_hs = p.bias_rs = 0;
    p.dbias = nullptr;
    p.drop_t = 0;
    p.drop_key0 = p.drop_key1 = p.drop_offset = 0;
    p.drop_scale = 1.f;
    p.drop_mask = nullptr;
    p.drop_mask_w = 0;
    p.Dhv = p.Dh;
    p.Dv = p.D;
    if (ext) {
        if (ext->head_dim_v != 0) {
            if (!head_dims_ok(p.Dh, ext->head_dim_v)) return FA_ERR_UNSUPPORTED;
            p.Dhv = ext->head_dim_v;
        }
        wl = ext->window_left;
        wr = ext->window_right;
        if (wl < -1 || wr < -1) return FA_ERR_INVALID_ARG;
        if (ext->alibi_slopes) {
            if ((reinterpret_cast<uintptr_t>(ext->alibi_slopes) & 3u) ||
                (ext->alibi_batch_stride != 0 && ext->alibi_batch_stride != p.Hq))
                return FA_ERR_INVALID_ARG;
            p.alibi = ext->alibi_slopes;
            p.alibi_bstride = ext->alibi_batch_stride;
        }
        if ((reinterpret_cast<uintptr_t>(ext->seqused_q) & 3u) ||
            (reinterpret_cast<uintptr_t>(ext->seqused_k) & 3u))
            return FA_ERR_INVALID_ARG;
        p.seqused_q = ext->seqused_q;
        p.seqused_k = ext->seqused_k;
        if (ext->bias) {
            if (p.varlen) return FA_ERR_UNSUPPORTED;
            if (!aligned16(ext->bias) || ext->bias_batch_stride < 0 || ext->bias_head_stride < 0 ||
                ext->bias_row_stride < p.Sk || (ext->bias_batch_stride & 7) ||
                (ext->bias_head_stride & 7) || (ext->bias_row_stride & 7))
                return FA_ERR_INVALID_ARG;
            p.bias = ext->bias;
            p.bias_bs = ext->bias_batch_stride;
            p.bias_hs = ext->bias_head_stride;
            p.bias_rs = ext->bias_row_stride;
        }
        if (ext->dbias) {
            if (p.varlen) return FA_ERR_UNSUPPORTED;
            if ((reinterpret_cast<uintptr_t>(ext->dbias) & 1u)) return FA_ERR_INVALID_ARG;
            p.dbias = ext->dbias;
        }
        const float dp = ext->dropout_p;
        if (!(dp >= 0.f && dp < 1.f)) return FA_ERR_INVALID_ARG;
        p.drop_t = std::min(255, (int)(dp * 256.f + 0.5f));
        p.drop_key0 = (uint32_t)ext->dropout_seed;
        p.drop_key1 = (uint32_t)(ext->dropout_seed >> 32);
        p.drop_offset = ext->dropout_offset;
        p.drop_scale = 256.f / (float)(256 - p.drop_t);
        if (ext->dropout_mask && p.drop_t > 0) {
            if (reinterpret_cast<uintptr_t>(ext->dropout_mask) & 3u) return FA_ERR_INVALID_ARG;
            p.drop_mask = ext->dropout_mask;
            p.drop_mask_w = (p.Sk + 31) / 32;
        }
    }
    p.win_lo = (wl < 0 || wl >= fa::kNoWindow) ? fa::kNoWindow : wl;
    p.win_hi = (wr < 0 || wr >= fa::kNoWindow) ? fa::kNoWindow : wr;
    if (causal) p.win_hi = std::min(p.win_hi, 0);
    if (wide_dims(p.Dh, p.Dhv)) {
        // the wide kernel's tile widths (128 or 256 on each side); it has the
        // band masks (causal, both window edges) and used lengths
        p.D = p.Dh <= 128 ? 128 : 256;
        p.Dv = value_tile(p.Dh, p.Dhv);
        if (p.alibi || p.bias || p.dbias || p.drop_t > 0) return FA_ERR_UNSUPPORTED;
    }
    return FA_OK;
}

fa_status prepare(const void *q, const void *k, const void *v, const void *o, const void *dout,
                  const float *lse, void *dq, void *dk, void *dv, int B, int Sq, int Sk, int Hq,
                  int Hkv, int D, float scale, int causal, const int *cu_q, const int *cu_k,
                  int deterministic, fa_dtype dtype, void *ws, size_t ws_bytes,
                  cudaStream_t stream, Prepared *out, const fa_ext *ext = nullptr) {
    fa_status st = check_shape(B, Sq, Sk, Hq, Hkv, D, dtype, cu_q, cu_k);
    if (st != FA_OK) return st;
    if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return FA_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return FA_ERR_INVALID_ARG;
    Layout L;
    if (!plan(B, Sq, Sk, Hq, Hkv, D, cu_q != nullptr, deterministic, &L)) return FA_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return FA_ERR_INVALID_ARG;
    uint8_t *w = static_cast<uint8_t *>(ws);
    fa::BwdParams &p = out->p;
    std::memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.B = B; p.Sq = Sq; p.Sk = Sk; p.Hq = Hq; p.Hkv = Hkv; p.D = bwd_pad_d(D, Sk, cu_q != nullptr);
    p.Dh = D;
    p.G = Hq / Hkv;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.deterministic = deterministic ? 1 : 0;
    p.varlen = cu_q != nullptr;
    p.cu_q = cu_q; p.cu_k = cu_k;
    // the extensions are host arguments too: checked before the device is
    if ((st = apply_ext(p, causal, ext)) != FA_OK) return st;
    if ((st = check_ext_totals(ext, cu_q != nullptr, B, Sq, Sk)) != FA_OK) return st;
    // the wide kernel adds dQ without the deterministic order
    if (deterministic && wide_dims(p.Dh, p.Dhv)) return FA_ERR_UNSUPPORTED;
    st = check_device();
    if (st != FA_OK) return st;
    long long tq = (long long)B * Sq, tk = (long long)B * Sk;
    if (cu_q) {
        if ((st = packed_totals(ext, cu_q, cu_k, B, Sq, Sk, stream, &tq, &tk)) != FA_OK) return st;
        p.total_q = tq;
        p.total_k = tk;
    }
    p.err = reinterpret_cast<int *>(w + L.err);
    p.ntiles = reinterpret_cast<int *>(w + L.ntiles);
    p.unit_counter = reinterpret_cast<int *>(w + L.ntiles) + 1;
    p.tiles = reinterpret_cast<int4 *>(w + L.tiles);
    p.max_tiles = L.max_tiles;
    p.num_units = L.max_tiles;
    // Unit order of the dense main kernel: the smallest group of (batch, kv
    // head) pairs -- a divisor of B * Hkv, so that no short group comes last --
    // whose units number at least 1.5 times the grid.
    // Deterministic mode adds each row block's contributions in n-block
    // order, so the units of one (sequence, kv head) wait on one another;
    // there, all pairs are interleaved (plain n-block-major order), so that
    // few units of any one chain run at the same time.
    // Varlen (the scheduler kernel builds the list): groups of consecutive
    // sequences of at least 1.5 grids of units each, the same idea; in
    // deterministic mode none (0: the plain order).
    p.unit_group = B * Hkv;
    if (!cu_q && !deterministic) {
        const int nblk = (Sk + fa::kBlockN - 1) / fa::kBlockN;
        const long long grid = std::min<long long>(L.max_tiles, sm_count());
        for (int g = 1; g <= B * Hkv; ++g)
            if ((B * Hkv) % g == 0 && 2LL * g * nblk >= 3 * grid) { p.unit_group = g; break; }
    } else if (cu_q) {
        const long long grid = std::min<long long>(L.max_tiles, sm_count());
        p.unit_group = deterministic ? 0 : (int)std::max<long long>(1, 3 * grid / 2);
    }
    p.dvec = reinterpret_cast<float *>(w + L.dvec);
    p.lse2 = reinterpret_cast<float *>(w + L.lse2);
    p.dqacc = reinterpret_cast<float *>(w + L.dqacc);
    p.sem = deterministic ? reinterpret_cast<int *>(w + L.sem) : nullptr;
    p.rows = L.rows;
    p.rows_per_head = L.rows_per_head;
    p.sq_round = L.sq_round;
    p.budget_ns = g_budget_ns.load();
    out->L = L;
    out->total_q = tq;
    out->total_k = tk;
    return FA_OK;
}

fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

fa_status run_preprocess(const Prepared &P, fa_dtype dtype, cudaStream_t stream) {
    if (!P.p.o || !P.p.dout || !P.p.lse) return FA_ERR_INVALID_ARG;
    return cuda_status(fa::launch_preprocess(P.p, dtype == FA_BF16, stream));
}

// dBias (dense, main kernel only): the main kernel writes dS of the tiles it
// visits, the rest is 0.  A kernel that decodes the same units writes those
// zeros when 16-byte stores fit the tensor; else the whole tensor is zeroed
// first.
fa_status zero_dbias(const Prepared &P, cudaStream_t stream) {
    const fa::BwdParams &p = P.p;
    if ((reinterpret_cast<uintptr_t>(p.dbias) & 15u) == 0 && (p.Sk & 7) == 0)
        return cuda_status(fa::launch_dbias_zero(p, fa::main_block_m(p.D), stream));
    const size_t n = (size_t)p.B * p.Hq * p.Sq * p.Sk * 2;
    return cudaMemsetAsync(p.dbias, 0, n, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_main(const Prepared &P, fa_dtype dtype, cudaStream_t stream) {
    const fa::BwdParams &p = P.p;
    const bool wide = wide_dims(p.Dh, p.Dhv);
    const int bm = wide ? fa::wide_block_m() : fa::main_block_m(p.D);
    const int bf16 = dtype == FA_BF16;
    CUtensorMap mq, mk, mv, mdo;
    const long long rq = p.varlen ? P.total_q : p.Sq, rk = p.varlen ? P.total_k : p.Sk;
    const int nb = p.varlen ? 1 : p.B;
    if (rq <= 0 || rk <= 0) return FA_ERR_INVALID_ARG;
    if (!p.q || !p.k || !p.v || !p.dout || !p.dk || !p.dv) return FA_ERR_INVALID_ARG;
    if (!encode_rows_map(&mq, p.q, p.Dh, p.Hq, rq, nb, bm, bf16) ||
        !encode_rows_map(&mdo, p.dout, p.Dhv, p.Hq, rq, nb, bm, bf16) ||
        !encode_rows_map(&mk, p.k, p.Dh, p.Hkv, rk, nb, fa::kBlockN, bf16) ||
        !encode_rows_map(&mv, p.v, p.Dhv, p.Hkv, rk, nb, fa::kBlockN, bf16))
        return FA_ERR_CUDA;
    if (p.varlen) {
        // the unit list depends on the device-resident cu_seqlens
        if (fa::launch_schedule(p, stream) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (wide) {
        // units: key-block units times column halves
        const long long units = (long long)p.max_tiles * fa::wide_halves(p.D, p.Dv);
        const int grid = (int)std::min<long long>(units, sm_count());
        return cuda_status(fa::launch_bwd_wide(p, mq, mk, mv, mdo, bf16, grid, stream));
    }
    // dK / dV leave the main kernel through tensor stores of the same geometry as K / V
    CUtensorMap mdk, mdv;
    if (!encode_rows_map(&mdk, p.dk, p.Dh, p.Hkv, rk, nb, fa::kBlockN, bf16) ||
        !encode_rows_map(&mdv, p.dv, p.Dhv, p.Hkv, rk, nb, fa::kBlockN, bf16))
        return FA_ERR_CUDA;
    const int grid = (int)std::min<long long>(p.max_tiles, sm_count());
    return cuda_status(fa::launch_bwd_main(p, mq, mk, mv, mdo, mdk, mdv, bf16, grid, stream));
}

fa_status run_postprocess(const Prepared &P, fa_dtype dtype, cudaStream_t stream) {
    if (!P.p.dq) return FA_ERR_INVALID_ARG;
    return cuda_status(fa::launch_postprocess(P.p, dtype == FA_BF16, stream));
}

fa_status read_error_word(int *err_dev, cudaStream_t stream, bool clear) {
    int h = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemcpy(&h, err_dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (clear && h != 0 && cudaMemset(err_dev, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    if (h & 4) return FA_ERR_INVALID_ARG;   // kErrBadLength: cu_seqlens against the sizes given
    return h ? FA_ERR_TIMEOUT : FA_OK;
}

}  // namespace

extern "C" {

const char *fa_status_string(fa_status s) {
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed no-alloc array";
    }
    return "unknown status";
}

long long fa_set_wait_timeout_ns(long long ns) {
    if (ns <= 0) return g_budget_ns.load();
    return g_budget_ns.exchange(ns);
}

size_t fa_bwd_workspace_bytes(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                              int deterministic) {
    Layout L;
    if (!head_dims_ok(D, 0)) return 0;
    if (!plan(B, Sq, Sk, Hq, Hkv, D, varlen, deterministic, &L)) return 0;
    return L.total;
}

fa_status fa_bwd_workspace_layout(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                                  int deterministic, size_t *dvec_off, size_t *lse2_off,
                                  size_t *dqacc_off, size_t *rows) {
    Layout L;
    if (!head_dims_ok(D, 0)) return FA_ERR_UNSUPPORTED;
    if (!plan(B, Sq, Sk, Hq, Hkv, D, varlen, deterministic, &L)) return FA_ERR_INVALID_ARG;
    if (dvec_off) *dvec_off = L.dvec / 4;
    if (lse2_off) *lse2_off = L.lse2 / 4;
    if (dqacc_off) *dqacc_off = L.dqacc / 4;
    if (rows) *rows = (size_t)L.rows;
    return FA_OK;
}

fa_status fa_bwd_workspace_sync_layout(int B, int Sq, int Sk, int Hq, int Hkv, int D, int varlen,
                                       int deterministic, size_t *err_off, size_t *sem_off,
                                       size_t *n_sem) {
    Layout L;
    if (!head_dims_ok(D, 0)) return FA_ERR_UNSUPPORTED;
    if (!plan(B, Sq, Sk, Hq, Hkv, D, varlen, deterministic, &L)) return FA_ERR_INVALID_ARG;
    if (err_off) *err_off = L.err;
    if (sem_off) *sem_off = deterministic ? L.sem : 0;
    if (n_sem) *n_sem = deterministic ? (size_t)(L.rows / 64) : 0;
    return FA_OK;
}

fa_status fa_bwd_preprocess(const void *o, const void *dout, const float *lse, int B, int Sq,
                            int Sk, int Hq, int Hkv, int D, const int *cu_seqlens_q,
                            const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!o || !dout || !lse) return FA_ERR_INVALID_ARG;
    Prepared P;
    fa_status st = prepare(nullptr, nullptr, nullptr, o, dout, lse, nullptr, nullptr, nullptr, B,
                           Sq, Sk, Hq, Hkv, D, 1.f, 0, cu_seqlens_q, cu_seqlens_k, deterministic,
                           dtype, workspace, workspace_bytes, stream, &P);
    if (st != FA_OK) return st;
    return run_preprocess(P, dtype, stream);
}

fa_status fa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dk,
                      void *dv, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                      float softmax_scale, int causal, const int *cu_seqlens_q,
                      const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!q || !k || !v || !dout || !dk || !dv) return FA_ERR_INVALID_ARG;
    Prepared P;
    fa_status st = prepare(q, k, v, nullptr, dout, nullptr, nullptr, dk, dv, B, Sq, Sk, Hq, Hkv,
                           D, softmax_scale, causal, cu_seqlens_q, cu_seqlens_k, deterministic,
                           dtype, workspace, workspace_bytes, stream, &P);
    if (st != FA_OK) return st;
    return run_main(P, dtype, stream);
}

fa_status fa_bwd_postprocess(void *dq, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                             float softmax_scale, const int *cu_seqlens_q,
                             const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!dq) return FA_ERR_INVALID_ARG;
    Prepared P;
    fa_status st = prepare(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr,
                           nullptr, B, Sq, Sk, Hq, Hkv, D, softmax_scale, 0, cu_seqlens_q,
                           cu_seqlens_k, deterministic, dtype, workspace, workspace_bytes, stream,
                           &P);
    if (st != FA_OK) return st;
    return run_postprocess(P, dtype, stream);
}

fa_status fa_bwd_with_workspace(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                int B, int Sq, int Sk, int Hq, int Hkv, int D,
                                float softmax_scale, int causal, const int *cu_seqlens_q,
                                const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!workspace) return FA_ERR_INVALID_ARG;   // (fa_bwd_ext would take the library's)
    return fa_bwd_ext(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D, softmax_scale,
                      causal, cu_seqlens_q, cu_seqlens_k, nullptr, deterministic, dtype,
                      workspace, workspace_bytes, stream);
}

fa_status fa_bwd_ext(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                     int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                     const int *cu_seqlens_q, const int *cu_seqlens_k, const fa_ext *ext,
                     int deterministic, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    fa_status st;
    if (!workspace) {
        // the library's own workspace, grown on demand
        st = check_shape(B, Sq, Sk, Hq, Hkv, D, dtype, cu_seqlens_q, cu_seqlens_k);
        if (st != FA_OK) return st;
        workspace_bytes = fa_bwd_workspace_bytes(B, Sq, Sk, Hq, Hkv, D,
                                                 cu_seqlens_q != nullptr, deterministic);
        if (workspace_bytes == 0) return FA_ERR_INVALID_ARG;
        if ((st = library_workspace(workspace_bytes, stream, &workspace)) != FA_OK) return st;
    }
    Prepared P;
    st = prepare(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D, softmax_scale, causal,
                 cu_seqlens_q, cu_seqlens_k, deterministic, dtype, workspace, workspace_bytes,
                 stream, &P, ext);
    if (st != FA_OK) return st;
    if ((st = run_preprocess(P, dtype, stream)) != FA_OK) return st;
    if (P.p.dbias && (st = zero_dbias(P, stream)) != FA_OK) return st;
    if ((st = run_main(P, dtype, stream)) != FA_OK) return st;
    if ((st = run_postprocess(P, dtype, stream)) != FA_OK) return st;
    if (deterministic) return read_error_word(P.p.err, stream, false);
    return FA_OK;
}

fa_status fa_bwd_stages_ext(int stages, const void *q, const void *k, const void *v,
                            const void *o, const void *dout, const float *lse, void *dq,
                            void *dk, void *dv, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                            float softmax_scale, int causal, const int *cu_seqlens_q,
                            const int *cu_seqlens_k, const fa_ext *ext, int deterministic,
                            fa_dtype dtype, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    const int all = FA_STAGE_PRE | FA_STAGE_MAIN | FA_STAGE_POST;
    if (stages <= 0 || (stages & ~all) || !workspace) return FA_ERR_INVALID_ARG;
    Prepared P;
    fa_status st = prepare(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D, softmax_scale,
                           causal, cu_seqlens_q, cu_seqlens_k, deterministic, dtype, workspace,
                           workspace_bytes, stream, &P, ext);
    if (st != FA_OK) return st;
    if ((stages & FA_STAGE_PRE) && (st = run_preprocess(P, dtype, stream)) != FA_OK) return st;
    if (stages & FA_STAGE_MAIN) {
        if (P.p.dbias && (st = zero_dbias(P, stream)) != FA_OK) return st;
        if ((st = run_main(P, dtype, stream)) != FA_OK) return st;
    }
    if ((stages & FA_STAGE_POST) && (st = run_postprocess(P, dtype, stream)) != FA_OK) return st;
    return FA_OK;
}

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, void *dq, void *dk, void *dv, int B, int Sq, int Sk, int Hq,
                 int Hkv, int D, float softmax_scale, int causal, const int *cu_seqlens_q,
                 const int *cu_seqlens_k, int deterministic, fa_dtype dtype,
                 cudaStream_t stream) {
    fa_status st = check_shape(B, Sq, Sk, Hq, Hkv, D, dtype, cu_seqlens_q, cu_seqlens_k);
    if (st != FA_OK) return st;
    const size_t need = fa_bwd_workspace_bytes(B, Sq, Sk, Hq, Hkv, D, cu_seqlens_q != nullptr,
                                               deterministic);
    if (need == 0) return FA_ERR_INVALID_ARG;
    void *ws = nullptr;
    st = library_workspace(need, stream, &ws);
    if (st != FA_OK) return st;
    return fa_bwd_with_workspace(q, k, v, o, dout, lse, dq, dk, dv, B, Sq, Sk, Hq, Hkv, D,
                                 softmax_scale, causal, cu_seqlens_q, cu_seqlens_k, deterministic,
                                 dtype, ws, need, stream);
}

fa_status fa_device_status(void *workspace, cudaStream_t stream) {
    void *ws = workspace ? workspace : library_workspace_peek();
    fa_status st = FA_OK;
    if (!workspace) {
        // the forward pass records its timeouts in a word of its own
        int *fwd_err = fa::fwd_error_word();
        if (!fwd_err) return FA_ERR_CUDA;
        st = read_error_word(fwd_err, stream, true);
        if (st == FA_ERR_CUDA) return st;
    }
    if (!ws) {
        return cudaStreamSynchronize(stream) == cudaSuccess ? st : FA_ERR_CUDA;
    }
    fa_status st2 = read_error_word(reinterpret_cast<int *>(ws), stream, true);
    return st2 != FA_OK ? st2 : st;
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Sq,
                 int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                 const int *cu_seqlens_q, const int *cu_seqlens_k, fa_dtype dtype,
                 cudaStream_t stream) {
    return fa_fwd_ext(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, softmax_scale, causal, cu_seqlens_q,
                      cu_seqlens_k, nullptr, dtype, stream);
}

fa_status fa_fwd_ext(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int Sq, int Sk, int Hq, int Hkv, int D, float softmax_scale, int causal,
                     const int *cu_seqlens_q, const int *cu_seqlens_k, const fa_ext *ext,
                     fa_dtype dtype, cudaStream_t stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, Sq, Sk, Hq, Hkv, D, dtype, cu_seqlens_q, cu_seqlens_k);
    if (st != FA_OK) return st;
    if (!(std::isfinite(softmax_scale) && softmax_scale > 0.f)) return FA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, o, lse};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return FA_ERR_INVALID_ARG;
    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v;
    p.B = B; p.Sq = Sq; p.Sk = Sk; p.Hq = Hq; p.Hkv = Hkv; p.D = pad_d(D); p.Dh = D;
    p.G = Hq / Hkv;
    p.scale = softmax_scale;
    p.scale_log2 = softmax_scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.varlen = cu_seqlens_q != nullptr;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    if ((st = apply_ext(p, causal, ext)) != FA_OK) return st;
    if ((st = check_ext_totals(ext, p.varlen, B, Sq, Sk)) != FA_OK) return st;
    if ((st = check_device()) != FA_OK) return st;
    p.err = fa::fwd_error_word();
    if (!p.err) return FA_ERR_CUDA;
    p.budget_ns = g_budget_ns.load();
    long long rq = Sq, rk = Sk;
    if (p.varlen) {
        st = packed_totals(ext, cu_seqlens_q, cu_seqlens_k, B, Sq, Sk, stream, &rq, &rk);
        if (st != FA_OK) return st;
        p.total_q = rq;
        p.total_k = rk;
        if (rq == 0) return FA_OK;
    }
    // a map needs at least one row; with no keys at all no K/V tile is loaded
    rk = std::max<long long>(rk, 1);
    const int bf16 = dtype == FA_BF16;
    const int nb = p.varlen ? 1 : B;
    CUtensorMap mq, mk, mv;
    const int bn = fa::fwd_block_n(p.D, p.Dv);
    if (!encode_rows_map(&mq, q, D, Hq, rq, nb, fa::fwd_block_m(), bf16) ||
        !encode_rows_map(&mk, k, D, Hkv, rk, nb, bn, bf16) ||
        !encode_rows_map(&mv, v, p.Dhv, Hkv, rk, nb, bn, bf16))
        return FA_ERR_CUDA;
    return cuda_status(fa::launch_fwd_tc(p, mq, mk, mv, o, lse, Sq, bf16, stream));
}

}  // extern "C"
