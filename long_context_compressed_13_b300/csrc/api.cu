// C ABI of the lcattn library: host-side validation, workspace sizing and
// dispatch to the kernels.  Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "lc_common.cuh"

namespace lc {

lc_status compress_launch(const void *K, const void *V, const float *GK, const float *GV,
                          int64_t T_, int d, int m, lc_dtype dt, void *Kc, void *Vc,
                          int64_t rope_pos0, cudaStream_t st);
lc_status rope_launch(void *X, int64_t n, int hv, int d, int64_t pos0, int inverse, lc_dtype dt,
                      cudaStream_t st);
lc_status compress_tok_launch(const void *X, const float *Z, int64_t T_, int d, int m,
                              lc_dtype dt, void *Xc, int64_t rope_pos0, cudaStream_t st);
lc_status decode_append_launch(const AppendArgs &a, lc_dtype dt, cudaStream_t st);
lc_status index_launch(const void *qI, const float *w, const void *kI, const lc_batch &b, int HI,
                       int dI, int m, lc_dtype dt, float *scores, int64_t ld, int32_t *dev_err,
                       cudaStream_t st);
lc_status topk_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                      int32_t *topk, int32_t *dev_err, cudaStream_t st);
lc_status index_tc_materialize(const void *qI, const float *w, const void *kI, const lc_batch &b,
                               int HI, int dI, int m, lc_dtype dt, float *scores, int64_t ld,
                               int32_t *dev_err, cudaStream_t st);
lc_status index_topk_tc_launch(const void *qI, const float *w, const void *kI,
                               const lc_batch &b, int HI, int dI, int m, lc_dtype dt, int k,
                               int32_t *topk, void *ws, size_t ws_bytes, int32_t *dev_err,
                               cudaStream_t st);
size_t index_tc_workspace(const lc_batch &b, int k);
lc_status mx_quantize_launch(const void *X, int64_t n, int fmt, lc_dtype dt, uint8_t *codes,
                             uint8_t *scales, cudaStream_t st);
lc_status index_rows_launch(const void *qI, const float *w, const void *kI, const lc_batch &b,
                            int HI, int dI, int m, lc_dtype dt, float *scores, int64_t ld,
                            int64_t r0, int64_t nrows, int32_t *dev_err, cudaStream_t st);
lc_status topk_rows_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                           int32_t *topk, int64_t r0, int64_t nrows, int32_t *dev_err,
                           cudaStream_t st);
lc_status index_mx_launch(int fmt, const uint8_t *qc, const uint8_t *qs, const float *w,
                          const uint8_t *kc, const uint8_t *ks, const lc_batch &b, int HI, int m,
                          float *scores, int64_t ld, int64_t r0, int64_t nrows, int32_t *dev_err,
                          cudaStream_t st);
lc_status hca_tc_launch(const void *Q, const void *Kc, const void *Vc, const void *Kraw,
                        const void *Vraw, const lc_batch &b, int H, int d, int m, int W,
                        float scale, const float *sink, int rope, lc_dtype dt, void *O,
                        float *lse, int32_t *dev_err, cudaStream_t st);
lc_status sparse_tc_launch(const void *Q, const void *Kc, const void *Vc, const int32_t *topk,
                           int k, const void *Kraw, const void *Vraw, const lc_batch &b, int H,
                           int d, int m, int W, float scale, const float *sink, int rope,
                           lc_dtype dt, void *O, float *lse, int32_t *dev_err, cudaStream_t st);
lc_status attn_simt_launch(bool sparse, const void *Q, const void *Kc, const void *Vc,
                           const int32_t *topk, int k, const void *Kraw, const void *Vraw,
                           const lc_batch &b, int H, int d, int m, int W, float scale,
                           const float *sink, int rope, lc_dtype dt, void *O, float *lse,
                           int32_t *dev_err, cudaStream_t st);

static std::atomic<uint64_t> g_launches{0};
static std::atomic<uint32_t> g_stall_mask{0};
static std::atomic<long long> g_stall_clocks{0};

long long debug_stall_clocks(uint32_t kernel_bit) {
    return (g_stall_mask.load() & kernel_bit) ? g_stall_clocks.load() : 0;
}

int sm_count() {
    constexpr int kMax = 64;
    static std::atomic<int> cache[kMax];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMax) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMax) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

static std::atomic<int32_t> g_last_cuda{0};

static thread_local const char *g_last_kernel = "";

void note_launch(const char *name) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    g_last_kernel = name;
}

lc_status check_launch() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        g_last_cuda.store((int32_t)e);
        return LC_ERR_CUDA;
    }
    return LC_OK;
}

lc_status check_launch_error(cudaError_t e) {
    g_last_cuda.store((int32_t)e);
    return LC_ERR_CUDA;
}

static bool debug_sync() {
    static int v = -1;
    if (v < 0) {
        const char *s = std::getenv("LC_DEBUG_SYNC");
        v = (s && s[0] == '1') ? 1 : 0;
    }
    return v == 1;
}

// With LC_DEBUG_SYNC=1: wait for the call's kernels and surface device errors.
lc_status finish(lc_status s, cudaStream_t st, int32_t *dev_err) {
    if (s != LC_OK || !debug_sync()) return s;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        g_last_cuda.store((int32_t)e);
        return LC_ERR_CUDA;
    }
    if (dev_err) {
        int32_t h = 0;
        if (cudaMemcpy(&h, dev_err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
            return LC_ERR_CUDA;
        if (h & LC_DEVERR_TIMEOUT) return LC_ERR_TIMEOUT;
        if (h) return LC_ERR_DEVICE_CHECK;
    }
    return LC_OK;
}

bool batch_ok(const lc_batch *b) {
    return b && b->B >= 1 && b->cu_q && b->q_pos0 && b->cu_c && b->cu_raw && b->raw_pos0 &&
           b->total_q >= 0 && b->max_q >= 0 && b->max_c >= 0 && b->max_q <= b->total_q &&
           b->total_c >= b->max_c && b->total_raw >= 0;
}

static bool dtype_ok(lc_dtype dt) { return dt == LC_F32 || dt == LC_BF16; }

static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Scores kept in the workspace by the fused call without the tensor-core
// plan: all rows when that fits in INDEX_WS_CHUNK bytes, else as many rows as
// fit (at least one), taken in turn.
constexpr size_t INDEX_WS_CHUNK = (size_t)64 << 20;

static size_t index_ws_bytes(const lc_batch *b) {
    const size_t row = sizeof(float) * (size_t)b->max_c;
    const size_t all = row * (size_t)b->total_q;
    if (all <= INDEX_WS_CHUNK || row == 0) return align_up(all);
    return align_up(row > INDEX_WS_CHUNK ? row : INDEX_WS_CHUNK / row * row);
}

static lc_status compress_common(const void *K, const void *V, const float *G_K,
                                 const float *G_V, int64_t T, int32_t d, int32_t m,
                                 lc_dtype dt, void *Kc, void *Vc, int64_t rope_pos0,
                                 cudaStream_t st) {
    if (T < 0 || m < 1 || !dtype_ok(dt) || !G_K || !G_V || rope_pos0 < -1)
        return LC_ERR_INVALID_ARG;
    // with fewer than m tokens there is no entry to write: outputs may be empty
    if (T / m > 0 && (!K || !V || !Kc || !Vc)) return LC_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || m > 256) return LC_ERR_UNSUPPORTED;
    return finish(compress_launch(K, V, G_K, G_V, T, d, m, dt, Kc, Vc, rope_pos0, st), st,
                  nullptr);
}

}  // namespace lc

using namespace lc;

extern "C" {

lc_status csa_compress(const void *K, const void *V, const float *G_K, const float *G_V,
                       int64_t T, int32_t d, int32_t m, lc_dtype dtype, void *Kc, void *Vc,
                       int64_t rope_pos0, lc_stream stream) {
    return compress_common(K, V, G_K, G_V, T, d, m, dtype, Kc, Vc, rope_pos0,
                           (cudaStream_t)stream);
}

lc_status hca_compress(const void *K, const void *V, const float *G_K, const float *G_V,
                       int64_t T, int32_t d, int32_t m, lc_dtype dtype, void *Kc, void *Vc,
                       int64_t rope_pos0, lc_stream stream) {
    return compress_common(K, V, G_K, G_V, T, d, m, dtype, Kc, Vc, rope_pos0,
                           (cudaStream_t)stream);
}

lc_status rope_rotate(void *X, int64_t n, int32_t hv, int32_t d, int64_t pos0, int32_t inverse,
                      lc_dtype dtype, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (n < 0 || hv < 1 || pos0 < 0 || !dtype_ok(dtype) || (n > 0 && !X))
        return LC_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return LC_ERR_UNSUPPORTED;
    return finish(rope_launch(X, n, hv, d, pos0, inverse, dtype, st), st, nullptr);
}

lc_status token_gated_compress(const void *X, const float *Z, int64_t T, int32_t d, int32_t m,
                               lc_dtype dtype, void *Xc, int64_t rope_pos0, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (T < 0 || m < 1 || !dtype_ok(dtype) || rope_pos0 < -1) return LC_ERR_INVALID_ARG;
    if (T / m > 0 && (!X || !Z || !Xc)) return LC_ERR_INVALID_ARG;
    if (d < 32 || d > 1024 || d % 32 || m > 4096) return LC_ERR_UNSUPPORTED;
    if (rope_pos0 >= 0 && d < ROPE_DIMS) return LC_ERR_UNSUPPORTED;
    return finish(compress_tok_launch(X, Z, T, d, m, dtype, Xc, rope_pos0, st), st, nullptr);
}

lc_status decode_append(const lc_decode_layer *L, const void *K_new, const void *V_new,
                        const void *kI_new, const float *G_K, const float *G_V,
                        const float *G_I, lc_dtype dtype, int32_t *dev_err, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (!L || L->B < 1 || L->m < 1 || L->R < L->m || L->cap < 1 || L->HI < 0 ||
        !dtype_ok(dtype) || !L->n_tok || !L->Kring || !L->Vring || !L->Kc || !L->Vc ||
        !L->q_pos0 || !L->cu_raw || !L->raw_pos0 || !K_new || !V_new || !G_K || !G_V)
        return LC_ERR_INVALID_ARG;
    if (L->HI > 0 && (L->dI < 1 || !L->kI_ring || !L->kI || !kI_new || !G_I))
        return LC_ERR_INVALID_ARG;
    if ((L->d != 64 && L->d != 128) || (int64_t)L->HI * L->dI > 1024) return LC_ERR_UNSUPPORTED;
    AppendArgs a{L->B, L->R, L->d, L->m, L->HI > 0 ? L->HI * L->dI : 0, L->cap, L->n_tok,
                 L->Kring, L->Vring, L->kI_ring, L->Kc, L->Vc, L->kI, L->q_pos0, L->cu_raw,
                 L->raw_pos0, K_new, V_new, kI_new, G_K, G_V, G_I, dev_err};
    return finish(decode_append_launch(a, dtype, st), st, dev_err);
}

lc_status lightning_index(const void *qI, const float *w, const void *kI, const lc_batch *batch,
                          int32_t HI, int32_t dI, int32_t m, lc_dtype dtype, float *scores,
                          int64_t ld, int32_t k, int32_t *topk, void *ws, size_t ws_bytes,
                          int32_t *dev_err, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (!qI || !w || !kI || !batch_ok(batch) || m < 1 || !dtype_ok(dtype) || (!scores && !topk))
        return LC_ERR_INVALID_ARG;
    if (scores && ld < batch->max_c) return LC_ERR_INVALID_ARG;
    if (topk && k < 1) return LC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kI) & 15u) != 0) return LC_ERR_INVALID_ARG;  // 16-B loads
    if ((HI != 1 && HI != 2 && HI != 4 && HI != 8) || (dI != 32 && dI != 64) ||
        (topk && k > 4096))
        return LC_ERR_UNSUPPORTED;
    if (batch->total_q == 0) return LC_OK;
    if (!scores) {
        // fused selection on the tensor cores when the shape allows it
        lc_status s = index_topk_tc_launch(qI, w, kI, *batch, HI, dI, m, dtype, k, topk, ws,
                                           ws_bytes, dev_err, st);
        if (s != LC_ERR_UNSUPPORTED) return finish(s, st, dev_err);
    }
    float *sc = scores;
    int64_t sld = ld;
    if (!scores) {
        // at least one row of scores; lc_workspace_size's size holds all rows
        // or INDEX_WS_CHUNK bytes of them
        const size_t need = sizeof(float) * (size_t)batch->max_c;
        if (need > 0 && (!ws || ws_bytes < need)) return LC_ERR_WORKSPACE;
        sc = reinterpret_cast<float *>(ws);
        sld = batch->max_c;
        if (sld == 0) {
            lc_status s = topk_launch(sc, 0, *batch, m, k, topk, dev_err, st);
            return finish(s, st, dev_err);
        }
        const int64_t fit = (int64_t)(ws_bytes / (sizeof(float) * (size_t)sld));
        if (fit < batch->total_q) {
            // the scores of `fit` rows at a time, each chunk selected before the next
            lc_status s = LC_OK;
            for (int64_t r0 = 0; r0 < batch->total_q && s == LC_OK; r0 += fit) {
                const int64_t n = std::min(fit, batch->total_q - r0);
                s = index_rows_launch(qI, w, kI, *batch, HI, dI, m, dtype, sc, sld, r0, n,
                                      dev_err, st);
                if (s == LC_OK) s = topk_rows_launch(sc, sld, *batch, m, k, topk, r0, n, dev_err, st);
            }
            return finish(s, st, dev_err);
        }
    }
    lc_status s = LC_ERR_UNSUPPORTED;
    if (scores) s = index_tc_materialize(qI, w, kI, *batch, HI, dI, m, dtype, sc, sld, dev_err, st);
    if (s == LC_ERR_UNSUPPORTED)
        s = index_launch(qI, w, kI, *batch, HI, dI, m, dtype, sc, sld, dev_err, st);
    if (s == LC_OK && topk) s = topk_launch(sc, sld, *batch, m, k, topk, dev_err, st);
    return finish(s, st, dev_err);
}

lc_status mx_quantize(const void *X, int64_t n, int32_t fmt, lc_dtype dtype, uint8_t *codes,
                      uint8_t *scales, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    if (n < 0 || n % 32 != 0 || (fmt != LC_MXFP8 && fmt != LC_MXFP4) || !dtype_ok(dtype) ||
        (n > 0 && (!X || !codes || !scales)))
        return LC_ERR_INVALID_ARG;
    return finish(mx_quantize_launch(X, n, fmt, dtype, codes, scales, st), st, nullptr);
}

lc_status lightning_index_mx(int32_t fmt, const uint8_t *qc, const uint8_t *qs, const float *w,
                             const uint8_t *kc, const uint8_t *ks, const lc_batch *batch,
                             int32_t HI, int32_t dI, int32_t m, float *scores, int64_t ld,
                             int32_t k, int32_t *topk, void *ws, size_t ws_bytes,
                             int32_t *dev_err, lc_stream stream) {
    cudaStream_t st = (cudaStream_t)stream;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if ((fmt != LC_MXFP8 && fmt != LC_MXFP4) || !qc || !qs || !w || !kc || !ks ||
        !batch_ok(batch) || m < 1 || (!scores && !topk) || !al16(qc) || !al16(kc) ||
        (reinterpret_cast<uintptr_t>(ks) & 1u) != 0)
        return LC_ERR_INVALID_ARG;
    if (scores && ld < batch->max_c) return LC_ERR_INVALID_ARG;
    if (topk && k < 1) return LC_ERR_INVALID_ARG;
    if ((HI != 4 && HI != 8) || dI != 64 || (topk && k > 4096) || batch->total_q > 65535)
        return LC_ERR_UNSUPPORTED;
    if (batch->total_q == 0) return LC_OK;
    float *sc = scores;
    int64_t sld = ld;
    int64_t fit = batch->total_q;  // rows whose scores are kept at a time
    if (!scores) {
        const size_t need = sizeof(float) * (size_t)batch->max_c;  // at least one row
        if (need > 0 && (!ws || ws_bytes < need)) return LC_ERR_WORKSPACE;
        sc = reinterpret_cast<float *>(ws);
        sld = batch->max_c;
        if (sld > 0)
            fit = std::min(fit, (int64_t)(ws_bytes / (sizeof(float) * (size_t)sld)));
    }
    lc_status s = LC_OK;
    for (int64_t r0 = 0; r0 < batch->total_q && s == LC_OK; r0 += fit) {
        const int64_t n = std::min(fit, batch->total_q - r0);
        if (sld > 0)
            s = index_mx_launch(fmt, qc, qs, w, kc, ks, *batch, HI, m, sc, sld, r0, n, dev_err,
                                st);
        if (s == LC_OK && topk) s = topk_rows_launch(sc, sld, *batch, m, k, topk, r0, n, dev_err, st);
    }
    return finish(s, st, dev_err);
}

lc_status topk_select(const float *scores, int64_t ld, const lc_batch *batch, int32_t m,
                      int32_t k, int32_t *topk, void *ws, size_t ws_bytes, int32_t *dev_err,
                      lc_stream stream) {
    (void)ws;
    (void)ws_bytes;
    cudaStream_t st = (cudaStream_t)stream;
    if (!batch_ok(batch) || !topk || k < 1 || m < 1 || ld < batch->max_c ||
        (!scores && batch->max_c > 0))
        return LC_ERR_INVALID_ARG;
    if (k > 4096) return LC_ERR_UNSUPPORTED;
    lc_status s = topk_launch(scores, ld, *batch, m, k, topk, dev_err, st);
    return finish(s, st, dev_err);
}

lc_status sparse_mqa_attn(const void *Q, const void *Kc, const void *Vc, const int32_t *topk,
                          int32_t k, const void *Kraw, const void *Vraw, const lc_batch *batch,
                          int32_t H, int32_t d, int32_t m, int32_t W, float scale,
                          const float *sink, int32_t rope, lc_dtype dtype, void *O, float *lse,
                          void *ws, size_t ws_bytes, int32_t *dev_err, lc_stream stream) {
    (void)ws;
    (void)ws_bytes;
    cudaStream_t st = (cudaStream_t)stream;
    if (!Q || !Kc || !Vc || !topk || !O || !batch_ok(batch) || k < 1 || m < 1 || W < 0 ||
        !dtype_ok(dtype) || !(scale > 0.f) || (W > 0 && (!Kraw || !Vraw)) ||
        (rope != 0 && rope != 1))
        return LC_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || H < 8 || H > 128 || H % 8 || W > 4096 || k > 4096)
        return LC_ERR_UNSUPPORTED;
    lc_status s = sparse_tc_launch(Q, Kc, Vc, topk, k, Kraw, Vraw, *batch, H, d, m, W, scale,
                                   sink, rope, dtype, O, lse, dev_err, st);
    if (s == LC_ERR_UNSUPPORTED)
        s = attn_simt_launch(true, Q, Kc, Vc, topk, k, Kraw, Vraw, *batch, H, d, m, W, scale,
                             sink, rope, dtype, O, lse, dev_err, st);
    return finish(s, st, dev_err);
}

lc_status hca_dense_attn(const void *Q, const void *Kc, const void *Vc, const void *Kraw,
                         const void *Vraw, const lc_batch *batch, int32_t H, int32_t d,
                         int32_t m, int32_t W, float scale, const float *sink, int32_t rope,
                         lc_dtype dtype, void *O, float *lse, void *ws, size_t ws_bytes,
                         int32_t *dev_err, lc_stream stream) {
    (void)ws;
    (void)ws_bytes;
    cudaStream_t st = (cudaStream_t)stream;
    if (!Q || !O || !batch_ok(batch) || m < 1 || W < 0 || !dtype_ok(dtype) || !(scale > 0.f) ||
        (batch->max_c > 0 && (!Kc || !Vc)) || (W > 0 && (!Kraw || !Vraw)) ||
        (rope != 0 && rope != 1))
        return LC_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || H < 8 || H > 128 || H % 8 || W > 4096)
        return LC_ERR_UNSUPPORTED;
    lc_status s = hca_tc_launch(Q, Kc, Vc, Kraw, Vraw, *batch, H, d, m, W, scale, sink, rope,
                                dtype, O, lse, dev_err, st);
    if (s == LC_ERR_UNSUPPORTED)
        s = attn_simt_launch(false, Q, Kc, Vc, nullptr, 0, Kraw, Vraw, *batch, H, d, m, W, scale,
                             sink, rope, dtype, O, lse, dev_err, st);
    return finish(s, st, dev_err);
}

size_t lc_workspace_size(int32_t op, const lc_batch *batch, int32_t H, int32_t d, int32_t HI,
                         int32_t dI, int32_t k) {
    (void)H;
    (void)d;
    (void)HI;
    (void)dI;
    (void)k;
    if (!batch) return 0;
    switch (op) {
        case LC_OP_LIGHTNING_INDEX: {
            // the fused tensor-core plan where the shape takes it (bf16 inputs),
            // else scores of bounded row chunks
            const bool tc = (HI == 4 || HI == 8) && dI == 64 && batch->max_q >= 64 &&
                            batch->max_c > 0;
            const size_t a = index_ws_bytes(batch), b = tc ? index_tc_workspace(*batch, k) : 0;
            return a > b ? a : b;
        }
        default: return 0;
    }
}

const char *lc_status_string(int32_t status) {
    switch (status) {
        case LC_OK: return "ok";
        case LC_ERR_INVALID_ARG: return "invalid argument";
        case LC_ERR_UNSUPPORTED: return "unsupported shape or option";
        case LC_ERR_CUDA: return "CUDA error";
        case LC_ERR_TIMEOUT: return "a bounded device wait timed out";
        case LC_ERR_DEVICE_CHECK: return "device-side check failed (see dev_err)";
        case LC_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int32_t lc_last_cuda_error(void) { return g_last_cuda.load(); }

uint64_t lc_launch_count(void) { return g_launches.load(); }

const char *lc_last_kernel(void) { return g_last_kernel; }

void lc_debug_stall(uint32_t kernels, int64_t clocks) {
    g_stall_clocks.store(clocks > 0 ? (long long)clocks : 0);
    g_stall_mask.store(clocks > 0 ? kernels : 0u);
}

const char *lc_version(void) { return "lcattn 0.1 sm_103a"; }

}  // extern "C"
