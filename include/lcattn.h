/*
 * lcattn — Compressed Sparse Attention (CSA) and Heavily Compressed Attention
 * (HCA) for one NVIDIA B300 (sm_103a).
 *
 * The method (page "DeepSeek-V4 技术解析：架构革新与 Coding Agent 后训练优化",
 * §1.1 混合注意力：CSA 与 HCA 的协同; page "DeepSeek-V4 技术报告解读：百万Token
 * 上下文是怎么做到的", §三大架构改动 1-2): the KV of every m tokens is folded
 * into one compressed entry; a Lightning Indexer scores every query against
 * the compressed entries; a causal top-k keeps the k best; MQA attention runs
 * over the kept entries plus an uncompressed sliding window.  HCA folds every
 * m' >> m tokens and attends densely over all visible entries plus the window.
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     the comment says otherwise.  The library never allocates, frees, or
 *     keeps a pointer past the call; scratch memory is the caller's
 *     `ws` buffer of at least lc_workspace_size() bytes.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream):
 *     it validates its host-side arguments, enqueues kernels and returns.
 *     It never synchronises unless the environment variable LC_DEBUG_SYNC=1
 *     is set, in which case it waits for its kernels and reports device-side
 *     errors through the return value.
 *   - Layouts are row-major with a contiguous last dimension.  `lc_dtype`
 *     selects the type of the activations (Q, K, V, compressed entries,
 *     indexer q/k, O); gate logits, head weights, scores and LSE are fp32.
 *     All arithmetic is fp32; outputs are rounded once (round-to-nearest-even).
 *   - Errors: invalid host arguments return LC_ERR_INVALID_ARG and enqueue
 *     nothing; a shape outside the supported set returns LC_ERR_UNSUPPORTED;
 *     a CUDA launch failure returns LC_ERR_CUDA (see lc_last_cuda_error()).
 *     Kernels never trap.  A bad value found on the device (an entry index out
 *     of range or not yet visible, a window position the raw cache does not
 *     hold, an inconsistent batch descriptor) is skipped and OR-ed as a bit of
 *     lc_dev_error into *dev_err when dev_err is not NULL.
 *
 * Notation: t = absolute position of a query row; entry j of a sequence is
 * visible from t iff (j+1)*m - 1 <= t, so n_vis(t) = floor((t+1)/m); the
 * window of t is raw positions max(0, t-W+1) .. t.
 */
#ifndef LCATTN_H
#define LCATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *lc_stream; /* a cudaStream_t */

typedef enum {
    LC_OK = 0,
    LC_ERR_INVALID_ARG = 1,
    LC_ERR_UNSUPPORTED = 2,
    LC_ERR_CUDA = 3,
    LC_ERR_TIMEOUT = 4,       /* a bounded device wait expired */
    LC_ERR_DEVICE_CHECK = 5,  /* LC_DEBUG_SYNC=1 only: *dev_err != 0 */
    LC_ERR_WORKSPACE = 6      /* ws too small for this call */
} lc_status;

typedef enum { LC_F32 = 0, LC_BF16 = 1 } lc_dtype;

/* Bits OR-ed into *dev_err by kernels. */
typedef enum {
    LC_DEVERR_INDEX = 1,   /* selected entry index >= stored entries or not visible */
    LC_DEVERR_WINDOW = 2,  /* window position outside the sequence's raw rows */
    LC_DEVERR_BATCH = 4,   /* batch descriptor inconsistent (e.g. n_vis > entries) */
    LC_DEVERR_TIMEOUT = 8, /* a bounded wait inside a kernel gave up */
    LC_DEVERR_SINK = 16    /* a sink logit is NaN or +inf (that head gets no sink) */
} lc_dev_error;

/* Ragged batch.  Every array is on the DEVICE (int64); the three maxima are
 * host values used to size grids.  Sequence b owns query rows
 * cu_q[b] .. cu_q[b+1]-1 at consecutive absolute positions q_pos0[b], ...;
 * compressed entries cu_c[b] .. cu_c[b+1]-1 (sequence-local entry j is row
 * cu_c[b]+j of Kc/Vc/kI); raw rows cu_raw[b] .. cu_raw[b+1]-1 holding
 * positions raw_pos0[b], raw_pos0[b]+1, ... (the window's source).  The
 * host fields must agree with the device arrays; the tensor-core kernels size
 * their TMA descriptors from total_c and total_raw. */
typedef struct {
    int32_t B;
    const int64_t *cu_q;     /* [B+1] */
    const int64_t *q_pos0;   /* [B]   */
    const int64_t *cu_c;     /* [B+1] */
    const int64_t *cu_raw;   /* [B+1] */
    const int64_t *raw_pos0; /* [B]   */
    int64_t total_q;         /* host: cu_q[B] */
    int64_t max_q;           /* host: max over b of rows of sequence b */
    int64_t max_c;           /* host: max over b of entries of sequence b */
    int64_t total_c;         /* host: cu_c[B] (rows of Kc/Vc/kI) */
    int64_t total_raw;       /* host: cu_raw[B] (rows of Kraw/Vraw) */
} lc_batch;

/* CSA token compressor (page "DeepSeek-V4 技术解析…", §1.1, CSA paragraph:
 * a token-level compressor merges the KV of every m tokens into one entry).
 * Form (the pages give none): softmax-gated pooling with position gates,
 *   Kc[j,c] = sum_{p<m} softmax_p(G_K[:,c])[p] * K[j*m+p, c],  j < floor(T/m)
 * and the same for V with G_V.  A tail of T mod m tokens makes no entry.
 *   K, V   [T, d] dtype          G_K, G_V [m, d] fp32 (may alias)
 *   Kc, Vc [floor(T/m), d] dtype (written; must not overlap the inputs)
 *   rope_pos0: -1, or the absolute position of input row 0: then every entry
 *          also gets partial RoPE (LC_ROPE_DIMS below) at the position of its
 *          last token, rope_pos0 + (j+1)*m - 1 (K and V alike).
 * Supported: d in {64, 128}; 1 <= m <= 256; T >= 0. */
lc_status csa_compress(const void *K, const void *V, const float *G_K, const float *G_V,
                       int64_t T, int32_t d, int32_t m, lc_dtype dtype, void *Kc, void *Vc,
                       int64_t rope_pos0, lc_stream stream);

/* HCA compressor (same page, §1.1, HCA paragraph: every m' tokens become one
 * entry, m' much larger than m).  Same arithmetic and arguments as
 * csa_compress; kept as its own entry point because the HCA ratio (128)
 * selects a different launch shape. */
lc_status hca_compress(const void *K, const void *V, const float *G_K, const float *G_V,
                       int64_t T, int32_t d, int32_t m, lc_dtype dtype, void *Kc, void *Vc,
                       int64_t rope_pos0, lc_stream stream);

/* Token-gated compressor (same page, §1.1, CSA paragraph: the token-level
 * compressor is learned, so every token brings its own gate logits).  With
 * Z [T, d] fp32 holding one gate logit per token and channel,
 *   Xc[j,c] = sum_{p<m} softmax_p(Z[j*m+p, c]) * X[j*m+p, c],  j < floor(T/m).
 * Compresses K, V or the token-level indexer keys (d = H_I * d_I) into their
 * entries; a tail of T mod m tokens makes no entry.
 *   X [T, d] dtype;  Z [T, d] fp32;  Xc [floor(T/m), d] dtype (written)
 *   rope_pos0: as for csa_compress (for attention K and V, whose last 64
 *          channels are the rotary ones; -1 for indexer keys).
 * Supported: d % 32 == 0, 32 <= d <= 1024 (d >= 64 with RoPE); 1 <= m <= 4096;
 * T >= 0. */
lc_status token_gated_compress(const void *X, const float *Z, int64_t T, int32_t d, int32_t m,
                               lc_dtype dtype, void *Xc, int64_t rope_pos0, lc_stream stream);

/* Partial RoPE (same page, §1.1, engineering details: RoPE acts only on the
 * last 64 dimensions; the core-attention output gets the inverse RoPE to
 * restore relative positions).  Pairs (2i, 2i+1), i < 32, of the last 64
 * dimensions of a vector at position p are rotated by p * theta_i,
 * theta_i = 10000^(-i/32).  With RoPE, queries rotate at their position t,
 * compressed entries at their last token's position (csa_compress), raw
 * window tokens at their own positions, values like keys, and the attention
 * output rotates back by -t.
 * rope_rotate rotates in place rows i = 0 .. n-1 of X [n, hv, d] (hv vectors
 * per row) at positions pos0 + i, or back (inverse = 1): use it on the raw
 * window cache, whose tokens are stored rotated.
 * Supported: d in {64, 128}; hv >= 1; pos0 >= 0. */
#define LC_ROPE_DIMS 64
lc_status rope_rotate(void *X, int64_t n, int32_t hv, int32_t d, int64_t pos0, int32_t inverse,
                      lc_dtype dtype, lc_stream stream);

/* Lightning Indexer (same page, §1.1, CSA paragraph: a light indexer scores
 * the compressed KV blocks against the query), with the form
 *   I[r,j] = sum_{h<HI} w[r,h] * max(0, qI[r,h,:] . kI[cu_c[b]+j,h,:])
 * for j < n_vis(t_r); other columns < ld are -inf.
 *   qI [total_q, HI, dI] dtype;  w [total_q, HI] fp32;  kI [cu_c[B], HI, dI] dtype
 *   scores [total_q, ld] fp32, ld >= max_c, or NULL
 *   topk   [total_q, k] int32 or NULL: when non-NULL the call also selects
 *          (as topk_select) and, if scores is NULL, keeps the scores in ws:
 *          with bf16 inputs, H_I in {4, 8}, d_I = 64 and a sequence of at
 *          least 64 query rows, the fused tensor-core selection (ws at least
 *          lc_workspace_size); otherwise the scores of as many rows as ws
 *          holds at a time (ws at least one row, max_c * 4 bytes).
 * At least one of scores / topk must be non-NULL; kI must be 16-byte aligned.
 * Supported: HI in {1,2,4,8}; dI in {32,64}; 1 <= k <= 4096. */
lc_status lightning_index(const void *qI, const float *w, const void *kI, const lc_batch *batch,
                          int32_t HI, int32_t dI, int32_t m, lc_dtype dtype, float *scores,
                          int64_t ld, int32_t k, int32_t *topk, void *ws, size_t ws_bytes,
                          int32_t *dev_err, lc_stream stream);

/* Low-precision indexer (page "DeepSeek V4 详解：1M 上下文背后，真正发生了什么",
 * §"mHC、Muon、FP4": FP4 runs in the CSA indexer's QK path, and the quantized
 * selector keeps almost all of the exact selection; "DeepSeek-V4 技术解析…",
 * §1.1: the indexer computes in FP4).  q_I and k_I are stored in an OCP MX
 * (microscaling, v1.0) format: blocks of 32 consecutive values share one
 * power-of-two scale X = 2^(floor(log2 amax) - emax), kept as an E8M0 byte
 * (exponent + 127; an all-zero block gets 2^-127), and each value becomes
 * the element nearest to v / X (ties to the even mantissa), clamped to the
 * largest finite element.
 *   LC_MXFP8  E4M3 elements (largest 448, emax 8), one byte per value;
 *   LC_MXFP4  E2M1 elements (largest 6, emax 2), two values per byte, the
 *             even-indexed value in the low nibble. */
#define LC_MXFP8 8
#define LC_MXFP4 4

/* X [n] (dtype; n % 32 == 0; block i = values 32i .. 32i+31) ->
 *   codes [n] bytes (LC_MXFP8) or [n / 2] bytes (LC_MXFP4), scales [n / 32]
 *   E8M0 bytes.  Values must be finite.  n = 0 enqueues nothing. */
lc_status mx_quantize(const void *X, int64_t n, int32_t fmt, lc_dtype dtype, uint8_t *codes,
                      uint8_t *scales, lc_stream stream);

/* lightning_index on MX-quantized indexer queries and keys, each head's d_I
 * values being d_I / 32 blocks:
 *   I[r,j] = sum_h w[r,h] * max(0, q^[r,h,:] . k^[cu_c[b]+j,h,:]),
 *   v^ = element * X (the dequantized value), fp32 accumulation;
 *   qc, qs: mx_quantize of qI [total_q, HI, dI]; kc, ks: of kI [cu_c[B], HI, dI];
 *   scores, ld, k, topk, ws, ws_bytes: as lightning_index (the selection is
 *   the exact top-k of these scores; ws: lc_workspace_size of
 *   LC_OP_LIGHTNING_INDEX).  qc and kc must be 16-byte aligned, ks 2-byte
 *   aligned.
 * Supported: dI = 64; HI in {4, 8}; total_q <= 65535; 1 <= k <= 4096. */
lc_status lightning_index_mx(int32_t fmt, const uint8_t *qc, const uint8_t *qs, const float *w,
                             const uint8_t *kc, const uint8_t *ks, const lc_batch *batch,
                             int32_t HI, int32_t dI, int32_t m, float *scores, int64_t ld,
                             int32_t k, int32_t *topk, void *ws, size_t ws_bytes,
                             int32_t *dev_err, lc_stream stream);

/* Causal top-k selector (same page, §1.1: the top-k selector keeps the most
 * relevant compressed entries, 1024 in the Pro setting).  For row r keep the
 * min(k, n_vis(t_r)) columns j < n_vis(t_r) that rank first under the total
 * order (larger score first; equal scores: lower j first; -0.0 equals +0.0),
 * written as ascending sequence-local j, then -1 up to k.  Scores must be
 * finite in the visible columns (not checked).
 *   scores [total_q, ld] fp32;  topk [total_q, k] int32 */
lc_status topk_select(const float *scores, int64_t ld, const lc_batch *batch, int32_t m,
                      int32_t k, int32_t *topk, void *ws, size_t ws_bytes, int32_t *dev_err,
                      lc_stream stream);

/* CSA core attention (same page, §1.1: MQA core attention over the kept
 * entries; extra sliding-window branch; a learnable attention-sink logit per
 * head that can push the head's total attention toward 0).  For query row
 * r, head h, with z_s = scale * Q[r,h].K_s and sink logit s_h:
 *   S = { Kc/Vc row cu_c[b]+topk[r,i] : topk[r,i] >= 0 }  then
 *       { raw row of position p : max(0,t-W+1) <= p <= t }
 *   O[r,h]   = sum_{s in S} e^{z_s} V_s / (e^{s_h} + sum_{s in S} e^{z_s})
 *   lse[r,h] = log(e^{s_h} + sum_{s in S} e^{z_s})
 * Without a sink (sink NULL, or s_h = -inf) this is one softmax over S; an
 * empty S gives O = 0 and lse = s_h (-inf without a sink).
 *   Q [total_q, H, d]; Kc, Vc [cu_c[B], d]; Kraw, Vraw [cu_raw[B], d] (dtype)
 *   topk [total_q, k] int32 (-1 = unused slot); O [total_q, H, d] dtype;
 *   sink [H] fp32 (natural-log units, like z) or NULL; at least H values,
 *        on the same device as Q; each finite or -inf (no sink for that
 *        head); a NaN or +inf value raises LC_DEVERR_SINK and that head is
 *        computed without a sink;
 *   rope 0 or 1: with 1, Q is rotated at t (partial RoPE, see rope_rotate)
 *        and O rotated back at t; Kc/Vc and Kraw/Vraw must hold rotated
 *        entries and tokens (csa_compress with rope_pos0, rope_rotate);
 *   lse [total_q, H] fp32 or NULL.
 * Supported: d in {64,128}; H % 8 == 0, 8 <= H <= 128; 0 <= W <= 4096. */
lc_status sparse_mqa_attn(const void *Q, const void *Kc, const void *Vc, const int32_t *topk,
                          int32_t k, const void *Kraw, const void *Vraw, const lc_batch *batch,
                          int32_t H, int32_t d, int32_t m, int32_t W, float scale,
                          const float *sink, int32_t rope, lc_dtype dtype, void *O, float *lse,
                          void *ws, size_t ws_bytes, int32_t *dev_err, lc_stream stream);

/* HCA dense attention (same page, §1.1, HCA paragraph: dense attention over
 * every compressed entry).  As sparse_mqa_attn (sink and rope included) with
 *   S = { entries j < n_vis(t) in order }  then the window. */
lc_status hca_dense_attn(const void *Q, const void *Kc, const void *Vc, const void *Kraw,
                         const void *Vraw, const lc_batch *batch, int32_t H, int32_t d,
                         int32_t m, int32_t W, float scale, const float *sink, int32_t rope,
                         lc_dtype dtype, void *O, float *lse, void *ws, size_t ws_bytes,
                         int32_t *dev_err, lc_stream stream);

/* Incremental decode state of one layer (page "DeepSeek V4 详解：1M 上下文背后，
 * 真正发生了什么", §"第二刀"：the KV cache is a classical cache of compressed
 * entries plus a per-request state cache of fixed size holding the sliding
 * window and the tail of tokens that do not fill a block yet).  Every array
 * is on the device and owned by the caller; per request b:
 *   classical cache: entry j at row b*cap + j of Kc, Vc [B*cap, d] and, for a
 *     CSA layer, of the indexer keys kI [B*cap, HI*dI];
 *   state cache: a mirrored ring of the last R raw tokens, K/V rows
 *     b*2R + p%R and b*2R + p%R + R both hold position p (Kring, Vring
 *     [B*2R, d]); for a CSA layer, kI_ring [B*m, HI*dI] holds the token-level
 *     indexer keys of the open block at slot p % m;
 *   n_tok[b]: tokens held (the next token's position);
 *   q_pos0 [B], cu_raw [B+1], raw_pos0 [B]: batch-descriptor arrays that
 *     decode_append rewrites.  With cu_q = 0..B and cu_c[b] = b*cap they form
 *     the lc_batch (total_q = B, max_q = 1, max_c = cap, total_c = B*cap,
 *     total_raw = B*2R) that the step's index and attention calls take: the
 *     query of request b at its newest position, its window read from the
 *     ring. */
typedef struct {
    int32_t B, R, d, m;   /* requests, ring rows (>= m and >= the window), head dim, ratio */
    int32_t HI, dI;       /* indexer heads and dim of a CSA layer; HI = 0: none */
    int64_t cap;          /* entries per request in the classical cache */
    int64_t *n_tok;
    void *Kring, *Vring, *kI_ring, *Kc, *Vc, *kI;
    int64_t *q_pos0, *cu_raw, *raw_pos0;
} lc_decode_layer;

/* Appends one token per request: K_new, V_new [B, d] (and kI_new [B, HI*dI]
 * for a CSA layer) go into the state cache; a token that closes a block (its
 * position t has (t+1) % m == 0) also writes the block's entry
 * (the csa_compress pooling with gates G_K, G_V [m, d] and, for the indexer
 * keys, G_I [m, HI*dI]); then the batch arrays advance to the new token.
 * A block past the classical cache's capacity is skipped and raises
 * LC_DEVERR_BATCH.  No RoPE (entries and ring hold unrotated values).
 * Supported: d in {64, 128}; 1 <= m <= R; HI*dI <= 1024. */
lc_status decode_append(const lc_decode_layer *layer, const void *K_new, const void *V_new,
                        const void *kI_new, const float *G_K, const float *G_V,
                        const float *G_I, lc_dtype dtype, int32_t *dev_err, lc_stream stream);

/* Index + top-k that allocates nothing (the pages have no counterpart: this
 * is an addition for callers that cannot allocate device memory, such as a
 * host program whose device memory belongs to another runtime's pool, or a
 * latency-critical loop where cudaMalloc/cudaFree could synchronise the
 * device).  Same arguments and results as lightning_index with scores ==
 * NULL and topk != NULL, but the fp32 score matrix [total_q, max_c] lives in
 * a fixed array of LC_NOALLOC_SCRATCH_BYTES compiled into the library instead
 * of a caller workspace.
 *   - Each device that loads the library's image holds that array until the
 *     process exits.
 *   - The first call on a device looks the array's device address up (with
 *     that device current) and keeps it; make that first call before any
 *     stream capture.  The address is not looked up again, so this entry
 *     point must not be called after a cudaDeviceReset of that device in the
 *     same process.
 *   - LC_DEBUG_SYNC=1 makes it wait and report device errors like the
 *     other calls.
 *   - Every call on a device shares the one array, so calls that overlap on
 *     the GPU (other streams, other host threads) race.  Nothing needs
 *     clearing between calls: each call writes every score it reads.
 *   - total_q * max_c * 4 > LC_NOALLOC_SCRATCH_BYTES returns LC_ERR_WORKSPACE
 *     and enqueues nothing.
 *   - No cudaMalloc, cudaFree or allocating library routine is called. */
#define LC_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
lc_status lightning_index_topk_noalloc(const void *qI, const float *w, const void *kI,
                                       const lc_batch *batch, int32_t HI, int32_t dI, int32_t m,
                                       lc_dtype dtype, int32_t k, int32_t *topk,
                                       int32_t *dev_err, lc_stream stream);

/* Bytes of `ws` a call needs (0 = none).  `op` is one of lc_op; unused
 * arguments are ignored.  Host only; reads only the batch's host fields.
 * LC_OP_LIGHTNING_INDEX: the fused tensor-core plan where the shape takes it,
 * and at most 64 MiB of score rows otherwise (the whole score matrix is
 * never required). */
typedef enum {
    LC_OP_LIGHTNING_INDEX = 0, /* with topk != NULL and scores == NULL */
    LC_OP_TOPK_SELECT = 1,
    LC_OP_SPARSE_MQA_ATTN = 2,
    LC_OP_HCA_DENSE_ATTN = 3
} lc_op;
size_t lc_workspace_size(int32_t op, const lc_batch *batch, int32_t H, int32_t d, int32_t HI,
                         int32_t dI, int32_t k);

/* Diagnostics (host only). */
const char *lc_status_string(int32_t status);
int32_t lc_last_cuda_error(void);   /* cudaError_t of the last failed launch */
uint64_t lc_launch_count(void);     /* kernels this library has launched so far */
const char *lc_last_kernel(void);   /* name of the last kernel launched by this host
                                       thread ("" before the first launch) */
const char *lc_version(void);

/* Test hook for the bounded device waits (the pages have no counterpart).
 * While set, every launch of the tensor-core kernels named by `kernels`
 * (a mask of lc_stall_kernel) starts with its MMA issuer waiting, for at most
 * `clocks` SM clocks, on a barrier that nothing completes, before any copy is
 * consumed or any MMA issued.  The wait gives up, the CTA abandons its work,
 * frees its tensor memory and raises LC_DEVERR_TIMEOUT, so the call's output
 * is not computed.  clocks <= 0 turns the hook off.  Host only; not for
 * production use. */
typedef enum {
    LC_STALL_INDEX_TC = 1,   /* tensor-core Lightning Indexer */
    LC_STALL_SPARSE_TC = 2,  /* tensor-core CSA attention */
    LC_STALL_HCA_TC = 4      /* tensor-core HCA attention */
} lc_stall_kernel;
void lc_debug_stall(uint32_t kernels, int64_t clocks);

#ifdef __cplusplus
}
#endif
#endif /* LCATTN_H */
