// Lightning Indexer on the tensor cores (tcgen05 + TMEM), bf16 q/k with
// d_I = 64, H_I in {4, 8}, any ragged batch, plus the fused exact top-k that
// never writes the full score matrix.
//
// k_index_tc: one CTA = 128 query rows x a contiguous range of entries.
//   q_I of the 128 rows stays in shared memory (one 16 KB TMA box per head)
//   for the CTA's lifetime, so all 512 TMEM columns hold score buffers.
//   warp 16     TMA producer: q_I once, then per tile of 128 entries one 16 KB
//               box per head into a ring of four head boxes (one per score
//               buffer)
//   warps 17-18 MMA issuers (warp 17 also owns TMEM): per tile, head by
//               head, one M=128, N=128, K=64 product q_h k_h^T into one of four
//               128-column TMEM score buffers (score buffer g % 4 for the g-th
//               head of the CTA); warp 17 issues the even heads and warp 18
//               the odd ones, so the short tensor-core queue stays fed while
//               one issuer waits; a buffer is reused four heads later.  One
//               commit per head: its arrival on k_empty of the head box's
//               ring slot both frees the box for the producer and tells the
//               epilogue that the head's scores are in TMEM (a commit costs
//               the tensor pipe about 40 cycles)
//   warps 0-15  epilogue: warp w owns TMEM lanes 32(w%4).. (its query rows)
//               and columns 32(w/4).. of each buffer; it folds the heads in
//               order, acc = fma(w_h / 2, s_h + |s_h|, acc) (= w_h max(s_h, 0)
//               in all but overflow cases), two columns per packed fp32x2
//               add and FMA, then either stores the 32 scores of the tile
//               (MATERIALIZE) or appends the entries whose score reaches the
//               row's threshold to the row's candidates (FILTER).  The
//               threshold test is a sign-bit collect of acc - theta; each
//               lane then takes one of its candidates per round, its score
//               picked from the registers by a select tree on the column's
//               bits (about 1.5 rounds per warp and tile).  A buffer is
//               handed back to its issuer through an mbarrier (one arrival
//               per warp) as soon as the warp's TMEM read completes.
// The fused top-k of a row (see index_topk_tc_launch):
//   1. the top 16 bits of the order keys of every s-th entry's score
//      (SAMPLE16 over a strided tensor map, visible columns only);
//   2. theta = the rho-th largest sampled key (a lower bound of it, from the
//      truncated keys), below the k-th largest key of the full row with
//      overwhelming probability;
//   3. FILTER pass over all entries: candidates = entries with key >= theta,
//      written to slots private to (row, CTA column), reserved by a
//      shared-memory atomic, with a shared overflow region per row;
//   4. exact top-k of the candidates, valid when the row has between k and
//      `cap` candidates: then every member of the true top-k is a candidate;
//   5. rows outside that range (rare: massive ties or an unlucky sample) go
//      to a list that a fixed grid redoes exactly from recomputed scores, a
//      row buffer per CTA.
// Both passes run the same arithmetic, so a sampled score and the FILTER
// pass's score of the same entry are bit-identical.
#include <cmath>

#include "lc_common.cuh"
#include "sm100.cuh"
#include "topk_common.cuh"

namespace lc {

using namespace sm100;

lc_status sample_threshold16_launch(const uint16_t *samp, int64_t lds, const lc_batch &b, int m,
                                    int stride, int k, int rho, uint32_t *theta, int32_t *count,
                                    int32_t *nfail, cudaStream_t st);
lc_status cand_pick_warp_launch(const lc_batch &b, int m, int k, int cap, int ocap, int nwmax,
                                const int32_t *count, const uint2 *cand, const int32_t *lcnt,
                                const uint2 *priv, int gy, int cloc, int32_t *topk,
                                int32_t *flist, int32_t *nfail, int32_t *dev_err,
                                cudaStream_t st);
lc_status topk_fallback_launch(const void *qI, const float *w, const void *kI, const lc_batch &b,
                               int HI, int m, int k, const int32_t *flist, const int32_t *nfail,
                               float *buf, int64_t ldb, int grid, int32_t *topk,
                               cudaStream_t st);

namespace {
constexpr int IBM = 128;          // query rows per CTA
constexpr int IBN = 128;          // entries per tile
constexpr int IDI = 64;           // indexer head dim
constexpr int NEPI = 512;         // epilogue threads (16 warps)
constexpr int I_THREADS = NEPI + 96;  // + producer warp + two MMA warps
constexpr int EPI_COLS = 32;      // columns of a score buffer per epilogue thread
constexpr int NBUF = 4;           // TMEM score buffers (one head each)
constexpr int NSB = 4;            // shared-memory head boxes in flight (one per score buffer)
constexpr uint32_t I_TMEM_COLS = 512;
// threads of the CTA-per-row candidate pick: 256 lets four CTAs share an SM
// (their shared memory is the limit) and halves each block-wide barrier
// (126 us per 4096-row step against 147 with 512)
constexpr int PICK_NT = 256;
static_assert(NSB == NBUF, "the epilogue waits on the key box's slot of its score buffer");
constexpr int MODE_MATERIALIZE = 0, MODE_FILTER = 1, MODE_SAMPLE16 = 2;

struct IdxCfg {
    static constexpr uint32_t HEAD_BOX = IBN * 128;         // 128 entries x 128 B
    static constexpr uint32_t Q_BOX = IBM * 128;             // 128 query rows x 128 B
    static constexpr uint32_t SM_Q = 0;                      // 8 heads of q_I
    static constexpr uint32_t SM_K = SM_Q + 8 * Q_BOX;       // ring of head boxes
    static constexpr uint32_t SM_BAR = SM_K + NSB * HEAD_BOX;
    static constexpr uint32_t SM_LCNT = SM_BAR + 256;          // FILTER: per-row slot counters
    static constexpr uint32_t SMEM = SM_LCNT + IBM * 4;
};

struct IdxBars {
    // k_empty[s]: the MMA of the box in slot s is complete (producer and epilogue)
    uint64_t q_full, k_full[NSB], k_empty[NSB];
    // releases of each score buffer: every epilogue warp arrives once its
    // reads of a use of the buffer are complete
    uint64_t freed[NBUF];
    uint64_t fin[2];          // each MMA issuer's last commit
    uint64_t stall;           // test hook: a barrier nothing completes
    uint32_t taddr;
    int abort;
};
static_assert(sizeof(IdxBars) <= IdxCfg::SM_LCNT - IdxCfg::SM_BAR, "indexer barriers");



// Lane 0 of the warp arrives on `bar` (a predicated instruction, no branch);
// called after tcgen05.wait::ld and tcgen05.fence::before_thread_sync so the
// MMA issuer that waits on `bar` may overwrite the buffer just read.
__device__ __forceinline__ void arrive_lane0(uint64_t *bar, int lane) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.eq.s32 p, %1, 0;\n\t"
        "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar)),
        "r"(lane)
        : "memory");
}

// Column c (0..31) of an epilogue thread's scores, held as pairs (column 2j
// in p[j].x, 2j+1 in p[j].y), taken by a select tree on the bits of c, so
// that a candidate's score needs neither a dynamically indexed register nor
// a round trip through shared memory.
__device__ __forceinline__ float col_of(const float2 (&p)[EPI_COLS / 2], int c) {
    float2 l8[8], l4[4], l2[2];
#pragma unroll
    for (int i = 0; i < 8; ++i) l8[i] = (c & 16) ? p[i + 8] : p[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) l4[i] = (c & 8) ? l8[i + 4] : l8[i];
#pragma unroll
    for (int i = 0; i < 2; ++i) l2[i] = (c & 4) ? l4[i + 2] : l4[i];
    const float2 q = (c & 2) ? l2[1] : l2[0];
    return (c & 1) ? q.y : q.x;
}

// Inverse of order_key: the float whose key is `key` (+0 for the key of
// +-0).  Key 0 (below every finite score) maps to -inf.
__device__ __forceinline__ float key_to_float(uint32_t key) {
    if (key == 0u) return -INFINITY;
    const uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
    return __uint_as_float(u);
}
}  // namespace

struct IdxTcArgs {
    Batch bt;                // device batch arrays (any number of sequences)
    int64_t total_q;         // host: query rows of the batch (grid size)
    const __nv_bfloat16 *qI; // [total_q, HI, 64]
    int stride;              // map entry e of a sequence is its entry e*stride
    int m;
    int64_t chunk;           // map entries per CTA (multiple of IBN)
    int64_t col_end;         // MATERIALIZE, SAMPLE16: map columns [0, col_end)
    const float *w;          // [Nq, HI]
    float *out;              // MATERIALIZE: [Nq, ld]
    uint16_t *out16;         // SAMPLE16: [Nq, ld] top 16 bits of the order keys
    int64_t ld;
    int vec_out;             // MATERIALIZE: out and ld allow 16-byte stores
    const uint32_t *theta;   // FILTER: [Nq] order-key thresholds
    uint2 *cand;             // FILTER: [Nq, ocap] overflow slots (order key, entry index)
    int32_t *count;          // FILTER: [Nq] overflow slots used (zeroed beforehand)
    uint2 *priv;             // FILTER: [Nq, gy, cloc] slots private to (row, CTA column)
    int32_t *lcnt;           // FILTER: [Nq, gy] private slots used
    int gy, cloc;
    int ocap;                // overflow slots per row
    int32_t *dev_err;
    long long stall;         // test hook (0: off): both MMA issuers first wait this
                             // many clocks on a barrier nothing completes
};

template <int MODE, int HI>
__global__ void __launch_bounds__(I_THREADS, 1)
    k_index_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               IdxTcArgs a) {
    using C = IdxCfg;
    extern __shared__ __align__(1024) uint8_t smem[];
    IdxBars &bars = *reinterpret_cast<IdxBars *>(smem + C::SM_BAR);
    volatile int *abort = &bars.abort;
    const unsigned FULL = 0xffffffffu;

    // the CTA's sequence and its 128-row tile there: sequence b owns
    // ceil(rows_b / 128) consecutive CTAs along x; the grid has up to one
    // surplus CTA per sequence, which leaves before any barrier
    const SeqTile sq = locate_tile(a.bt, blockIdx.x, 1, IBM);
    if (sq.b == a.bt.B) return;
    const int64_t tile = sq.tile, q_beg = sq.q_beg, nq = sq.nq;
    const int64_t q_pos0 = sq.q_pos0, c_beg = sq.c_beg, Tc = sq.c_end - sq.c_beg;
    const int64_t row0 = tile * IBM;  // sequence-local; global row = q_beg + local
    const int64_t last_row = min(row0 + IBM, nq) - 1;
    int64_t nv_last = n_vis(q_pos0 + last_row, a.m);
    if (nv_last > Tc) nv_last = Tc;
    const int64_t nvm = (nv_last + a.stride - 1) / a.stride;  // visible map entries (max)
    const int64_t c0 = (int64_t)blockIdx.y * a.chunk;
    const int64_t c_end = MODE != MODE_FILTER ? min(c0 + a.chunk, a.col_end)
                                              : min(c0 + a.chunk, nvm);
    const int64_t comp_end = min(c_end, nvm);  // computed columns [c0, comp_end)
    const int n_t = comp_end > c0 ? (int)((comp_end - c0 + IBN - 1) / IBN) : 0;
    const int n_all = n_t * HI;  // head boxes / score buffers of this CTA
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (n_t == 0) {
        // Nothing to compute (every column of the CTA is past its rows' visible
        // entries): write what the CTA owes and leave before any mbarrier or
        // tcgen05 instruction, so that every CTA that runs one holds tensor
        // memory.  MATERIALIZE: columns [c0, c_end) of the rows are -inf.
        // FILTER: the rows have no candidate in this CTA column.
        // SAMPLE16: nothing (only visible columns are stored, and none is here)
        if (MODE == MODE_MATERIALIZE) {
            for (int r = warp; r < IBM && row0 + r < nq; r += I_THREADS / 32) {
                float *dst = a.out + (q_beg + row0 + r) * a.ld;
                for (int64_t e = c0 + lane; e < c_end; e += 32) dst[e] = -INFINITY;
            }
        } else if (MODE == MODE_FILTER) {
            for (int r = tid; r < IBM; r += I_THREADS)
                if (row0 + r < nq) a.lcnt[(size_t)(q_beg + row0 + r) * a.gy + blockIdx.y] = 0;
        }
        return;
    }

    if (tid == 0) {
        bars.abort = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
        if (bars.abort) flag(a.dev_err, LC_DEVERR_TIMEOUT);
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.stall, 1);
        mbar_init(&bars.fin[0], 1);
        mbar_init(&bars.fin[1], 1);
        for (int s = 0; s < NSB; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) mbar_init(&bars.freed[b], NEPI / 32);
        fence_barrier_init();
    }
    int *lcount = reinterpret_cast<int *>(smem + C::SM_LCNT);  // FILTER: slots used per row
    for (int i = tid; i < IBM; i += I_THREADS) lcount[i] = 0;
    constexpr int W_PROD = NEPI / 32, W_MMA = NEPI / 32 + 1, W_MMA2 = NEPI / 32 + 2;
    if (warp == W_MMA) {
        tmem_alloc(&bars.taddr, I_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = bars.taddr;
    const bool dead = bars.abort != 0;

    if (warp == W_PROD) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && !dead) {
            prefetch_tmap(&mK);
            mbar_expect_tx(&bars.q_full, HI * C::Q_BOX);
#pragma unroll
            for (int h = 0; h < HI; ++h)
                tma_load_2d(smem + C::SM_Q + h * C::Q_BOX, &mQ, &bars.q_full, h * IDI,
                            (int32_t)(q_beg + row0));
            int issued = 0;
            for (int g = 0; g < n_all; ++g) {
                const int s = g % NSB, i = g / HI, h = g % HI;
                if (g >= NSB && !mbar_wait(&bars.k_empty[s], ((g - NSB) / NSB) & 1, abort)) break;
                mbar_expect_tx(&bars.k_full[s], C::HEAD_BOX);
                if (MODE == MODE_SAMPLE16)
                    // the sequence's entry c_beg + e*stride: phase c_beg % stride,
                    // strided row c_beg / stride + e of the 3-D view
                    tma_load_3d(smem + C::SM_K + s * C::HEAD_BOX, &mK, &bars.k_full[s], h * IDI,
                                (int32_t)(c_beg % a.stride),
                                (int32_t)(c_beg / a.stride + c0 + (int64_t)i * IBN));
                else
                    tma_load_2d(smem + C::SM_K + s * C::HEAD_BOX, &mK, &bars.k_full[s], h * IDI,
                                (int32_t)(c_beg + c0 + (int64_t)i * IBN));
                ++issued;
            }
            int dummy = 0;
            for (int g = max(0, issued - NSB); g < issued; ++g)
                mbar_wait(&bars.k_full[g % NSB], (g / NSB) & 1, &dummy, 400000000LL);
            mbar_wait(&bars.q_full, 0, &dummy, 400000000LL);
            // the MMAs' releases of the last boxes: no commit may still be on its
            // way to this CTA's barriers when it exits (skipped after an abort,
            // when some of those MMAs are never issued)
            for (int g = max(0, issued - NSB); g < issued && !*abort; ++g)
                mbar_wait(&bars.k_empty[g % NSB], (g / NSB) & 1, abort);
        }
    } else if (warp == W_MMA || warp == W_MMA2) {
        // ------------------------------------------------------ MMA issuers
        const int par = warp - W_MMA;  // head boxes g with g % 2 == par
        if (lane == 0 && !dead) {
            constexpr uint32_t IDESC = idesc_bf16_f32(IBM, IBN, 0, 0);
            bool ok = (a.stall == 0 || mbar_wait(&bars.stall, 0, abort, a.stall)) &&
                      mbar_wait(&bars.q_full, 0, abort);
            tc_fence_after();
            // operand descriptors of the first q box and the first ring slot; each
            // MMA adds its box and K-step offset
            const uint64_t qd0 = sw128_desc(smem_u32(smem + C::SM_Q), 16, 1024);
            const uint64_t kd0 = sw128_desc(smem_u32(smem + C::SM_K), 16, 1024);
            int mine = 0;  // MMAs this thread issued
            for (int g = par; ok && g < n_all; g += 2) {
                const int s = g % NSB, h = g % HI, b = g % NBUF, u = g / NBUF;
                // The release of buffer b (the epilogue's read of head g-4) comes
                // first: the epilogue reads heads in order, so it also read head
                // g-NSB, whose box is the previous use of slot s (the MMA that
                // read it is complete and the box had landed).  Only then is
                // k_full[s] at most one phase behind box g, which a parity wait
                // needs: waited first, it could pass on the completed phase
                // before that one while box g-NSB is still landing.
                if ((u > 0 && !mbar_wait(&bars.freed[b], (uint32_t)(u - 1) & 1u, abort)) ||
                    !mbar_wait(&bars.k_full[s], (g / NSB) & 1, abort))
                    break;
                tc_fence_after();
                const uint64_t qd = desc_add(qd0, h * C::Q_BOX);
                const uint64_t kd = desc_add(kd0, s * C::HEAD_BOX);
#pragma unroll
                for (int kk = 0; kk < IDI / 16; ++kk)
                    mma_bf16(taddr + b * IBN, desc_add(qd, kk * 32), desc_add(kd, kk * 32), IDESC,
                             kk > 0);
                mma_commit(&bars.k_empty[s]);
                ++mine;
            }
            // none of this thread's MMAs may still run when the tensor memory is
            // freed (after an abort the epilogue no longer waits for them)
            if (mine > 0) {
                int dummy = 0;
                mma_commit(&bars.fin[par]);
                mbar_wait(&bars.fin[par], 0, &dummy, 400000000LL);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int quad = warp & 3, part = warp >> 2;
        const int64_t lrow = row0 + quad * 32 + lane;  // sequence-local
        const bool row_ok = lrow < nq;
        const int64_t row = q_beg + lrow;              // global
        const int64_t t = q_pos0 + (row_ok ? lrow : last_row);
        int64_t nv = n_vis(t, a.m);
        if (nv > Tc) nv = Tc;
        const int64_t nvr = (nv + a.stride - 1) / a.stride;  // this row's visible map entries
        float wh[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) wh[h] = row_ok ? __ldg(a.w + row * HI + h) : 0.f;
        float thf = 0.f;
        if (MODE == MODE_FILTER) thf = row_ok ? key_to_float(__ldg(a.theta + row)) : INFINITY;
        const uint32_t lane_addr = taddr + ((uint32_t)(quad * 32) << 16);
        const uint32_t buf_addr = lane_addr + part * EPI_COLS;
        bool ok = !dead;
        float2 acc[EPI_COLS / 2];
        // head g's MMA is complete once phase g / NSB of k_empty[g % NSB] (the
        // release of its key box; the slot is the score buffer, NSB == NBUF) is.
        // That barrier is never two phases ahead here: its next phase is box
        // g + NSB's, whose MMA waits for this epilogue's release of head g
        for (int i = 0; ok && i < n_t; ++i) {
#pragma unroll
            for (int c = 0; c < EPI_COLS / 2; ++c) acc[c] = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < HI; ++h) {
                // the score buffer of the g-th head is compile-time for HI = 8
                // slot, buffer and phase of the g-th head are compile-time for HI = 8
                const int g = i * HI + h, b = g % NBUF;
                const uint32_t kph = (uint32_t)(g / NBUF) & 1u;
                // the (suspending) try-wait normally succeeds; the bounded loop is the slow path
                if (!__all_sync(FULL, mbar_try_wait(&bars.k_empty[b], kph)) &&
                    !__all_sync(FULL, mbar_wait(&bars.k_empty[b], kph, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[EPI_COLS];
                tmem_ld32(buf_addr + b * IBN, v);
                tmem_wait_ld();
                tc_fence_before();
                arrive_lane0(&bars.freed[b], lane);
                // w * max(s, 0) == (w / 2) * (s + |s|) (exact unless s + |s| overflows
                // or w / 2 is subnormal): the ReLU runs as a packed add with
                // absolute-value operands on the FMA pipe
                const float2 w2 = make_float2(0.5f * wh[h], 0.5f * wh[h]);
#pragma unroll
                for (int c = 0; c < EPI_COLS / 2; ++c) {
                    const float2 s2 = make_float2(v[2 * c], v[2 * c + 1]);
                    const float2 r2 = __fadd2_rn(s2, make_float2(fabsf(s2.x), fabsf(s2.y)));
                    acc[c] = __ffma2_rn(w2, r2, acc[c]);
                }
            }
            if (!ok) break;
            if (!row_ok) continue;
            const int64_t e0 = c0 + (int64_t)i * IBN + part * EPI_COLS;  // map entry of column 0
            if (MODE == MODE_MATERIALIZE) {
                float *dst = a.out + row * a.ld + e0;
                const int64_t vis = nvr - e0, lim = c_end - e0;
                if (a.vec_out && vis >= EPI_COLS && lim >= EPI_COLS) {
#pragma unroll
                    for (int u = 0; u < EPI_COLS / 4; ++u)
                        reinterpret_cast<float4 *>(dst)[u] =
                            make_float4(acc[2 * u].x, acc[2 * u].y, acc[2 * u + 1].x,
                                        acc[2 * u + 1].y);
                } else {
#pragma unroll
                    for (int c = 0; c < EPI_COLS; ++c) {
                        const float s = (c & 1) ? acc[c >> 1].y : acc[c >> 1].x;
                        if (c < lim) dst[c] = c < vis ? s : -INFINITY;
                    }
                }
            } else if (MODE == MODE_SAMPLE16) {
                // the top 16 bits of each visible column's order key (a key
                // truncated this way is a lower bound of the full key)
                uint16_t *dst = a.out16 + row * a.ld + e0;
                const int64_t vis = min(nvr, c_end) - e0;
                if (vis >= EPI_COLS) {
                    uint32_t p[EPI_COLS / 2];
#pragma unroll
                    for (int c = 0; c < EPI_COLS / 2; ++c)
                        p[c] = (order_key(acc[c].x) >> 16) | (order_key(acc[c].y) & 0xffff0000u);
#pragma unroll
                    for (int u = 0; u < EPI_COLS / 8; ++u)
                        reinterpret_cast<uint4 *>(dst)[u] =
                            make_uint4(p[4 * u], p[4 * u + 1], p[4 * u + 2], p[4 * u + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < EPI_COLS; ++c) {
                        const float sv = (c & 1) ? acc[c >> 1].y : acc[c >> 1].x;
                        if (c < vis) dst[c] = (uint16_t)(order_key(sv) >> 16);
                    }
                }
            } else {
                // bit c of `below` (after the reversal) = column c is under theta
                const float2 nt = make_float2(-thf, -thf);
                uint32_t below = 0;
#pragma unroll
                for (int c = 0; c < EPI_COLS / 2; ++c) {
                    const float2 d = __fadd2_rn(acc[c], nt);
                    below = __funnelshift_l(__float_as_uint(d.x), below, 1);
                    below = __funnelshift_l(__float_as_uint(d.y), below, 1);
                }
                uint32_t cand = __brev(~below);
                const int64_t lim = min(nvr, c_end) - e0;
                if (lim < EPI_COLS) cand &= lim <= 0 ? 0u : ((1u << lim) - 1u);
                if (cand) {
                    // slots lb .. lb+n-1 of the row in this CTA: the first `cloc` are
                    // private to (row, CTA column) and reserved by a shared-memory
                    // atomic; the rest overflow into the row's shared slots
                    const int n = __popc(cand);
                    const int lb = atomicAdd(lcount + quad * 32 + lane, n);
                    uint2 *pr = a.priv + ((size_t)row * a.gy + blockIdx.y) * a.cloc;
                    uint2 *cr = a.cand + row * a.ocap;
                    int ob = 0;  // overflow slot of local slot s: s + ob
                    if (lb + n > a.cloc) {
                        const int first = max(lb, a.cloc);
                        ob = atomicAdd(a.count + row, lb + n - first) - first;
                    }
                    int base = lb;
                    // one candidate per lane and round, lowest column first
                    while (cand) {
                        const int c = __ffs(cand) - 1;
                        cand &= cand - 1;
                        const uint2 kv =
                            make_uint2(order_key(col_of(acc, c)), (uint32_t)(e0 + c));
                        if (base < a.cloc)
                            pr[base] = kv;
                        else if (base + ob < a.ocap)
                            cr[base + ob] = kv;
                        ++base;
                    }
                }
            }
        }
        if (MODE == MODE_FILTER) {
            // every emission of the CTA is complete: publish the private counts
            asm volatile("bar.sync 1, %0;" ::"n"(NEPI) : "memory");
            if (part == 0 && row_ok)
                a.lcnt[(size_t)row * a.gy + blockIdx.y] = min(lcount[quad * 32 + lane], a.cloc);
        }
        if (!ok) {
            if (row_ok) flag(a.dev_err, LC_DEVERR_TIMEOUT);
        } else if (MODE == MODE_MATERIALIZE && row_ok) {
            // columns of this CTA past the last computed tile
            float *dst = a.out + row * a.ld;
            for (int64_t e = max(c0, comp_end) + part; e < c_end; e += 4) dst[e] = -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(taddr, I_TMEM_COLS);
    }
}

// Ascending bitonic sort of P (power of two) uint32 values in shared memory.
template <int NT>
__device__ __forceinline__ void bitonic_sort_u32_asc(uint32_t *a, int P) {
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < (P >> 1); i += NT) {
                const int lo = 2 * stride * (i / stride) + (i % stride);
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const uint32_t x = a[lo], y = a[hi];
                if ((x > y) == up) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
        }
    }
    __syncthreads();
}

// Exact top-k of each row's candidates, one CTA per row (for rows too long
// for the warp-per-row kernel's bitmaps): radix selection of the k-th largest
// key K* in shared memory; the candidates above K* and the `need` lowest-index
// candidates equal to K* are collected (in any order, one shared atomic per
// warp) and written out in ascending index order: through a bitmap over the
// row's visible entries when it fits in the `R` words that held the keys and
// indices (only the words holding a chosen entry are touched, found through
// a summary bitmap of them), else by a bitonic sort.  A row's candidates are
// the private slots
// of each of its gy CTA columns (lcnt of them in each) followed by its
// overflow slots (count, in a region of ocap slots); rows with a total
// outside [k, cap], or an overflow past its region, are appended to the
// failed-row list.  Shared memory: R >= 2 cap words (keys, indices, later the
// bitmap), PK collected indices, P tie slots (PK, P: powers of two >= k,
// cap); the tie slots double as the radix selection's spare and, at the end,
// as the summary bitmap (R / 32 <= P words).
template <int NT>
__global__ void __launch_bounds__(NT) k_cand_pick(Batch bt, int m, int k, int cap, int ocap,
                                                   int R, int PK, int P,
                                                   const int32_t *__restrict__ count,
                                                   const uint2 *__restrict__ cand,
                                                   const int32_t *__restrict__ lcnt,
                                                   const uint2 *__restrict__ priv, int gy,
                                                   int cloc, int32_t *__restrict__ topk,
                                                   int32_t *flist, int32_t *nfail,
                                                   int32_t *dev_err) {
    constexpr int NW = NT / 32;
    const unsigned FULL = 0xffffffffu;
    extern __shared__ uint32_t sbuf[];
    uint32_t *keys = sbuf;                                      // [cap]
    uint32_t *idx = sbuf + cap;                                 // [cap]
    uint32_t *bm = sbuf;                                        // [R], after the collection
    uint32_t *sel = sbuf + R;                                   // [PK]
    uint32_t *tl = sel + PK;                                    // [P]
    __shared__ RadixScratch rs;
    __shared__ int s_n, s_ties, s_priv, wsum[NW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r = blockIdx.x;
    const int bq = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[bq] + (r - bt.cu_q[bq]);
    const int64_t Tc = bt.cu_c[bq + 1] - bt.cu_c[bq];
    int64_t nv = n_vis(t, m);
    if (nv > Tc) nv = Tc;
    int32_t *out = topk + r * k;
    if (nv <= k) {
        for (int i = threadIdx.x; i < k; i += NT) out[i] = i < nv ? i : -1;
        return;
    }
    // candidates: the private slots of the row's CTA columns, then its overflow slots
    if (threadIdx.x == 0) {
        s_priv = 0;
        s_n = 0;
        s_ties = 0;
    }
    __syncthreads();
    const int n_over = count[r];
    // each CTA column's count and, with at most NT columns (the usual case),
    // their block-wide prefix (the place of each column's segment) at once
    __shared__ int seg_off[NT];
    int n_priv;
    if (gy <= NT) {
        const int c = threadIdx.x < gy ? lcnt[r * gy + threadIdx.x] : 0;
        seg_off[threadIdx.x] = block_exclusive_scan<NT>(c, wsum, &n_priv);
    } else {
        int c = 0;
        for (int y = threadIdx.x; y < gy; y += NT) c += lcnt[r * gy + y];
        c = __reduce_add_sync(FULL, c);
        if (lane == 0 && c) atomicAdd(&s_priv, c);
        __syncthreads();
        n_priv = s_priv;
    }
    const int n = n_priv + n_over;
    if (n < k || n > cap || n_over > ocap) {
        if (threadIdx.x == 0) flist[atomicAdd(nfail, 1)] = (int32_t)r;
        return;
    }
    // the private segments, NT CTA columns at a time; the index array first
    // holds the owner (group-local CTA column) of each place, so that every
    // thread loads its share of all segments at once, one memory round trip
    // per group
    int filled = 0;
    for (int y0 = 0; y0 < gy; y0 += NT) {
        int tot = n_priv;
        if (gy > NT) {
            const int y = y0 + threadIdx.x;
            const int c = y < gy ? lcnt[r * gy + y] : 0;
            seg_off[threadIdx.x] = block_exclusive_scan<NT>(c, wsum, &tot);
        }
        __syncthreads();
        if (filled + tot > cap) {
            flag(dev_err, LC_DEVERR_BATCH);  // counts changed under us: never expected
            break;
        }
        const int nseg = min(NT, gy - y0);
        for (int sg = warp; sg < nseg; sg += NW) {
            const int b0 = seg_off[sg], b1 = sg + 1 < nseg ? seg_off[sg + 1] : tot;
            for (int i = b0 + lane; i < b1; i += 32) idx[filled + i] = (uint32_t)sg;
        }
        __syncthreads();
        for (int j0 = threadIdx.x; j0 < tot; j0 += 4 * NT) {
            uint2 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * NT;
                if (j < tot) {
                    const int sg = (int)idx[filled + j];
                    v[u] = priv[((size_t)r * gy + y0 + sg) * cloc + (j - seg_off[sg])];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * NT;
                if (j < tot) {
                    keys[filled + j] = v[u].x;
                    idx[filled + j] = v[u].y;
                }
            }
        }
        filled += tot;
        __syncthreads();  // seg_off is rewritten by the next group
    }
    for (int i = threadIdx.x; i < n_over; i += NT) {
        const uint2 ki = cand[r * ocap + i];
        keys[n_priv + i] = ki.x;
        idx[n_priv + i] = ki.y;
    }
    for (int i = threadIdx.x; i < PK; i += NT) sel[i] = 0xFFFFFFFFu;  // bitonic padding
    __syncthreads();
    int need;
    const uint32_t kstar = radix_kth_largest_smem<NT>(keys, n, k, rs, &need, tl);
    // candidates above K* are in; the ties at K* go to a list
    for (int j0 = threadIdx.x & ~31; j0 < n; j0 += NT) {
        const int j = j0 + lane;
        const uint32_t key = j < n ? keys[j] : 0u;
        const bool up = j < n && key > kstar, eq = j < n && key == kstar;
        const uint32_t mu = __ballot_sync(FULL, up), me = __ballot_sync(FULL, eq);
        int bu = 0, be = 0;
        if (lane == 0) {
            if (mu) bu = atomicAdd(&s_n, __popc(mu));
            if (me) be = atomicAdd(&s_ties, __popc(me));
        }
        bu = __shfl_sync(FULL, bu, 0);
        be = __shfl_sync(FULL, be, 0);
        const uint32_t lt = (1u << lane) - 1u;
        if (up) sel[bu + __popc(mu & lt)] = idx[j];
        if (eq) tl[be + __popc(me & lt)] = idx[j];
    }
    __syncthreads();
    const int above = s_n, ties = s_ties;
    if (ties == need) {
        for (int i = threadIdx.x; i < ties; i += NT) sel[above + i] = tl[i];
    } else {
        // more ties than places (rare): the lowest indices win
        int Pt = 1;
        while (Pt < ties) Pt <<= 1;
        for (int i = ties + threadIdx.x; i < Pt; i += NT) tl[i] = 0xFFFFFFFFu;
        bitonic_sort_u32_asc<NT>(tl, Pt);
        for (int i = threadIdx.x; i < need; i += NT) sel[above + i] = tl[i];
    }
    const int nw = (int)((nv + 31) >> 5);
    if (nw > R) {
        bitonic_sort_u32_asc<NT>(sel, PK);
        for (int i = threadIdx.x; i < k; i += NT) out[i] = (int32_t)sel[i];
        return;
    }
    // ascending order through a bitmap of the chosen entries (keys and indices
    // are dead) and a summary bitmap of its non-zero words (in the tie slots,
    // dead too): only the words that hold a chosen entry are cleared, marked
    // and read back
    uint32_t *sm = tl;
    const int ns = (nw + 31) >> 5;
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += NT) {
        const uint32_t e = sel[i];
        if (e < (uint32_t)nv) bm[e >> 5] = 0u;
    }
    for (int w = threadIdx.x; w < ns; w += NT) sm[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += NT) {
        const uint32_t e = sel[i];
        if (e < (uint32_t)nv) {
            atomicOr(&bm[e >> 5], 1u << (e & 31u));
            atomicOr(&sm[e >> 10], 1u << ((e >> 5) & 31u));
        } else {
            flag(dev_err, LC_DEVERR_BATCH);  // a chosen index outside the row: never expected
        }
    }
    __syncthreads();
    // the non-zero bitmap words in ascending order, listed in `sel` (dead
    // now; at most k of them): warp w lists those of summary words [sb, se)
    const int per_w = (ns + NW - 1) / NW;
    const int sb = min(warp * per_w, ns), se = min(sb + per_w, ns);
    int cnt = 0;
    for (int s0 = sb + lane; s0 < se; s0 += 32) cnt += __popc(sm[s0]);
    cnt = __reduce_add_sync(FULL, cnt);
    if (lane == 0) wsum[warp] = cnt;
    __syncthreads();
    int off = 0, nz = 0;
    for (int u = 0; u < NW; ++u) {
        if (u < warp) off += wsum[u];
        nz += wsum[u];
    }
    for (int s0 = sb; s0 < se; s0 += 32) {
        const int sw = s0 + lane;
        uint32_t x = sw < se ? sm[sw] : 0u;
        const int c = __popc(x);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = off + incl - c;
        for (; x; x &= x - 1) sel[pos++] = (uint32_t)(sw * 32 + __ffs(x) - 1);
        off += __shfl_sync(FULL, incl, 31);
    }
    __syncthreads();
    // the listed words, an equal share per warp, lanes on consecutive words;
    // each chosen entry's place is the count of chosen entries before it
    const int per_l = (nz + NW - 1) / NW;
    const int lb = min(warp * per_l, nz), le = min(lb + per_l, nz);
    cnt = 0;
    for (int i = lb + lane; i < le; i += 32) cnt += __popc(bm[sel[i]]);
    cnt = __reduce_add_sync(FULL, cnt);
    if (lane == 0) wsum[warp] = cnt;  // the first counts were read before the last barrier
    __syncthreads();
    off = 0;
    for (int u = 0; u < warp; ++u) off += wsum[u];
    for (int i0 = lb; i0 < le; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t w = i < le ? sel[i] : 0u;
        uint32_t bits = i < le ? bm[w] : 0u;
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = off + incl - c;
        for (; bits; bits &= bits - 1) {
            if (pos < k) out[pos] = (int32_t)(w * 32 + __ffs(bits) - 1);
            ++pos;
        }
        off += __shfl_sync(FULL, incl, 31);
    }
}

namespace {
int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

int64_t pick_chunk(int64_t Nq, int64_t n_cols);

struct FusedPlan {
    int stride, rho, cap, ocap, P, PK, R, gy, cloc, nwmax, fb_grid;
    int64_t ns, lds, chunk, ldb;
    size_t off_samp, off_theta, off_count, off_flist, off_nfail, off_cand, off_lcnt, off_priv,
        total;
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Rows whose visible entries fit the warp-per-row pick's bitmaps (two words
// per 32 entries, a warp each, eight warps a CTA, 227 KB at most).
constexpr int NW_WARP_MAX = 1024;

FusedPlan plan_fused(const lc_batch &b, int k) {
    FusedPlan p{};
    const int64_t n = b.max_c;
    // the sampling stride: at most 32, at least 2k samples per longest row
    // (the candidate count is then rho * stride +- stride * sqrt(rho), far
    // above k: a row whose count still falls short goes to the fallback)
    p.stride = 1;
    while (p.stride < 32 && n / (2 * p.stride) >= 2 * (int64_t)k) p.stride *= 2;
    if (p.stride == 1) {
        p.rho = k;
    } else {
        const double x = 2.0 + std::sqrt(4.0 + (double)k / p.stride);
        p.rho = (int)std::ceil(x * x);
    }
    int cap = 4 * k;
    if (cap < 2 * p.rho * p.stride) cap = 2 * p.rho * p.stride;
    if (cap < 2048) cap = 2048;
    cap = (cap + 31) & ~31;
    if (cap > 16384) cap = 16384;
    p.cap = cap;
    // the overflow region per row: half of cap (a row whose overflow passes
    // it is redone by the fallback)
    p.ocap = cap / 2;
    p.P = pow2_at_least(cap);
    p.PK = pow2_at_least(k);
    // k_cand_pick orders its output through a bitmap of the row when that fits
    p.R = 2 * cap;
    const int64_t nw = (n + 31) / 32;
    if (nw > p.R && 4 * (nw + p.PK + p.P) <= 200 * 1024) p.R = (int)nw;
    p.nwmax = nw <= NW_WARP_MAX ? (int)nw : 0;  // 0: the CTA-per-row pick
    p.ns = (n + p.stride - 1) / p.stride;
    p.lds = (p.ns + 7) & ~(int64_t)7;  // uint16 keys, 16-byte rows
    const size_t Nq = (size_t)b.total_q;
    p.chunk = pick_chunk(b.total_q, n);
    p.gy = (int)((n + p.chunk - 1) / p.chunk);
    int64_t cl = (2 * (int64_t)p.cap * p.chunk + n - 1) / n;
    cl = (cl + 31) / 32 * 32;
    if (cl < 32) cl = 32;
    if (cl > p.cap) cl = p.cap;
    p.cloc = (int)cl;
    // the fallback's row buffers reuse the sample region (dead by then); at
    // least one row, at most two CTAs per SM
    p.ldb = (n + 3) & ~(int64_t)3;
    size_t samp = sizeof(uint16_t) * Nq * (size_t)p.lds;
    const size_t one_row = sizeof(float) * (size_t)p.ldb;
    if (samp < one_row) samp = one_row;
    p.fb_grid = (int)std::min<size_t>(296, samp / one_row);
    size_t o = 0;
    p.off_samp = o;  o += al256(samp);
    p.off_theta = o; o += al256(sizeof(uint32_t) * Nq);
    p.off_count = o; o += al256(sizeof(int32_t) * Nq);
    p.off_flist = o; o += al256(sizeof(int32_t) * Nq);
    p.off_nfail = o; o += al256(sizeof(int32_t));
    p.off_cand = o;  o += al256(sizeof(uint2) * Nq * (size_t)p.ocap);
    p.off_lcnt = o;  o += al256(sizeof(int32_t) * Nq * (size_t)p.gy);
    p.off_priv = o;  o += al256(sizeof(uint2) * Nq * (size_t)p.gy * (size_t)p.cloc);
    p.total = o;
    return p;
}

bool index_tc_eligible(const void *qI, const void *kI, const lc_batch &b, int HI, int dI,
                       lc_dtype dt) {
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return dt == LC_BF16 && dI == IDI && (HI == 4 || HI == 8) && b.max_q >= 64 &&
           b.max_c > 0 && al16(qI) && al16(kI) && b.total_q < (1ll << 31) &&
           b.max_c < (1ll << 31);
}

template <int MODE, int HI>
lc_status launch_tc(const CUtensorMap &mQ, const CUtensorMap &mK, const IdxTcArgs &a, int64_t n_cols,
                    cudaStream_t st) {
    constexpr uint32_t SMEM = IdxCfg::SMEM;
    static_assert(SMEM <= 227 * 1024, "indexer shared memory");
    auto kfn = k_index_tc<MODE, HI>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) !=
            cudaSuccess)
            return LC_ERR_CUDA;
        attr = true;
    }
    const int64_t gy = (n_cols + a.chunk - 1) / a.chunk;
    if (gy < 1 || gy > 65535) return LC_ERR_UNSUPPORTED;
    // every sequence's row tiles, at most one partial tile each: the surplus
    // CTAs exit at once
    const int64_t gx = (a.total_q + IBM - 1) / IBM + a.bt.B;
    if (gx >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    dim3 grid((unsigned)gx, (unsigned)gy);
    LC_LAUNCH_AS(MODE == MODE_FILTER      ? "k_index_tc<filter>"
                 : MODE == MODE_SAMPLE16 ? "k_index_tc<sample16>"
                                         : "k_index_tc<materialize>",
                 kfn, grid, dim3(I_THREADS), SMEM, st, mQ, mK, a);
    return check_launch();
}

template <int MODE>
lc_status launch_tc_hi(int HI, const CUtensorMap &mQ, const CUtensorMap &mK, const IdxTcArgs &a,
                       int64_t n_cols, cudaStream_t st) {
    return HI == 8 ? launch_tc<MODE, 8>(mQ, mK, a, n_cols, st)
                   : launch_tc<MODE, 4>(mQ, mK, a, n_cols, st);
}

// entries per CTA: about eight waves of CTAs over the 148 SMs, at least 16 tiles each
int64_t pick_chunk(int64_t Nq, int64_t n_cols) {
    const int64_t row_tiles = (Nq + IBM - 1) / IBM;
    int64_t want_y = (148 * 8 + row_tiles - 1) / row_tiles;
    if (want_y < 1) want_y = 1;
    int64_t chunk = (n_cols + want_y - 1) / want_y;
    chunk = (chunk + IBN - 1) / IBN * IBN;
    // a CTA first moves its 128 query rows into shared memory; amortise that
    // over at least 16 tiles
    if (chunk < 16 * IBN) chunk = 16 * IBN;
    while ((n_cols + chunk - 1) / chunk > 65535) chunk *= 2;
    return chunk;
}

IdxTcArgs base_args(const lc_batch &b, const void *qI, const float *w, int m,
                    int32_t *dev_err) {
    IdxTcArgs a{};
    a.bt = to_dev(b);
    a.total_q = b.total_q;
    a.qI = static_cast<const __nv_bfloat16 *>(qI);
    a.stride = 1;
    a.m = m;
    a.w = w;
    a.dev_err = dev_err;
    a.stall = debug_stall_clocks(LC_STALL_INDEX_TC);
    return a;
}
}  // namespace

size_t index_tc_workspace(const lc_batch &b, int k) {
    if (k < 1) return 0;
    return plan_fused(b, k).total;
}

// Scores [total_q, ld] on the tensor cores, or LC_ERR_UNSUPPORTED.
lc_status index_tc_materialize(const void *qI, const float *w, const void *kI, const lc_batch &b,
                               int HI, int dI, int m, lc_dtype dt, float *scores, int64_t ld,
                               int32_t *dev_err, cudaStream_t st) {
    if (!index_tc_eligible(qI, kI, b, HI, dI, dt)) return LC_ERR_UNSUPPORTED;
    CUtensorMap mQ, mK;
    if (!make_tmap_bf16_2d(&mQ, qI, (uint64_t)b.total_q, (uint64_t)HI * IDI, HI * IDI * 2, IDI,
                           IBM) ||
        !make_tmap_bf16_2d(&mK, kI, (uint64_t)b.total_c, (uint64_t)HI * IDI, HI * IDI * 2, IDI,
                           IBN))
        return LC_ERR_CUDA;
    IdxTcArgs a = base_args(b, qI, w, m, dev_err);
    a.col_end = ld;
    a.out = scores;
    a.ld = ld;
    a.vec_out = (reinterpret_cast<uintptr_t>(scores) & 15u) == 0 && (ld & 3) == 0;
    a.chunk = pick_chunk(b.total_q, ld);
    return launch_tc_hi<MODE_MATERIALIZE>(HI, mQ, mK, a, ld, st);
}

// Fused exact top-k on the tensor cores (ws holds the plan's buffers), or
// LC_ERR_UNSUPPORTED.
lc_status index_topk_tc_launch(const void *qI, const float *w, const void *kI,
                               const lc_batch &b, int HI, int dI, int m, lc_dtype dt, int k,
                               int32_t *topk, void *ws, size_t ws_bytes, int32_t *dev_err,
                               cudaStream_t st) {
    if (!index_tc_eligible(qI, kI, b, HI, dI, dt)) return LC_ERR_UNSUPPORTED;
    const FusedPlan p = plan_fused(b, k);
    if (!ws || ws_bytes < p.total) return LC_ERR_WORKSPACE;
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint16_t *samp = reinterpret_cast<uint16_t *>(base + p.off_samp);
    uint32_t *theta = reinterpret_cast<uint32_t *>(base + p.off_theta);
    int32_t *count = reinterpret_cast<int32_t *>(base + p.off_count);
    int32_t *flist = reinterpret_cast<int32_t *>(base + p.off_flist);
    int32_t *nfail = reinterpret_cast<int32_t *>(base + p.off_nfail);
    uint2 *cand = reinterpret_cast<uint2 *>(base + p.off_cand);
    int32_t *lcnt = reinterpret_cast<int32_t *>(base + p.off_lcnt);
    uint2 *priv = reinterpret_cast<uint2 *>(base + p.off_priv);
    float *fbuf = reinterpret_cast<float *>(base + p.off_samp);  // after the sample is read
    const int64_t Tc = b.total_c;
    const uint64_t pitch = (uint64_t)HI * IDI * 2;

    CUtensorMap mQ, mKs, mK;
    if (!make_tmap_bf16_2d(&mQ, qI, (uint64_t)b.total_q, (uint64_t)HI * IDI, pitch, IDI, IBM) ||
        !make_tmap_bf16_2d(&mK, kI, (uint64_t)Tc, (uint64_t)HI * IDI, pitch, IDI, IBN) ||
        !make_tmap_bf16_strided_rows(&mKs, kI, (uint64_t)Tc, (uint64_t)HI * IDI, pitch,
                                     (uint32_t)p.stride, IDI, IBN))
        return LC_ERR_CUDA;
    lc_status s;
    // 1. 16-bit keys of every s-th entry's score (visible columns only)
    {
        IdxTcArgs a = base_args(b, qI, w, m, dev_err);
        a.stride = p.stride;
        a.col_end = p.ns;
        a.out16 = samp;
        a.ld = p.lds;
        a.chunk = pick_chunk(b.total_q, p.ns);
        s = launch_tc_hi<MODE_SAMPLE16>(HI, mQ, mKs, a, p.ns, st);
        if (s != LC_OK) return s;
    }
    // 2. thresholds (and the per-row overflow counts and the failed-row count zeroed)
    s = sample_threshold16_launch(samp, p.lds, b, m, p.stride, k, p.rho, theta, count, nfail, st);
    if (s != LC_OK) return s;
    // 3. candidates
    {
        IdxTcArgs a = base_args(b, qI, w, m, dev_err);
        a.theta = theta;
        a.count = count;
        a.cand = cand;
        a.ocap = p.ocap;
        a.priv = priv;
        a.lcnt = lcnt;
        a.gy = p.gy;
        a.cloc = p.cloc;
        a.chunk = p.chunk;
        if ((b.max_c + p.chunk - 1) / p.chunk != p.gy) return LC_ERR_INVALID_ARG;  // gridDim.y == gy
        s = launch_tc_hi<MODE_FILTER>(HI, mQ, mK, a, b.max_c, st);
        if (s != LC_OK) return s;
    }
    // 4. exact selection among the candidates
    if (p.nwmax > 0) {
        s = cand_pick_warp_launch(b, m, k, p.cap, p.ocap, p.nwmax, count, cand, lcnt, priv, p.gy,
                                  p.cloc, topk, flist, nfail, dev_err, st);
        if (s != LC_OK) return s;
    } else {
        const size_t smem = sizeof(uint32_t) * (size_t)(p.R + p.PK + p.P);
        static size_t attr = 0;
        if (smem > 48 * 1024 && smem > attr) {
            if (cudaFuncSetAttribute(k_cand_pick<PICK_NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess)
                return LC_ERR_CUDA;
            attr = smem;
        }
        LC_LAUNCH_AS("k_cand_pick", k_cand_pick<PICK_NT>, dim3((unsigned)b.total_q), dim3(PICK_NT),
                     smem, st, to_dev(b), m, k,
                  p.cap, p.ocap, p.R, p.PK, p.P, count, cand, lcnt, priv, p.gy, p.cloc, topk,
                  flist, nfail, dev_err);
        if ((s = check_launch()) != LC_OK) return s;
    }
    // 5. exact top-k of the failed rows from recomputed scores (no work when none failed)
    return topk_fallback_launch(qI, w, kI, b, HI, m, k, flist, nfail, fbuf, p.ldb, p.fb_grid,
                                topk, st);
}

}  // namespace lc

