// HCA dense attention on the 5th-generation tensor cores, bf16, head dim 128,
// any ragged batch (page "DeepSeek-V4 技术解析…", §1.1, HCA paragraph:
// attention over every compressed entry, plus the sliding-window branch).
//
// A work tile is two M = 128 tiles of one sequence's query rows of
// Q[total_q*H, 128] (256 consecutive rows, 256/H tokens); it walks the union
// of their keys: the compressed entries 0 .. n_vis(t_last)-1, then the raw
// window positions, in tiles of BN = 128 keys.  Both query tiles share every
// K/V tile, so each key is read from L2 once per 256 query rows.  The CTAs
// are persistent (one per SM) and take the work tiles in turn; the next
// tile's Q and first K/V tiles load, and its first S products run, while the
// softmax warps finish the current one.
//   warp 9       producer: per work tile Q0, Q1 (once the previous tile's S
//                products are done), then K and V tiles into a 2-stage ring
//   warp 8       TMEM owner and MMA issuer, in the order
//                  S0(j+1) = Q0 K^T, PV1(j), S1(j+1), PV0(j+1), ...
//                so that one softmax warpgroup works while the tensor core
//                serves the other; S (M=128, N=128, K=128) lands in TMEM and
//                the softmax writes P (bf16) back over it, where the PV MMA
//                (M=128, N=128, K=128) reads it as its A operand
//   warps 0-3    softmax of query tile 0, warps 4-7 of query tile 1: thread
//                r owns row r (TMEM lane r).  Pass 1 reads S and takes the
//                row max; the reference max only moves when the max grows by
//                more than 2^8 (then O and l are rescaled, which is safe
//                because S(j) completing implies PV(j-1) completed); pass 2
//                reads S again, forms p = 2^(s*scale*log2e - m), the row sum
//                and the packed bf16 P.  Masks are applied only on tiles that
//                straddle a row's visible range.
// TMEM: O0 [0,128) | O1 [128,256) | S0/P0 [256,384) | S1/P1 [384,512).  A
// work tile's first PV into O_g waits until the softmax warps of tile g have
// read the previous tile's O_g out (o_free).
// Every wait is bounded; on a timeout the CTA raises LC_DEVERR_TIMEOUT,
// skips the rest and still frees its TMEM.
#include <algorithm>

#include "lc_common.cuh"
#include "sm100.cuh"

namespace lc {

using namespace sm100;

namespace {
constexpr int HBM_ = 128, HBN = 128, HHD = 128;
constexpr int H_THREADS = 384;                         // three warpgroups
// Registers are allocated to a CTA in whole warpgroups: launched at 168 a
// thread (384 x 168 <= 65,536), warpgroup 2 (MMA issuer, producer, two idle
// warps) gives back down to H_REG_LO and the two softmax warpgroups grow to
// H_REG_HI, which their 128-float rows of S need without spilling.
constexpr uint32_t H_REG_LAUNCH = 168, H_REG_HI = 200, H_REG_LO = 104;
static_assert(128 * (2 * H_REG_HI + H_REG_LO) <= H_THREADS * H_REG_LAUNCH &&
                  2 * 128 * (H_REG_HI - H_REG_LAUNCH) <= 128 * (H_REG_LAUNCH - H_REG_LO),
              "register split must fit the launch allocation");
constexpr uint32_t H_TILE = HBN * 128;                 // one 64-column half of a 128-row tile
constexpr uint32_t HS_Q = 0;                           // 2 tiles x 2 halves
constexpr uint32_t HS_K = HS_Q + 4 * H_TILE;           // 2 stages x 2 halves
constexpr uint32_t HS_V = HS_K + 4 * H_TILE;           // 2 stages x 2 halves
constexpr uint32_t HS_BAR = HS_V + 4 * H_TILE;
constexpr uint32_t HS_ROPE = HS_BAR + 256;            // RoPE: (cos, sin) [tokens][32]
constexpr uint32_t HS_TOTAL = HS_ROPE + 32 * 32 * 8;
constexpr uint32_t H_TMEM_COLS = 512;
constexpr uint32_t HT_O = 0, HT_S = 256;               // + 128 * tile
constexpr float H_LOG2E = 1.4426950408889634f;
// work tiles of at most this many key tiles go to persistent CTAs
constexpr int64_t HCA_SHORT_KEY_TILES = 16;
constexpr float H_RESCALE = 8.f;

struct HBars {
    uint64_t q_full, q_empty, k_full[2], v_full[2], kv_empty[2], s_full[2], p_full[2],
        o_done[2], o_free[2];   // phases count across the CTA's work tiles
    uint64_t stall;           // test hook: a barrier nothing completes
    uint64_t q_ready;         // RoPE: the softmax warps rotated Q0 and Q1
    uint32_t taddr;
    int abort;
};
static_assert(sizeof(HBars) <= HS_ROPE - HS_BAR, "HCA barriers");

__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16_u(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

}  // namespace

struct HcaArgs {
    Batch bt;             // device batch arrays (any number of sequences)
    int have_c, have_r;   // compressed entries / raw window present
    int H;
    int m, W;
    float scale_log2;
    const float *sink;    // [H] per-head sink logits or NULL
    __nv_bfloat16 *O;
    float *lse;
    int32_t *dev_err;
    int rope;             // partial RoPE: Q rotated at t, O rotated back at t
    long long stall;      // test hook (0: off): the MMA issuer first waits this
                          // many clocks on a barrier nothing completes
};

// One work tile: 256 consecutive query rows (token x head) of one sequence
// and the key tiles they walk.  valid = false past the batch's last tile.
struct HcaTile {
    bool valid;
    int64_t q_row_beg, row0, rows_here;  // the sequence's first Q/O row; tile rows (local)
    int64_t q_pos0, raw_pos0, c_beg, raw_beg, Tc, Nraw, t_first, t_last, wlo;
    int nct, n_tiles;
};

__device__ __forceinline__ HcaTile hca_tile(const HcaArgs &a, int64_t w) {
    HcaTile T;
    const SeqTile sq = locate_tile(a.bt, w, a.H, 2 * HBM_);
    T.valid = sq.b < a.bt.B;
    if (!T.valid) return T;
    const int64_t n_rows = sq.nq * a.H;
    T.q_row_beg = sq.q_beg * a.H;
    T.row0 = sq.tile * (2 * HBM_);
    T.rows_here = min((int64_t)(2 * HBM_), n_rows - T.row0);
    T.q_pos0 = sq.q_pos0;
    T.raw_pos0 = sq.raw_pos0;
    T.c_beg = sq.c_beg;
    T.raw_beg = sq.raw_beg;
    T.Tc = a.have_c ? sq.c_end - sq.c_beg : 0;
    T.Nraw = a.have_r ? sq.raw_end - sq.raw_beg : 0;
    T.t_first = T.q_pos0 + T.row0 / a.H;
    T.t_last = T.q_pos0 + (T.row0 + T.rows_here - 1) / a.H;
    int64_t n_ent = n_vis(T.t_last, a.m);
    if (n_ent > T.Tc) n_ent = T.Tc;
    T.nct = (int)((n_ent + HBN - 1) / HBN);
    T.wlo = 0;
    int nwt = 0;
    if (a.W > 0) {
        T.wlo = max((int64_t)0, T.t_first - a.W + 1);
        nwt = (int)((T.t_last - T.wlo + 1 + HBN - 1) / HBN);
    }
    T.n_tiles = T.nct + nwt;
    return T;
}

// MULTI: CTA c takes work tiles c, c + gridDim.x, ... in turn (else the one
// tile blockIdx.x, with no loop around it).  Every
// barrier's phase counts across work tiles (q_full / q_empty / q_ready /
// o_free once per work tile with keys, the K/V stages, S and P and O once
// per key tile), so the next tile's Q and first K/V tiles load, and its
// first S products run, while the softmax warps finish the previous tile.
template <bool MULTI>
__global__ void __launch_bounds__(H_THREADS, 1)
    k_hca_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKc,
             const __grid_constant__ CUtensorMap mVc, const __grid_constant__ CUtensorMap mKr,
             const __grid_constant__ CUtensorMap mVr, HcaArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    HBars &bars = *reinterpret_cast<HBars *>(smem + HS_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = &bars.abort;
    const unsigned FULL = 0xffffffffu;

    // the CTA's first work tile, looked up while the barriers are set up; a
    // CTA past the last tile leaves before any barrier
    const HcaTile T0 = hca_tile(a, blockIdx.x);
    if (!T0.valid) return;

    if (tid == 0) {
        bars.abort = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
        if (bars.abort) flag(a.dev_err, LC_DEVERR_TIMEOUT);  // layout assumption broken
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        mbar_init(&bars.q_ready, 8);  // one arrival per softmax warp
        mbar_init(&bars.stall, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.p_full[s], 4);  // one arrival per softmax warp
            mbar_init(&bars.o_done[s], 1);
            mbar_init(&bars.o_free[s], 4);  // one arrival per softmax warp
        }
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(&bars.taddr, H_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = bars.taddr;
    const bool dead = bars.abort != 0;

    if (warp >= 8) {
      // warpgroup 2: one register decrease for its four warps, then the roles
      setmaxnreg_dec<H_REG_LO>();
      if (warp == 9) {
        // ------------------------------------------------------ producer
        if (lane == 0 && !dead) {
            prefetch_tmap(&mQ);
            int J = 0, nq = 0;  // key tiles and work tiles with keys so far
            // a later tile is looked up when the previous one is done (the
            // batch arrays' lines stay in L1 across the CTA's tiles)
            for (int64_t w = blockIdx.x; !*abort; w += gridDim.x) {
                const HcaTile T = w == blockIdx.x ? T0 : hca_tile(a, w);
                if (!T.valid) break;
                if (T.n_tiles == 0) {
                    if (MULTI) continue;
                    break;
                }
                // the previous tile's S products have read its Q
                if (nq > 0 && !mbar_wait(&bars.q_empty, (nq - 1) & 1, abort)) break;
                mbar_expect_tx(&bars.q_full, 4 * H_TILE);
                for (int g = 0; g < 2; ++g)
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_2d(smem + HS_Q + (2 * g + hf) * H_TILE, &mQ, &bars.q_full,
                                    hf * 64, (int32_t)(T.q_row_beg + T.row0 + g * HBM_));
                ++nq;
                for (int j = 0; j < T.n_tiles; ++j, ++J) {
                    const int s = J & 1;
                    if (J >= 2 && !mbar_wait(&bars.kv_empty[s], ((J - 2) >> 1) & 1, abort)) break;
                    const CUtensorMap *mk, *mv;
                    int32_t y;
                    if (j < T.nct) {
                        mk = &mKc;
                        mv = &mVc;
                        y = (int32_t)(T.c_beg + (int64_t)j * HBN);
                    } else {
                        mk = &mKr;
                        mv = &mVr;
                        y = (int32_t)(T.raw_beg + T.wlo + (int64_t)(j - T.nct) * HBN - T.raw_pos0);
                    }
                    uint8_t *kd = smem + HS_K + s * 2 * H_TILE, *vd = smem + HS_V + s * 2 * H_TILE;
                    mbar_expect_tx(&bars.k_full[s], 2 * H_TILE);
                    tma_load_2d(kd, mk, &bars.k_full[s], 0, y);
                    tma_load_2d(kd + H_TILE, mk, &bars.k_full[s], 64, y);
                    mbar_expect_tx(&bars.v_full[s], 2 * H_TILE);
                    tma_load_2d(vd, mv, &bars.v_full[s], 0, y);
                    tma_load_2d(vd + H_TILE, mv, &bars.v_full[s], 64, y);
                }
                if (!MULTI) break;
            }
            // copies still in flight must land before the CTA exits
            int dummy = 0;
            for (int j = max(0, J - 2); j < J; ++j) {
                mbar_wait(&bars.k_full[j & 1], (j >> 1) & 1, &dummy, 400000000LL);
                mbar_wait(&bars.v_full[j & 1], (j >> 1) & 1, &dummy, 400000000LL);
            }
            if (nq > 0) mbar_wait(&bars.q_full, (nq - 1) & 1, &dummy, 400000000LL);
            // the MMAs' releases of the last tiles: no commit may still be on
            // its way to this CTA's barriers when it exits (skipped after an
            // abort, when some of those MMAs are never issued)
            for (int j = max(0, J - 2); j < J && !*abort; ++j)
                mbar_wait(&bars.kv_empty[j & 1], (j >> 1) & 1, abort);
            if (MULTI && nq > 0 && !*abort) mbar_wait(&bars.q_empty, (nq - 1) & 1, abort);
        }
      } else if (warp == 8) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !dead) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(HBM_, HBN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(HBM_, HHD, 0, 1);
            const uint32_t q_base = smem_u32(smem + HS_Q);
            auto issue_s = [&](int g, int J) {
                const uint32_t k_base = smem_u32(smem + HS_K + (J & 1) * 2 * H_TILE);
                const uint32_t qg = q_base + g * 2 * H_TILE;
#pragma unroll
                for (int kk = 0; kk < HHD / 16; ++kk) {
                    const uint64_t ad = sw128_desc(qg + (kk >> 2) * H_TILE + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        sw128_desc(k_base + (kk >> 2) * H_TILE + (kk & 3) * 32, 16, 1024);
                    mma_bf16(taddr + HT_S + g * 128, ad, bd, IDESC_S, kk > 0);
                }
                mma_commit(&bars.s_full[g]);
            };
            auto issue_pv = [&](int g, int J, bool first) {
                const uint32_t v_base = smem_u32(smem + HS_V + (J & 1) * 2 * H_TILE);
#pragma unroll
                for (int kk = 0; kk < HBN / 16; ++kk) {
                    const uint64_t bd = sw128_desc(v_base + kk * 16 * 128, H_TILE, 1024);
                    mma_bf16_ta(taddr + HT_O + g * 128, taddr + HT_S + g * 128 + kk * 8, bd,
                                IDESC_O, (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars.o_done[g]);
            };
            bool ok = a.stall == 0 || mbar_wait(&bars.stall, 0, abort, a.stall);
            int J = 0, nq = 0;
            for (int64_t w = blockIdx.x; ok; w += gridDim.x) {
                const HcaTile T = w == blockIdx.x ? T0 : hca_tile(a, w);
                if (!T.valid) break;
                if (T.n_tiles == 0) {
                    if (MULTI) continue;
                    break;
                }
                if (!mbar_wait(a.rope ? &bars.q_ready : &bars.q_full, nq & 1, abort) ||
                    !mbar_wait(&bars.k_full[J & 1], (J >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_s(0, J);
                issue_s(1, J);
                if (MULTI && T.n_tiles == 1) mma_commit(&bars.q_empty);  // every S of the tile issued
                for (int j = 0; j < T.n_tiles; ++j) {
                    const int Jj = J + j, s = Jj & 1;
                    // PV0(j) (after the previous tile's O0 is read out), then
                    // S0(j+1) as soon as its K tile is in
                    if (!mbar_wait(&bars.v_full[s], (Jj >> 1) & 1, abort) ||
                        !mbar_wait(&bars.p_full[0], Jj & 1, abort) ||
                        (j == 0 && nq > 0 && !mbar_wait(&bars.o_free[0], (nq - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(0, Jj, j == 0);
                    const bool more = j + 1 < T.n_tiles;
                    if (more) {
                        if (!mbar_wait(&bars.k_full[s ^ 1], ((Jj + 1) >> 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(0, Jj + 1);
                    }
                    if (!mbar_wait(&bars.p_full[1], Jj & 1, abort) ||
                        (j == 0 && nq > 0 && !mbar_wait(&bars.o_free[1], (nq - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, Jj, j == 0);
                    mma_commit(&bars.kv_empty[s]);
                    if (more) {
                        issue_s(1, Jj + 1);
                        if (MULTI && j + 2 == T.n_tiles) mma_commit(&bars.q_empty);
                    }
                }
                J += T.n_tiles;
                ++nq;
                if (!MULTI) break;
            }
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<H_REG_HI>();
        // ------------------------------------------------------ softmax warpgroups
        const int g = warp >> 2;                       // query tile
        const int r = tid & 127;                       // row in the tile (TMEM lane)
        const uint32_t lane_base = taddr + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + HT_S + g * 128, o_addr = lane_base + HT_O + g * 128;
        const float sl2 = a.scale_log2;
        bool ok = !dead, flagged = false;
        int J = 0, nq = 0;
        // after a timeout (ok false) the loop still walks the remaining tiles,
        // doing nothing but the RoPE path's named barriers
        // a later tile is looked up when the previous one is done
        for (int64_t w = blockIdx.x;; w += gridDim.x) {
            const HcaTile T = w == blockIdx.x ? T0 : hca_tile(a, w);
            if (!T.valid) break;
            const int64_t row = T.row0 + g * HBM_ + r;  // sequence-local
            const bool row_ok = (int64_t)(g * HBM_ + r) < T.rows_here;
            const int64_t t = T.q_pos0 + (row_ok ? row : T.row0 + T.rows_here - 1) / a.H;
            int64_t nv = n_vis(t, a.m);
            if (nv > T.Tc) nv = T.Tc;
            if (!row_ok) nv = 0;
            const int64_t w_lo = a.W > 0 ? max((int64_t)0, t - a.W + 1) : t + 1;
            // window positions the raw cache does not hold are skipped and flagged
            int64_t c_lo = max(w_lo, T.raw_pos0), c_hi = min(t, T.raw_pos0 + T.Nraw - 1);
            if (row_ok && a.W > 0 && (c_lo > w_lo || c_hi < t)) flag(a.dev_err, LC_DEVERR_WINDOW);
            if (!row_ok) c_hi = c_lo - 1;
            float m_used = -INFINITY, l = 0.f;
            // RoPE: (cos, sin) of the angles of the tile's tokens t_first .. t_last
            const float2 *rope_tab = reinterpret_cast<const float2 *>(smem + HS_ROPE);
            const float2 *my_cs = rope_tab + (t - T.t_first) * 32;
            if (a.rope && T.n_tiles > 0) {
                // rotate the query rows in place before the tile's first S MMA
                // (the previous tile's epilogue, the table's last reader, is
                // done).  Both warpgroups pass these two named barriers for
                // every tile with keys, also after a timeout, so neither waits
                // at one the other has left behind.
                asm volatile("bar.sync 2, 256;" ::: "memory");
                if (ok && !__all_sync(FULL, mbar_wait(&bars.q_full, nq & 1, abort))) ok = false;
                const int ntok = (int)(T.t_last - T.t_first + 1);
                float2 *tab = reinterpret_cast<float2 *>(smem + HS_ROPE);
                for (int u = tid; u < ntok * 32; u += 256)
                    tab[u] = rope_cs(T.t_first + u / 32, rope_theta(u % 32));
                asm volatile("bar.sync 2, 256;" ::: "memory");
                if (ok && row_ok) rope_smem_row(smem + HS_Q + (2 * g + 1) * H_TILE, r, my_cs);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(&bars.q_ready);
            }
            for (int j = 0; ok && j < T.n_tiles; ++j) {
                const int Jj = J + j;
                if (!__all_sync(FULL, mbar_wait(&bars.s_full[g], Jj & 1, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // valid columns [lo, hi) of this tile for this row
                int lo, hi;
                if (j < T.nct) {
                    const int64_t e0 = (int64_t)j * HBN;
                    lo = 0;
                    hi = (int)max((int64_t)0, min((int64_t)HBN, nv - e0));
                } else {
                    const int64_t p0 = T.wlo + (int64_t)(j - T.nct) * HBN;
                    lo = (int)min((int64_t)HBN, max((int64_t)0, c_lo - p0));
                    hi = (int)max((int64_t)0, min((int64_t)HBN, c_hi + 1 - p0));
                }
                const bool full = lo == 0 && hi == HBN;
                // the whole row of S in registers: four loads in flight, one wait
                float v[HBN];
                tmem_ld32(s_addr, *reinterpret_cast<float(*)[32]>(v));
                tmem_ld32(s_addr + 32, *reinterpret_cast<float(*)[32]>(v + 32));
                tmem_ld32(s_addr + 64, *reinterpret_cast<float(*)[32]>(v + 64));
                tmem_ld32(s_addr + 96, *reinterpret_cast<float(*)[32]>(v + 96));
                tmem_wait_ld();
                if (!full) {
#pragma unroll
                    for (int c = 0; c < HBN; ++c)
                        if (c < lo || c >= hi) v[c] = -INFINITY;
                }
                float mt = -INFINITY;
#pragma unroll
                for (int c = 0; c < HBN; c += 2) mt = max3f(mt, v[c], v[c + 1]);
                const float m_new = fmaxf(m_used, mt * sl2);
                const bool grow = m_new > m_used + H_RESCALE;
                // rows that already hold a finite reference rescale O and l; S(j)
                // being complete means PV(j-1) is complete, so O is at rest
                const bool need = grow && m_used != -INFINITY;
                if (__any_sync(FULL, need)) {
                    const float f = need ? ex2(m_used - m_new) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < HHD; c += 32) {
                        float o[32];
                        tmem_ld32(o_addr + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) o[u] *= f;
                        tmem_st32(o_addr + c, o);
                    }
                    tmem_wait_st();
                    l *= f;
                }
                if (grow) m_used = m_new;
                // p = 2^(s*scale*log2e - m) (masked columns hold -inf and give 0),
                // row sum, bf16 P over the S columns already read
                const float neg = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll
                for (int c0 = 0; c0 < HBN; c0 += 32) {
                    uint32_t pk[16];
                    float2 l2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        // packed fp32x2 scale-and-shift and row-sum adds
                        const float2 x = __ffma2_rn(make_float2(v[c0 + c], v[c0 + c + 1]),
                                                    make_float2(sl2, sl2), make_float2(neg, neg));
                        const float2 p = make_float2(ex2(x.x), ex2(x.y));
                        l2 = __fadd2_rn(l2, p);
                        pk[c / 2] = pack_bf16x2(p.x, p.y);
                    }
                    l += l2.x + l2.y;
                    tmem_st16_u(s_addr + c0 / 2, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[g]);
            }
            // epilogue (ok is warp-uniform here): O out of TMEM, released to
            // the next tile's first PV, then normalised and stored
            float o[HHD];
            if (ok && T.n_tiles > 0) {
                if (!__all_sync(FULL,
                                mbar_wait(&bars.o_done[g], (J + T.n_tiles - 1) & 1, abort))) {
                    ok = false;
                } else {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < HHD; c += 32)
                        tmem_ld32(o_addr + c, *reinterpret_cast<float(*)[32]>(o + c));
                    tmem_wait_ld();
                    if (MULTI) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars.o_free[g]);
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < HHD; ++c) o[c] = 0.f;
            }
            if (!ok) {
                if (!flagged && !dead) flag(a.dev_err, LC_DEVERR_TIMEOUT);
                flagged = true;
                if (MULTI) continue;
                break;
            }
            const float of = fold_sink(
                m_used, l, row_ok ? sink_log2(a.sink, (int)(row % a.H), a.dev_err) : -INFINITY);
            const float inv = l > 0.f ? of / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.O + (T.q_row_beg + row) * HHD);
#pragma unroll
            for (int c = 0; c < HHD; c += 32) {
                if (a.rope && T.n_tiles > 0 && c >= HHD - ROPE_DIMS)
                    rope_out32(*reinterpret_cast<float(*)[32]>(o + c), c, HHD, my_cs);
                if (row_ok) {
#pragma unroll
                    for (int u = 0; u < 32; u += 8) {
                        uint4 pv = make_uint4(pack_bf16x2(o[c + u] * inv, o[c + u + 1] * inv),
                                              pack_bf16x2(o[c + u + 2] * inv, o[c + u + 3] * inv),
                                              pack_bf16x2(o[c + u + 4] * inv, o[c + u + 5] * inv),
                                              pack_bf16x2(o[c + u + 6] * inv, o[c + u + 7] * inv));
                        dst[(c + u) / 8] = pv;
                    }
                }
            }
            if (row_ok && a.lse)
                a.lse[T.q_row_beg + row] = l > 0.f ? (m_used + log2f(l)) / H_LOG2E : -INFINITY;
            if (T.n_tiles > 0) {
                J += T.n_tiles;
                ++nq;
            }
            if (!MULTI) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(taddr, H_TMEM_COLS);
    }
}

namespace {
bool al16h(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// HCA on the tensor cores: bf16, d = 128, any ragged batch, H dividing 128.
// LC_ERR_UNSUPPORTED when the shape does not fit (the caller falls back).
lc_status hca_tc_launch(const void *Q, const void *Kc, const void *Vc, const void *Kraw,
                        const void *Vraw, const lc_batch &b, int H, int d, int m, int W,
                        float scale, const float *sink, int rope, lc_dtype dt, void *O,
                        float *lse, int32_t *dev_err, cudaStream_t st) {
    if (dt != LC_BF16 || d != HHD || (HBM_ % H) != 0) return LC_ERR_UNSUPPORTED;
    if (!al16h(Q) || !al16h(O) || (Kc && !al16h(Kc)) || (Vc && !al16h(Vc)) ||
        (Kraw && !al16h(Kraw)) || (Vraw && !al16h(Vraw)))
        return LC_ERR_UNSUPPORTED;
    if (b.total_q * H >= (1ll << 31) || b.total_c >= (1ll << 31) || b.total_raw >= (1ll << 31))
        return LC_ERR_UNSUPPORTED;
    const int64_t n_rows = b.total_q * H;
    if (n_rows == 0) return LC_OK;
    const bool have_c = b.total_c > 0 && Kc && Vc;
    const bool have_r = W > 0 && b.total_raw > 0 && Kraw && Vraw;
    CUtensorMap maps[5];
    if (!make_tmap_bf16_2d(&maps[0], Q, (uint64_t)n_rows, HHD, HHD * 2, 64, HBM_) ||
        !make_tmap_bf16_2d(&maps[1], have_c ? Kc : Q, have_c ? b.total_c : 1, HHD, HHD * 2, 64,
                           HBN) ||
        !make_tmap_bf16_2d(&maps[2], have_c ? Vc : Q, have_c ? b.total_c : 1, HHD, HHD * 2, 64,
                           HBN) ||
        !make_tmap_bf16_2d(&maps[3], have_r ? Kraw : Q, have_r ? b.total_raw : 1, HHD, HHD * 2,
                           64, HBN) ||
        !make_tmap_bf16_2d(&maps[4], have_r ? Vraw : Q, have_r ? b.total_raw : 1, HHD, HHD * 2,
                           64, HBN))
        return LC_ERR_CUDA;
    HcaArgs a{};
    a.bt = to_dev(b);
    a.have_c = have_c;
    a.have_r = have_r;
    a.H = H;
    a.m = m;
    a.W = have_r ? W : 0;
    a.scale_log2 = scale * H_LOG2E;
    a.sink = sink;
    a.O = reinterpret_cast<__nv_bfloat16 *>(O);
    a.lse = lse;
    a.dev_err = dev_err;
    a.rope = rope;
    a.stall = debug_stall_clocks(LC_STALL_HCA_TC);
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(k_hca_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)HS_TOTAL) != cudaSuccess ||
            cudaFuncSetAttribute(k_hca_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)HS_TOTAL) != cudaSuccess)
            return LC_ERR_CUDA;
        attr_done = true;
    }
    // The work tiles are at most ceil(rows / 256) plus one partial tile per
    // sequence.  Tiles with few key tiles (short contexts) are dominated by
    // their pipeline fill and drain: one persistent CTA per SM then walks
    // every gridDim.x-th tile, overlapping one tile's tail with the next one's
    // start.  Longer tiles take one CTA each (the hardware's CTA scheduling
    // keeps the SMs evenly loaded).
    const int64_t tiles = (n_rows + 2 * HBM_ - 1) / (2 * HBM_) + b.B;
    const int64_t key_tiles = (b.max_c + HBN - 1) / HBN + (W > 0 ? (W + HBN - 1) / HBN + 1 : 0);
    const int64_t sms = sm_count();
    if (sms <= 0) return LC_ERR_CUDA;
    const bool multi = key_tiles <= HCA_SHORT_KEY_TILES && tiles > sms;
    const int64_t grid64 = multi ? sms : tiles;
    if (grid64 >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    const unsigned grid = (unsigned)grid64;
    // one tile per CTA: the loop-free instance (the multi-tile one's loop
    // cost long tiles about a tenth of their speed)
    if (multi)
        LC_LAUNCH_AS("k_hca_tc", k_hca_tc<true>, dim3(grid), dim3(H_THREADS), HS_TOTAL, st,
                     maps[0], maps[1], maps[2], maps[3], maps[4], a);
    else
        LC_LAUNCH_AS("k_hca_tc", k_hca_tc<false>, dim3(grid), dim3(H_THREADS), HS_TOTAL, st,
                     maps[0], maps[1], maps[2], maps[3], maps[4], a);
    return check_launch();
}

}  // namespace lc
