// HCA dense attention on the 5th-generation tensor cores, bf16, head dim 128,
// any ragged batch (page "DeepSeek-V4 技术解析…", §1.1, HCA paragraph:
// attention over every compressed entry, plus the sliding-window branch).
//
// A CTA owns two M = 128 tiles of one sequence's query rows of Q[total_q*H,
// 128] (256 consecutive rows, 256/H tokens; a sequence's rows are covered by
// its own run of CTAs) and walks the union of their keys: the
// compressed entries 0 .. n_vis(t_last)-1, then the raw window positions,
// in tiles of BN = 128 keys.  Both query tiles share every K/V tile, so each
// key is read from L2 once per 256 query rows.
//   warp 9       producer: Q0, Q1 once, then K and V tiles into a 2-stage ring
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
// TMEM: O0 [0,128) | O1 [128,256) | S0/P0 [256,384) | S1/P1 [384,512).
// Every wait is bounded; on a timeout the CTA raises LC_DEVERR_TIMEOUT,
// skips the rest and still frees its TMEM.
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
constexpr uint32_t H_REG_LAUNCH = 168, H_REG_HI = 192, H_REG_LO = 96;
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
constexpr float H_RESCALE = 8.f;

struct HBars {
    uint64_t q_full, k_full[2], v_full[2], kv_empty[2], s_full[2], p_full[2], o_done[2];
    uint64_t stall;           // test hook: a barrier nothing completes
    uint64_t q_ready;         // RoPE: the softmax warps rotated Q0 and Q1
    uint32_t taddr;
    int abort;
};

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

__global__ void __launch_bounds__(H_THREADS, 1)
    k_hca_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKc,
             const __grid_constant__ CUtensorMap mVc, const __grid_constant__ CUtensorMap mKr,
             const __grid_constant__ CUtensorMap mVr, HcaArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    HBars &bars = *reinterpret_cast<HBars *>(smem + HS_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = &bars.abort;
    const unsigned FULL = 0xffffffffu;

    // ---- the CTA's sequence and its 256-row tile there (rows = token x head):
    // sequence b owns ceil(rows_b / 256) consecutive CTAs; the grid has up
    // to one surplus CTA per sequence, which leaves before any barrier
    const SeqTile sq = locate_tile(a.bt, blockIdx.x, a.H, 2 * HBM_);
    if (sq.b == a.bt.B) return;
    const int64_t tile = sq.tile, n_rows = sq.nq * a.H;
    const int64_t q_row_beg = sq.q_beg * a.H;  // the sequence's first row of Q / O
    const int64_t q_pos0 = sq.q_pos0, raw_pos0 = sq.raw_pos0;
    const int64_t c_beg = sq.c_beg, raw_beg = sq.raw_beg;
    const int64_t Tc = a.have_c ? sq.c_end - c_beg : 0;
    const int64_t Nraw = a.have_r ? sq.raw_end - raw_beg : 0;
    const int64_t row0 = tile * (2 * HBM_);  // sequence-local
    const int64_t rows_here = min((int64_t)(2 * HBM_), n_rows - row0);
    const int64_t t_first = q_pos0 + row0 / a.H;
    const int64_t t_last = q_pos0 + (row0 + rows_here - 1) / a.H;
    int64_t n_ent = n_vis(t_last, a.m);
    if (n_ent > Tc) n_ent = Tc;
    const int nct = (int)((n_ent + HBN - 1) / HBN);
    int64_t wlo = 0;
    int nwt = 0;
    if (a.W > 0) {
        wlo = max((int64_t)0, t_first - a.W + 1);
        nwt = (int)((t_last - wlo + 1 + HBN - 1) / HBN);
    }
    const int n_tiles = nct + nwt;

    if (tid == 0) {
        bars.abort = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
        if (bars.abort) flag(a.dev_err, LC_DEVERR_TIMEOUT);  // layout assumption broken
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_ready, 8);  // one arrival per softmax warp
        mbar_init(&bars.stall, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.p_full[s], 4);  // one arrival per softmax warp
            mbar_init(&bars.o_done[s], 1);
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
        if (lane == 0 && !dead && n_tiles > 0) {
            prefetch_tmap(&mQ);
            mbar_expect_tx(&bars.q_full, 4 * H_TILE);
            for (int g = 0; g < 2; ++g)
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_2d(smem + HS_Q + (2 * g + hf) * H_TILE, &mQ, &bars.q_full, hf * 64,
                                (int32_t)(q_row_beg + row0 + g * HBM_));
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int s = j & 1;
                if (j >= 2 && !mbar_wait(&bars.kv_empty[s], ((j - 2) >> 1) & 1, abort)) break;
                const CUtensorMap *mk, *mv;
                int32_t y;
                if (j < nct) {
                    mk = &mKc;
                    mv = &mVc;
                    y = (int32_t)(c_beg + (int64_t)j * HBN);
                } else {
                    mk = &mKr;
                    mv = &mVr;
                    y = (int32_t)(raw_beg + wlo + (int64_t)(j - nct) * HBN - raw_pos0);
                }
                uint8_t *kd = smem + HS_K + s * 2 * H_TILE, *vd = smem + HS_V + s * 2 * H_TILE;
                mbar_expect_tx(&bars.k_full[s], 2 * H_TILE);
                tma_load_2d(kd, mk, &bars.k_full[s], 0, y);
                tma_load_2d(kd + H_TILE, mk, &bars.k_full[s], 64, y);
                mbar_expect_tx(&bars.v_full[s], 2 * H_TILE);
                tma_load_2d(vd, mv, &bars.v_full[s], 0, y);
                tma_load_2d(vd + H_TILE, mv, &bars.v_full[s], 64, y);
                ++issued;
            }
            // copies still in flight must land before the CTA exits
            int dummy = 0;
            for (int j = max(0, issued - 2); j < issued; ++j) {
                mbar_wait(&bars.k_full[j & 1], (j >> 1) & 1, &dummy, 400000000LL);
                mbar_wait(&bars.v_full[j & 1], (j >> 1) & 1, &dummy, 400000000LL);
            }
            mbar_wait(&bars.q_full, 0, &dummy, 400000000LL);
            // the MMAs' releases of the last tiles: no commit may still be on
            // its way to this CTA's barriers when it exits (skipped after an
            // abort, when some of those MMAs are never issued)
            for (int j = max(0, issued - 2); j < issued && !*abort; ++j)
                mbar_wait(&bars.kv_empty[j & 1], (j >> 1) & 1, abort);
        }
      } else if (warp == 8) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !dead && n_tiles > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(HBM_, HBN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(HBM_, HHD, 0, 1);
            const uint32_t q_base = smem_u32(smem + HS_Q);
            auto issue_s = [&](int g, int j) {
                const uint32_t k_base = smem_u32(smem + HS_K + (j & 1) * 2 * H_TILE);
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
            auto issue_pv = [&](int g, int j) {
                const uint32_t v_base = smem_u32(smem + HS_V + (j & 1) * 2 * H_TILE);
#pragma unroll
                for (int kk = 0; kk < HBN / 16; ++kk) {
                    const uint64_t bd = sw128_desc(v_base + kk * 16 * 128, H_TILE, 1024);
                    mma_bf16_ta(taddr + HT_O + g * 128, taddr + HT_S + g * 128 + kk * 8, bd,
                                IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars.o_done[g]);
            };
            bool ok = (a.stall == 0 || mbar_wait(&bars.stall, 0, abort, a.stall)) &&
                      mbar_wait(a.rope ? &bars.q_ready : &bars.q_full, 0, abort) &&
                      mbar_wait(&bars.k_full[0], 0, abort);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int s = j & 1;
                // PV0(j), then S0(j+1) as soon as its K tile is in
                if (!mbar_wait(&bars.v_full[s], (j >> 1) & 1, abort) ||
                    !mbar_wait(&bars.p_full[0], j & 1, abort))
                    break;
                tc_fence_after();
                issue_pv(0, j);
                const bool more = j + 1 < n_tiles;
                if (more) {
                    if (!mbar_wait(&bars.k_full[s ^ 1], ((j + 1) >> 1) & 1, abort)) break;
                    tc_fence_after();
                    issue_s(0, j + 1);
                }
                if (!mbar_wait(&bars.p_full[1], j & 1, abort)) break;
                tc_fence_after();
                issue_pv(1, j);
                mma_commit(&bars.kv_empty[s]);
                if (more) issue_s(1, j + 1);
            }
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<H_REG_HI>();
        // ------------------------------------------------------ softmax warpgroups
        const int g = warp >> 2;                       // query tile
        const int r = tid & 127;                       // row in the tile (TMEM lane)
        const int64_t row = row0 + g * HBM_ + r;
        const bool row_ok = (int64_t)(g * HBM_ + r) < rows_here;
        const int64_t t = q_pos0 + (row_ok ? row : row0 + rows_here - 1) / a.H;
        int64_t nv = n_vis(t, a.m);
        if (nv > Tc) nv = Tc;
        if (!row_ok) nv = 0;
        const int64_t w_lo = a.W > 0 ? max((int64_t)0, t - a.W + 1) : t + 1;
        // window positions the raw cache does not hold are skipped and flagged
        int64_t c_lo = max(w_lo, raw_pos0), c_hi = min(t, raw_pos0 + Nraw - 1);
        if (row_ok && a.W > 0 && (c_lo > w_lo || c_hi < t)) flag(a.dev_err, LC_DEVERR_WINDOW);
        if (!row_ok) c_hi = c_lo - 1;
        const uint32_t lane_base = taddr + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + HT_S + g * 128, o_addr = lane_base + HT_O + g * 128;
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = !dead;
        // RoPE: (cos, sin) of the angles of the CTA's tokens t_first .. t_last
        const float2 *rope_tab = reinterpret_cast<const float2 *>(smem + HS_ROPE);
        const float2 *my_cs = rope_tab + (t - t_first) * 32;
        if (a.rope && ok && n_tiles > 0) {
            // rotate the query rows in place before the first S MMA
            if (!__all_sync(FULL, mbar_wait(&bars.q_full, 0, abort))) ok = false;
            const int ntok = (int)(t_last - t_first + 1);
            float2 *tab = reinterpret_cast<float2 *>(smem + HS_ROPE);
            for (int u = tid; u < ntok * 32; u += 256)
                tab[u] = rope_cs(t_first + u / 32, rope_theta(u % 32));
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (ok && row_ok) rope_smem_row(smem + HS_Q + (2 * g + 1) * H_TILE, r, my_cs);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.q_ready);
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
            if (!__all_sync(FULL, mbar_wait(&bars.s_full[g], j & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // valid columns [lo, hi) of this tile for this row
            int lo, hi;
            if (j < nct) {
                const int64_t e0 = (int64_t)j * HBN;
                lo = 0;
                hi = (int)max((int64_t)0, min((int64_t)HBN, nv - e0));
            } else {
                const int64_t p0 = wlo + (int64_t)(j - nct) * HBN;
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
        // epilogue (ok is warp-uniform here)
        if (ok && n_tiles > 0 &&
            !__all_sync(FULL, mbar_wait(&bars.o_done[g], (n_tiles - 1) & 1, abort)))
            ok = false;
        if (!ok) {
            if (row_ok) flag(a.dev_err, LC_DEVERR_TIMEOUT);
        } else {
            tc_fence_after();
            const float of = fold_sink(
                m_used, l, row_ok ? sink_log2(a.sink, (int)(row % a.H), a.dev_err) : -INFINITY);
            const float inv = l > 0.f ? of / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.O + (q_row_beg + row) * HHD);
#pragma unroll 1
            for (int c = 0; c < HHD; c += 32) {
                float o[32];
                if (n_tiles > 0) {
                    tmem_ld32(o_addr + c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = 0.f;
                }
                if (a.rope && n_tiles > 0 && c >= HHD - ROPE_DIMS) rope_out32(o, c, HHD, my_cs);
                if (row_ok) {
#pragma unroll
                    for (int u = 0; u < 32; u += 8) {
                        uint4 v = make_uint4(pack_bf16x2(o[u] * inv, o[u + 1] * inv),
                                             pack_bf16x2(o[u + 2] * inv, o[u + 3] * inv),
                                             pack_bf16x2(o[u + 4] * inv, o[u + 5] * inv),
                                             pack_bf16x2(o[u + 6] * inv, o[u + 7] * inv));
                        dst[(c + u) / 8] = v;
                    }
                }
            }
            if (row_ok && a.lse)
                a.lse[q_row_beg + row] = l > 0.f ? (m_used + log2f(l)) / H_LOG2E : -INFINITY;
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
        if (cudaFuncSetAttribute(k_hca_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)HS_TOTAL) != cudaSuccess)
            return LC_ERR_CUDA;
        attr_done = true;
    }
    // every sequence's tiles, at most one partial tile each: the surplus CTAs exit
    const int64_t grid64 = (n_rows + 2 * HBM_ - 1) / (2 * HBM_) + b.B;
    if (grid64 >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    const unsigned grid = (unsigned)grid64;
    LC_LAUNCH(k_hca_tc, dim3(grid), dim3(H_THREADS), HS_TOTAL, st, maps[0], maps[1], maps[2],
              maps[3], maps[4], a);
    return check_launch();
}

}  // namespace lc
