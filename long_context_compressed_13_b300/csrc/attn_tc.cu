// MQA attention on the 5th-generation tensor cores (tcgen05 + TMEM), bf16
// inputs, head dim 128: HCA dense attention and CSA sparse attention.
//
// A CTA owns one M = 128 tile of query rows of Q[total_q*H, 128]:
//   HCA    128 consecutive rows (128/H tokens of one sequence); keys are the
//          compressed entries 0 .. n_vis(t_last)-1, loaded as TMA boxes;
//   CSA    the H rows of one token (rows H..127 of the tile are padding);
//          keys are the token's selected entries, fetched row by row with
//          TMA tile::gather4 (4 rows per instruction, 128-byte swizzle).
// Both then take the raw window positions of their tokens as TMA boxes.
// Keys are walked in tiles of BN = 64:
//   warp 4       producer: Q once, then K/V tiles into a 2-stage ring; for
//                CSA tiles the whole warp gathers and publishes a 64-bit
//                validity mask per tile
//   warp 5       TMEM owner and MMA issuer: S = Q K^T (M=128, N=64, K=128)
//                into one of two TMEM S buffers, O += P V (M=128, N=128,
//                K=64) into the TMEM O accumulator
//   warps 0-3    softmax: thread r owns row r (TMEM lane r); masks, online
//                max with lazy rescaling of O (only when the max grows by
//                more than 2^8), P as bf16 into shared memory for the PV MMA,
//                and the final O / l, lse epilogue
// Two CTAs fit on one SM (112 KB of shared memory, 256 TMEM columns each), so
// one CTA's softmax overlaps the other's MMAs.  Every wait is bounded; on a
// timeout the CTA raises LC_DEVERR_TIMEOUT, skips the rest and still frees
// its TMEM.
#include "lc_common.cuh"
#include "sm100.cuh"

namespace lc {

using namespace sm100;

namespace {
constexpr int BM = 128, BN = 64, HD = 128;
constexpr int THREADS = 192;
constexpr uint32_t SM_Q = 0;                   // 2 x [128 rows x 128 B]
constexpr uint32_t SM_K = 32768;               // 2 stages x 2 x [64 x 128 B]
constexpr uint32_t SM_V = SM_K + 2 * 16384;    // 2 stages x 2 x [64 x 128 B]
constexpr uint32_t SM_P = SM_V + 2 * 16384;    // [128 rows x 128 B]
constexpr uint32_t SM_BAR = SM_P + 16384;      // barriers and scalars
constexpr uint32_t SM_TOTAL = SM_BAR + 256;
constexpr uint32_t TMEM_COLS = 256;            // S0 | S1 | O(128)
constexpr uint32_t T_S = 0, T_O = 128;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.f;

struct Bars {
    uint64_t q_full, k_full[2], v_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done;
    uint64_t mask_full[2];
    uint64_t mask[2];  // CSA: valid keys of the tile held by each stage
    uint32_t taddr;
    int abort;
};

__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t r0, int32_t r1, int32_t r2,
                                            int32_t r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::"
        "bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1),
        "r"(r2), "r"(r3)
        : "memory");
}

__device__ __forceinline__ uint64_t low_bits(int n) { return n >= 64 ? ~0ull : (1ull << n) - 1; }
}  // namespace

struct AttnTcArgs {
    int64_t n_rows;   // total_q * H
    int H;
    Batch bt;         // device batch arrays
    int64_t Tc;       // HCA: stored compressed entries (one sequence)
    int64_t Nraw;     // HCA: stored raw rows (one sequence)
    const int32_t *topk;  // CSA: [total_q, k]
    int k;
    int m, W;
    float scale_log2;
    __nv_bfloat16 *O;
    float *lse;
    int32_t *dev_err;
};

template <bool SPARSE>
__global__ void __launch_bounds__(THREADS, 2)
    k_attn_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKc,
              const __grid_constant__ CUtensorMap mVc, const __grid_constant__ CUtensorMap mKr,
              const __grid_constant__ CUtensorMap mVr, AttnTcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Bars &bars = *reinterpret_cast<Bars *>(smem + SM_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = &bars.abort;
    const unsigned FULL = 0xffffffffu;

    // ---- the tile's rows, tokens and key list
    int64_t row0, rows_here, t_first, t_last, c_beg, Tc, raw_beg, Nraw, raw_pos0, qrow = 0;
    if (SPARSE) {
        qrow = blockIdx.x;  // one query token
        const int b = seq_of_row(a.bt, qrow);
        t_first = t_last = a.bt.q_pos0[b] + (qrow - a.bt.cu_q[b]);
        row0 = qrow * a.H;
        rows_here = a.H;
        c_beg = a.bt.cu_c[b];
        Tc = a.bt.cu_c[b + 1] - c_beg;
        raw_beg = a.bt.cu_raw[b];
        Nraw = a.bt.cu_raw[b + 1] - raw_beg;
        raw_pos0 = a.bt.raw_pos0[b];
    } else {
        const int64_t q_pos0 = a.bt.q_pos0[0];
        row0 = (int64_t)blockIdx.x * BM;
        rows_here = min((int64_t)BM, a.n_rows - row0);
        t_first = q_pos0 + row0 / a.H;
        t_last = q_pos0 + (row0 + rows_here - 1) / a.H;
        c_beg = 0;
        Tc = a.Tc;
        raw_beg = 0;
        Nraw = a.Nraw;
        raw_pos0 = a.bt.raw_pos0[0];
    }
    int nct;  // key tiles before the window: compressed (HCA) or selected (CSA)
    if (SPARSE) {
        nct = (a.k + BN - 1) / BN;
    } else {
        int64_t n_ent = n_vis(t_last, a.m);
        if (n_ent > Tc) n_ent = Tc;
        nct = (int)((n_ent + BN - 1) / BN);
    }
    int64_t wlo = 0;
    int nwt = 0;
    if (a.W > 0) {
        wlo = max((int64_t)0, t_first - a.W + 1);
        nwt = (int)((t_last - wlo + 1 + BN - 1) / BN);
    }
    const int n_tiles = nct + nwt;

    if (tid == 0) {
        bars.abort = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
        if (bars.abort) flag(a.dev_err, LC_DEVERR_TIMEOUT);  // layout assumption broken
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.s_free[s], 4);  // one arrival per softmax warp
            mbar_init(&bars.mask_full[s], 1);
        }
        mbar_init(&bars.p_full, 4);
        mbar_init(&bars.o_done, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(&bars.taddr, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = bars.taddr;
    const bool dead = bars.abort != 0;

    if (warp == 4) {
        // ------------------------------------------------------ producer warp
        if (!dead && n_tiles > 0) {
            if (lane == 0) {
                prefetch_tmap(&mQ);
                mbar_expect_tx(&bars.q_full, 2 * BM * 128);
                tma_load_2d(smem + SM_Q, &mQ, &bars.q_full, 0, (int32_t)row0);
                tma_load_2d(smem + SM_Q + BM * 128, &mQ, &bars.q_full, 64, (int32_t)row0);
            }
            int64_t nv = n_vis(t_last, a.m);
            if (nv > Tc) nv = Tc;
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i & 1;
                if (i >= 2 &&
                    !__all_sync(FULL, mbar_wait(&bars.kv_empty[s], ((i - 2) >> 1) & 1, abort)))
                    break;
                uint8_t *kd = smem + SM_K + s * 16384, *vd = smem + SM_V + s * 16384;
                if (SPARSE && i < nct) {
                    // selected entries of this tile: keys lane and lane + 32
                    const int slot0 = i * BN + lane, slot1 = slot0 + 32;
                    const int64_t j0 = slot0 < a.k ? a.topk[qrow * a.k + slot0] : -1;
                    const int64_t j1 = slot1 < a.k ? a.topk[qrow * a.k + slot1] : -1;
                    const bool v0 = j0 >= 0 && j0 < nv, v1 = j1 >= 0 && j1 < nv;
                    if ((j0 >= nv) || (j1 >= nv)) flag(a.dev_err, LC_DEVERR_INDEX);
                    // masked slots fetch row 0 of the map, which always exists
                    const int32_t g0 = v0 ? (int32_t)(c_beg + j0) : 0;
                    const int32_t g1 = v1 ? (int32_t)(c_beg + j1) : 0;
                    const uint64_t mask = (uint64_t)__ballot_sync(FULL, v0) |
                                          ((uint64_t)__ballot_sync(FULL, v1) << 32);
                    // lane -> 4-row group (lane >> 1) and d half (lane & 1)
                    const int grp = lane >> 1, half = lane & 1;
                    int32_t r[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int key = grp * 4 + u;
                        const int32_t x0 = __shfl_sync(FULL, g0, key & 31);
                        const int32_t x1 = __shfl_sync(FULL, g1, key & 31);
                        r[u] = key < 32 ? x0 : x1;
                    }
                    if (lane == 0) {
                        mbar_expect_tx(&bars.k_full[s], 2 * BN * 128);
                        mbar_expect_tx(&bars.v_full[s], 2 * BN * 128);
                    }
                    __syncwarp();
                    tma_gather4(kd + half * BN * 128 + grp * 512, &mKc, &bars.k_full[s],
                                half * 64, r[0], r[1], r[2], r[3]);
                    tma_gather4(vd + half * BN * 128 + grp * 512, &mVc, &bars.v_full[s],
                                half * 64, r[0], r[1], r[2], r[3]);
                    if (lane == 0) {
                        bars.mask[s] = mask;
                        mbar_arrive(&bars.mask_full[s]);
                    }
                } else if (lane == 0) {
                    const CUtensorMap *mk, *mv;
                    int32_t y;
                    if (i < nct) {
                        mk = &mKc;
                        mv = &mVc;
                        y = (int32_t)(c_beg + (int64_t)i * BN);
                    } else {
                        mk = &mKr;
                        mv = &mVr;
                        y = (int32_t)(raw_beg + wlo + (int64_t)(i - nct) * BN - raw_pos0);
                    }
                    mbar_expect_tx(&bars.k_full[s], 2 * BN * 128);
                    tma_load_2d(kd, mk, &bars.k_full[s], 0, y);
                    tma_load_2d(kd + BN * 128, mk, &bars.k_full[s], 64, y);
                    mbar_expect_tx(&bars.v_full[s], 2 * BN * 128);
                    tma_load_2d(vd, mv, &bars.v_full[s], 0, y);
                    tma_load_2d(vd + BN * 128, mv, &bars.v_full[s], 64, y);
                    mbar_arrive(&bars.mask_full[s]);  // keeps the mask phases in step
                }
                __syncwarp();
                ++issued;
            }
            // copies still in flight must land before the CTA exits
            if (lane == 0) {
                int dummy = 0;
                for (int i = max(0, issued - 2); i < issued; ++i) {
                    mbar_wait(&bars.k_full[i & 1], (i >> 1) & 1, &dummy, 400000000LL);
                    mbar_wait(&bars.v_full[i & 1], (i >> 1) & 1, &dummy, 400000000LL);
                }
                mbar_wait(&bars.q_full, 0, &dummy, 400000000LL);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !dead && n_tiles > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, HD, 0, 1);
            const uint32_t q_base = smem_u32(smem + SM_Q);
            auto issue_s = [&](int i) -> bool {
                const int s = i & 1;
                if (!mbar_wait(&bars.k_full[s], (i >> 1) & 1, abort)) return false;
                if (i >= 2 && !mbar_wait(&bars.s_free[s], ((i - 2) >> 1) & 1, abort)) return false;
                tc_fence_after();
                const uint32_t k_base = smem_u32(smem + SM_K + s * 16384);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t ad =
                        sw128_desc(q_base + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        sw128_desc(k_base + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
                    mma_bf16(taddr + T_S + s * BN, ad, bd, IDESC_S, kk > 0);
                }
                mma_commit(&bars.s_full[s]);
                return true;
            };
            bool ok = mbar_wait(&bars.q_full, 0, abort) && issue_s(0);
            const uint32_t p_base = smem_u32(smem + SM_P);
            for (int i = 0; ok && i < n_tiles; ++i) {
                const int s = i & 1;
                if (i + 1 < n_tiles && !issue_s(i + 1)) break;
                if (!mbar_wait(&bars.p_full, i & 1, abort)) break;
                if (!mbar_wait(&bars.v_full[s], (i >> 1) & 1, abort)) break;
                tc_fence_after();
                const uint32_t v_base = smem_u32(smem + SM_V + s * 16384);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t ad = sw128_desc(p_base + kk * 32, 16, 1024);
                    const uint64_t bd = sw128_desc(v_base + kk * 16 * 128, BN * 128, 1024);
                    mma_bf16(taddr + T_O, ad, bd, IDESC_O, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars.o_done);
                mma_commit(&bars.kv_empty[s]);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax warps
        const bool row_ok = tid < rows_here;
        const int64_t row = row0 + tid;
        const int64_t t =
            SPARSE ? t_first
                   : a.bt.q_pos0[0] + (row0 + (row_ok ? tid : rows_here - 1)) / a.H;
        int64_t nv = n_vis(t, a.m);
        if (nv > Tc) nv = Tc;
        const int64_t w_lo = a.W > 0 ? max((int64_t)0, t - a.W + 1) : t + 1;
        // window positions the raw cache does not hold are skipped and flagged
        const int64_t c_lo = max(w_lo, raw_pos0), c_hi = min(t, raw_pos0 + Nraw - 1);
        if (row_ok && a.W > 0 && (c_lo > w_lo || c_hi < t)) flag(a.dev_err, LC_DEVERR_WINDOW);
        const uint32_t lane_addr = taddr + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = !dead;
        uint8_t *prow = smem + SM_P + tid * 128;
        // tcgen05.ld/st are warp-collective: every decision that guards them
        // is made uniform across the warp
        for (int i = 0; ok && i < n_tiles; ++i) {
            const int b = i & 1;
            if (!__all_sync(FULL, mbar_wait(&bars.s_full[b], (i >> 1) & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[BN];
            {
                float v0[32], v1[32];
                tmem_ld32(lane_addr + T_S + b * BN, v0);
                tmem_ld32(lane_addr + T_S + b * BN + 32, v1);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = v0[c];
                    s[32 + c] = v1[c];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.s_free[b]);
            // valid keys: a 64-bit mask (CSA selected tiles) or a column range
            uint64_t vmask;
            if (SPARSE && i < nct) {
                if (!__all_sync(FULL, mbar_wait(&bars.mask_full[b], (i >> 1) & 1, abort))) {
                    ok = false;
                    break;
                }
                vmask = *reinterpret_cast<volatile uint64_t *>(&bars.mask[b]);
            } else {
                int lo, hi;
                if (i < nct) {
                    const int64_t j0 = (int64_t)i * BN;
                    lo = 0;
                    hi = (int)max((int64_t)0, min((int64_t)BN, nv - j0));
                } else {
                    const int64_t p0 = wlo + (int64_t)(i - nct) * BN;
                    lo = (int)min((int64_t)BN, max((int64_t)0, c_lo - p0));
                    hi = (int)max((int64_t)0, min((int64_t)BN, c_hi + 1 - p0));
                }
                vmask = hi > lo ? (low_bits(hi) & ~low_bits(lo)) : 0ull;
            }
            if (!row_ok) vmask = 0;
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                if (!((vmask >> c) & 1ull)) s[c] = -INFINITY;
                mt = fmaxf(mt, s[c]);
            }
            const float m_new = fmaxf(m_used, mt * a.scale_log2);
            const bool grow = m_new > m_used + RESCALE_LOG2;
            // grow the reference max; O and l are rescaled only for rows that
            // already hold a finite reference (others have O = 0, l = 0)
            const bool need = grow && m_used != -INFINITY;
            bool waited = false;
            if (__any_sync(FULL, need)) {
                if (!__all_sync(FULL, mbar_wait(&bars.o_done, (i - 1) & 1, abort))) {
                    ok = false;
                    break;
                }
                waited = true;
                tc_fence_after();
                const float f = need ? exp2f(m_used - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < HD; c += 32) {
                    float o[32];
                    tmem_ld32(lane_addr + T_O + c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] *= f;
                    tmem_st32(lane_addr + T_O + c, o);
                }
                tmem_wait_st();
                l *= f;
            }
            if (grow) m_used = m_new;
            uint32_t pk[BN / 2];
            const float neg = -m_used;
            if (m_used == -INFINITY) {
#pragma unroll
                for (int c = 0; c < BN / 2; ++c) pk[c] = 0u;
            } else {
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    const float p0 = exp2f(fmaf(s[c], a.scale_log2, neg));
                    const float p1 = exp2f(fmaf(s[c + 1], a.scale_log2, neg));
                    l += p0 + p1;
                    pk[c / 2] = pack_bf16x2(p0, p1);
                }
            }
            if (i > 0 && !waited &&
                !__all_sync(FULL, mbar_wait(&bars.o_done, (i - 1) & 1, abort))) {
                ok = false;
                break;
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 v = make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
                *reinterpret_cast<uint4 *>(prow + ((ch ^ (tid & 7)) * 16)) = v;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_full);
        }
        // epilogue (ok is warp-uniform here)
        if (ok && n_tiles > 0 &&
            !__all_sync(FULL, mbar_wait(&bars.o_done, (n_tiles - 1) & 1, abort)))
            ok = false;
        if (!ok) {
            if (row_ok) flag(a.dev_err, LC_DEVERR_TIMEOUT);
        } else {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.O + row * HD);
#pragma unroll 1
            for (int c = 0; c < HD; c += 32) {
                float o[32];
                if (n_tiles > 0) {
                    tmem_ld32(lane_addr + T_O + c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = 0.f;
                }
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
            if (row_ok && a.lse) a.lse[row] = l > 0.f ? (m_used + log2f(l)) / LOG2E_F : -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(taddr, TMEM_COLS);
    }
}

namespace {
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <bool SPARSE>
lc_status launch_attn_tc(const CUtensorMap (&maps)[5], const AttnTcArgs &a, unsigned grid,
                         cudaStream_t st) {
    auto kfn = k_attn_tc<SPARSE>;
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SM_TOTAL) != cudaSuccess)
            return LC_ERR_CUDA;
        cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        attr_done = true;
    }
    LC_LAUNCH(kfn, dim3(grid), dim3(THREADS), SM_TOTAL, st, maps[0], maps[1], maps[2], maps[3],
              maps[4], a);
    return check_launch();
}

// Tensor maps of Q and of the compressed / raw K and V (dummy maps on Q for
// sources that are absent; they are never read then).  `gather` selects the
// one-row boxes of tile::gather4 for the compressed entries.
bool make_maps(CUtensorMap (&maps)[5], const void *Q, int64_t q_rows, const void *Kc,
               const void *Vc, int64_t c_rows, const void *Kr, const void *Vr, int64_t r_rows,
               bool gather) {
    const bool have_c = c_rows > 0 && Kc && Vc;
    const bool have_r = r_rows > 0 && Kr && Vr;
    const uint32_t cbox = gather ? 1 : BN;
    return make_tmap_bf16_2d(&maps[0], Q, (uint64_t)q_rows, HD, HD * 2, 64, BM) &&
           make_tmap_bf16_2d(&maps[1], have_c ? Kc : Q, have_c ? c_rows : 1, HD, HD * 2, 64,
                             cbox) &&
           make_tmap_bf16_2d(&maps[2], have_c ? Vc : Q, have_c ? c_rows : 1, HD, HD * 2, 64,
                             cbox) &&
           make_tmap_bf16_2d(&maps[3], have_r ? Kr : Q, have_r ? r_rows : 1, HD, HD * 2, 64, BN) &&
           make_tmap_bf16_2d(&maps[4], have_r ? Vr : Q, have_r ? r_rows : 1, HD, HD * 2, 64, BN);
}
}  // namespace

// CSA sparse attention on the tensor cores: bf16, d = 128, H <= 128, any
// ragged batch (one CTA per query token).  LC_ERR_UNSUPPORTED otherwise.
lc_status sparse_tc_launch(const void *Q, const void *Kc, const void *Vc, const int32_t *topk,
                           int k, const void *Kraw, const void *Vraw, const lc_batch &b, int H,
                           int d, int m, int W, float scale, lc_dtype dt, void *O, float *lse,
                           int32_t *dev_err, cudaStream_t st) {
    if (dt != LC_BF16 || d != HD || H > BM || b.total_q > 0x7fffffff ||
        b.total_c >= 0x7fffffff || b.total_raw >= 0x7fffffff)
        return LC_ERR_UNSUPPORTED;
    if (!al16(Q) || !al16(O) || !al16(Kc) || !al16(Vc) || (Kraw && !al16(Kraw)) ||
        (Vraw && !al16(Vraw)))
        return LC_ERR_UNSUPPORTED;
    if (b.total_q == 0) return LC_OK;
    const bool have_r = W > 0 && b.total_raw > 0 && Kraw && Vraw;
    CUtensorMap maps[5];
    if (!make_maps(maps, Q, b.total_q * H, Kc, Vc, b.total_c, Kraw, Vraw,
                   have_r ? b.total_raw : 0, true))
        return LC_ERR_CUDA;
    AttnTcArgs a{};
    a.n_rows = b.total_q * H;
    a.H = H;
    a.bt = to_dev(b);
    a.topk = topk;
    a.k = k;
    a.m = m;
    a.W = have_r ? W : 0;
    a.scale_log2 = scale * LOG2E_F;
    a.O = reinterpret_cast<__nv_bfloat16 *>(O);
    a.lse = lse;
    a.dev_err = dev_err;
    return launch_attn_tc<true>(maps, a, (unsigned)b.total_q, st);
}

}  // namespace lc
