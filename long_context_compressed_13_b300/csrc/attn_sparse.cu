// CSA core attention on the 5th-generation tensor cores, bf16, head dim 128
// (page "DeepSeek-V4 技术解析…", §1.1, CSA paragraph: MQA core attention over
// the entries kept by the top-k selector plus the sliding-window branch).
//
// A CTA owns one query token: its H <= 128 heads are the rows of one M = 128
// tile (rows H..127 are padding).  The token's keys are its selected entries,
// 128 slots per tile, gathered with 16-byte cp.async copies (16 lanes per
// 256-byte row, written straight into the 128-byte-swizzled operand layout;
// a TMA gather moves only 4 rows per instruction and is far slower), then its
// raw window positions as TMA boxes.
//   warps 4-7    producers: Q once, then K and V tiles into a 3-stage ring;
//                for a selected tile each warp looks up 32 of the slots' rows,
//                publishes its quarter of the tile's 128-bit slot validity
//                mask and gathers those rows (four warps keep more copies in
//                flight than two: the gather's issue rate bounds the kernel);
//                each producer thread's copies complete on the stage barrier
//   warp 8       TMEM owner and MMA issuer, in the order
//                  S(0), S(1), PV(0), S(2), PV(1), S(3), ...
//                S (M=128, N=128, K=128) alternates between two TMEM buffers,
//                so the next tile's scores are ready while the softmax works;
//                the softmax writes P (bf16) over the S it read, and PV
//                (M=128, N=128, K=128) reads it as its A operand
//   warps 0-3    softmax: thread r owns row r (TMEM lane r); with RoPE they
//                first rotate the token's query rows in shared memory; the
//                whole row of
//                S is read with four loads and one wait; the reference max
//                only moves when the max grows by more than 2^8 (then O and l
//                are rescaled after PV(j-1) has completed); p = 2^(s*scale*
//                log2e - m), the row sum, packed bf16 P into TMEM.
// TMEM: O [0,128) | S0/P0 [128,256) | S1/P1 [256,384).
// Every wait is bounded; on a timeout the CTA raises LC_DEVERR_TIMEOUT,
// skips the rest and still frees its TMEM.
#include "lc_common.cuh"
#include "sm100.cuh"

namespace lc {

using namespace sm100;

namespace {
constexpr int SBM = 128, SBN = 128, SHD = 128;
constexpr int NPW = 4;                                 // producer warps
constexpr int W_MMA_S = 4 + NPW;                       // MMA issuer warp
constexpr int S_THREADS = 384;                         // three warpgroups
static_assert(NPW == 4, "warpgroup 1 holds the producer warps");
// Registers are allocated to a CTA in whole warpgroups: launched at 168 a
// thread (384 x 168 <= 65,536), warpgroups 1 (producers) and 2 (MMA issuer,
// three idle warps) give back down to S_REG_LO and the softmax warpgroup grows
// to S_REG_HI, which its 128-float rows of S need without spilling.
constexpr uint32_t S_REG_LAUNCH = 168, S_REG_HI = 200, S_REG_LO = 120;
static_assert(128 * (S_REG_HI + 2 * S_REG_LO) <= S_THREADS * S_REG_LAUNCH &&
                  128 * (S_REG_HI - S_REG_LAUNCH) <= 2 * 128 * (S_REG_LAUNCH - S_REG_LO),
              "register split must fit the launch allocation");
constexpr int NPROD = 32 * NPW;                        // producer threads
constexpr int SPT = 128 / NPROD;                       // slots of a tile per producer thread
constexpr int S_NST = 3;                               // K/V stages
constexpr uint32_t S_TILE = SBN * 128;                 // one 64-column half of a 128-row tile
constexpr uint32_t SS_Q = 0;                           // 2 halves
constexpr uint32_t SS_K = SS_Q + 2 * S_TILE;           // S_NST stages x 2 halves
constexpr uint32_t SS_V = SS_K + S_NST * 2 * S_TILE;   // S_NST stages x 2 halves
constexpr uint32_t SS_BAR = SS_V + S_NST * 2 * S_TILE;
constexpr uint32_t SS_TOTAL = SS_BAR + 512;
constexpr uint32_t S_TMEM_COLS = 512;
constexpr uint32_t ST_O = 0, ST_S = 128;               // + 128 * buffer
constexpr float S_LOG2E = 1.4426950408889634f;
constexpr float S_RESCALE = 8.f;

struct SBars {
    uint64_t q_full, k_full[S_NST], v_full[S_NST], kv_empty[S_NST], mask_full[S_NST];
    uint64_t s_full[2], p_full, o_done;
    uint64_t stall;           // test hook: a barrier nothing completes
    uint64_t q_ready;         // RoPE: the softmax warps rotated Q
    uint32_t mask[S_NST][4];  // valid slots of the selected tile held by each stage
    uint32_t taddr;
    int abort;
    float2 rope_cs[32];       // RoPE: (cos, sin) of the token's angles
};
static_assert(sizeof(SBars) <= 512, "barrier block");

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrives on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ float ex2s(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3s(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
}  // namespace

struct SparseArgs {
    int H;
    const __nv_bfloat16 *Kc, *Vc;  // compressed entries (gathered rows)
    Batch bt;             // device batch arrays
    const int32_t *topk;  // [total_q, k]
    int k;
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

__global__ void __launch_bounds__(S_THREADS, 1)
    k_sparse_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKr,
                const __grid_constant__ CUtensorMap mVr, SparseArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    SBars &bars = *reinterpret_cast<SBars *>(smem + SS_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = &bars.abort;
    const unsigned FULL = 0xffffffffu;

    // ---- the token, its entries and its window
    const int64_t qrow = blockIdx.x;
    const int b = seq_of_row(a.bt, qrow);
    const int64_t t = a.bt.q_pos0[b] + (qrow - a.bt.cu_q[b]);
    const int64_t c_beg = a.bt.cu_c[b], Tc = a.bt.cu_c[b + 1] - c_beg;
    const int64_t raw_beg = a.bt.cu_raw[b], Nraw = a.bt.cu_raw[b + 1] - raw_beg;
    const int64_t raw_pos0 = a.bt.raw_pos0[b];
    int64_t nv = n_vis(t, a.m);
    if (nv > Tc) nv = Tc;
    const int nct = (a.k + SBN - 1) / SBN;
    int64_t wlo = 0;
    int nwt = 0;
    if (a.W > 0) {
        wlo = max((int64_t)0, t - a.W + 1);
        nwt = (int)((t - wlo + 1 + SBN - 1) / SBN);
    }
    const int n_tiles = nct + nwt;

    if (tid == 0) {
        bars.abort = (smem_u32(smem) & 1023u) != 0 ? 1 : 0;
        if (bars.abort) flag(a.dev_err, LC_DEVERR_TIMEOUT);  // layout assumption broken
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.stall, 1);
        for (int s = 0; s < S_NST; ++s) {
            mbar_init(&bars.k_full[s], NPROD);  // one arrival per producer thread
            mbar_init(&bars.v_full[s], NPROD);
            mbar_init(&bars.kv_empty[s], 1);
            mbar_init(&bars.mask_full[s], NPW);  // one per producer warp
        }
        mbar_init(&bars.s_full[0], 1);
        mbar_init(&bars.s_full[1], 1);
        mbar_init(&bars.p_full, 4);  // one arrival per softmax warp
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.q_ready, 4);  // one arrival per softmax warp
        fence_barrier_init();
    }
    if (warp == W_MMA_S) {
        tmem_alloc(&bars.taddr, S_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = bars.taddr;
    const bool dead = bars.abort != 0;

    if (warp >= 4) {
      // warpgroups 1 and 2: one register decrease per warpgroup, then the roles
      setmaxnreg_dec<S_REG_LO>();
      if (warp < 4 + NPW) {
        // ------------------------------------------------------ producer warps
        const int pt = tid - 128;  // producer thread 0 .. NPROD-1
        if (!dead && n_tiles > 0) {
            if (pt == 0) {
                prefetch_tmap(&mQ);
                mbar_expect_tx(&bars.q_full, 2 * S_TILE);
                tma_load_2d(smem + SS_Q, &mQ, &bars.q_full, 0, (int32_t)(qrow * a.H));
                tma_load_2d(smem + SS_Q + S_TILE, &mQ, &bars.q_full, 64, (int32_t)(qrow * a.H));
            }
            const char *kc_base = reinterpret_cast<const char *>(a.Kc) + (lane & 15) * 16;
            const char *vc_base = reinterpret_cast<const char *>(a.Vc) + (lane & 15) * 16;
            // the selected entries of this warp's slots NPROD u + 32(warp-4) + lane
            // (u < SPT) of a tile; the next tile's are loaded while the current
            // tile is gathered
            const int32_t *sel_row = a.topk + qrow * a.k;
            auto load_sel = [&](int i, int32_t (&jj)[SPT]) {
#pragma unroll
                for (int u = 0; u < SPT; ++u) {
                    const int slot = i * SBN + NPROD * u + pt;
                    jj[u] = (i < nct && slot < a.k) ? __ldg(sel_row + slot) : -1;
                }
            };
            int32_t jn[SPT];
            load_sel(0, jn);
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % S_NST;
                int32_t jc[SPT];
#pragma unroll
                for (int u = 0; u < SPT; ++u) jc[u] = jn[u];
                load_sel(i + 1, jn);
                if (i >= S_NST &&
                    !__all_sync(FULL, mbar_wait(&bars.kv_empty[s], ((i - S_NST) / S_NST) & 1, abort)))
                    break;
                uint8_t *kd = smem + SS_K + s * 2 * S_TILE, *vd = smem + SS_V + s * 2 * S_TILE;
                if (i < nct) {
                    // rows of this warp's slots, gathered by this warp, the
                    // indices passed by shuffles
                    int32_t g[SPT];
#pragma unroll
                    for (int u = 0; u < SPT; ++u) {
                        const int64_t j = jc[u];
                        const bool ok = j >= 0 && j < nv;
                        if (j >= nv) flag(a.dev_err, LC_DEVERR_INDEX);
                        // an empty or invalid slot fetches row 0, which always exists
                        g[u] = ok ? (int32_t)(c_beg + j) : 0;
                        const uint32_t bal = __ballot_sync(FULL, ok);
                        if (lane == 0) bars.mask[s][NPW * u + (warp - 4)] = bal;
                    }
                    if (lane == 0) mbar_arrive(&bars.mask_full[s]);
                    // gather: per pass two rows, 16 lanes x 16 bytes each, into the
                    // swizzled half `hf` of the stage
                    const int hw = lane >> 4, chunk = lane & 15, hf = chunk >> 3, cc = chunk & 7;
                    const uint32_t kdst = smem_u32(kd) + hf * S_TILE, vdst = smem_u32(vd) + hf * S_TILE;
#pragma unroll 8
                    for (int pass = 0; pass < 16 * SPT; ++pass) {
                        const int q = 2 * pass + hw, u = q >> 5, l = q & 31;
                        int32_t gu = g[0];
#pragma unroll
                        for (int v = 1; v < SPT; ++v)
                            if (u == v) gu = g[v];
                        const int64_t gi = __shfl_sync(FULL, gu, l);
                        const int r = NPROD * u + 32 * (warp - 4) + l;
                        const uint32_t off = (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
                        cp_async16(kdst + off, kc_base + gi * (SHD * 2));
                        cp_async16(vdst + off, vc_base + gi * (SHD * 2));
                    }
                    cp_async_arrive(&bars.k_full[s]);
                    cp_async_arrive(&bars.v_full[s]);
                } else {
                    if (pt == 0) {
                        const int32_t y =
                            (int32_t)(raw_beg + wlo + (int64_t)(i - nct) * SBN - raw_pos0);
                        mbar_expect_tx(&bars.k_full[s], 2 * S_TILE);
                        tma_load_2d(kd, &mKr, &bars.k_full[s], 0, y);
                        tma_load_2d(kd + S_TILE, &mKr, &bars.k_full[s], 64, y);
                        mbar_expect_tx(&bars.v_full[s], 2 * S_TILE);
                        tma_load_2d(vd, &mVr, &bars.v_full[s], 0, y);
                        tma_load_2d(vd + S_TILE, &mVr, &bars.v_full[s], 64, y);
                    } else {
                        mbar_arrive(&bars.k_full[s]);
                        mbar_arrive(&bars.v_full[s]);
                    }
                    if (lane == 0) mbar_arrive(&bars.mask_full[s]);  // keeps the phases in step
                }
                ++issued;
            }
            // copies still in flight must land before the CTA exits
            int dummy = 0;
            for (int i = max(0, issued - S_NST); i < issued; ++i) {
                mbar_wait(&bars.k_full[i % S_NST], (i / S_NST) & 1, &dummy, 400000000LL);
                mbar_wait(&bars.v_full[i % S_NST], (i / S_NST) & 1, &dummy, 400000000LL);
            }
            if (pt == 0) mbar_wait(&bars.q_full, 0, &dummy, 400000000LL);
            // the MMAs' releases of the last tiles: no commit may still be on
            // its way to this CTA's barriers when it exits (skipped after an
            // abort, when some of those MMAs are never issued)
            for (int i = max(0, issued - S_NST); i < issued && !*abort; ++i)
                mbar_wait(&bars.kv_empty[i % S_NST], (i / S_NST) & 1, abort);
        }
    } else if (warp == W_MMA_S) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !dead && n_tiles > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(SBM, SBN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(SBM, SHD, 0, 1);
            const uint32_t q_base = smem_u32(smem + SS_Q);
            auto issue_s = [&](int j) -> bool {
                const int s = j % S_NST;
                if (!mbar_wait(&bars.k_full[s], (j / S_NST) & 1, abort)) return false;
                fence_proxy_async_smem();  // gathered rows were written by cp.async
                tc_fence_after();
                const uint32_t k_base = smem_u32(smem + SS_K + s * 2 * S_TILE);
#pragma unroll
                for (int kk = 0; kk < SHD / 16; ++kk) {
                    const uint64_t ad =
                        sw128_desc(q_base + (kk >> 2) * S_TILE + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        sw128_desc(k_base + (kk >> 2) * S_TILE + (kk & 3) * 32, 16, 1024);
                    mma_bf16(taddr + ST_S + (j & 1) * 128, ad, bd, IDESC_S, kk > 0);
                }
                mma_commit(&bars.s_full[j & 1]);
                return true;
            };
            bool ok = (a.stall == 0 || mbar_wait(&bars.stall, 0, abort, a.stall)) &&
                      mbar_wait(a.rope ? &bars.q_ready : &bars.q_full, 0, abort) && issue_s(0) &&
                      (n_tiles < 2 || issue_s(1));
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int s = j % S_NST;
                if (!mbar_wait(&bars.v_full[s], (j / S_NST) & 1, abort) ||
                    !mbar_wait(&bars.p_full, j & 1, abort))
                    break;
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t v_base = smem_u32(smem + SS_V + s * 2 * S_TILE);
#pragma unroll
                for (int kk = 0; kk < SBN / 16; ++kk) {
                    const uint64_t bd = sw128_desc(v_base + kk * 16 * 128, S_TILE, 1024);
                    mma_bf16_ta(taddr + ST_O, taddr + ST_S + (j & 1) * 128 + kk * 8, bd, IDESC_O,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars.o_done);
                mma_commit(&bars.kv_empty[s]);
                // S(j+2) reuses the buffer of S(j): PV(j) was queued before it
                if (j + 2 < n_tiles && !issue_s(j + 2)) break;
            }
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<S_REG_HI>();
        // ------------------------------------------------------ softmax warps
        const bool row_ok = tid < a.H;
        const int64_t row = qrow * a.H + tid;
        const int64_t w_lo = a.W > 0 ? max((int64_t)0, t - a.W + 1) : t + 1;
        // window positions the raw cache does not hold are skipped and flagged
        const int64_t c_lo = max(w_lo, raw_pos0), c_hi = min(t, raw_pos0 + Nraw - 1);
        if (tid == 0 && a.W > 0 && (c_lo > w_lo || c_hi < t)) flag(a.dev_err, LC_DEVERR_WINDOW);
        const uint32_t lane_base = taddr + ((uint32_t)(warp * 32) << 16);
        const uint32_t o_addr = lane_base + ST_O;
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = !dead;
        // od = phases of o_done observed (PV(0..od-1) complete).  Phases are
        // waited one at a time and never fall two behind: before P(j) is
        // published PV(j) cannot have started, so at most PV(j-1) is pending.
        if (a.rope && ok && n_tiles > 0) {
            // partial RoPE of the token's query heads, in place, before the
            // first S MMA: angles of position t, then each thread rotates its row
            if (!__all_sync(FULL, mbar_wait(&bars.q_full, 0, abort))) ok = false;
            if (tid < 32) bars.rope_cs[tid] = rope_cs(t, rope_theta(tid));
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (ok && row_ok) rope_smem_row(smem + SS_Q + S_TILE, tid, bars.rope_cs);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.q_ready);
        }
        int od = 0;
        auto wait_pv = [&](int upto) -> bool {  // until PV(0..upto-1) complete
            while (od < upto) {
                if (!__all_sync(FULL, mbar_wait(&bars.o_done, od & 1, abort))) return false;
                ++od;
            }
            return true;
        };
        for (int j = 0; ok && j < n_tiles; ++j) {
            const uint32_t s_addr = lane_base + ST_S + (j & 1) * 128;
            if (!__all_sync(FULL, mbar_wait(&bars.s_full[j & 1], (j >> 1) & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // valid columns: slot mask (selected tiles) or the window range
            uint32_t vm[4];
            if (j < nct) {
                if (!__all_sync(FULL, mbar_wait(&bars.mask_full[j % S_NST], (j / S_NST) & 1, abort))) {
                    ok = false;
                    break;
                }
                const volatile uint32_t *mk = bars.mask[j % S_NST];
#pragma unroll
                for (int u = 0; u < 4; ++u) vm[u] = mk[u];
            } else {
                if (!__all_sync(FULL, mbar_wait(&bars.mask_full[j % S_NST], (j / S_NST) & 1, abort))) {
                    ok = false;
                    break;
                }
                const int64_t p0 = wlo + (int64_t)(j - nct) * SBN;
                const int lo = (int)min((int64_t)SBN, max((int64_t)0, c_lo - p0));
                const int hi = (int)max((int64_t)0, min((int64_t)SBN, c_hi + 1 - p0));
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int a0 = max(lo - 32 * u, 0), b0 = min(hi - 32 * u, 32);
                    vm[u] = b0 <= a0 ? 0u
                                     : ((b0 >= 32 ? 0xffffffffu : ((1u << b0) - 1u)) &
                                        (a0 >= 32 ? 0u : ~((1u << a0) - 1u)));
                }
            }
            if (!row_ok) vm[0] = vm[1] = vm[2] = vm[3] = 0u;
            const bool full = (vm[0] & vm[1] & vm[2] & vm[3]) == 0xffffffffu;
            // the whole row of S in registers: four loads in flight, one wait
            float v[SBN];
            tmem_ld32(s_addr, *reinterpret_cast<float(*)[32]>(v));
            tmem_ld32(s_addr + 32, *reinterpret_cast<float(*)[32]>(v + 32));
            tmem_ld32(s_addr + 64, *reinterpret_cast<float(*)[32]>(v + 64));
            tmem_ld32(s_addr + 96, *reinterpret_cast<float(*)[32]>(v + 96));
            tmem_wait_ld();
            if (!full) {
#pragma unroll
                for (int c = 0; c < SBN; ++c)
                    if (!((vm[c >> 5] >> (c & 31)) & 1u)) v[c] = -INFINITY;
            }
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < SBN; c += 2) mt = max3s(mt, v[c], v[c + 1]);
            const float m_new = fmaxf(m_used, mt * sl2);
            const bool grow = m_new > m_used + S_RESCALE;
            const bool need = grow && m_used != -INFINITY;
            if (__any_sync(FULL, need)) {
                // O holds PV(0..j-1); wait for PV(j-1) before rescaling it
                if (!wait_pv(j)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float f = need ? ex2s(m_used - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < SHD; c += 32) {
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
            for (int c0 = 0; c0 < SBN; c0 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float p0 = ex2s(fmaf(v[c0 + c], sl2, neg));
                    const float p1 = ex2s(fmaf(v[c0 + c + 1], sl2, neg));
                    l += p0 + p1;
                    pk[c / 2] = pack_bf16x2(p0, p1);
                }
                tmem_st16_u(s_addr + c0 / 2, pk);
            }
            tmem_wait_st();
            // keep the o_done phase count in step (PV(j-1) is long done here)
            if (!wait_pv(j)) {
                ok = false;
                break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_full);
        }
        // epilogue (ok is warp-uniform here)
        if (ok && n_tiles > 0 && !wait_pv(n_tiles)) ok = false;
        if (!ok) {
            if (row_ok) flag(a.dev_err, LC_DEVERR_TIMEOUT);
        } else {
            tc_fence_after();
            const float of =
                fold_sink(m_used, l, row_ok ? sink_log2(a.sink, tid, a.dev_err) : -INFINITY);
            const float inv = l > 0.f ? of / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.O + row * SHD);
#pragma unroll 1
            for (int c = 0; c < SHD; c += 32) {
                float o[32];
                if (n_tiles > 0) {
                    tmem_ld32(o_addr + c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = 0.f;
                }
                if (a.rope && n_tiles > 0 && c >= SHD - ROPE_DIMS)
                    rope_out32(o, c, SHD, bars.rope_cs);
                if (row_ok) {
#pragma unroll
                    for (int u = 0; u < 32; u += 8) {
                        uint4 vv = make_uint4(pack_bf16x2(o[u] * inv, o[u + 1] * inv),
                                              pack_bf16x2(o[u + 2] * inv, o[u + 3] * inv),
                                              pack_bf16x2(o[u + 4] * inv, o[u + 5] * inv),
                                              pack_bf16x2(o[u + 6] * inv, o[u + 7] * inv));
                        dst[(c + u) / 8] = vv;
                    }
                }
            }
            if (row_ok && a.lse) a.lse[row] = l > 0.f ? (m_used + log2f(l)) / S_LOG2E : -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA_S) {
        tc_fence_after();
        tmem_dealloc(taddr, S_TMEM_COLS);
    }
}

namespace {
bool al16s(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// CSA sparse attention on the tensor cores: bf16, d = 128, H <= 128, any
// ragged batch (one CTA per query token).  LC_ERR_UNSUPPORTED otherwise.
lc_status sparse_tc_launch(const void *Q, const void *Kc, const void *Vc, const int32_t *topk,
                           int k, const void *Kraw, const void *Vraw, const lc_batch &b, int H,
                           int d, int m, int W, float scale, const float *sink, int rope,
                           lc_dtype dt, void *O, float *lse, int32_t *dev_err, cudaStream_t st) {
    if (dt != LC_BF16 || d != SHD || H > SBM || b.total_c < 1 || b.total_q > 0x7fffffff ||
        b.total_q * H >= 0x7fffffff || b.total_c >= 0x7fffffff || b.total_raw >= 0x7fffffff)
        return LC_ERR_UNSUPPORTED;
    if (!al16s(Q) || !al16s(O) || !al16s(Kc) || !al16s(Vc) || (Kraw && !al16s(Kraw)) ||
        (Vraw && !al16s(Vraw)))
        return LC_ERR_UNSUPPORTED;
    if (b.total_q == 0) return LC_OK;
    const bool have_r = W > 0 && b.total_raw > 0 && Kraw && Vraw;
    CUtensorMap maps[3];
    if (!make_tmap_bf16_2d(&maps[0], Q, (uint64_t)(b.total_q * H), SHD, SHD * 2, 64, SBM) ||
        !make_tmap_bf16_2d(&maps[1], have_r ? Kraw : Q, have_r ? b.total_raw : 1, SHD, SHD * 2,
                           64, SBN) ||
        !make_tmap_bf16_2d(&maps[2], have_r ? Vraw : Q, have_r ? b.total_raw : 1, SHD, SHD * 2,
                           64, SBN))
        return LC_ERR_CUDA;
    SparseArgs a{};
    a.H = H;
    a.Kc = reinterpret_cast<const __nv_bfloat16 *>(Kc);
    a.Vc = reinterpret_cast<const __nv_bfloat16 *>(Vc);
    a.bt = to_dev(b);
    a.topk = topk;
    a.k = k;
    a.m = m;
    a.W = have_r ? W : 0;
    a.scale_log2 = scale * S_LOG2E;
    a.sink = sink;
    a.O = reinterpret_cast<__nv_bfloat16 *>(O);
    a.lse = lse;
    a.dev_err = dev_err;
    a.rope = rope;
    a.stall = debug_stall_clocks(LC_STALL_SPARSE_TC);
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(k_sparse_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SS_TOTAL) != cudaSuccess)
            return LC_ERR_CUDA;
        attr_done = true;
    }
    LC_LAUNCH(k_sparse_tc, dim3((unsigned)b.total_q), dim3(S_THREADS), SS_TOTAL, st, maps[0],
              maps[1], maps[2], a);
    return check_launch();
}

}  // namespace lc
