// Selection kernels of the fused index + top-k (the exact causal top-k of
// page "DeepSeek-V4 技术解析…", §1.1: the top-k selector keeps the best
// compressed entries), after the tensor-core passes of index_tc.cu:
//
// k_sample_threshold16  one warp per query row.  The sample pass stored the
//     top 16 bits of each sampled score's order key (visible columns only);
//     two 8-bit radix digits find T16, the rho-th largest of them, and
//     theta = T16 << 16.  Truncation only lowers a key, so at least rho
//     sampled entries have full keys >= theta: theta is a lower bound of the
//     rho-th largest sampled key, the bound the candidate pass needs.
// k_cand_pick_warp  one warp per query row whose visible entries fit the
//     warp's bitmaps: four 8-bit radix digits over the row's candidates
//     (read where the candidate pass left them: the private slots of each
//     CTA column, then the row's overflow slots) give the k-th largest key
//     K* and how many ties at K* rank within the top k; candidates above K*
//     are marked in bitmap A, candidates at K* in bitmap E, both indexed by
//     entry; one pass over the words writes A plus the lowest-index ties of E
//     in ascending entry order.  A row whose candidate count lies outside
//     [k, cap] (or whose overflow exceeded its region) is appended to the
//     list of failed rows.
// k_topk_fallback  a fixed grid over the failed rows: each CTA recomputes its
//     row's scores into its own row buffer (bf16 keys, fp32 arithmetic, a
//     warp per entry) and takes the exact top-k there.  No work when the
//     list is empty.
#include <cuda_bf16.h>

#include "topk_common.cuh"

namespace lc {

namespace {
constexpr int SEL_WARPS = 8;  // rows per CTA of the warp-per-row kernels
const unsigned FULL = 0xffffffffu;
}  // namespace

__global__ void __launch_bounds__(SEL_WARPS * 32) k_sample_threshold16(
    const uint16_t *__restrict__ samp, int64_t lds, Batch bt, int m, int stride, int k, int rho,
    int64_t total_q, uint32_t *__restrict__ theta, int32_t *__restrict__ count,
    int32_t *__restrict__ nfail) {
    __shared__ uint32_t hist[SEL_WARPS][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (blockIdx.x == 0 && threadIdx.x == 0) *nfail = 0;
    const int64_t r = (int64_t)blockIdx.x * SEL_WARPS + warp;
    if (r >= total_q) return;  // the whole warp
    const int bq = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[bq] + (r - bt.cu_q[bq]);
    const int64_t Tc = bt.cu_c[bq + 1] - bt.cu_c[bq];
    int64_t nv = n_vis(t, m);
    if (nv > Tc) nv = Tc;
    const int64_t nvs = (nv + stride - 1) / stride;
    uint32_t th = 0;
    if (nv > k && rho <= nvs) {
        const uint16_t *row = samp + r * lds;  // 16-byte aligned (lds % 8 == 0)
        const int n = (int)nvs;
        // the whole warp steps together, four 16-byte loads per lane in flight
        auto visit = [&](auto f) {
            for (int b8 = 0; 8 * b8 < n; b8 += 128) {
                uint4 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j8 = b8 + 32 * q + lane;
                    v[q] = 8 * j8 < n ? *reinterpret_cast<const uint4 *>(row + 8 * j8)
                                      : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j8 = b8 + 32 * q + lane;
                    const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        f((w[u >> 1] >> (16 * (u & 1))) & 0xffffu, 8 * j8 + u < n);
                }
            }
        };
        int need = rho;
        const uint32_t d1 = warp_radix_digit(hist[warp], visit, 0u, 0u, 8, need);
        const uint32_t d2 = warp_radix_digit(hist[warp], visit, d1 << 8, 0xff00u, 0, need);
        th = ((d1 << 8) | d2) << 16;
    }
    if (lane == 0) {
        theta[r] = th;
        count[r] = 0;
    }
}

// Shared memory per warp: hist[256], A[nwmax], E[nwmax] (words).
__global__ void __launch_bounds__(SEL_WARPS * 32) k_cand_pick_warp(
    Batch bt, int m, int k, int cap, int ocap, int nwmax, int64_t total_q,
    const int32_t *__restrict__ count, const uint2 *__restrict__ cand,
    const int32_t *__restrict__ lcnt, const uint2 *__restrict__ priv, int gy, int cloc,
    int32_t *__restrict__ topk, int32_t *__restrict__ flist, int32_t *__restrict__ nfail,
    int32_t *dev_err) {
    extern __shared__ uint32_t sm_sel[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r = (int64_t)blockIdx.x * SEL_WARPS + warp;
    if (r >= total_q) return;
    uint32_t *hist = sm_sel + warp * (256 + 2 * nwmax);
    uint32_t *A = hist + 256, *E = A + nwmax;
    const int bq = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[bq] + (r - bt.cu_q[bq]);
    const int64_t Tc = bt.cu_c[bq + 1] - bt.cu_c[bq];
    int64_t nv = n_vis(t, m);
    if (nv > Tc) nv = Tc;
    int32_t *out = topk + r * k;
    if (nv <= k) {
        for (int i = lane; i < k; i += 32) out[i] = i < nv ? i : -1;
        return;
    }
    const int nw = (int)((nv + 31) >> 5);
    // the first 32 segments' counts, one per lane (shuffled out below)
    const int lc0 = lane < gy ? lcnt[r * gy + lane] : 0;
    int n_priv = lc0;
    for (int y = lane + 32; y < gy; y += 32) n_priv += lcnt[r * gy + y];
    n_priv = __reduce_add_sync(FULL, n_priv);
    const int n_over = count[r];
    const int n = n_priv + n_over;
    if (n < k || n > cap || n_over > ocap || nw > nwmax) {
        if (lane == 0) flist[atomicAdd(nfail, 1)] = (int32_t)r;
        return;
    }
    // every candidate of the row: (order key, entry index); all 32 lanes step
    // together, lanes past a segment's end get valid = false.  Each lane has
    // four loads in flight before it visits them (the visits are shared-memory
    // atomics, which the loads would otherwise wait behind one by one)
    auto each = [&](auto f) {
        auto run = [&](const uint2 *seg, int c) {
            for (int i0 = 0; i0 < c; i0 += 128) {
                uint2 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + 32 * u + lane;
                    v[u] = i < c ? seg[i] : make_uint2(0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (i0 + 32 * u < c) f(v[u], i0 + 32 * u + lane < c);
            }
        };
        for (int y = 0; y < gy; ++y)
            run(priv + ((size_t)r * gy + y) * cloc,
                y < 32 ? __shfl_sync(FULL, lc0, y) : lcnt[r * gy + y]);
        run(cand + (size_t)r * ocap, n_over);
    };
    auto keys = [&](auto f) { each([&](uint2 kv, bool ok) { f(kv.x, ok); }); };
    int need = k;
    uint32_t prefix = 0, mask = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t dg = warp_radix_digit(hist, keys, prefix, mask, shift, need);
        prefix |= dg << shift;
        mask |= 255u << shift;
    }
    const uint32_t kstar = prefix;
    for (int w = lane; w < nw; w += 32) {
        A[w] = 0u;
        E[w] = 0u;
    }
    __syncwarp();
    each([&](uint2 kv, bool ok) {
        if (!ok) return;
        const uint32_t e = kv.y;
        if (e >= (uint32_t)nv) {
            flag(dev_err, LC_DEVERR_BATCH);  // a candidate outside the row: never expected
            return;
        }
        if (kv.x > kstar)
            atomicOr(&A[e >> 5], 1u << (e & 31u));
        else if (kv.x == kstar)
            atomicOr(&E[e >> 5], 1u << (e & 31u));
    });
    __syncwarp();
    // ascending output: the marked entries above K*, plus the `need`
    // lowest-index entries at K*
    int pos = 0, ties_left = need;
    for (int w0 = 0; w0 < nw; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t a = w < nw ? A[w] : 0u;
        uint32_t e = w < nw ? E[w] : 0u;
        const int te = __popc(e);
        int tin = te;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, tin, o);
            if (lane >= o) tin += y;
        }
        const int take = min(te, max(0, ties_left - (tin - te)));
        uint32_t keep = 0u;
        for (int i = 0; i < take; ++i) {
            const uint32_t low = e & (0u - e);
            keep |= low;
            e ^= low;
        }
        uint32_t sel = a | keep;
        const int c = __popc(sel);
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, inc, o);
            if (lane >= o) inc += y;
        }
        int p = pos + inc - c;
        while (sel) {
            const int bit = __ffs(sel) - 1;
            sel &= sel - 1;
            if (p < k) out[p] = w * 32 + bit;
            ++p;
        }
        pos += __shfl_sync(FULL, inc, 31);
        ties_left -= min(ties_left, __shfl_sync(FULL, tin, 31));
    }
    for (int i = pos + lane; i < k; i += 32) out[i] = -1;  // never taken: pos == k
}

// Exact top-k of the rows in flist[0 .. *nfail) from recomputed scores.
// buf: gridDim.x rows of ldb floats, one per CTA.
template <int HI>
__global__ void __launch_bounds__(512) k_topk_fallback(const __nv_bfloat16 *__restrict__ qI,
                                                       const float *__restrict__ w,
                                                       const __nv_bfloat16 *__restrict__ kI,
                                                       Batch bt, int m, int k,
                                                       const int32_t *__restrict__ flist,
                                                       const int32_t *__restrict__ nfail,
                                                       float *buf, int64_t ldb,
                                                       int32_t *__restrict__ topk) {
    constexpr int NT = 512, NW = NT / 32, DI = 64;
    constexpr int LPH = 32 / HI, DPL = DI / LPH;  // lanes per head, dims per lane (8 or 16)
    __shared__ float sq[HI * DI];
    __shared__ float sw[HI];
    __shared__ RadixScratch rs;
    __shared__ int warp_sums[NW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = lane / LPH, sl = lane % LPH;
    const int total = *nfail;
    float *row = buf + (int64_t)blockIdx.x * ldb;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
        const int64_t r = flist[i];
        const int bq = seq_of_row(bt, r);
        const int64_t t = bt.q_pos0[bq] + (r - bt.cu_q[bq]);
        const int64_t c_beg = bt.cu_c[bq], Tc = bt.cu_c[bq + 1] - c_beg;
        int64_t nv = n_vis(t, m);
        if (nv > Tc) nv = Tc;
        if (nv > ldb) nv = ldb;
        __syncthreads();  // the previous row's reads of sq, sw and row are done
        for (int j = threadIdx.x; j < HI * DI; j += NT)
            sq[j] = __bfloat162float(qI[r * HI * DI + j]);
        if (threadIdx.x < HI) sw[threadIdx.x] = w[r * HI + threadIdx.x];
        __syncthreads();
        for (int64_t j = warp; j < nv; j += NW) {
            const __nv_bfloat16 *kr = kI + ((c_beg + j) * HI + h) * DI + sl * DPL;
            float d = 0.f;
#pragma unroll
            for (int u = 0; u < DPL; u += 8) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(kr + u));
                const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    d = fmaf(sq[h * DI + sl * DPL + u + 2 * q], __uint_as_float(x[q] << 16), d);
                    d = fmaf(sq[h * DI + sl * DPL + u + 2 * q + 1],
                             __uint_as_float(x[q] & 0xffff0000u), d);
                }
            }
#pragma unroll
            for (int o = 1; o < LPH; o <<= 1) d += __shfl_xor_sync(FULL, d, o);
            float p = sw[h] * fmaxf(d, 0.f);
#pragma unroll
            for (int o = LPH; o < 32; o <<= 1) p += __shfl_xor_sync(FULL, p, o);
            if (lane == 0) row[j] = p;
        }
        __syncthreads();
        radix_topk_row<NT, false>(row, nv, k, topk + r * k, rs, warp_sums);
    }
}

// Host side ------------------------------------------------------------------

lc_status sample_threshold16_launch(const uint16_t *samp, int64_t lds, const lc_batch &b, int m,
                                    int stride, int k, int rho, uint32_t *theta, int32_t *count,
                                    int32_t *nfail, cudaStream_t st) {
    const int64_t blocks = (b.total_q + SEL_WARPS - 1) / SEL_WARPS;
    if (blocks >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    LC_LAUNCH(k_sample_threshold16, dim3((unsigned)blocks), dim3(SEL_WARPS * 32), 0, st, samp,
              lds, to_dev(b), m, stride, k, rho, b.total_q, theta, count, nfail);
    return check_launch();
}

size_t cand_pick_warp_smem(int nwmax) {
    return sizeof(uint32_t) * (size_t)SEL_WARPS * (256 + 2 * (size_t)nwmax);
}

lc_status cand_pick_warp_launch(const lc_batch &b, int m, int k, int cap, int ocap, int nwmax,
                                const int32_t *count, const uint2 *cand, const int32_t *lcnt,
                                const uint2 *priv, int gy, int cloc, int32_t *topk,
                                int32_t *flist, int32_t *nfail, int32_t *dev_err,
                                cudaStream_t st) {
    const size_t smem = cand_pick_warp_smem(nwmax);
    static size_t attr = 0;
    if (smem > 48 * 1024 && smem > attr) {
        if (cudaFuncSetAttribute(k_cand_pick_warp, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return LC_ERR_CUDA;
        attr = smem;
    }
    const int64_t blocks = (b.total_q + SEL_WARPS - 1) / SEL_WARPS;
    if (blocks >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    LC_LAUNCH(k_cand_pick_warp, dim3((unsigned)blocks), dim3(SEL_WARPS * 32), smem, st, to_dev(b),
              m, k, cap, ocap, nwmax, b.total_q, count, cand, lcnt, priv, gy, cloc, topk, flist,
              nfail, dev_err);
    return check_launch();
}

lc_status topk_fallback_launch(const void *qI, const float *w, const void *kI, const lc_batch &b,
                               int HI, int m, int k, const int32_t *flist, const int32_t *nfail,
                               float *buf, int64_t ldb, int grid, int32_t *topk,
                               cudaStream_t st) {
    if (grid < 1) return LC_ERR_WORKSPACE;
    const auto *q = static_cast<const __nv_bfloat16 *>(qI);
    const auto *kk = static_cast<const __nv_bfloat16 *>(kI);
    if (HI == 8)
        LC_LAUNCH_AS("k_topk_fallback", k_topk_fallback<8>, dim3((unsigned)grid), dim3(512), 0,
                     st, q, w, kk, to_dev(b), m, k, flist, nfail, buf, ldb, topk);
    else
        LC_LAUNCH_AS("k_topk_fallback", k_topk_fallback<4>, dim3((unsigned)grid), dim3(512), 0,
                     st, q, w, kk, to_dev(b), m, k, flist, nfail, buf, ldb, topk);
    return check_launch();
}

}  // namespace lc
