// Exact causal top-k per row under the total order (score desc, index asc).
//
// k_topk_radix, one CTA per row (rows of a prefill batch):
//   1. radix select (4 passes of 8 bits over the order-preserving uint32 keys
//      of the visible scores) finds the k-th largest key K* and how many keys
//      equal to K* must be kept (`need`);
//   2. one ordered compaction pass keeps every key > K* and the first `need`
//      keys == K* in index order; writing positions come from block-wide
//      prefix sums, so the output is already in ascending index order.
//   Scores are read 5 times; the row stays hot in L2 for rows up to a few MB.
//
// k_topk_cluster, one thread-block cluster of C CTAs per row (a few long
// rows, e.g. a decode batch, where one CTA per row would leave most SMs idle):
//   CTA c of the cluster owns the contiguous slice [n c / C, n (c+1) / C) of
//   the row's n visible columns and stages its order keys in shared memory.
//   Each radix pass builds the slice's 256-bin histogram; after a cluster
//   barrier every CTA sums the C histograms through distributed shared memory,
//   so all CTAs pick the same digit.  For the compaction each CTA counts its
//   keys > K* and == K*; from the counts of the CTAs before it (read the same
//   way) it knows how many ties it may keep and where its part of the output
//   starts, then compacts its slice in index order as above.
#include <cooperative_groups.h>

#include "topk_common.cuh"

namespace lc {

namespace {
constexpr int TK_THREADS = 512;
}

// Query row r0 + blockIdx.x, its scores in row blockIdx.x of `scores`.
__global__ void __launch_bounds__(TK_THREADS) k_topk_radix(const float *__restrict__ scores,
                                                           int64_t ld, Batch bt, int m, int k,
                                                           int32_t *__restrict__ topk,
                                                           int64_t r0, int32_t *dev_err) {
    __shared__ RadixScratch rs;
    __shared__ int warp_sums[TK_THREADS / 32];
    const int64_t r = r0 + blockIdx.x;
    const int b = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[b] + (r - bt.cu_q[b]);
    const int64_t Tc = bt.cu_c[b + 1] - bt.cu_c[b];
    int64_t n = n_vis(t, m);
    if (n > Tc) {
        if (threadIdx.x == 0) flag(dev_err, LC_DEVERR_BATCH);
        n = Tc;
    }
    if (n > ld) n = ld;
    int32_t *out = topk + r * k;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += TK_THREADS) out[i] = i < n ? i : -1;
        return;
    }
    radix_topk_row<TK_THREADS>(scores + (int64_t)blockIdx.x * ld, n, k, out, rs, warp_sums);
}

namespace cg = cooperative_groups;

namespace {
constexpr int TC_THREADS = 512;
// keys of a slice staged in shared memory (32 KB): an 8-CTA cluster stages
// rows of up to 65,536 entries (the decode batch's longest), and four CTAs
// fit on an SM, so 64 rows x 8 CTAs run as one wave (with 64 KB slices, three
// per SM, they ran as 1.15 waves: 41 against 56 us for the batch-64 decode)
constexpr int TC_STAGE_KEYS = 8192;
}  // namespace

__global__ void __launch_bounds__(TC_THREADS) k_topk_cluster(const float *__restrict__ scores,
                                                             int64_t ld, Batch bt, int m, int k,
                                                             int32_t *__restrict__ topk,
                                                             int64_t r0, int32_t *dev_err) {
    constexpr int NT = TC_THREADS, NW = NT / 32;
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ uint32_t skeys[];          // [TC_STAGE_KEYS]
    __shared__ uint32_t hist[2][256];            // this CTA's histogram (double-buffered)
    __shared__ uint32_t tot[256];                // the cluster's histogram
    __shared__ int counts[2];                    // keys > K*, keys == K* of this slice
    __shared__ uint32_t s_digit;
    __shared__ int s_need;
    __shared__ int warp_sums[NW];
    const int C = (int)cl.num_blocks(), c = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t rl = blockIdx.x / C;           // every CTA of a cluster has the same row
    const int64_t r = r0 + rl;                   // its scores: row rl of `scores`
    const int b = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[b] + (r - bt.cu_q[b]);
    const int64_t Tc = bt.cu_c[b + 1] - bt.cu_c[b];
    int64_t n = n_vis(t, m);
    if (n > Tc) {
        if (c == 0 && tid == 0) flag(dev_err, LC_DEVERR_BATCH);
        n = Tc;
    }
    if (n > ld) n = ld;
    int32_t *out = topk + r * k;
    if (n <= k) {  // the whole cluster takes this branch
        for (int64_t i = (int64_t)c * NT + tid; i < k; i += (int64_t)C * NT)
            out[i] = i < n ? (int32_t)i : -1;
        return;
    }
    const float *row = scores + rl * ld;
    const int64_t lo = n * c / C, hi = n * (c + 1) / C;
    const int len = (int)(hi - lo);
    const bool staged = len <= TC_STAGE_KEYS;
    if (staged) {
        for (int j = tid; j < len; j += NT) skeys[j] = order_key(__ldg(row + lo + j));
    }
    auto key_at = [&](int j) -> uint32_t {
        return staged ? skeys[j] : order_key(__ldg(row + lo + j));
    };

    // ---- radix selection of the k-th largest key over the whole row
    uint32_t prefix = 0, mask = 0;
    int need = k;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *h = hist[pass & 1];
        for (int i = tid; i < 256; i += NT) h[i] = 0u;
        __syncthreads();  // also orders the staging stores before the first pass
        for (int j = tid; j < len; j += NT) {
            const uint32_t key = key_at(j);
            if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1u);
        }
        // every CTA's histogram of this pass is complete and visible; the
        // other buffer is free again (its readers passed this barrier)
        cl.sync();
        if (tid < 256) {
            uint32_t sum = 0;
            for (int q = 0; q < C; ++q) sum += *cl.map_shared_rank(&h[tid], q);
            tot[tid] = sum;
        }
        __syncthreads();
        if (warp == 0) {
            // suffix sums over the 256 bins, 8 bins per lane, highest first
            uint32_t cnt[8];
            uint32_t mine = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                cnt[u] = tot[255 - (lane * 8 + u)];
                mine += cnt[u];
            }
            uint32_t incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - mine;
            if (excl < (uint32_t)need && incl >= (uint32_t)need) {
                uint32_t cum = excl;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (cum + cnt[u] >= (uint32_t)need) {
                        s_digit = 255u - (uint32_t)(lane * 8 + u);
                        s_need = need - (int)cum;
                        break;
                    }
                    cum += cnt[u];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        need = s_need;
    }
    const uint32_t kstar = prefix;

    // ---- this slice's keys above and at K*, then the counts of the CTAs before it
    int gt = 0, eq = 0;
    for (int j = tid; j < len; j += NT) {
        const uint32_t key = key_at(j);
        gt += key > kstar;
        eq += key == kstar;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (tid == 0) counts[0] = counts[1] = 0;
    __syncthreads();
    if (lane == 0) {
        atomicAdd(&counts[0], gt);
        atomicAdd(&counts[1], eq);
    }
    cl.sync();
    int64_t out0 = 0, eq_before = 0;
    for (int q = 0; q < c; ++q) {
        const int g = *cl.map_shared_rank(&counts[0], q);
        const int e = *cl.map_shared_rank(&counts[1], q);
        const int64_t tk = min((int64_t)e, max((int64_t)0, (int64_t)need - eq_before));
        out0 += g + tk;
        eq_before += e;
    }
    const int my_eq = counts[1];
    const int my_ties = (int)min((int64_t)my_eq, max((int64_t)0, (int64_t)need - eq_before));
    const int my_take = counts[0] + my_ties;
    // no CTA reads another's shared memory after this point
    cl.sync();

    // ---- ordered compaction of the slice: keys > K*, then the first ties
    int written = 0, eq_seen = 0;
#pragma unroll 1
    for (int j0 = 0; j0 < len && written < my_take; j0 += NT) {
        const int j = j0 + tid;
        uint32_t key = 0;
        if (j < len) key = key_at(j);
        const int is_gt = (j < len) && key > kstar;
        const int is_eq = (j < len) && key == kstar;
        int eq_tot;
        const int eq_pre = block_exclusive_scan<NT>(is_eq, warp_sums, &eq_tot);
        const int take = is_gt || (is_eq && eq_seen + eq_pre < my_ties);
        int take_tot;
        const int pos = block_exclusive_scan<NT>(take, warp_sums, &take_tot);
        if (take && written + pos < my_take) out[out0 + written + pos] = (int32_t)(lo + j);
        written += take_tot;
        eq_seen += eq_tot;
    }
}

// Top-k of query rows r0 .. r0 + nrows - 1, whose scores are rows 0 .. nrows
// - 1 of `scores`.
lc_status topk_rows_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                           int32_t *topk, int64_t r0, int64_t nrows, int32_t *dev_err,
                           cudaStream_t st) {
    if (nrows <= 0) return LC_OK;
    // a few long rows: one 8-CTA cluster per row keeps the SMs busy
    constexpr int C = 8;
    if (nrows <= 2 * 148 && b.max_c >= 4096 && nrows * C < (1ll << 31)) {
        static bool attr = false;
        if (!attr) {
            if (cudaFuncSetAttribute(k_topk_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(TC_STAGE_KEYS * sizeof(uint32_t))) != cudaSuccess)
                return LC_ERR_CUDA;
            attr = true;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nrows * C));
        cfg.blockDim = dim3(TC_THREADS);
        cfg.dynamicSmemBytes = TC_STAGE_KEYS * sizeof(uint32_t);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, k_topk_cluster, scores, ld, to_dev(b), m,
                                                 k, topk, r0, dev_err);
        note_launch("k_topk_cluster");
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return check_launch_error(e);
        }
        return check_launch();
    }
    LC_LAUNCH(k_topk_radix, dim3((unsigned)nrows), dim3(TK_THREADS), 0, st, scores, ld,
              to_dev(b), m, k, topk, r0, dev_err);
    return check_launch();
}

lc_status topk_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                      int32_t *topk, int32_t *dev_err, cudaStream_t st) {
    return topk_rows_launch(scores, ld, b, m, k, topk, 0, b.total_q, dev_err, st);
}

}  // namespace lc
