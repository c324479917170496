// Exact causal top-k per row under the total order (score desc, index asc).
// One CTA per row:
//   1. radix select (4 passes of 8 bits over the order-preserving uint32 keys
//      of the visible scores) finds the k-th largest key K* and how many keys
//      equal to K* must be kept (`need`);
//   2. one ordered compaction pass keeps every key > K* and the first `need`
//      keys == K* in index order; writing positions come from block-wide
//      prefix sums, so the output is already in ascending index order.
// Scores are read 5 times; the row stays hot in L2 for rows up to a few MB.
#include "topk_common.cuh"

namespace lc {

namespace {
constexpr int TK_THREADS = 512;
}

// row_mask (nullable): rows with row_mask[r] == 0 are skipped.
__global__ void __launch_bounds__(TK_THREADS) k_topk_radix(const float *__restrict__ scores,
                                                           int64_t ld, Batch bt, int m, int k,
                                                           int32_t *__restrict__ topk,
                                                           const int32_t *__restrict__ row_mask,
                                                           int32_t *dev_err) {
    __shared__ RadixScratch rs;
    __shared__ int warp_sums[TK_THREADS / 32];
    const int64_t r = blockIdx.x;
    if (row_mask && row_mask[r] == 0) return;
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
    const float *row = scores + r * ld;
    int need;
    const uint32_t kstar = radix_kth_largest<TK_THREADS>(row, n, k, rs, &need);

    // ordered compaction: keys > K*, then the first `need` keys == K*
    int written = 0, eq_seen = 0;
#pragma unroll 1
    for (int64_t j0 = 0; j0 < n && written < k; j0 += TK_THREADS) {
        const int64_t j = j0 + threadIdx.x;
        uint32_t key = 0;
        if (j < n) key = order_key(__ldg(row + j));
        const int gt = (j < n) && key > kstar;
        const int eq = (j < n) && key == kstar;
        int eq_tot;
        const int eq_before = block_exclusive_scan<TK_THREADS>(eq, warp_sums, &eq_tot);
        const int take = gt || (eq && eq_seen + eq_before < need);
        int take_tot;
        const int pos = block_exclusive_scan<TK_THREADS>(take, warp_sums, &take_tot);
        if (take && written + pos < k) out[written + pos] = (int32_t)j;
        written += take_tot;
        eq_seen += eq_tot;
    }
}

lc_status topk_launch_masked(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                             int32_t *topk, const int32_t *row_mask, int32_t *dev_err,
                             cudaStream_t st) {
    if (b.total_q == 0) return LC_OK;
    LC_LAUNCH(k_topk_radix, dim3((unsigned)b.total_q), dim3(TK_THREADS), 0, st, scores, ld,
              to_dev(b), m, k, topk, row_mask, dev_err);
    return check_launch();
}

lc_status topk_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                      int32_t *topk, int32_t *dev_err, cudaStream_t st) {
    return topk_launch_masked(scores, ld, b, m, k, topk, nullptr, dev_err, st);
}

}  // namespace lc
