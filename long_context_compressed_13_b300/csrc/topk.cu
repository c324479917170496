// Exact causal top-k per row under the total order (score desc, index asc).
// One CTA per row:
//   1. radix select, 4 passes of 8 bits over the order-preserving uint32 keys
//      of the visible scores, finds the k-th largest key K* and how many keys
//      equal to K* must be kept (`need`);
//   2. one ordered compaction pass keeps every key > K* and the first `need`
//      keys == K* in index order; writing positions come from block-wide
//      prefix sums, so the output is already in ascending index order.
// Scores are read 5 times; the row stays hot in L2 for rows up to a few MB.
#include "lc_common.cuh"

namespace lc {

namespace {
constexpr int TK_THREADS = 512;
constexpr int TK_WARPS = TK_THREADS / 32;

// Exclusive block-wide prefix sum of v; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = lane < TK_WARPS ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        if (lane < TK_WARPS) warp_sums[lane] = s;  // inclusive warp prefix
    }
    __syncthreads();
    const int before = wid ? warp_sums[wid - 1] : 0;
    *total = warp_sums[TK_WARPS - 1];
    __syncthreads();
    return before + x - v;
}
}  // namespace

__global__ void __launch_bounds__(TK_THREADS) k_topk_radix(const float *__restrict__ scores,
                                                           int64_t ld, Batch bt, int m, int k,
                                                           int32_t *__restrict__ topk,
                                                           int32_t *dev_err) {
    __shared__ uint32_t hist[256];
    __shared__ int warp_sums[TK_WARPS];
    __shared__ uint32_t s_digit;
    __shared__ int s_need;
    const int64_t r = blockIdx.x;
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

    uint32_t prefix = 0, mask = 0;
    int need = k;  // keys still to take among those matching prefix
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += TK_THREADS) hist[i] = 0;
        __syncthreads();
        for (int64_t j = threadIdx.x; j < n; j += TK_THREADS) {
            const uint32_t key = order_key(__ldg(row + j));
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // find the digit holding the need-th largest key: suffix sums over
            // 256 bins, 8 bins per lane, highest digits first
            const int lane = threadIdx.x;
            uint32_t c[8];
            uint32_t mine = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                c[u] = hist[255 - (lane * 8 + u)];
                mine += c[u];
            }
            uint32_t incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - mine;
            const bool here = excl < (uint32_t)need && incl >= (uint32_t)need;
            if (here) {
                uint32_t cum = excl;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (cum + c[u] >= (uint32_t)need) {
                        s_digit = 255u - (uint32_t)(lane * 8 + u);
                        s_need = need - (int)cum;
                        break;
                    }
                    cum += c[u];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        need = s_need;
        __syncthreads();
    }

    // ordered compaction: keys > prefix, then the first `need` keys == prefix
    int written = 0, eq_seen = 0;
#pragma unroll 1
    for (int64_t j0 = 0; j0 < n && written < k; j0 += TK_THREADS) {
        const int64_t j = j0 + threadIdx.x;
        uint32_t key = 0;
        if (j < n) key = order_key(__ldg(row + j));
        const int gt = (j < n) && key > prefix;
        const int eq = (j < n) && key == prefix;
        int eq_tot;
        const int eq_before = block_exclusive_scan(eq, warp_sums, &eq_tot);
        const int take = gt || (eq && eq_seen + eq_before < need);
        int take_tot;
        const int pos = block_exclusive_scan(take, warp_sums, &take_tot);
        if (take && written + pos < k) out[written + pos] = (int32_t)j;
        written += take_tot;
        eq_seen += eq_tot;
    }
}

lc_status topk_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                      int32_t *topk, int32_t *dev_err, cudaStream_t st) {
    if (b.total_q == 0) return LC_OK;
    LC_LAUNCH(k_topk_radix, dim3((unsigned)b.total_q), dim3(TK_THREADS), 0, st, scores, ld,
              to_dev(b), m, k, topk, dev_err);
    return check_launch();
}

}  // namespace lc
