// Block-level helpers shared by the top-k kernels: prefix sums and radix
// selection of the k-th largest order key.  NT = threads per block.
#pragma once

#include "lc_common.cuh"

namespace lc {

// Exclusive block-wide prefix sum of v; *total receives the block sum.
// warp_sums needs NT/32 ints of shared memory.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    constexpr int NW = NT / 32;
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
        int s = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        if (lane < NW) warp_sums[lane] = s;  // inclusive prefix over warps
    }
    __syncthreads();
    const int before = wid ? warp_sums[wid - 1] : 0;
    *total = warp_sums[NW - 1];
    __syncthreads();
    return before + x - v;
}

struct RadixScratch {
    uint32_t hist[256];
    uint32_t digit;
    int need;
    int cnt;   // keys in the chosen bin
    int fill;  // compaction cursor
};

// The `need`-th largest order key (1-based) among order_key(row[0..n-1]),
// by four 8-bit radix passes (most significant digit first).  Returns the
// key; *need_left receives how many keys equal to it rank within the top
// `need`.  Requires 1 <= need <= n.  All threads of the block call it.
template <int NT>
__device__ uint32_t radix_kth_largest(const float *__restrict__ row, int64_t n, int need,
                                      RadixScratch &rs, int *need_left) {
    uint32_t prefix = 0, mask = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += NT) rs.hist[i] = 0;
        __syncthreads();
        for (int64_t j = threadIdx.x; j < n; j += NT) {
            const uint32_t key = order_key(__ldg(row + j));
            if ((key & mask) == prefix) atomicAdd(&rs.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // suffix sums over the 256 bins, 8 bins per lane, highest first
            const int lane = threadIdx.x;
            uint32_t c[8];
            uint32_t mine = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                c[u] = rs.hist[255 - (lane * 8 + u)];
                mine += c[u];
            }
            uint32_t incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - mine;
            if (excl < (uint32_t)need && incl >= (uint32_t)need) {
                uint32_t cum = excl;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (cum + c[u] >= (uint32_t)need) {
                        rs.digit = 255u - (uint32_t)(lane * 8 + u);
                        rs.need = need - (int)cum;
                        break;
                    }
                    cum += c[u];
                }
            }
        }
        __syncthreads();
        prefix |= rs.digit << shift;
        mask |= 255u << shift;
        need = rs.need;
        __syncthreads();
    }
    *need_left = need;
    return prefix;
}

// As radix_kth_largest, over n order keys held in shared memory.  With
// `spare` (room for n keys, NT a multiple of 32), the keys that still match
// after the first pass are copied there when they are at most half of all,
// and the last three passes scan only them.
template <int NT>
__device__ uint32_t radix_kth_largest_smem(const uint32_t *keys, int n, int need,
                                           RadixScratch &rs, int *need_left,
                                           uint32_t *spare = nullptr) {
    uint32_t prefix = 0, mask = 0;
    const uint32_t *src = keys;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += NT) rs.hist[i] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += NT) {
            const uint32_t key = src[j];
            if ((key & mask) == prefix) atomicAdd(&rs.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            uint32_t c[8];
            uint32_t mine = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                c[u] = rs.hist[255 - (lane * 8 + u)];
                mine += c[u];
            }
            uint32_t incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - mine;
            if (excl < (uint32_t)need && incl >= (uint32_t)need) {
                uint32_t cum = excl;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (cum + c[u] >= (uint32_t)need) {
                        rs.digit = 255u - (uint32_t)(lane * 8 + u);
                        rs.need = need - (int)cum;
                        rs.cnt = (int)c[u];
                        break;
                    }
                    cum += c[u];
                }
            }
            if (lane == 0) rs.fill = 0;
        }
        __syncthreads();
        prefix |= rs.digit << shift;
        mask |= 255u << shift;
        need = rs.need;
        const int nsel = rs.cnt;
        __syncthreads();
        if (spare != nullptr && pass == 0 && 2 * nsel <= n) {
            // the keys of the chosen bin, in any order; one shared atomic per warp
            const int lane = threadIdx.x & 31;
            for (int j0 = threadIdx.x & ~31; j0 < n; j0 += NT) {
                const int j = j0 + lane;
                const uint32_t key = j < n ? src[j] : 0u;
                const bool in = j < n && (key & mask) == prefix;
                const uint32_t bal = __ballot_sync(0xffffffffu, in);
                int base = 0;
                if (lane == 0 && bal) base = atomicAdd(&rs.fill, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (in) spare[base + __popc(bal & ((1u << lane) - 1u))] = key;
            }
            __syncthreads();
            src = spare;
            n = nsel;
        }
    }
    *need_left = need;
    return prefix;
}

}  // namespace lc
