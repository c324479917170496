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
    uint32_t all_and, all_or;  // common bits of the keys (shared-memory selection)
};

// The `need`-th largest order key (1-based) among order_key(row[0..n-1]),
// by four 8-bit radix passes (most significant digit first).  Returns the
// key; *need_left receives how many keys equal to it rank within the top
// `need`.  Requires 1 <= need <= n.  All threads of the block call it.
// RO = false reads the row with plain loads (for a row this kernel itself
// wrote: the read-only cache path does not see such writes).
template <bool RO>
__device__ __forceinline__ float ld_score(const float *p) {
    if (RO) return __ldg(p);
    return *p;
}

template <int NT, bool RO = true>
__device__ uint32_t radix_kth_largest(const float *__restrict__ row, int64_t n, int need,
                                      RadixScratch &rs, int *need_left) {
    uint32_t prefix = 0, mask = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += NT) rs.hist[i] = 0;
        __syncthreads();
        for (int64_t j = threadIdx.x; j < n; j += NT) {
            const uint32_t key = order_key(ld_score<RO>(row + j));
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

// As radix_kth_largest, over n order keys held in shared memory.  The bits
// that every key shares are found first (an AND and an OR over the keys) and
// need no pass; the 8-bit digits start at the highest bit where keys differ
// (keys of a selection share their top bits: byte-aligned digits would send
// nearly every key of the first pass to one or two histogram bins).  With
// `spare` (room for n keys, NT a multiple of 32), the keys that still match
// after the first pass are copied there when they are at most half of all,
// and the later passes scan only them.  Once at most 64 keys are left, all
// matching the digits found so far, one warp ranks them directly.
template <int NT>
__device__ uint32_t radix_kth_largest_smem(const uint32_t *keys, int n, int need,
                                           RadixScratch &rs, int *need_left,
                                           uint32_t *spare = nullptr) {
    if (threadIdx.x == 0) {
        rs.all_and = 0xffffffffu;
        rs.all_or = 0u;
    }
    __syncthreads();
    {
        uint32_t a = 0xffffffffu, o = 0u;
        for (int j = threadIdx.x; j < n; j += NT) {
            a &= keys[j];
            o |= keys[j];
        }
        a = __reduce_and_sync(0xffffffffu, a);
        o = __reduce_or_sync(0xffffffffu, o);
        if ((threadIdx.x & 31) == 0) {
            atomicAnd(&rs.all_and, a);
            atomicOr(&rs.all_or, o);
        }
    }
    __syncthreads();
    const uint32_t diff = rs.all_and ^ rs.all_or;
    int hi = 32 - __clz(diff);  // bits [0, hi) still open (0: all keys are equal)
    uint32_t mask = hi == 32 ? 0u : ~((1u << hi) - 1u);
    uint32_t prefix = rs.all_and & mask;
    const uint32_t *src = keys;
    bool first = true, all_match = true;  // all_match: every key of src matches prefix
#pragma unroll 1
    while (hi > 0) {
        if (all_match && n <= 64) {
            // few keys left, all matching the prefix: one warp ranks them by
            // counting (the need-th largest x has fewer than need keys above
            // it and at least need at or above it)
            if (threadIdx.x < 32) {
                const int lane = threadIdx.x;
                const uint32_t a = lane < n ? src[lane] : 0u;
                const uint32_t b = lane + 32 < n ? src[lane + 32] : 0u;
                int ga = 0, ea = 0, gb = 0, eb = 0;
                for (int j = 0; j < n; ++j) {
                    const uint32_t x = src[j];
                    ga += x > a;
                    ea += x == a;
                    gb += x > b;
                    eb += x == b;
                }
                const bool ha = lane < n && ga < need && ga + ea >= need;
                const bool hb = lane + 32 < n && gb < need && gb + eb >= need;
                const unsigned wa = __ballot_sync(0xffffffffu, ha);
                const unsigned wb = __ballot_sync(0xffffffffu, hb);
                const int who = wa ? __ffs(wa) - 1 : __ffs(wb) - 1;  // one of them is set
                if (lane == who) {
                    rs.digit = wa ? a : b;
                    rs.need = need - (wa ? ga : gb);
                }
            }
            __syncthreads();
            prefix = rs.digit;
            need = rs.need;
            __syncthreads();
            break;
        }
        const int lo = hi > 8 ? hi - 8 : 0;  // the digit: bits [lo, hi)
        const uint32_t dmask = (1u << (hi - lo)) - 1u;
        for (int i = threadIdx.x; i < 256; i += NT) rs.hist[i] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += NT) {
            const uint32_t key = src[j];
            if ((key & mask) == prefix) atomicAdd(&rs.hist[(key >> lo) & dmask], 1u);
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
        prefix |= rs.digit << lo;
        mask |= dmask << lo;
        need = rs.need;
        const int nsel = rs.cnt;
        __syncthreads();
        if (spare != nullptr && first && 2 * nsel <= n) {
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
            all_match = true;
        } else {
            all_match = false;
        }
        first = false;
        hi = lo;
    }
    *need_left = need;
    return prefix;
}

// Exact top-k of one row of n visible scores (n > k) under the total order
// (larger score first, then lower index), written as ascending indices to
// out[0..k): radix selection of the k-th largest key K* and of how many
// keys equal to K* rank within the top k, then one ordered compaction pass
// (keys > K*, and the first `need` keys == K*) whose write positions come
// from block-wide prefix sums.  All NT threads of the block call it.
template <int NT, bool RO = true>
__device__ void radix_topk_row(const float *__restrict__ row, int64_t n, int k, int32_t *out,
                               RadixScratch &rs, int *warp_sums) {
    int need;
    const uint32_t kstar = radix_kth_largest<NT, RO>(row, n, k, rs, &need);
    int written = 0, eq_seen = 0;
#pragma unroll 1
    for (int64_t j0 = 0; j0 < n && written < k; j0 += NT) {
        const int64_t j = j0 + threadIdx.x;
        uint32_t key = 0;
        if (j < n) key = order_key(ld_score<RO>(row + j));
        const int gt = (j < n) && key > kstar;
        const int eq = (j < n) && key == kstar;
        int eq_tot;
        const int eq_before = block_exclusive_scan<NT>(eq, warp_sums, &eq_tot);
        const int take = gt || (eq && eq_seen + eq_before < need);
        int take_tot;
        const int pos = block_exclusive_scan<NT>(take, warp_sums, &take_tot);
        if (take && written + pos < k) out[written + pos] = (int32_t)j;
        written += take_tot;
        eq_seen += eq_tot;
    }
}

// One radix digit of a warp-level selection: among the keys that match
// `prefix` under `mask`, the digit (key >> shift) & 255 of the need-th
// largest, from a histogram in the warp's own 256 shared-memory words `h`.
// visit(f) must call f(key, valid) on all 32 lanes together (warp-uniform
// trip counts), once with valid = true for every key of the set (each lane
// its share); lanes without a key pass valid = false.  On return `need` is
// the rank of the wanted key within the chosen digit's bin.  Requires
// 1 <= need <= (keys matching prefix); all 32 lanes call it.
template <typename Visit>
__device__ __forceinline__ uint32_t warp_radix_digit(uint32_t *h, Visit visit, uint32_t prefix,
                                                     uint32_t mask, int shift, int &need) {
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < 256; i += 32) h[i] = 0u;
    __syncwarp();
    visit([&](uint32_t key, bool valid) {
        if (valid && (key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1u);
    });
    __syncwarp();
    // suffix sums over the 256 bins, 8 bins per lane, highest first
    uint32_t c[8], mine = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        c[u] = h[255 - (lane * 8 + u)];
        mine += c[u];
    }
    uint32_t incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += y;
    }
    const uint32_t excl = incl - mine;
    const bool has = excl < (uint32_t)need && incl >= (uint32_t)need;
    uint32_t digit = 0;
    int rank = need;
    if (has) {
        uint32_t cum = excl;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (cum + c[u] >= (uint32_t)need) {
                digit = 255u - (uint32_t)(lane * 8 + u);
                rank = need - (int)cum;
                break;
            }
            cum += c[u];
        }
    }
    const unsigned who = __ballot_sync(FULL, has);
    const int src = who ? __ffs(who) - 1 : 0;
    digit = __shfl_sync(FULL, digit, src);
    need = __shfl_sync(FULL, rank, src);
    __syncwarp();  // h may be reused by the next digit
    return digit;
}

}  // namespace lc
