// Shared device/host helpers of the lcattn CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lcattn.h"

namespace lc {

// ---------------------------------------------------------------- launches
// Every kernel launch goes through LC_LAUNCH (or LC_LAUNCH_AS, which names a
// kernel reached through a function-pointer variable) so the library can
// report how many kernels it enqueued and which one it enqueued last.
void note_launch(const char *name);
lc_status check_launch();
lc_status check_launch_error(cudaError_t e);  // records e, returns LC_ERR_CUDA

#define LC_LAUNCH_AS(name, kernel, grid, block, smem, stream, ...)                \
    do {                                                                          \
        kernel<<<(grid), (block), (smem), (cudaStream_t)(stream)>>>(__VA_ARGS__); \
        ::lc::note_launch(name);                                                  \
    } while (0)
#define LC_LAUNCH(kernel, grid, block, smem, stream, ...) \
    LC_LAUNCH_AS(#kernel, kernel, grid, block, smem, stream, __VA_ARGS__)

// Test hook (lc_debug_stall): clocks the MMA issuer of the named tensor-core
// kernel waits at its start on a barrier nothing completes (0 = off).
long long debug_stall_clocks(uint32_t kernel_bit);

// ---------------------------------------------------------------- dtypes
template <typename T> struct io;
template <> struct io<float> {
    static __device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) {
        return __float2bfloat16_rn(x);
    }
};

// ---------------------------------------------------------------- batch
// Device view of lc_batch.
struct Batch {
    int32_t B;
    const int64_t *cu_q, *q_pos0, *cu_c, *cu_raw, *raw_pos0;
};

static inline Batch to_dev(const lc_batch &b) {
    return Batch{b.B, b.cu_q, b.q_pos0, b.cu_c, b.cu_raw, b.raw_pos0};
}

// Sequence owning query row r (binary search over cu_q).
__device__ __forceinline__ int seq_of_row(const Batch &bt, int64_t r) {
    int lo = 0, hi = bt.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(bt.cu_q + mid) <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Entries visible from absolute position t under ratio m.
__device__ __forceinline__ int64_t n_vis(int64_t t, int m) { return (t + 1) / m; }

__device__ __forceinline__ void flag(int32_t *dev_err, int bits) {
    if (dev_err) atomicOr(dev_err, bits);
}

// Order-preserving map of an fp32 score to uint32: larger score, larger key.
// -0.0 is folded onto +0.0 first so the two tie.
__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;  // +-0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The sink logit of head h in log2 units, -inf for no sink (sink NULL or
// -inf).  A NaN or +inf sink is not a usable logit: it is flagged as
// LC_DEVERR_SINK and the head is treated as having no sink.
__device__ __forceinline__ float sink_log2(const float *sink, int h, int32_t *dev_err) {
    if (!sink) return -INFINITY;
    const float s = __ldg(sink + h);
    if (!(s < INFINITY)) {  // NaN or +inf
        flag(dev_err, LC_DEVERR_SINK);
        return -INFINITY;
    }
    return s * 1.4426950408889634f;
}

// Folds a per-head attention-sink logit sk2 (log2 units; -inf: none) into a
// softmax row's running max m and sum l (log2 units, l = 0 when the row had
// no key): the sink is one more logit of the denominator with no value.
// Returns the factor that rescales the row's unnormalised output.
__device__ __forceinline__ float fold_sink(float &m, float &l, float sk2) {
    if (!(sk2 > -INFINITY)) return 1.f;
    const float mf = fmaxf(m, sk2);
    const float f = l > 0.f ? exp2f(m - mf) : 0.f;
    l = l * f + exp2f(sk2 - mf);
    m = mf;
    return f;
}

}  // namespace lc
