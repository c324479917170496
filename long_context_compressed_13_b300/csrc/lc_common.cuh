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
// Streaming multiprocessors of the current device (looked up once per
// device); 0 when the query fails.
int sm_count();

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

// ---------------------------------------------------------------- decode state
// Arguments of the decode-state append kernel (decode_append).
struct AppendArgs {
    int B, R, d, m, dk;            // dk = HI * dI, 0 without an indexer
    int64_t cap;
    int64_t *n_tok;
    void *Kring, *Vring, *kI_ring, *Kc, *Vc, *kI;
    int64_t *q_pos0, *cu_raw, *raw_pos0;
    const void *K_new, *V_new, *kI_new;
    const float *G_K, *G_V, *G_I;
    int32_t *dev_err;
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

// The tile of a CTA of a grid in which sequence b owns ceil(rows_b / per_cta)
// consecutive CTAs (rows_b = its query rows x rows_per_q), in blockIdx.x
// order, and that sequence's fields.  b == bt.B: a surplus CTA (the grid
// adds one per sequence for the partial tiles).  Sequence 0's fields are
// loaded together with the first bounds, so a one-sequence batch costs one
// round trip of global loads before the CTA can start its copies.
struct SeqTile {
    int b;
    int64_t tile;                 // tile index within the sequence
    int64_t q_beg, nq, q_pos0;    // first global query row, rows, position of row 0
    int64_t c_beg, c_end;         // entries [c_beg, c_end)
    int64_t raw_beg, raw_end, raw_pos0;
};

__device__ __forceinline__ SeqTile locate_tile(const Batch &bt, int64_t cta, int64_t rows_per_q,
                                               int64_t per_cta) {
    SeqTile s;
    const int64_t q1 = __ldg(bt.cu_q + 1);
    s.q_beg = __ldg(bt.cu_q);
    s.q_pos0 = __ldg(bt.q_pos0);
    s.c_beg = __ldg(bt.cu_c);
    s.c_end = __ldg(bt.cu_c + 1);
    s.raw_beg = __ldg(bt.cu_raw);
    s.raw_end = __ldg(bt.cu_raw + 1);
    s.raw_pos0 = __ldg(bt.raw_pos0);
    s.nq = q1 - s.q_beg;
    s.tile = cta;
    s.b = 0;
    int64_t nt = (s.nq * rows_per_q + per_cta - 1) / per_cta;
    while (s.tile >= nt) {
        s.tile -= nt;
        if (++s.b == bt.B) return s;
        s.q_beg = __ldg(bt.cu_q + s.b);
        s.nq = __ldg(bt.cu_q + s.b + 1) - s.q_beg;
        nt = (s.nq * rows_per_q + per_cta - 1) / per_cta;
    }
    if (s.b > 0) {
        s.q_pos0 = __ldg(bt.q_pos0 + s.b);
        s.c_beg = __ldg(bt.cu_c + s.b);
        s.c_end = __ldg(bt.cu_c + s.b + 1);
        s.raw_beg = __ldg(bt.cu_raw + s.b);
        s.raw_end = __ldg(bt.cu_raw + s.b + 1);
        s.raw_pos0 = __ldg(bt.raw_pos0 + s.b);
    }
    return s;
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

// ---------------------------------------------------------------- partial RoPE
// RoPE on the last 64 dimensions of a head vector (page "DeepSeek-V4 技术解析…",
// §1.1, engineering details): 32 interleaved pairs (2i, 2i+1) rotated by the
// angle p * theta_i, theta_i = 10000^(-i/32).  Positions reach 2^20 and more,
// so the angle is formed and reduced modulo 2 pi in fp64 before the fp32
// sine and cosine.
constexpr int ROPE_DIMS = 64;

__device__ __forceinline__ double rope_theta(int i) {
    return exp2(-(double)i * 0.41524101186092029);  // log2(10000) / 32
}

// (cos, sin) of p * theta.
__device__ __forceinline__ float2 rope_cs(int64_t p, double theta) {
    const double a = (double)p * theta;
    const double k = rint(a * 0.15915494309189535);  // 1 / (2 pi)
    double r = fma(-k, 6.283185307179586, a);       // 2 pi, high part
    r = fma(-k, 2.4492935982947064e-16, r);         // 2 pi, low part
    float sn, cs;
    sincosf((float)r, &sn, &cs);
    return make_float2(cs, sn);
}

// Rotates the pair (x, y) by the angle whose (cos, sin) is cs; inverse
// rotates by minus that angle.
__device__ __forceinline__ void rope_pair(float &x, float &y, float2 cs, bool inverse) {
    const float sn = inverse ? -cs.y : cs.y;
    const float nx = x * cs.x - y * sn;
    const float ny = x * sn + y * cs.x;
    x = nx;
    y = ny;
}

// Partial RoPE of one bf16 row of 64 rotary values held in shared memory in
// the 128-byte-swizzled operand layout (16-byte chunk c of row r at chunk
// position c ^ (r & 7)): row r starts at `half`, cs[i] holds the (cos, sin)
// of pair i.  Rounds each rotated value to bf16 once.
__device__ __forceinline__ void rope_smem_row(uint8_t *half, int r, const float2 *cs) {
    uint8_t *row = half + (size_t)r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 *p = reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4));
        uint4 v = *p;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w[u]);
            float x = __low2float(h), y = __high2float(h);
            rope_pair(x, y, cs[4 * c + u], false);
            h = __floats2bfloat162_rn(x, y);
            w[u] = *reinterpret_cast<uint32_t *>(&h);
        }
        *p = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Inverse partial RoPE of 32 consecutive output columns c0 .. c0+31 of one row
// (c0 a multiple of 32 at or past d - 64), cs as above.
__device__ __forceinline__ void rope_out32(float (&o)[32], int c0, int d, const float2 *cs) {
    const int i0 = (c0 - (d - ROPE_DIMS)) >> 1;
#pragma unroll
    for (int u = 0; u < 32; u += 2) rope_pair(o[u], o[u + 1], cs[i0 + u / 2], true);
}

// Partial RoPE of one channel of a compressed entry at position p, inside a
// warp whose lanes hold consecutive channels (even channel in an even lane):
// channels d-64 .. d-1 form the pairs; the partner's value comes by shuffle.
// Every lane of the warp calls it.
__device__ __forceinline__ float rope_entry(float v, int ch, int d, int64_t p) {
    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
    const int rc = ch - (d - ROPE_DIMS);
    if (rc < 0) return v;
    const float2 cs = rope_cs(p, rope_theta(rc >> 1));
    float x = (rc & 1) ? other : v, y = (rc & 1) ? v : other;
    rope_pair(x, y, cs, false);
    return (rc & 1) ? y : x;
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
