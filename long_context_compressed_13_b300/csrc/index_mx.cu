// Low-precision Lightning Indexer (page "DeepSeek V4 详解：1M 上下文背后，真正发生了
// 什么", §"mHC、Muon、FP4": FP4 runs in the CSA indexer's QK path and the
// quantized selector keeps almost all of the exact selection; page
// "DeepSeek-V4 技术解析…", §1.1: the indexer computes in FP4).
//
// Storage follows the OCP Microscaling (MX) formats v1.0: blocks of 32
// consecutive values share a power-of-two scale X = 2^(floor(log2 amax) -
// emax) kept as an E8M0 byte; each value is the element nearest to v / X
// (ties to even), clamped to the largest element.  MXFP8 has E4M3 elements
// (one byte each), MXFP4 E2M1 elements (two per byte, the even-indexed value
// in the low nibble).
//
// k_mx_quantize   one warp per block of 32 values: warp max of |v|, the
//                 shared exponent from the exponent of amax, the elements by
//                 the round-to-nearest-even conversions of cuda_fp8.h /
//                 cuda_fp4.h (satfinite), one coalesced store of the codes.
// k_index_stream_mx  the decode-shaped indexer of indexer.cu on MX keys: one
//                 CTA per (query row, range of entries); a lane owns one
//                 (entry, head) pair of a warp step (32 / H_I entries per
//                 step, read as one contiguous span): it loads the head's 64
//                 key codes (64 B MXFP8, 32 B MXFP4) and its two block scales,
//                 converts code pairs to f16x2 (exact: every element is a
//                 half) and accumulates each 32-value block's dot product:
//                 MXFP4 with packed half FMAs over groups of 8 pairs (exact:
//                 the products are multiples of 1/4 below 37, a group's sums
//                 stay below 512) added in fp32; MXFP8 with mixed-precision
//                 FMAs (f16 multiplicands, exact products, fp32 addend); then
//                 each block is scaled by 2^(q exponent + k exponent).  Shuffles over the H_I lanes of an entry add the
//                 ReLU-weighted heads.  HBM-bound: per entry H_I * (d_I * bits
//                 / 8 + d_I / 32) bytes.
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "lc_common.cuh"

namespace lc {

namespace {

constexpr int MX_FP8 = 8, MX_FP4 = 4;

// Shared exponent of a block with largest magnitude amax: floor(log2 amax) -
// emax, clamped to the E8M0 range; -127 for an all-zero block.
__device__ __forceinline__ int mx_shared_exp(float amax, int emax) {
    if (!(amax > 0.f)) return -127;
    const int e = ilogbf(amax) - emax;  // exact: the exponent of amax
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// v * 2^-e, exact whenever the result is a normal fp32 (always, for the
// values that do not round to zero in the element format).
__device__ __forceinline__ float scale_down(float v, int e) { return scalbnf(v, -e); }

template <typename T, int FMT>
__global__ void __launch_bounds__(256) k_mx_quantize(const T *__restrict__ X, int64_t nblk,
                                                     uint8_t *__restrict__ codes,
                                                     uint8_t *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (blk >= nblk) return;  // whole warps leave together
    const float v = io<T>::to_f(X[blk * 32 + lane]);
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const int e = mx_shared_exp(a, FMT == MX_FP8 ? 8 : 2);
    const float x = scale_down(v, e);
    if (FMT == MX_FP8) {
        codes[blk * 32 + lane] = (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    } else {
        const uint32_t c = (uint32_t)__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest) & 15u;
        const uint32_t hi = __shfl_down_sync(0xffffffffu, c, 1);
        if ((lane & 1) == 0) codes[blk * 16 + (lane >> 1)] = (uint8_t)(c | (hi << 4));
    }
    if (lane == 0) scales[blk] = (uint8_t)(e + 127);
}

// Element pairs -> f16x2 (every E4M3 and E2M1 element is exactly a half).
// E4M3: two bytes of a 32-bit word (half 0 or 1); E2M1: one byte (two nibbles,
// the even-indexed value in the low nibble becomes the low half).
// One conversion instruction per pair (cvt .f16x2 from .e4m3x2 / .e2m1x2):
// the lower element goes to the lower half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t word, int half) {
    const uint16_t s = (uint16_t)(half ? (word >> 16) : (word & 0xffffu));
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(s));
    return h;
}
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t word, int byte) {
    const uint32_t b = (word >> (8 * byte)) & 0xffu;
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h)
        : "r"(b));
    return h;
}

// acc += a.lo * b.lo + a.hi * b.hi for f16x2 a, b: products of two halves are
// exact in the fused multiply-add, which rounds once to fp32 (mixed-precision
// FMA with f16 multiplicands and an f32 addend).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// One head's 64 element codes: MXFP8 64 bytes, MXFP4 32 bytes.
template <int FMT>
struct HeadCodes {
    static constexpr int NV4 = FMT * 64 / 8 / 16;  // 16-byte loads
    uint4 v[NV4];
    __device__ __forceinline__ void load(const uint8_t *p) {
#pragma unroll
        for (int i = 0; i < NV4; ++i) v[i] = __ldg(reinterpret_cast<const uint4 *>(p) + i);
    }
    __device__ __forceinline__ uint32_t word(int i) const {  // 32-bit word i of the codes
        const uint4 &x = v[i >> 2];
        return (i & 3) == 0 ? x.x : (i & 3) == 1 ? x.y : (i & 3) == 2 ? x.z : x.w;
    }
    // values 2i, 2i+1 as f16x2 (i < 32)
    __device__ __forceinline__ uint32_t pair(int i) const {
        if (FMT == MX_FP8) return e4m3x2_to_f16x2(word(i >> 1), i & 1);
        return e2m1x2_to_f16x2(word(i >> 2), i & 3);
    }
};

template <int FMT, int HI>
__global__ void __launch_bounds__(256) k_index_stream_mx(const uint8_t *__restrict__ qc,
                                                         const uint8_t *__restrict__ qs,
                                                         const float *__restrict__ w,
                                                         const uint8_t *__restrict__ kc,
                                                         const uint8_t *__restrict__ ks,
                                                         Batch bt, int m,
                                                         float *__restrict__ scores, int64_t ld,
                                                         int64_t chunk, int64_t r0,
                                                         int32_t *dev_err) {
    constexpr int CB = 64 * FMT / 8;      // code bytes per head
    constexpr int EPS = 32 / HI;          // entries per warp step
    constexpr int U = FMT == MX_FP4 ? 4 : 2;  // warp steps in flight (16-byte loads: 8)
    const unsigned FULL = 0xffffffffu;
    const int64_t r = r0 + blockIdx.y;  // written to scores row blockIdx.y
    const int b = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[b] + (r - bt.cu_q[b]);
    const int64_t c_beg = bt.cu_c[b], Tc = bt.cu_c[b + 1] - c_beg;
    int64_t nv = n_vis(t, m);
    if (nv > Tc) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(dev_err, LC_DEVERR_BATCH);
        nv = Tc;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int es = lane / HI, h = lane % HI;  // entry of the step, head
    // this lane's head of q: 64 element values as 32 f16x2, two block exponents
    uint32_t qh[32];
    {
        HeadCodes<FMT> c;
        c.load(qc + (r * HI + h) * CB);
#pragma unroll
        for (int i = 0; i < 32; ++i) qh[i] = c.pair(i);
    }
    const int qe0 = (int)__ldg(qs + (r * HI + h) * 2) - 127;
    const int qe1 = (int)__ldg(qs + (r * HI + h) * 2 + 1) - 127;
    const float wh = __ldg(w + r * HI + h);
    const int64_t e_lo = (int64_t)blockIdx.x * chunk;
    const int64_t e_hi = min(e_lo + chunk, ld);
    const int64_t v_hi = min(e_hi, nv);
    float *out = scores + (int64_t)blockIdx.y * ld;
    const uint8_t *kbase = kc + (c_beg * HI + h) * CB;
    const uint16_t *sbase = reinterpret_cast<const uint16_t *>(ks) + c_beg * HI + h;
    for (int64_t base = e_lo + (int64_t)warp * EPS * U; base < v_hi; base += 8 * EPS * U) {
        HeadCodes<FMT> kv[U];
        uint32_t sk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = base + u * EPS + es;
            if (e < v_hi) {
                kv[u].load(kbase + e * HI * CB);
                sk[u] = __ldg(sbase + e * HI);
            } else {
#pragma unroll
                for (int i = 0; i < HeadCodes<FMT>::NV4; ++i) kv[u].v[i] = make_uint4(0, 0, 0, 0);
                sk[u] = 0x7f7fu;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float a0 = 0.f, a1 = 0.f;  // the two 32-value blocks
            if (FMT == MX_FP4) {
                // E2M1 x E2M1 products are multiples of 1/4 of magnitude <= 36,
                // so a packed half FMA chain of 8 products per half stays
                // below 512 and is exact; each group of 16 products then
                // joins the block's fp32 sum
#pragma unroll
                for (int grp = 0; grp < 4; ++grp) {
                    __half2 acc = __float2half2_rn(0.f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t kp = kv[u].pair(8 * grp + i), qp = qh[8 * grp + i];
                        acc = __hfma2(*reinterpret_cast<const __half2 *>(&qp),
                                      *reinterpret_cast<const __half2 *>(&kp), acc);
                    }
                    const float2 f = __half22float2(acc);
                    if (grp < 2)
                        a0 += f.x + f.y;
                    else
                        a1 += f.x + f.y;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) a0 = fma2_f16_f32(qh[i], kv[u].pair(i), a0);
#pragma unroll
                for (int i = 16; i < 32; ++i) a1 = fma2_f16_f32(qh[i], kv[u].pair(i), a1);
            }
            const int ke0 = (int)(sk[u] & 0xffu) - 127, ke1 = (int)(sk[u] >> 8) - 127;
            const float d = scalbnf(a0, qe0 + ke0) + scalbnf(a1, qe1 + ke1);
            float p = wh * fmaxf(d, 0.f);
#pragma unroll
            for (int o = 1; o < HI; o <<= 1) p += __shfl_xor_sync(FULL, p, o);
            const int64_t e = base + u * EPS + es;
            if (h == 0 && e < v_hi) out[e] = p;
        }
    }
    for (int64_t e = max(e_lo, nv) + threadIdx.x; e < e_hi; e += 256) out[e] = -INFINITY;
}

}  // namespace

template <typename T, int FMT>
static void launch_quantize(const void *X, int64_t nblk, uint8_t *codes, uint8_t *scales,
                            cudaStream_t st) {
    const int64_t blocks = (nblk + 7) / 8;  // 8 warps per CTA, one block of 32 each
    auto kfn = k_mx_quantize<T, FMT>;
    LC_LAUNCH_AS("k_mx_quantize", kfn, dim3((unsigned)blocks), dim3(256), 0, st,
                 static_cast<const T *>(X), nblk, codes, scales);
}

lc_status mx_quantize_launch(const void *X, int64_t n, int fmt, lc_dtype dt, uint8_t *codes,
                             uint8_t *scales, cudaStream_t st) {
    const int64_t nblk = n / 32;
    if (nblk == 0) return LC_OK;
    if ((nblk + 7) / 8 >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    if (dt == LC_F32)
        fmt == MX_FP8 ? launch_quantize<float, MX_FP8>(X, nblk, codes, scales, st)
                      : launch_quantize<float, MX_FP4>(X, nblk, codes, scales, st);
    else
        fmt == MX_FP8 ? launch_quantize<__nv_bfloat16, MX_FP8>(X, nblk, codes, scales, st)
                      : launch_quantize<__nv_bfloat16, MX_FP4>(X, nblk, codes, scales, st);
    return check_launch();
}

template <int FMT, int HI>
static void launch_index_mx(dim3 grid, const uint8_t *qc, const uint8_t *qs, const float *w,
                            const uint8_t *kc, const uint8_t *ks, const lc_batch &b, int m,
                            float *scores, int64_t ld, int64_t chunk, int64_t r0,
                            int32_t *dev_err, cudaStream_t st) {
    auto kfn = k_index_stream_mx<FMT, HI>;
    LC_LAUNCH_AS("k_index_stream_mx", kfn, grid, dim3(256), 0, st, qc, qs, w, kc, ks, to_dev(b),
                 m, scores, ld, chunk, r0, dev_err);
}

// Scores of query rows r0 .. r0 + nrows - 1 (into scores rows 0 .. nrows - 1)
// of the MX indexer (d_I = 64, H_I in {4, 8}).
lc_status index_mx_launch(int fmt, const uint8_t *qc, const uint8_t *qs, const float *w,
                          const uint8_t *kc, const uint8_t *ks, const lc_batch &b, int HI, int m,
                          float *scores, int64_t ld, int64_t r0, int64_t nrows, int32_t *dev_err,
                          cudaStream_t st) {
    if (nrows <= 0) return LC_OK;
    if (nrows > 65535 || (HI != 4 && HI != 8)) return LC_ERR_UNSUPPORTED;
    // about eight CTAs per SM over the rows, at least 1024 entries each
    const int64_t want_x = (148 * 8 + nrows - 1) / nrows;
    int64_t chunk = (ld + want_x - 1) / want_x;
    if (chunk < 1024) chunk = 1024;
    chunk = (chunk + 255) / 256 * 256;
    const int64_t gx = (ld + chunk - 1) / chunk;
    if (gx > 65535) return LC_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)nrows);
    if (fmt == MX_FP8)
        HI == 8 ? launch_index_mx<MX_FP8, 8>(grid, qc, qs, w, kc, ks, b, m, scores, ld, chunk, r0,
                                            dev_err, st)
                : launch_index_mx<MX_FP8, 4>(grid, qc, qs, w, kc, ks, b, m, scores, ld, chunk, r0,
                                            dev_err, st);
    else
        HI == 8 ? launch_index_mx<MX_FP4, 8>(grid, qc, qs, w, kc, ks, b, m, scores, ld, chunk, r0,
                                            dev_err, st)
                : launch_index_mx<MX_FP4, 4>(grid, qc, qs, w, kc, ks, b, m, scores, ld, chunk, r0,
                                            dev_err, st);
    return check_launch();
}

}  // namespace lc
