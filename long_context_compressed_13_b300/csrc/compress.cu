// Softmax-gated pooling compressor shared by CSA (m = 4) and HCA (m' = 128).
// Kc[j,c] = sum_p softmax_p(G[:,c])[p] * K[j*m+p, c]; one output element per
// thread, gate weights computed once per block into shared memory.  HBM-bound:
// reads m*d elements and writes d elements per entry.
#include "lc_common.cuh"

namespace lc {

// One launch for both tensors: blockIdx.y = 0 compresses K with G_K, 1 compresses V
// with G_V.  The block first stages its gate logits G [m][d] in shared memory
// (coalesced), then P = blockDim.x / d threads per channel reduce the max and
// the sum over the m positions (lanes of one warp, combined by shuffles) and
// write the normalised weights in place.
template <typename T>
__global__ void __launch_bounds__(256) k_compress(const T *__restrict__ K, const T *__restrict__ V,
                                                  const float *__restrict__ GK,
                                                  const float *__restrict__ GV, int64_t Tc,
                                                  int d, int m, T *__restrict__ Kc,
                                                  T *__restrict__ Vc, int64_t rope_pos0) {
    extern __shared__ float wgt[];  // [m][d]
    const bool is_v = blockIdx.y != 0;
    const T *X = is_v ? V : K;
    const float *G = is_v ? GV : GK;
    T *Xc = is_v ? Vc : Kc;
    const int md = m * d;
    for (int i = threadIdx.x; i < md; i += blockDim.x) wgt[i] = __ldg(G + i);
    __syncthreads();
    const int P = blockDim.x / d;  // threads per channel: 2 (d = 128) or 4 (d = 64)
    const int c = threadIdx.x / P, part = threadIdx.x % P;
    float mx = -INFINITY;
    for (int p = part; p < m; p += P) mx = fmaxf(mx, wgt[p * d + c]);
    for (int o = 1; o < P; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float s = 0.f;
    for (int p = part; p < m; p += P) s += expf(wgt[p * d + c] - mx);
    for (int o = 1; o < P; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.f / s;
    __syncthreads();  // every max and sum is read before any weight is overwritten
    for (int p = part; p < m; p += P) wgt[p * d + c] = expf(wgt[p * d + c] - mx) * inv;
    __syncthreads();
    const int64_t total = Tc * d;
    // total is a multiple of 32 (d is), so every warp is either wholly inside
    // or wholly past the end: the partner channel of a RoPE pair is one lane away
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = e / d;
        const int ch = (int)(e - j * d);
        const T *src = X + j * m * d + ch;
        float acc = 0.f;
        for (int p = 0; p < m; ++p) acc = fmaf(wgt[p * d + ch], io<T>::ld(src + (int64_t)p * d), acc);
        if (rope_pos0 >= 0) acc = rope_entry(acc, ch, d, rope_pos0 + (j + 1) * m - 1);
        Xc[e] = io<T>::from_f(acc);
    }
}

// Long groups (m >= 32, the HCA ratio): one block per (entry, 32 channels);
// its eight warps split the m positions, lanes take consecutive channels
// (coalesced rows).  The gate softmax of the block's channels is reduced over
// the warps in shared memory, each warp sums its positions, and warp 0 adds
// the eight partial sums.  blockIdx.y = 0 compresses K, 1 compresses V.
template <typename T>
__global__ void __launch_bounds__(256) k_compress_long(const T *__restrict__ K,
                                                       const T *__restrict__ V,
                                                       const float *__restrict__ GK,
                                                       const float *__restrict__ GV, int64_t Tc,
                                                       int d, int m, T *__restrict__ Kc,
                                                       T *__restrict__ Vc, int64_t rope_pos0) {
    __shared__ float red[8][32];
    __shared__ float stat[2][32];
    const bool is_v = blockIdx.y != 0;
    const T *X = is_v ? V : K;
    const float *G = is_v ? GV : GK;
    T *Xc = is_v ? Vc : Kc;
    const int ngrp = d / 32;
    const int64_t j = blockIdx.x / ngrp;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = (int)(blockIdx.x % ngrp) * 32 + lane;
    const int per = (m + 7) / 8;
    const int p0 = min(m, w * per), p1 = min(m, p0 + per);
    float mx = -INFINITY;
    for (int p = p0; p < p1; ++p) mx = fmaxf(mx, __ldg(G + (int64_t)p * d + c));
    red[w][lane] = mx;
    __syncthreads();
    if (w == 0) {
        float v = red[0][lane];
        for (int u = 1; u < 8; ++u) v = fmaxf(v, red[u][lane]);
        stat[0][lane] = v;
    }
    __syncthreads();
    const float M = stat[0][lane];
    float s = 0.f;
    for (int p = p0; p < p1; ++p) s += expf(__ldg(G + (int64_t)p * d + c) - M);
    red[w][lane] = s;
    __syncthreads();
    if (w == 0) {
        float v = 0.f;
        for (int u = 0; u < 8; ++u) v += red[u][lane];
        stat[1][lane] = v;
    }
    __syncthreads();
    const float inv = 1.f / stat[1][lane];
    const T *src = X + (j * m) * d + c;
    float acc = 0.f;
#pragma unroll 8
    for (int p = p0; p < p1; ++p)
        acc = fmaf(expf(__ldg(G + (int64_t)p * d + c) - M) * inv, io<T>::ld(src + (int64_t)p * d),
                   acc);
    red[w][lane] = acc;
    __syncthreads();
    if (w == 0) {
        float v = 0.f;
        for (int u = 0; u < 8; ++u) v += red[u][lane];
        if (rope_pos0 >= 0) v = rope_entry(v, c, d, rope_pos0 + (j + 1) * m - 1);
        Xc[j * d + c] = io<T>::from_f(v);
    }
}

template <typename T>
static lc_status launch(const void *K, const void *V, const float *GK, const float *GV,
                        int64_t T_, int d, int m, void *Kc, void *Vc, int64_t rope_pos0,
                        cudaStream_t st) {
    const int64_t Tc = T_ / m;
    if (Tc == 0) return LC_OK;
    if (m >= 32 && d % 32 == 0 && Tc * (d / 32) < (1ll << 31)) {
        auto kl = k_compress_long<T>;
        LC_LAUNCH_AS("k_compress_long", kl, dim3((unsigned)(Tc * (d / 32)), 2), dim3(256), 0, st, (const T *)K,
                  (const T *)V, GK, GV, Tc, d, m, (T *)Kc, (T *)Vc, rope_pos0);
        return check_launch();
    }
    const size_t smem = sizeof(float) * (size_t)m * d;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(k_compress<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return LC_ERR_CUDA;
    }
    int64_t blocks = (Tc * d + 255) / 256;
    if (blocks > 148 * 4) blocks = 148 * 4;
    auto kfn = k_compress<T>;
    LC_LAUNCH_AS("k_compress", kfn, dim3((unsigned)blocks, 2), dim3(256), smem, st, (const T *)K, (const T *)V,
              GK, GV, Tc, d, m, (T *)Kc, (T *)Vc, rope_pos0);
    return check_launch();
}

lc_status compress_launch(const void *K, const void *V, const float *GK, const float *GV,
                          int64_t T_, int d, int m, lc_dtype dt, void *Kc, void *Vc,
                          int64_t rope_pos0, cudaStream_t st) {
    if (dt == LC_F32) return launch<float>(K, V, GK, GV, T_, d, m, Kc, Vc, rope_pos0, st);
    return launch<__nv_bfloat16>(K, V, GK, GV, T_, d, m, Kc, Vc, rope_pos0, st);
}

}  // namespace lc
