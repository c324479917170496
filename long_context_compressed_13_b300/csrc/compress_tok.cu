// Token-gated compressor (page "DeepSeek-V4 技术解析…", §1.1, CSA paragraph:
// a token-level compressor merges the KV of every m tokens into one entry; the
// real one is learned, so each token brings its own gate logits):
//   Xc[j,c] = sum_{p<m} softmax_p(Z[j*m+p, c]) * X[j*m+p, c]
// with Z [T, d] fp32, one logit per token and channel (for instance a
// projection of the token's hidden state).  The same call compresses K, V or
// the indexer keys (d = H_I * d_I).
//
// One block per (entry, 32 channels): its eight warps split the m tokens of
// the block (lanes take consecutive channels, so every row read is
// coalesced); each warp keeps an online softmax of its tokens (running max,
// sum of exponentials, weighted sum) and warp 0 merges the eight partial
// states.  HBM-bound: reads m*d*(4 + element size) bytes per entry.
#include "lc_common.cuh"

namespace lc {

template <typename T>
__global__ void __launch_bounds__(256) k_compress_tok(const T *__restrict__ X,
                                                      const float *__restrict__ Z, int64_t Tc,
                                                      int d, int m, T *__restrict__ Xc,
                                                      int64_t rope_pos0) {
    __shared__ float st_m[8][32], st_s[8][32], st_a[8][32];
    const int ngrp = d / 32;
    const int64_t j = blockIdx.x / ngrp;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = (int)(blockIdx.x % ngrp) * 32 + lane;
    const T *x = X + (j * m) * d + c;
    const float *z = Z + (j * m) * d + c;
    float mx = -INFINITY, s = 0.f, acc = 0.f;
#pragma unroll 4
    for (int p = w; p < m; p += 8) {
        const float zp = __ldg(z + (int64_t)p * d);
        const float xp = io<T>::ld(x + (int64_t)p * d);
        if (zp > mx) {  // new running max: rescale what was summed so far
            const float f = mx == -INFINITY ? 0.f : expf(mx - zp);
            s *= f;
            acc *= f;
            mx = zp;
        }
        const float e = expf(zp - mx);
        s += e;
        acc = fmaf(e, xp, acc);
    }
    st_m[w][lane] = mx;
    st_s[w][lane] = s;
    st_a[w][lane] = acc;
    __syncthreads();
    if (w == 0) {
        float M = -INFINITY;
        for (int u = 0; u < 8; ++u) M = fmaxf(M, st_m[u][lane]);
        float S = 0.f, A = 0.f;
        for (int u = 0; u < 8; ++u) {
            if (st_m[u][lane] == -INFINITY) continue;  // a warp with no token
            const float f = expf(st_m[u][lane] - M);
            S = fmaf(st_s[u][lane], f, S);
            A = fmaf(st_a[u][lane], f, A);
        }
        float v = A / S;
        if (rope_pos0 >= 0) v = rope_entry(v, c, d, rope_pos0 + (j + 1) * m - 1);
        Xc[j * d + c] = io<T>::from_f(v);
    }
}

lc_status compress_tok_launch(const void *X, const float *Z, int64_t T_, int d, int m,
                              lc_dtype dt, void *Xc, int64_t rope_pos0, cudaStream_t st) {
    const int64_t Tc = T_ / m;
    if (Tc == 0) return LC_OK;
    const int64_t blocks = Tc * (d / 32);
    if (blocks >= (1ll << 31)) return LC_ERR_UNSUPPORTED;
    if (dt == LC_F32)
        LC_LAUNCH_AS("k_compress_tok", k_compress_tok<float>, dim3((unsigned)blocks), dim3(256), 0,
                     st, (const float *)X, Z, Tc, d, m, (float *)Xc, rope_pos0);
    else
        LC_LAUNCH_AS("k_compress_tok", k_compress_tok<__nv_bfloat16>, dim3((unsigned)blocks),
                     dim3(256), 0, st, (const __nv_bfloat16 *)X, Z, Tc, d, m,
                     (__nv_bfloat16 *)Xc, rope_pos0);
    return check_launch();
}

}  // namespace lc
