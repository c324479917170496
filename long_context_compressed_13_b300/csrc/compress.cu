// Softmax-gated pooling compressor shared by CSA (m = 4) and HCA (m' = 128).
// Kc[j,c] = sum_p softmax_p(G[:,c])[p] * K[j*m+p, c]; one output element per
// thread, gate weights computed once per block into shared memory.  HBM-bound:
// reads m*d elements and writes d elements per entry.
#include "lc_common.cuh"

namespace lc {

template <typename T>
__global__ void __launch_bounds__(256) k_compress(const T *__restrict__ X,
                                                  const float *__restrict__ G, int64_t Tc,
                                                  int d, int m, T *__restrict__ Xc) {
    extern __shared__ float wgt[];  // [m][d]
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float mx = -INFINITY;
        for (int p = 0; p < m; ++p) mx = fmaxf(mx, G[(int64_t)p * d + c]);
        float s = 0.f;
        for (int p = 0; p < m; ++p) s += expf(G[(int64_t)p * d + c] - mx);
        float inv = 1.f / s;
        for (int p = 0; p < m; ++p) wgt[p * d + c] = expf(G[(int64_t)p * d + c] - mx) * inv;
    }
    __syncthreads();
    const int64_t total = Tc * d;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = e / d;
        const int c = (int)(e - j * d);
        const T *src = X + j * m * d + c;
        float acc = 0.f;
        for (int p = 0; p < m; ++p) acc = fmaf(wgt[p * d + c], io<T>::ld(src + (int64_t)p * d), acc);
        Xc[e] = io<T>::from_f(acc);
    }
}

template <typename T>
static lc_status launch(const void *X, const float *G, int64_t T_, int d, int m, void *Xc,
                        cudaStream_t st) {
    const int64_t Tc = T_ / m;
    if (Tc == 0) return LC_OK;
    const size_t smem = sizeof(float) * (size_t)m * d;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(k_compress<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return LC_ERR_CUDA;
    }
    int64_t blocks = (Tc * d + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    auto kfn = k_compress<T>;
    LC_LAUNCH(kfn, dim3((unsigned)blocks), dim3(256), smem, st, (const T *)X, G, Tc, d, m,
              (T *)Xc);
    return check_launch();
}

lc_status compress_launch(const void *X, const float *G, int64_t T_, int d, int m,
                          lc_dtype dt, void *Xc, cudaStream_t st) {
    if (dt == LC_F32) return launch<float>(X, G, T_, d, m, Xc, st);
    return launch<__nv_bfloat16>(X, G, T_, d, m, Xc, st);
}

}  // namespace lc
