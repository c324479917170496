// In-place partial RoPE of rows at consecutive positions (page "DeepSeek-V4
// 技术解析…", §1.1, engineering details: RoPE acts only on the last 64
// dimensions).  Used for the raw window cache, whose tokens are rotated once,
// when they are written, at their own positions.  One thread per (row, head
// vector, pair); HBM-bound (reads and writes 64 of every d values).
#include "lc_common.cuh"

namespace lc {

template <typename T>
__global__ void __launch_bounds__(256) k_rope_rows(T *__restrict__ X, int64_t n, int hv, int d,
                                                   int64_t pos0, int inverse) {
    const int64_t total = n * hv * (ROPE_DIMS / 2);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(e % (ROPE_DIMS / 2));
        const int64_t vec = e / (ROPE_DIMS / 2);  // row * hv + head
        const int64_t row = vec / hv;
        T *x = X + vec * d + (d - ROPE_DIMS) + 2 * i;
        float a = io<T>::to_f(x[0]), b = io<T>::to_f(x[1]);
        rope_pair(a, b, rope_cs(pos0 + row, rope_theta(i)), inverse != 0);
        x[0] = io<T>::from_f(a);
        x[1] = io<T>::from_f(b);
    }
}

lc_status rope_launch(void *X, int64_t n, int hv, int d, int64_t pos0, int inverse, lc_dtype dt,
                      cudaStream_t st) {
    const int64_t total = n * hv * (ROPE_DIMS / 2);
    if (total == 0) return LC_OK;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (dt == LC_F32)
        LC_LAUNCH_AS("k_rope_rows", k_rope_rows<float>, dim3((unsigned)blocks), dim3(256), 0, st,
                     (float *)X, n, hv, d, pos0, inverse);
    else
        LC_LAUNCH_AS("k_rope_rows", k_rope_rows<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256),
                     0, st, (__nv_bfloat16 *)X, n, hv, d, pos0, inverse);
    return check_launch();
}

}  // namespace lc
