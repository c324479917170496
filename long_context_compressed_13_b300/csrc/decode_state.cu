// Incremental decode state of one compressed-attention layer (page "DeepSeek
// V4 详解：1M 上下文背后，真正发生了什么", §"第二刀：KV cache 被当成系统在管": a
// classical KV cache holds the compressed entries, a per-request state cache
// of fixed size holds the sliding-window KV and the tail of tokens that do not
// yet fill a compression block; compressed blocks cover lcm(m, m') raw tokens
// so CSA and HCA share the layout).
//
// Layout per request b (every region of fixed capacity, so the other kernels
// read it with the ordinary batch descriptor and no page table):
//   classical cache  Kc, Vc [cap, d] (and the CSA indexer keys kI [cap, HI*dI])
//                    at rows b*cap ..: entry j of the request is row b*cap + j;
//   state cache      a mirrored ring of the last R raw tokens: position p sits
//                    at rows b*2R + p%R and b*2R + p%R + R, so any R consecutive
//                    positions are R consecutive rows; it serves the window
//                    (R >= W) and the open block's tokens (R >= m);
//                    token-level indexer keys of the open CSA block in
//                    kI_ring [m, HI*dI] at slot p % m.
// k_decode_append appends one token per request: both ring slots, the indexer
// slot, and, when the token closes a block, the block's entry (softmax-gated
// pooling with position gates, the compressor of csa_compress); then it
// advances the request's batch descriptor (query position t, window origin)
// so that the index and attention calls of the same step read the new token.
#include "lc_common.cuh"

namespace lc {


// Softmax over the m gate logits of channel c (column c of G [m, width]),
// pooled with values fetched by val(p).
template <typename F>
__device__ __forceinline__ float gated_pool(const float *G, int width, int c, int m, F val) {
    float mx = -INFINITY;
    for (int p = 0; p < m; ++p) mx = fmaxf(mx, __ldg(G + (int64_t)p * width + c));
    float s = 0.f, acc = 0.f;
    for (int p = 0; p < m; ++p) {
        const float e = expf(__ldg(G + (int64_t)p * width + c) - mx);
        s += e;
        acc = fmaf(e, val(p), acc);
    }
    return acc / s;
}

template <typename T>
__global__ void __launch_bounds__(256) k_decode_append(AppendArgs a) {
    const int b = blockIdx.x, tid = threadIdx.x;
    const int64_t t = a.n_tok[b];  // position of the new token
    const int64_t cap_pos = a.cap * a.m;
    const bool room = t < cap_pos;  // the classical cache has room for the token's block
    T *Kr = static_cast<T *>(a.Kring), *Vr = static_cast<T *>(a.Vring);
    const T *Kn = static_cast<const T *>(a.K_new), *Vn = static_cast<const T *>(a.V_new);
    const int64_t ring0 = (int64_t)b * 2 * a.R;
    const int64_t slot = ring0 + t % a.R;
    for (int c = tid; c < a.d; c += blockDim.x) {
        const T k = Kn[(int64_t)b * a.d + c], v = Vn[(int64_t)b * a.d + c];
        Kr[slot * a.d + c] = k;
        Kr[(slot + a.R) * a.d + c] = k;
        Vr[slot * a.d + c] = v;
        Vr[(slot + a.R) * a.d + c] = v;
    }
    T *kIr = static_cast<T *>(a.kI_ring);
    const T *kIn = static_cast<const T *>(a.kI_new);
    if (a.dk > 0)
        for (int c = tid; c < a.dk; c += blockDim.x)
            kIr[((int64_t)b * a.m + t % a.m) * a.dk + c] = kIn[(int64_t)b * a.dk + c];
    __syncthreads();  // the block's tokens are in place (this CTA wrote the newest)
    if ((t + 1) % a.m == 0) {
        const int64_t j = (t + 1) / a.m - 1;
        if (!room) {
            if (tid == 0) flag(a.dev_err, LC_DEVERR_BATCH);
        } else {
            const int64_t p0 = t + 1 - a.m;  // first position of the block
            T *Kc = static_cast<T *>(a.Kc), *Vc = static_cast<T *>(a.Vc);
            const int64_t row = (int64_t)b * a.cap + j;
            for (int c = tid; c < 2 * a.d; c += blockDim.x) {
                const bool isv = c >= a.d;
                const int cc = isv ? c - a.d : c;
                const T *ring = isv ? Vr : Kr;
                const float v = gated_pool(isv ? a.G_V : a.G_K, a.d, cc, a.m, [&](int p) {
                    return io<T>::to_f(ring[(ring0 + (p0 + p) % a.R) * a.d + cc]);
                });
                (isv ? Vc : Kc)[row * a.d + cc] = io<T>::from_f(v);
            }
            if (a.dk > 0) {
                T *kI = static_cast<T *>(a.kI);
                for (int c = tid; c < a.dk; c += blockDim.x) {
                    const float v = gated_pool(a.G_I, a.dk, c, a.m, [&](int p) {
                        return io<T>::to_f(kIr[((int64_t)b * a.m + p) * a.dk + c]);
                    });
                    kI[row * a.dk + c] = io<T>::from_f(v);
                }
            }
        }
    }
    if (tid == 0) {
        a.n_tok[b] = t + 1;
        a.q_pos0[b] = t;
        const int64_t lo = t + 1 > a.R ? t + 1 - a.R : 0;  // oldest position the ring holds
        a.raw_pos0[b] = lo;
        a.cu_raw[b] = ring0 + lo % a.R;
        if (b == a.B - 1) a.cu_raw[a.B] = (int64_t)a.B * 2 * a.R;
    }
}

lc_status decode_append_launch(const AppendArgs &a, lc_dtype dt, cudaStream_t st) {
    if (a.B == 0) return LC_OK;
    if (dt == LC_F32)
        LC_LAUNCH_AS("k_decode_append", k_decode_append<float>, dim3(a.B), dim3(256), 0, st, a);
    else
        LC_LAUNCH_AS("k_decode_append", k_decode_append<__nv_bfloat16>, dim3(a.B), dim3(256), 0,
                     st, a);
    return check_launch();
}

}  // namespace lc
