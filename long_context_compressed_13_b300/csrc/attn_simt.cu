// MQA attention over an explicit key list, SIMT fp32 path (every dtype; the
// only path for fp32 inputs and for shapes the tensor-core kernels skip).
//
// One CTA = one query row x HG heads.  The row's key list is
//   CSA: slots 0..k-1 = Kc/Vc rows of topk[r, :] (-1 = masked), then the window
//   HCA: slots 0..n_vis-1 = Kc/Vc rows 0..n_vis-1, then the window
// and is walked in tiles of 32 keys: gather K/V rows into shared memory,
// scores for all HG heads, an online-softmax update per head, then O += P.V.
// Scores carry scale*log2(e) so exp2f serves the softmax; lse is returned in
// natural-log units.
#include "lc_common.cuh"

namespace lc {

namespace {
constexpr int KT = 32;        // keys per tile
constexpr int AT = 256;       // threads per CTA
constexpr float LOG2E = 1.4426950408889634f;
}

struct AttnArgs {
    const void *Q, *Kc, *Vc, *Kraw, *Vraw;
    const int32_t *topk;
    int k;         // slots of topk per row (CSA); 0 for HCA
    int H, m, W;
    float scale;
    const float *sink;  // [H] per-head sink logits or NULL
    void *O;
    float *lse;
    int32_t *dev_err;
    int rope;           // partial RoPE: q rotated at t, O rotated back at t
};

template <typename T, int D, int HG, bool SPARSE>
__global__ void __launch_bounds__(AT) k_attn_simt(AttnArgs a, Batch bt) {
    extern __shared__ float sm[];
    float *sQ = sm;                         // [HG][D]   pre-scaled q
    float *sK = sQ + HG * D;                // [KT][D+1]
    float *sV = sK + KT * (D + 1);          // [KT][D]
    float *sP = sV + KT * D;                // [HG][KT+1]
    float *sM = sP + HG * (KT + 1);         // [HG] running max (log2 units)
    float *sL = sM + HG;                    // [HG] running sum
    float *sA = sL + HG;                    // [HG] rescale factor of this tile
    int64_t *sRow = reinterpret_cast<int64_t *>(sA + HG);  // [KT] source row, -1 masked
    int *sSrc = reinterpret_cast<int *>(sRow + KT);         // [KT] 0 compressed, 1 raw
    float2 *sCS = reinterpret_cast<float2 *>(sSrc + KT);     // [32] RoPE (cos, sin) at t

    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const int h0 = blockIdx.y * HG;
    const int b = seq_of_row(bt, r);
    const int64_t t = bt.q_pos0[b] + (r - bt.cu_q[b]);
    const int64_t c_beg = bt.cu_c[b], Tc = bt.cu_c[b + 1] - c_beg;
    const int64_t raw_beg = bt.cu_raw[b], Nraw = bt.cu_raw[b + 1] - raw_beg;
    const int64_t raw_pos0 = bt.raw_pos0[b];
    int64_t nv = n_vis(t, a.m);
    if (nv > Tc) {
        if (tid == 0 && blockIdx.y == 0 && !SPARSE) flag(a.dev_err, LC_DEVERR_BATCH);
        nv = Tc;
    }
    const int64_t nsel = SPARSE ? a.k : nv;
    const int64_t wlo = (a.W > 0) ? max((int64_t)0, t - a.W + 1) : t + 1;
    const int64_t nwin = t + 1 - wlo;
    const int64_t nkeys = nsel + nwin;

    const T *Q = reinterpret_cast<const T *>(a.Q);
    const float qs = a.scale * LOG2E;
    for (int i = tid; i < HG * D; i += AT)
        sQ[i] = io<T>::ld(Q + (r * a.H + h0) * D + i) * qs;
    if (tid < HG) {
        sM[tid] = -INFINITY;
        sL[tid] = 0.f;
    }
    if (a.rope) {
        // partial RoPE of the row's query heads at position t (fp32, in place)
        if (tid < 32) sCS[tid] = rope_cs(t, rope_theta(tid));
        __syncthreads();
        for (int u = tid; u < HG * 32; u += AT) {
            float *q = sQ + (u >> 5) * D + (D - ROPE_DIMS) + 2 * (u & 31);
            rope_pair(q[0], q[1], sCS[u & 31], false);
        }
    }

    constexpr int NO = HG * D / AT;  // outputs per thread in P.V
    constexpr int HSTEP = AT / D;    // head stride between a thread's outputs
    float acc[NO];
#pragma unroll
    for (int i = 0; i < NO; ++i) acc[i] = 0.f;
    const int oc = tid % D, oh = tid / D;

    const T *Kc = reinterpret_cast<const T *>(a.Kc), *Vc = reinterpret_cast<const T *>(a.Vc);
    const T *Kr = reinterpret_cast<const T *>(a.Kraw), *Vr = reinterpret_cast<const T *>(a.Vraw);
    const bool report = blockIdx.y == 0;

    for (int64_t k0 = 0; k0 < nkeys; k0 += KT) {
        __syncthreads();
        if (tid < KT) {
            const int64_t i = k0 + tid;
            int64_t row = -1;
            int src = 0;
            if (i < nsel) {
                int64_t j = SPARSE ? (int64_t)a.topk[r * a.k + i] : i;
                if (j >= 0) {
                    if (j < nv) {
                        row = c_beg + j;
                    } else if (report) {
                        flag(a.dev_err, LC_DEVERR_INDEX);
                    }
                }
            } else if (i < nkeys) {
                const int64_t rr = wlo + (i - nsel) - raw_pos0;
                if (rr >= 0 && rr < Nraw) {
                    row = raw_beg + rr;
                    src = 1;
                } else if (report) {
                    flag(a.dev_err, LC_DEVERR_WINDOW);
                }
            }
            sRow[tid] = row;
            sSrc[tid] = src;
        }
        __syncthreads();
        for (int e = tid; e < KT * D; e += AT) {
            const int kk = e / D, c = e - kk * D;
            const int64_t row = sRow[kk];
            float kv = 0.f, vv = 0.f;
            if (row >= 0) {
                const T *Ks = sSrc[kk] ? Kr : Kc;
                const T *Vs = sSrc[kk] ? Vr : Vc;
                kv = io<T>::ld(Ks + row * D + c);
                vv = io<T>::ld(Vs + row * D + c);
            }
            sK[kk * (D + 1) + c] = kv;
            sV[kk * D + c] = vv;
        }
        __syncthreads();
        // scores: thread -> key kk = tid % 32, heads tid/32 + 8*i
        {
            const int kk = tid & 31, hb = tid >> 5;
            constexpr int NH = HG / 8;
            float s[NH];
#pragma unroll
            for (int i = 0; i < NH; ++i) s[i] = 0.f;
            for (int c = 0; c < D; ++c) {
                const float kv = sK[kk * (D + 1) + c];
#pragma unroll
                for (int i = 0; i < NH; ++i) s[i] = fmaf(sQ[(hb + 8 * i) * D + c], kv, s[i]);
            }
            const bool valid = sRow[kk] >= 0;
#pragma unroll
            for (int i = 0; i < NH; ++i) sP[(hb + 8 * i) * (KT + 1) + kk] = valid ? s[i] : -INFINITY;
        }
        __syncthreads();
        // online softmax, one thread per head
        if (tid < HG) {
            float mx = sM[tid];
            float tmax = -INFINITY;
            for (int kk = 0; kk < KT; ++kk) tmax = fmaxf(tmax, sP[tid * (KT + 1) + kk]);
            const float mnew = fmaxf(mx, tmax);
            float alpha = 1.f, sum = 0.f;
            if (mnew != -INFINITY) {
                alpha = exp2f(mx - mnew);  // mx = -inf -> 0
                for (int kk = 0; kk < KT; ++kk) {
                    const float p = exp2f(sP[tid * (KT + 1) + kk] - mnew);
                    sP[tid * (KT + 1) + kk] = p;
                    sum += p;
                }
            } else {
                for (int kk = 0; kk < KT; ++kk) sP[tid * (KT + 1) + kk] = 0.f;
            }
            sM[tid] = mnew;
            sL[tid] = sL[tid] * alpha + sum;
            sA[tid] = alpha;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NO; ++i) {
            const int h = oh + HSTEP * i;
            float o = acc[i] * sA[h];
#pragma unroll 8
            for (int kk = 0; kk < KT; ++kk) o = fmaf(sP[h * (KT + 1) + kk], sV[kk * D + oc], o);
            acc[i] = o;
        }
    }
    __syncthreads();
    if (tid < HG) {
        // the head's sink logit joins the denominator; sA takes the output factor
        float mm = sM[tid], ll = sL[tid];
        sA[tid] = fold_sink(mm, ll, sink_log2(a.sink, h0 + tid, a.dev_err));
        sM[tid] = mm;
        sL[tid] = ll;
    }
    __syncthreads();
    T *O = reinterpret_cast<T *>(a.O);
#pragma unroll
    for (int i = 0; i < NO; ++i) {
        const int h = oh + HSTEP * i;
        const float l = sL[h];
        float o = l > 0.f ? acc[i] * sA[h] / l : 0.f;
        if (a.rope) {
            // rotate the output back at t: channel pairs sit in adjacent lanes
            const float other = __shfl_xor_sync(0xffffffffu, o, 1);
            const int rc = oc - (D - ROPE_DIMS);
            if (rc >= 0) {
                float x = (rc & 1) ? other : o, y = (rc & 1) ? o : other;
                rope_pair(x, y, sCS[rc >> 1], true);
                o = (rc & 1) ? y : x;
            }
        }
        O[(r * a.H + h0 + h) * D + oc] = io<T>::from_f(o);
    }
    if (a.lse && tid < HG) {
        const float l = sL[tid];
        a.lse[r * a.H + h0 + tid] = l > 0.f ? (sM[tid] + log2f(l)) / LOG2E : -INFINITY;
    }
}

template <typename T, int D, int HG, bool SPARSE>
static lc_status launch_hg(const AttnArgs &a, const lc_batch &b, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)HG * D + KT * (D + 1) + KT * D + HG * (KT + 1) +
                                         3 * HG) +
                        KT * (sizeof(int64_t) + sizeof(int)) + 32 * sizeof(float2);
    auto kfn = k_attn_simt<T, D, HG, SPARSE>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return LC_ERR_CUDA;
    dim3 grid((unsigned)b.total_q, (unsigned)(a.H / HG));
    LC_LAUNCH_AS("k_attn_simt", kfn, grid, dim3(AT), smem, st, a, to_dev(b));
    return check_launch();
}

template <typename T, int D, bool SPARSE>
static lc_status launch_d(const AttnArgs &a, const lc_batch &b, cudaStream_t st) {
    if (a.H % 64 == 0) return launch_hg<T, D, 64, SPARSE>(a, b, st);
    if (a.H % 32 == 0) return launch_hg<T, D, 32, SPARSE>(a, b, st);
    if (a.H % 16 == 0) return launch_hg<T, D, 16, SPARSE>(a, b, st);
    return launch_hg<T, D, 8, SPARSE>(a, b, st);
}

template <bool SPARSE>
static lc_status launch_attn(const AttnArgs &a, const lc_batch &b, int d, lc_dtype dt,
                             cudaStream_t st) {
    if (b.total_q == 0) return LC_OK;
    if (dt == LC_F32)
        return d == 64 ? launch_d<float, 64, SPARSE>(a, b, st) : launch_d<float, 128, SPARSE>(a, b, st);
    return d == 64 ? launch_d<__nv_bfloat16, 64, SPARSE>(a, b, st)
                   : launch_d<__nv_bfloat16, 128, SPARSE>(a, b, st);
}

lc_status attn_simt_launch(bool sparse, const void *Q, const void *Kc, const void *Vc,
                           const int32_t *topk, int k, const void *Kraw, const void *Vraw,
                           const lc_batch &b, int H, int d, int m, int W, float scale,
                           const float *sink, int rope, lc_dtype dt, void *O, float *lse,
                           int32_t *dev_err, cudaStream_t st) {
    AttnArgs a{Q, Kc, Vc, Kraw, Vraw, topk, sparse ? k : 0, H, m, W, scale, sink, O, lse, dev_err,
               rope};
    return sparse ? launch_attn<true>(a, b, d, dt, st) : launch_attn<false>(a, b, d, dt, st);
}

}  // namespace lc
