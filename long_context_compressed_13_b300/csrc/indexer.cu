// Lightning Indexer, SIMT fp32 paths.
//   I[r,j] = sum_h w[r,h] * max(0, qI[r,h,:] . kI[cu_c[b]+j,h,:])   j < n_vis(t_r)
//   I[r,j] = -inf                                                   n_vis(t_r) <= j < ld
// Two launch shapes:
//   k_index_tiled  many query rows per sequence (prefill): 64x64 (row, entry)
//                  tiles, q and k head slices staged in shared memory, one
//                  head at a time.
//   k_index_scan   few rows per sequence (decode): one row per grid.y, each
//                  thread streams one (entry, head) slice of kI with 16-byte
//                  loads (fp32 keys, d_I = 32 or H_I < 4);
//   k_index_stream the same rows for bf16 keys with d_I = 64, H_I in {4, 8}:
//                  coalesced 512-byte warp loads, HBM-bound.
#include <type_traits>

#include "lc_common.cuh"

namespace lc {

namespace {
constexpr int TQ = 64;  // rows per tile
constexpr int TE = 64;  // entries per tile
}

template <typename T>
__global__ void __launch_bounds__(256) k_index_tiled(const T *__restrict__ qI,
                                                     const float *__restrict__ w,
                                                     const T *__restrict__ kI, Batch bt, int HI,
                                                     int dI, int m, float *__restrict__ scores,
                                                     int64_t ld, int32_t *dev_err) {
    extern __shared__ float sm[];
    const int b = blockIdx.y;
    const int64_t q_beg = bt.cu_q[b], nq = bt.cu_q[b + 1] - q_beg;
    const int64_t row0 = (int64_t)blockIdx.x * TQ;
    const int64_t e0 = (int64_t)blockIdx.z * TE;
    if (row0 >= nq || e0 >= ld) return;
    const int64_t c_beg = bt.cu_c[b], Tc = bt.cu_c[b + 1] - c_beg;
    const int64_t t0 = bt.q_pos0[b] + row0;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int64_t last_row = min(row0 + TQ, nq) - 1;
    int64_t nv_max = n_vis(bt.q_pos0[b] + last_row, m);
    if (nv_max > Tc) {
        flag(dev_err, LC_DEVERR_BATCH);
        nv_max = Tc;
    }

    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;

    if (e0 < nv_max) {
        const int stride = dI + 1;
        float *sq = sm;                 // [TQ][dI+1]
        float *sk = sm + TQ * stride;   // [TE][dI+1]
        float *sw = sk + TE * stride;   // [TQ]
        for (int h = 0; h < HI; ++h) {
            for (int i = tid; i < TQ * dI; i += 256) {
                const int rr = i / dI, e = i - rr * dI;
                const int64_t row = row0 + rr;
                sq[rr * stride + e] =
                    row < nq ? io<T>::ld(qI + ((q_beg + row) * HI + h) * dI + e) : 0.f;
                const int64_t j = e0 + rr;
                sk[rr * stride + e] = j < nv_max ? io<T>::ld(kI + ((c_beg + j) * HI + h) * dI + e) : 0.f;
            }
            if (tid < TQ) sw[tid] = row0 + tid < nq ? w[(q_beg + row0 + tid) * HI + h] : 0.f;
            __syncthreads();
            float dot[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) dot[a][c] = 0.f;
            for (int e = 0; e < dI; ++e) {
                float qa[4], kb[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) qa[a] = sq[(ty * 4 + a) * stride + e];
#pragma unroll
                for (int c = 0; c < 4; ++c) kb[c] = sk[(tx + 16 * c) * stride + e];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) dot[a][c] = fmaf(qa[a], kb[c], dot[a][c]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float wa = sw[ty * 4 + a];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(wa, fmaxf(dot[a][c], 0.f), acc[a][c]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t row = row0 + ty * 4 + a;
        if (row >= nq) continue;
        int64_t nv = n_vis(t0 + ty * 4 + a, m);
        if (nv > Tc) nv = Tc;
        float *out = scores + (q_beg + row) * ld;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t j = e0 + tx + 16 * c;
            if (j < ld) out[j] = j < nv ? acc[a][c] : -INFINITY;
        }
    }
}

// Query rows r0 + blockIdx.y, r0 + blockIdx.y + gridDim.y, ... (nrows of
// them; row r0 + i is written to scores row i); threads cover (entry, head)
// pairs, HI lanes per entry reduce with shuffles.  DI * sizeof(T) bytes are
// read per thread with 16-byte vector loads.
template <typename T, int DI, int HI>
__global__ void __launch_bounds__(256) k_index_scan(const T *__restrict__ qI,
                                                    const float *__restrict__ w,
                                                    const T *__restrict__ kI, Batch bt, int m,
                                                    float *__restrict__ scores, int64_t ld,
                                                    int64_t r0, int64_t nrows,
                                                    int32_t *dev_err) {
    __shared__ float sq[HI][DI];
    __shared__ float sw[HI];
    constexpr int EPB = 256 / HI;                 // entries per block pass
    constexpr int NV = DI * (int)sizeof(T) / 16;  // 16-byte vectors per slice
    constexpr int EPV = 16 / (int)sizeof(T);      // elements per vector
    const int h = threadIdx.x % HI;
    const int el = threadIdx.x / HI;
    for (int64_t ri = blockIdx.y; ri < nrows; ri += gridDim.y) {
        const int64_t r = r0 + ri;
        const int b = seq_of_row(bt, r);
        const int64_t t = bt.q_pos0[b] + (r - bt.cu_q[b]);
        const int64_t c_beg = bt.cu_c[b], Tc = bt.cu_c[b + 1] - c_beg;
        int64_t nv = n_vis(t, m);
        if (nv > Tc) {
            if (blockIdx.x == 0 && threadIdx.x == 0) flag(dev_err, LC_DEVERR_BATCH);
            nv = Tc;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < HI * DI; i += blockDim.x)
            sq[i / DI][i % DI] = io<T>::ld(qI + r * HI * DI + i);
        if (threadIdx.x < HI) sw[threadIdx.x] = w[r * HI + threadIdx.x];
        __syncthreads();
        float *out = scores + ri * ld;
        for (int64_t j0 = (int64_t)blockIdx.x * EPB; j0 < ld; j0 += (int64_t)gridDim.x * EPB) {
            const int64_t j = j0 + el;
            float part = 0.f;
            if (j < nv) {
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(kI + ((c_beg + j) * HI + h) * DI);
                uint4 v[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i) v[i] = __ldg(src + i);
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const T *e = reinterpret_cast<const T *>(&v[i]);
#pragma unroll
                    for (int u = 0; u < EPV; ++u)
                        dot = fmaf(sq[h][i * EPV + u], io<T>::to_f(e[u]), dot);
                }
                part = sw[h] * fmaxf(dot, 0.f);
            }
#pragma unroll
            for (int off = HI / 2; off > 0; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            if (h == 0 && j < ld) out[j] = j < nv ? part : -INFINITY;
        }
    }
}

// Decode-shaped streaming indexer for bf16 keys with d_I = 64 and H_I in {4, 8}:
// one CTA per (query row, range of entries).  An entry's keys are H_I x 128 B;
// a warp reads them as H_I/4 instructions of 512 contiguous bytes (4 heads),
// lane = (head g within the four, 16-byte slice sl of the head).  Each lane
// keeps the matching 8 q_I values per head in registers, so the dot product
// is 8 FMAs per lane and load, reduced over the 8 lanes of a head and then
// over the heads with shuffles.  Lane i keeps the score of the i-th entry of
// each 32-entry block, which the warp stores with one coalesced write.
// Columns [n_vis, ld) get -inf.
template <int HI>
__global__ void __launch_bounds__(256) k_index_stream(const __nv_bfloat16 *__restrict__ qI,
                                                      const float *__restrict__ w,
                                                      const __nv_bfloat16 *__restrict__ kI,
                                                      Batch bt, int m, float *__restrict__ scores,
                                                      int64_t ld, int64_t chunk, int64_t r0,
                                                      int32_t *dev_err) {
    constexpr int L = HI / 4;  // 512-byte loads per entry
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
    const int g = lane >> 3, sl = lane & 7;
    float q[L][8], wl[L];
#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int h = 4 * l + g;
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(qI + (r * HI + h) * 64 + sl * 8));
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[l][2 * i] = __uint_as_float(u[i] << 16);
            q[l][2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
        wl[l] = __ldg(w + r * HI + h);
    }
    const int64_t e_lo = (int64_t)blockIdx.x * chunk;
    const int64_t e_hi = min(e_lo + chunk, ld);
    const int64_t v_hi = min(e_hi, nv);
    float *out = scores + (int64_t)blockIdx.y * ld;
    const __nv_bfloat16 *krow = kI + (c_beg * HI + g) * 64 + sl * 8;
    for (int64_t base = e_lo + 32 * warp; base < v_hi; base += 32 * 8) {
        const int n_here = (int)min((int64_t)32, v_hi - base);
        float mine = 0.f;
#pragma unroll 1
        for (int e4 = 0; e4 < 32; e4 += 4) {
            uint4 v[4][L];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int l = 0; l < L; ++l)
                    v[u][l] = e4 + u < n_here
                                  ? __ldg(reinterpret_cast<const uint4 *>(
                                        krow + ((base + e4 + u) * HI + 4 * l) * 64))
                                  : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float p = 0.f;
#pragma unroll
                for (int l = 0; l < L; ++l) {
                    const uint32_t x[4] = {v[u][l].x, v[u][l].y, v[u][l].z, v[u][l].w};
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        d = fmaf(q[l][2 * i], __uint_as_float(x[i] << 16), d);
                        d = fmaf(q[l][2 * i + 1], __uint_as_float(x[i] & 0xffff0000u), d);
                    }
                    d += __shfl_xor_sync(0xffffffffu, d, 1);
                    d += __shfl_xor_sync(0xffffffffu, d, 2);
                    d += __shfl_xor_sync(0xffffffffu, d, 4);
                    p = fmaf(wl[l], fmaxf(d, 0.f), p);
                }
                p += __shfl_xor_sync(0xffffffffu, p, 8);
                p += __shfl_xor_sync(0xffffffffu, p, 16);
                if (lane == e4 + u) mine = p;
            }
            if (e4 + 4 >= n_here) break;
        }
        if (lane < n_here) out[base + lane] = mine;
    }
    for (int64_t e = max(e_lo, nv) + threadIdx.x; e < e_hi; e += 256) out[e] = -INFINITY;
}

static bool stream_ok(const void *qI, const void *kI, int HI, int dI, lc_dtype dt) {
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return dt == LC_BF16 && dI == 64 && (HI == 4 || HI == 8) && al16(qI) && al16(kI);
}

static lc_status launch_stream(const void *qI, const float *w, const void *kI, const lc_batch &b,
                               int HI, int m, float *scores, int64_t ld, int64_t r0,
                               int64_t nrows, int32_t *dev_err, cudaStream_t st) {
    if (nrows > 65535) return LC_ERR_UNSUPPORTED;
    // about eight CTAs per SM over the rows, at least 1024 entries each
    const int64_t want_x = (148 * 8 + nrows - 1) / nrows;
    int64_t chunk = (ld + want_x - 1) / want_x;
    if (chunk < 1024) chunk = 1024;
    chunk = (chunk + 255) / 256 * 256;
    const int64_t gx = (ld + chunk - 1) / chunk;
    if (gx > 65535) return LC_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)nrows);
    if (HI == 8)
        LC_LAUNCH_AS("k_index_stream", k_index_stream<8>, grid, dim3(256), 0, st,
                     (const __nv_bfloat16 *)qI, w, (const __nv_bfloat16 *)kI, to_dev(b), m,
                     scores, ld, chunk, r0, dev_err);
    else
        LC_LAUNCH_AS("k_index_stream", k_index_stream<4>, grid, dim3(256), 0, st,
                     (const __nv_bfloat16 *)qI, w, (const __nv_bfloat16 *)kI, to_dev(b), m,
                     scores, ld, chunk, r0, dev_err);
    return check_launch();
}

template <typename T, int DI, int HI>
static void launch_scan(const void *qI, const float *w, const void *kI, const lc_batch &b, int m,
                        float *scores, int64_t ld, int64_t r0, int64_t nrows, int32_t *dev_err,
                        cudaStream_t st) {
    constexpr int EPB = 256 / HI;
    const int64_t rows = nrows < 65535 ? nrows : 65535;
    int64_t gx = (ld + EPB - 1) / EPB;
    int64_t want = (148 * 8 + rows - 1) / rows;  // ~8 blocks per SM overall
    if (gx > want) gx = want;
    if (gx < 1) gx = 1;
    auto kfn = k_index_scan<T, DI, HI>;
    LC_LAUNCH_AS("k_index_scan", kfn, dim3((unsigned)gx, (unsigned)rows), dim3(256), 0, st,
                 (const T *)qI, w, (const T *)kI, to_dev(b), m, scores, ld, r0, nrows, dev_err);
}

template <typename T, int DI>
static lc_status scan_hi(const void *qI, const float *w, const void *kI, const lc_batch &b, int HI,
                         int m, float *scores, int64_t ld, int64_t r0, int64_t nrows,
                         int32_t *dev_err, cudaStream_t st) {
    switch (HI) {
        case 1: launch_scan<T, DI, 1>(qI, w, kI, b, m, scores, ld, r0, nrows, dev_err, st); break;
        case 2: launch_scan<T, DI, 2>(qI, w, kI, b, m, scores, ld, r0, nrows, dev_err, st); break;
        case 4: launch_scan<T, DI, 4>(qI, w, kI, b, m, scores, ld, r0, nrows, dev_err, st); break;
        case 8: launch_scan<T, DI, 8>(qI, w, kI, b, m, scores, ld, r0, nrows, dev_err, st); break;
        default: return LC_ERR_UNSUPPORTED;
    }
    return check_launch();
}

// Per-row scores of query rows r0 .. r0 + nrows - 1 into scores rows 0 ..
// nrows - 1 (streaming kernels: any batch, rows in any sequence).
lc_status index_rows_launch(const void *qI, const float *w, const void *kI, const lc_batch &b,
                            int HI, int dI, int m, lc_dtype dt, float *scores, int64_t ld,
                            int64_t r0, int64_t nrows, int32_t *dev_err, cudaStream_t st) {
    if (nrows <= 0) return LC_OK;
    if (stream_ok(qI, kI, HI, dI, dt)) {
        const lc_status s = launch_stream(qI, w, kI, b, HI, m, scores, ld, r0, nrows, dev_err, st);
        if (s != LC_ERR_UNSUPPORTED) return s;
    }
    if (dt == LC_F32)
        return dI == 32
                   ? scan_hi<float, 32>(qI, w, kI, b, HI, m, scores, ld, r0, nrows, dev_err, st)
                   : scan_hi<float, 64>(qI, w, kI, b, HI, m, scores, ld, r0, nrows, dev_err, st);
    return dI == 32 ? scan_hi<__nv_bfloat16, 32>(qI, w, kI, b, HI, m, scores, ld, r0, nrows,
                                                 dev_err, st)
                    : scan_hi<__nv_bfloat16, 64>(qI, w, kI, b, HI, m, scores, ld, r0, nrows,
                                                 dev_err, st);
}

template <typename T>
static lc_status launch_index(const void *qI, const float *w, const void *kI, const lc_batch &b,
                              int HI, int dI, int m, float *scores, int64_t ld, int32_t *dev_err,
                              cudaStream_t st) {
    if (b.max_q < 16) {
        if (std::is_same<T, __nv_bfloat16>::value && stream_ok(qI, kI, HI, dI, LC_BF16)) {
            const lc_status s =
                launch_stream(qI, w, kI, b, HI, m, scores, ld, 0, b.total_q, dev_err, st);
            if (s != LC_ERR_UNSUPPORTED) return s;
        }
        if (dI == 32)
            return scan_hi<T, 32>(qI, w, kI, b, HI, m, scores, ld, 0, b.total_q, dev_err, st);
        return scan_hi<T, 64>(qI, w, kI, b, HI, m, scores, ld, 0, b.total_q, dev_err, st);
    }
    const size_t smem = sizeof(float) * ((size_t)(TQ + TE) * (dI + 1) + TQ);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_index_tiled<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return LC_ERR_CUDA;
    dim3 grid((unsigned)((b.max_q + TQ - 1) / TQ), (unsigned)b.B, (unsigned)((ld + TE - 1) / TE));
    if ((ld + TE - 1) / TE > 65535) return LC_ERR_UNSUPPORTED;
    auto kfn = k_index_tiled<T>;
    LC_LAUNCH_AS("k_index_tiled", kfn, grid, dim3(256), smem, st, (const T *)qI, w, (const T *)kI, to_dev(b), HI, dI,
              m, scores, ld, dev_err);
    return check_launch();
}

lc_status index_launch(const void *qI, const float *w, const void *kI, const lc_batch &b, int HI,
                       int dI, int m, lc_dtype dt, float *scores, int64_t ld, int32_t *dev_err,
                       cudaStream_t st) {
    if (dt == LC_F32) return launch_index<float>(qI, w, kI, b, HI, dI, m, scores, ld, dev_err, st);
    return launch_index<__nv_bfloat16>(qI, w, kI, b, HI, dI, m, scores, ld, dev_err, st);
}

}  // namespace lc
