/*
 * Plain CPU oracle for the CSA + HCA attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark call this file.  It shares no code, header or
 * constant with the CUDA library, and the product path never calls it.
 *
 * Every function is the literal definition of one step of the method, written
 * out in fp64 with no tiling, fusion or reordering.  Sources (page title,
 * section):
 *   - "DeepSeek-V4 技术解析：架构革新与 Coding Agent 后训练优化", §1.1
 *     (混合注意力：CSA 与 HCA 的协同): a token-level compressor folds the KV
 *     of every m tokens into one entry, a Lightning Indexer scores the query
 *     against compressed entries, a top-k selector keeps the best entries,
 *     MQA core attention runs over them; HCA folds m' >> m tokens and attends
 *     densely over all entries; an extra sliding-window branch adds raw
 *     local KV.
 *   - "DeepSeek-V4 技术报告解读：百万Token上下文是怎么做到的", §三大架构改动
 *     1-2: sequence shrinks to 1/m; top-k over compressed entries plus a few
 *     sliding-window entries; HCA attends densely over all compressed entries.
 * Where the pages leave the form open (the compressor's pooling, the
 * indexer's score, tie order, window extent) the readings adopted are:
 *   compressor  Xc[j,c] = sum_p softmax_p(G[:,c])[p] * X[j*m+p, c]
 *   visibility  entry j is visible from position t iff (j+1)*m - 1 <= t
 *   indexer     I[t,j]  = sum_h w[t,h] * max(0, q_I[t,h,:] . k_I[j,h,:])
 *   top-k       larger score first, equal scores -> lower index first;
 *               output ascending entry index, -1 padded
 *   window      raw positions max(0, t-W+1) .. t (W tokens, t included)
 *   attention   one softmax over (selected entries, then window tokens)
 *   sink        the same page, §1.1 (engineering details): a learnable
 *               per-head attention-sink logit lets a head push its total
 *               attention toward 0.  Read as one extra logit s_h that joins
 *               the softmax's denominator and carries no value:
 *               O = sum_i e^{z_i} V_i / (e^{s_h} + sum_i e^{z_i}),
 *               lse = log(e^{s_h} + sum_i e^{z_i}); no sink = s_h = -inf
 *   empty set   O = 0, lse = s_h (-inf without a sink)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Compressor (CSA with m = 4, HCA with m' = 128).
 * X [T, d], G [m, d] gate logits -> Xc [floor(T/m), d].
 * Only full blocks of m tokens become entries; a tail shorter than m does not. */
void oracle_compress(const double *X, const double *G, int64_t T, int32_t d,
                     int32_t m, double *Xc)
{
    int64_t Tc = T / m;
    double *wgt = (double *)malloc(sizeof(double) * (size_t)m * (size_t)d);
    for (int32_t c = 0; c < d; ++c) {
        double mx = -INFINITY;
        for (int32_t p = 0; p < m; ++p)
            if (G[(int64_t)p * d + c] > mx) mx = G[(int64_t)p * d + c];
        double s = 0.0;
        for (int32_t p = 0; p < m; ++p) s += exp(G[(int64_t)p * d + c] - mx);
        for (int32_t p = 0; p < m; ++p)
            wgt[(int64_t)p * d + c] = exp(G[(int64_t)p * d + c] - mx) / s;
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Tc; ++j) {
        for (int32_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int32_t p = 0; p < m; ++p)
                acc += wgt[(int64_t)p * d + c] * X[(j * m + p) * d + c];
            Xc[j * d + c] = acc;
        }
    }
    free(wgt);
}

/* Token-level compressor (the same page, §1.1, CSA paragraph: a token-level
 * compressor merges every m tokens' KV into one entry; the real one is
 * learned).  The gate logit of each channel comes from the token itself:
 * Z [T, d] holds one logit per token and channel (for instance a projection
 * of the token's hidden state), and
 *   Xc[j,c] = sum_p softmax_p(Z[j*m+p, c]) * X[j*m+p, c],  p = 0 .. m-1.
 * X [T, d], Z [T, d] -> Xc [floor(T/m), d]; only full blocks make entries. */
void oracle_compress_tok(const double *X, const double *Z, int64_t T, int32_t d,
                         int32_t m, double *Xc)
{
    int64_t Tc = T / m;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Tc; ++j) {
        for (int32_t c = 0; c < d; ++c) {
            double mx = -INFINITY;
            for (int32_t p = 0; p < m; ++p) {
                double z = Z[(j * m + p) * d + c];
                if (z > mx) mx = z;
            }
            double s = 0.0, acc = 0.0;
            for (int32_t p = 0; p < m; ++p) {
                double e = exp(Z[(j * m + p) * d + c] - mx);
                s += e;
                acc += e * X[(j * m + p) * d + c];
            }
            Xc[j * d + c] = acc / s;
        }
    }
}

/* Partial RoPE (the same page, §1.1, engineering details: RoPE acts only on
 * the last 64 dimensions, and the core-attention output gets the inverse
 * RoPE to restore relative positions).  Reading: the last R = 64 dimensions
 * of each d-vector form 32 interleaved pairs (2i, 2i+1), i = 0..31, rotated by
 * the angle p * theta_i with theta_i = base^(-2i/R), base = 10000:
 *   y[2i]   = x[2i] cos(a) - x[2i+1] sin(a)
 *   y[2i+1] = x[2i] sin(a) + x[2i+1] cos(a),   a = sign * p * theta_i;
 * sign = -1 is the inverse rotation.  The first d - R dimensions are copied.
 * X [n, hd, d] (hd vectors per row, all at the row's position pos[r]). */
void oracle_rope(const double *X, const int64_t *pos, int64_t n, int32_t hd, int32_t d,
                 int32_t R, double base, int32_t sign, double *Y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int32_t h = 0; h < hd; ++h) {
            const double *x = X + (r * hd + h) * d;
            double *y = Y + (r * hd + h) * d;
            for (int32_t c = 0; c < d - R; ++c) y[c] = x[c];
            const double *xr = x + (d - R);
            double *yr = y + (d - R);
            for (int32_t i = 0; i < R / 2; ++i) {
                double theta = pow(base, -2.0 * i / R);
                double a = (double)sign * (double)pos[r] * theta;
                double cs = cos(a), sn = sin(a);
                yr[2 * i] = xr[2 * i] * cs - xr[2 * i + 1] * sn;
                yr[2 * i + 1] = xr[2 * i] * sn + xr[2 * i + 1] * cs;
            }
        }
    }
}

/* ------------------------------------------------------------------------
 * Low-precision indexer ("DeepSeek V4 详解：1M 上下文背后，真正发生了什么",
 * §"mHC、Muon、FP4": FP4 runs in the CSA indexer's QK path, and the selector
 * keeps almost all of the exact selection; "DeepSeek-V4 技术解析…", §1.1:
 * the indexer computes in FP4).  The pages give neither the element format
 * nor the scaling, so the reading is the OCP Microscaling (MX) formats
 * specification v1.0: blocks of 32 consecutive values share one power-of-two
 * scale X = 2^(floor(log2(amax)) - emax_elem), stored as an E8M0 byte, and
 * each value becomes the element nearest to v / X (ties to the even
 * mantissa), clamped to the largest finite element.  Elements:
 *   E4M3 (MXFP8): bias 7, 3 mantissa bits, no infinity, largest 448
 *                 (emax_elem 8), smallest normal 2^-6, subnormal step 2^-9
 *   E2M1 (MXFP4): bias 1, 1 mantissa bit, largest 6 (emax_elem 2), smallest
 *                 normal 1, subnormal step 1/2
 * An all-zero block takes the smallest scale, 2^-127.  Shared exponents
 * outside the E8M0 range are clamped to [-127, 127].
 * ------------------------------------------------------------------------ */

/* Element format parameters: mantissa bits, smallest normal exponent,
 * largest finite value, emax, exponent bias. */
typedef struct { int mbits, emin, emax, bias; double maxv; } mx_elem;
static mx_elem mx_format(int32_t fmt)
{
    mx_elem f;
    if (fmt == 4) { f.mbits = 1; f.emin = 0; f.emax = 2; f.bias = 1; f.maxv = 6.0; }
    else          { f.mbits = 3; f.emin = -6; f.emax = 8; f.bias = 7; f.maxv = 448.0; }
    return f;
}

/* Nearest element to v (ties to the even mantissa), clamped to +-maxv;
 * *code receives the element's bit pattern (sign, exponent field, mantissa). */
static double mx_round(double v, mx_elem f, uint32_t *code)
{
    const int neg = signbit(v) != 0;
    double a = fabs(v), r;
    if (a >= f.maxv) {
        r = f.maxv;
    } else {
        int E;
        if (a < ldexp(1.0, f.emin)) {
            E = f.emin;                       /* subnormal range: fixed step */
        } else {
            (void)frexp(a, &E);               /* a = frac * 2^E, frac in [0.5, 1) */
            E -= 1;                           /* a in [2^E, 2^(E+1)) */
        }
        const double q = ldexp(1.0, E - f.mbits);
        r = nearbyint(a / q) * q;             /* round half to even: default mode */
        if (r > f.maxv) r = f.maxv;
    }
    uint32_t ef, mf;
    if (r < ldexp(1.0, f.emin)) {
        ef = 0;
        mf = (uint32_t)(r / ldexp(1.0, f.emin - f.mbits));
    } else {
        int E;
        (void)frexp(r, &E);
        E -= 1;
        ef = (uint32_t)(E + f.bias);
        mf = (uint32_t)((r / ldexp(1.0, E) - 1.0) * (double)(1 << f.mbits));
    }
    *code = ((uint32_t)neg << (f.mbits + (f.mbits == 3 ? 4 : 2))) | (ef << f.mbits) | mf;
    return neg ? -r : r;
}

/* MX quantization of n values (n a multiple of 32), fmt 8 = MXFP8 (E4M3),
 * 4 = MXFP4 (E2M1).  Outputs per value its element code and its dequantized
 * value code * X; per block of 32 the E8M0 scale byte (shared exponent + 127). */
void oracle_mx_quantize(const double *x, int64_t n, int32_t fmt, uint32_t *codes,
                        uint8_t *scales, double *deq)
{
    const mx_elem f = mx_format(fmt);
    for (int64_t b = 0; b < n / 32; ++b) {
        const double *v = x + b * 32;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) if (fabs(v[i]) > amax) amax = fabs(v[i]);
        int e = -127;
        if (amax > 0.0) {
            int E;
            (void)frexp(amax, &E);            /* floor(log2(amax)) = E - 1 */
            e = (E - 1) - f.emax;
            if (e < -127) e = -127;
            if (e > 127) e = 127;
        }
        scales[b] = (uint8_t)(e + 127);
        const double X = ldexp(1.0, e);
        for (int i = 0; i < 32; ++i) {
            uint32_t c;
            const double el = mx_round(v[i] / X, f, &c);
            codes[b * 32 + i] = c;
            deq[b * 32 + i] = el * X;
        }
    }
}

/* Number of compressed entries visible from absolute position t. */
static int64_t n_visible(int64_t t, int32_t m) { return (t + 1) / m; }

/* Lightning Indexer for one sequence.
 * qI [Nq, HI, dI], w [Nq, HI], kI [Tc, HI, dI], tpos [Nq] absolute positions.
 * I [Nq, Tc]: visible entries get the score, invisible ones -inf. */
void oracle_index(const double *qI, const double *w, const double *kI,
                  const int64_t *tpos, int64_t Nq, int64_t Tc, int32_t HI,
                  int32_t dI, int32_t m, double *I)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < Nq; ++r) {
        int64_t nv = n_visible(tpos[r], m);
        for (int64_t j = 0; j < Tc; ++j) {
            if (j >= nv) { I[r * Tc + j] = -INFINITY; continue; }
            double score = 0.0;
            for (int32_t h = 0; h < HI; ++h) {
                const double *q = qI + (r * HI + h) * dI;
                const double *k = kI + (j * HI + h) * dI;
                double dot = 0.0;
                for (int32_t e = 0; e < dI; ++e) dot += q[e] * k[e];
                score += w[r * HI + h] * (dot > 0.0 ? dot : 0.0);
            }
            I[r * Tc + j] = score;
        }
    }
}

typedef struct { double s; int64_t j; } scored;

/* Total order: larger score first; on equal score the lower index first.
 * C compares -0.0 and +0.0 as equal, so they tie as the reading requires. */
static int by_score_desc_index_asc(const void *a, const void *b)
{
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int by_int_asc(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Top-k selector: for each row keep the min(k, nvis[r]) visible entries
 * (columns 0 .. nvis[r]-1 of I) ranked first by the total order, written in
 * ascending index order, then -1 padding up to k. */
void oracle_topk(const double *I, int64_t Nq, int64_t ld, const int64_t *nvis,
                 int32_t k, int32_t *idx)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < Nq; ++r) {
        int64_t n = nvis[r];
        scored *all = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
        for (int64_t j = 0; j < n; ++j) { all[j].s = I[r * ld + j]; all[j].j = j; }
        qsort(all, (size_t)n, sizeof(scored), by_score_desc_index_asc);
        int64_t keep = n < k ? n : k;
        int32_t *out = idx + r * k;
        for (int64_t i = 0; i < keep; ++i) out[i] = (int32_t)all[i].j;
        qsort(out, (size_t)keep, sizeof(int32_t), by_int_asc);
        for (int64_t i = keep; i < k; ++i) out[i] = -1;
        free(all);
    }
}

/* Softmax attention of one query head over an explicit list of key rows.
 * logits_i = scale * q . K_i ; the sink logit (-inf: none) joins the
 * denominator only: O = sum_i e^{logit_i} V_i / (e^{sink} + sum_i e^{logit_i}),
 * lse = log of that denominator. */
static void attend_list(const double *q, const double *const *K,
                        const double *const *V, int64_t n, int32_t d,
                        double scale, double sink, double *o, double *lse)
{
    if (n == 0) {
        for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
        *lse = sink;
        return;
    }
    double *logit = (double *)malloc(sizeof(double) * (size_t)n);
    double mx = sink;
    for (int64_t i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int32_t c = 0; c < d; ++c) dot += q[c] * K[i][c];
        logit[i] = scale * dot;
        if (logit[i] > mx) mx = logit[i];
    }
    double sum = sink == -INFINITY ? 0.0 : exp(sink - mx);
    for (int64_t i = 0; i < n; ++i) { logit[i] = exp(logit[i] - mx); sum += logit[i]; }
    for (int32_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t i = 0; i < n; ++i) acc += logit[i] * V[i][c];
        o[c] = acc / sum;
    }
    *lse = mx + log(sum);
    free(logit);
}

/* Appends the window rows of position t: raw positions max(0,t-W+1) .. t,
 * stored at raw row (position - raw_pos0).  Returns the new count, or -1 if a
 * window position is not held by the raw cache. */
static int64_t add_window(const double *Kraw, const double *Vraw, int64_t Nraw,
                          int64_t raw_pos0, int64_t t, int32_t W, int32_t d,
                          const double **Kl, const double **Vl, int64_t n)
{
    if (W <= 0) return n;
    int64_t lo = t - W + 1 < 0 ? 0 : t - W + 1;
    for (int64_t p = lo; p <= t; ++p) {
        int64_t row = p - raw_pos0;
        if (row < 0 || row >= Nraw) return -1;
        Kl[n] = Kraw + row * d;
        Vl[n] = Vraw + row * d;
        ++n;
    }
    return n;
}

/* CSA core attention for one sequence (MQA: one K/V row serves every head).
 * Q [Nq, H, d]; Kc, Vc [Tc, d]; idx [Nq, k] sequence-local entry numbers,
 * -1 = padding (skipped); raw Kraw, Vraw [Nraw, d] holding positions
 * raw_pos0 ..; tpos [Nq].  Key set of row r: the selected entries in the order
 * listed, then the window.  sink [H] or NULL.  O [Nq, H, d], lse [Nq, H].
 * Returns 0, or the first row whose inputs are invalid + 1 (negated). */
int64_t oracle_sparse_attn(const double *Q, const double *Kc, const double *Vc,
                           int64_t Tc, const int32_t *idx, int32_t k,
                           const double *Kraw, const double *Vraw, int64_t Nraw,
                           int64_t raw_pos0, const int64_t *tpos, int64_t Nq,
                           int32_t H, int32_t d, int32_t W, double scale,
                           const double *sink, double *O, double *lse)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < Nq; ++r) {
        int64_t cap = (int64_t)k + (W > 0 ? W : 0);
        const double **Kl = (const double **)malloc(sizeof(double *) * (size_t)(cap + 1));
        const double **Vl = (const double **)malloc(sizeof(double *) * (size_t)(cap + 1));
        int64_t n = 0;
        int ok = 1;
        for (int32_t i = 0; i < k; ++i) {
            int32_t j = idx[r * k + i];
            if (j < 0) continue;
            if ((int64_t)j >= Tc) { ok = 0; break; }
            Kl[n] = Kc + (int64_t)j * d;
            Vl[n] = Vc + (int64_t)j * d;
            ++n;
        }
        if (ok) n = add_window(Kraw, Vraw, Nraw, raw_pos0, tpos[r], W, d, Kl, Vl, n);
        if (!ok || n < 0) {
#pragma omp critical
            { if (bad == 0 || r + 1 < bad) bad = r + 1; }
        } else {
            for (int32_t h = 0; h < H; ++h)
                attend_list(Q + (r * H + h) * d, Kl, Vl, n, d, scale,
                            sink ? sink[h] : -INFINITY, O + (r * H + h) * d,
                            lse + r * H + h);
        }
        free(Kl);
        free(Vl);
    }
    return -bad;
}

/* HCA attention for one sequence: every visible entry j < floor((t+1)/m),
 * in entry order, then the window; otherwise as oracle_sparse_attn. */
int64_t oracle_hca_attn(const double *Q, const double *Kc, const double *Vc,
                        int64_t Tc, int32_t m, const double *Kraw,
                        const double *Vraw, int64_t Nraw, int64_t raw_pos0,
                        const int64_t *tpos, int64_t Nq, int32_t H, int32_t d,
                        int32_t W, double scale, const double *sink, double *O,
                        double *lse)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < Nq; ++r) {
        int64_t nv = n_visible(tpos[r], m);
        int64_t cap = nv + (W > 0 ? W : 0);
        const double **Kl = (const double **)malloc(sizeof(double *) * (size_t)(cap + 1));
        const double **Vl = (const double **)malloc(sizeof(double *) * (size_t)(cap + 1));
        int64_t n = 0;
        int ok = nv <= Tc;
        for (int64_t j = 0; ok && j < nv; ++j) {
            Kl[n] = Kc + j * d;
            Vl[n] = Vc + j * d;
            ++n;
        }
        if (ok) n = add_window(Kraw, Vraw, Nraw, raw_pos0, tpos[r], W, d, Kl, Vl, n);
        if (!ok || n < 0) {
#pragma omp critical
            { if (bad == 0 || r + 1 < bad) bad = r + 1; }
        } else {
            for (int32_t h = 0; h < H; ++h)
                attend_list(Q + (r * H + h) * d, Kl, Vl, n, d, scale,
                            sink ? sink[h] : -INFINITY, O + (r * H + h) * d,
                            lse + r * H + h);
        }
        free(Kl);
        free(Vl);
    }
    return -bad;
}
