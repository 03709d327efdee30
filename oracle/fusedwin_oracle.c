/*
 * fusedwin_oracle.c -- the oracle: plain, slow, single-threaded CPU loops that
 * define what the three fused sliding-window operators compute.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The CUDA product path never calls it
 * and shares no code, header or table with it.
 *
 * Arithmetic convention.  Inputs are float32.  Every linear stage (conv2d,
 * conv-transpose) is summed in float64 (each float32 x float32 product is exact
 * in float64), and every stage's result is rounded to float32, the storage type
 * of the PyTorch models the pages describe; the next stage starts from that
 * float32 value.  Elementwise stages (tanh, scale, bias, softmax, sigmoid) are
 * evaluated in float64 and rounded to float32.  MaxPool is a pure float32
 * comparison and rounds nothing.
 *
 * Sources (POPCORNBENCH reasoning traces, all for the same PyTorch models):
 *   [P1] "Kimi-K2.6 l2_p82": Conv2d(8->64,k3) -> tanh -> *2.0 -> +bias[64,1,1]
 *        -> MaxPool2d(4), x [128,8,256,256]; problem statement and output-size
 *        derivation (conv 254, pool 63); the model's forward order.
 *   [P2] "Kimi-K2.6 l1_p42": MaxPool2d(k=4,s=1,p=1,d=1), x [32,64,512,512];
 *        problem statement (pooled size formula, 511) and the -inf padding
 *        semantics quoted from the PyTorch documentation.
 *   [P3] "Kimi-K2.6 l2_p91": ConvTranspose2d(64->128,k4,s2,p1,op1) -> softmax
 *        over dim 1 -> +bias[128,1,1] -> *2.0 -> sigmoid, x [128,64,64,64];
 *        the transposed-convolution index map oh = ih*s + kh - p and the
 *        output-size formula (129).
 *
 * Readings taken where the pages are silent:
 *   - MaxPool ties keep the first tap in row-major (kh, kw) order; a NaN tap
 *     propagates (the first NaN in that order is kept); padded taps are -inf.
 *   - The fused conv+pool applies tanh/scale/bias to EVERY conv output before
 *     pooling, literally in the model's order; no reordering is done here.
 *   - Pool windows use floor mode (ragged rows/cols are dropped), no padding.
 *   - Extensions beyond the pages (the generic MaxPool2d options the l1_p42 trace
 *     names only as PyTorch's non-default behaviour): ceil mode and argmax
 *     indices, following PyTorch's documented MaxPool2d definition -- in ceil
 *     mode the size rounds up, and a window that would start in the right
 *     padding is dropped; an index is the flat ih*W + iw of the tap the value
 *     came from (same tie and NaN rules; -1 when a window has no input tap).
 *
 * Parity pins for every function here live in the CPU test-suite (brute force,
 * library special cases, closed forms, invariants, the adjoint identity).
 *
 * Threads.  The file is built twice from this one source: single-threaded (the
 * oracle proper; the OpenMP pragmas are ignored) and with -fopenmp, which only
 * spreads independent images / channels / planes over the host cores to time the
 * definition at full size.  No pragma changes an operation or its order within
 * an output, so both builds give bit-identical results.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

/* ---------------------------------------------------------------- sizes -- */

/* Floor division for a possibly negative numerator and a positive divisor. */
static long floordiv(long a, long b) {
    long q = a / b;
    if ((a % b != 0) && (a < 0)) q -= 1;
    return q;
}

/* Conv2d output size, dilation 1 ([P1] output-size derivation: 256 -> 254). */
long oracle_conv2d_out_size(long H, long k, long s, long p) {
    if (k < 1 || s < 1 || p < 0) return -1;
    return floordiv(H + 2 * p - k, s) + 1;
}

/* MaxPool2d output size, floor mode ([P2] pooled size formula: 512 -> 511;
 * [P1] 254 -> 63 with the default stride = kernel). */
long oracle_pool_out_size(long H, long k, long s, long p, long d) {
    if (k < 1 || s < 1 || p < 0 || d < 1) return -1;
    return floordiv(H + 2 * p - d * (k - 1) - 1, s) + 1;
}

/* MaxPool2d output size in ceil mode (extension, see the readings above):
 * ceil((H + 2p - d(k-1) - 1) / s) + 1, minus one when that last window would
 * start at or past H + p (inside the right padding). */
long oracle_pool_out_size_ceil(long H, long k, long s, long p, long d) {
    if (k < 1 || s < 1 || p < 0 || d < 1) return -1;
    const long span = H + 2 * p - d * (k - 1) - 1;
    long o = -floordiv(-span, s) + 1;  /* ceil(span / s) + 1 */
    if (o >= 1 && (o - 1) * s >= H + p) o -= 1;
    return o;
}

/* ConvTranspose2d output size, dilation 1 ([P3] output-size formula: 64 -> 129). */
long oracle_convt_out_size(long H, long k, long s, long p, long op) {
    if (k < 1 || s < 1 || p < 0 || op < 0) return -1;
    return (H - 1) * s - 2 * p + (k - 1) + op + 1;
}

/* ------------------------------------------------------------- conv2d ---- */

/* One output of a Conv2d (cross-correlation, as nn.Conv2d computes it):
 *   y[n,co,oh,ow] = cb[co] + sum_{ci,kh,kw} x[n,ci,oh*s-p+kh, ow*s-p+kw] * w[co,ci,kh,kw]
 * with taps outside the input contributing zero (zero padding).
 * x: [N,Cin,H,W], w: [Cout,Cin,KH,KW], cb: [Cout] or NULL.  Result in float64. */
double oracle_conv2d_one(const float *x, long Cin, long H, long W,
                         const float *w, const float *cb, long KH, long KW,
                         long s, long p, long n, long co, long oh, long ow) {
    double acc = cb ? (double)cb[co] : 0.0;
    for (long ci = 0; ci < Cin; ++ci)
        for (long kh = 0; kh < KH; ++kh)
            for (long kw = 0; kw < KW; ++kw) {
                long ih = oh * s - p + kh, iw = ow * s - p + kw;
                if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
                double xv = x[((n * Cin + ci) * H + ih) * W + iw];
                double wv = w[((co * Cin + ci) * KH + kh) * KW + kw];
                acc += xv * wv;
            }
    return acc;
}

/* Full Conv2d in float64: y [N,Cout,Ho,Wo]. */
int oracle_conv2d(const float *x, long N, long Cin, long H, long W,
                  const float *w, const float *cb, long Cout, long KH, long KW,
                  long s, long p, double *y) {
    long Ho = oracle_conv2d_out_size(H, KH, s, p);
    long Wo = oracle_conv2d_out_size(W, KW, s, p);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (long n = 0; n < N; ++n)
        for (long co = 0; co < Cout; ++co)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow)
                    y[((n * Cout + co) * Ho + oh) * Wo + ow] =
                        oracle_conv2d_one(x, Cin, H, W, w, cb, KH, KW, s, p, n, co, oh, ow);
    return ORACLE_OK;
}

/* ------------------------------------------------------------ maxpool ---- */

/* Running-max update: a larger value replaces the current one, a NaN replaces
 * a non-NaN current value, ties keep the current (earlier) tap. */
static float max_update(float m, float v) {
    if (isnan(m)) return m;
    if (isnan(v) || v > m) return v;
    return m;
}

/* One MaxPool2d output over a single [H,W] plane:
 *   out[oh,ow] = max_{kh,kw} xpad[oh*s - p + kh*d, ow*s - p + kw*d]
 * where taps outside the plane are -inf ([P2] -inf padding).  Taps are visited
 * in row-major (kh, kw) order. */
float oracle_maxpool2d_one(const float *plane, long H, long W, long k, long s,
                           long p, long d, long oh, long ow) {
    float m = -INFINITY;
    for (long kh = 0; kh < k; ++kh)
        for (long kw = 0; kw < k; ++kw) {
            long ih = oh * s - p + kh * d, iw = ow * s - p + kw * d;
            float v = (ih >= 0 && ih < H && iw >= 0 && iw < W) ? plane[ih * W + iw] : -INFINITY;
            m = max_update(m, v);
        }
    return m;
}

/* One MaxPool2d output and its argmax (extension): the value as in
 * oracle_maxpool2d_one; *idx = ih*W + iw of the input tap that value came from --
 * the first in-bounds tap initialises the running (value, index), later taps
 * replace it by the running-max rule -- or -1 when no tap is in bounds. */
float oracle_maxpool2d_one_idx(const float *plane, long H, long W, long k, long s,
                               long p, long d, long oh, long ow, long *idx) {
    float m = -INFINITY;
    long at = -1;
    for (long kh = 0; kh < k; ++kh)
        for (long kw = 0; kw < k; ++kw) {
            const long ih = oh * s - p + kh * d;
            const long iw = ow * s - p + kw * d;
            if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;  /* -inf: never the first max */
            float v = plane[ih * W + iw];
            /* the running-max rule of max_update, keeping the tap's index with the value */
            if (at < 0 || (!isnan(m) && (isnan(v) || v > m))) {
                m = v;
                at = ih * W + iw;
            }
        }
    *idx = at;
    return m;
}

/* MaxPool2d with ceil mode and indices (extension): out and idx [N,C,Ho,Wo]
 * (idx may be NULL), Ho/Wo from oracle_pool_out_size(_ceil). */
int oracle_maxpool2d_ex(const float *x, long N, long C, long H, long W, long k, long s, long p,
                        long d, int ceil_mode, float *out, long *idx) {
    long Ho = ceil_mode ? oracle_pool_out_size_ceil(H, k, s, p, d) : oracle_pool_out_size(H, k, s, p, d);
    long Wo = ceil_mode ? oracle_pool_out_size_ceil(W, k, s, p, d) : oracle_pool_out_size(W, k, s, p, d);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
    for (long nc = 0; nc < N * C; ++nc) {
        const float *plane = x + nc * H * W;
        for (long oh = 0; oh < Ho; ++oh)
            for (long ow = 0; ow < Wo; ++ow) {
                long at;
                const long o = (nc * Ho + oh) * Wo + ow;
                out[o] = oracle_maxpool2d_one_idx(plane, H, W, k, s, p, d, oh, ow, &at);
                if (idx) idx[o] = at;
            }
    }
    return ORACLE_OK;
}

/* Full MaxPool2d: x [N,C,H,W] -> out [N,C,Ho,Wo]. */
int oracle_maxpool2d(const float *x, long N, long C, long H, long W,
                     long k, long s, long p, long d, float *out) {
    long Ho = oracle_pool_out_size(H, k, s, p, d);
    long Wo = oracle_pool_out_size(W, k, s, p, d);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
#pragma omp parallel for schedule(dynamic)
    for (long nc = 0; nc < N * C; ++nc) {
        const float *plane = x + nc * H * W;
        for (long oh = 0; oh < Ho; ++oh)
            for (long ow = 0; ow < Wo; ++ow)
                out[(nc * Ho + oh) * Wo + ow] = oracle_maxpool2d_one(plane, H, W, k, s, p, d, oh, ow);
    }
    return ORACLE_OK;
}

/* ----------------------------------------- fused conv+tanh+scale+bias+pool */

/* The elementwise chain of [P1]'s forward, applied to one float32 conv output:
 * tanh, then multiply by the scalar, then add the channel's bias; each stage
 * rounded to float32. */
static float tanh_scale_bias(float y, float scale, float b) {
    float t = (float)tanh((double)y);
    float u = (float)((double)t * (double)scale);
    return (float)((double)u + (double)b);
}

/* One output of [P1]'s model: MaxPool2d(pk, stride ps) over
 * bias[co] + scale * tanh(conv2d(x)[n,co]), conv stride 1 and padding 0.
 * The pool has no padding and dilation 1 (floor mode). */
float oracle_convpool_one(const float *x, long Cin, long H, long W,
                          const float *w, const float *cb, long KH, long KW,
                          float scale, const float *bias, long pk, long ps,
                          long n, long co, long i, long j) {
    float m = -INFINITY;
    for (long a = 0; a < pk; ++a)
        for (long b = 0; b < pk; ++b) {
            long oh = i * ps + a, ow = j * ps + b;
            float y = (float)oracle_conv2d_one(x, Cin, H, W, w, cb, KH, KW, 1, 0, n, co, oh, ow);
            m = max_update(m, tanh_scale_bias(y, scale, bias[co]));
        }
    return m;
}

/* Full fused model, stage by stage: conv (-> float32 tensor), tanh, scale,
 * bias, then MaxPool2d(pk, ps) of the whole intermediate tensor.
 * out: [N,Cout,Ho,Wo], Ho = floor((H-KH+1-pk)/ps)+1. */
int oracle_conv2d_tanh_scale_bias_maxpool(const float *x, long N, long Cin, long H, long W,
                                          const float *w, const float *cb, long Cout,
                                          long KH, long KW, float scale, const float *bias,
                                          long pk, long ps, float *out) {
    long Hc = oracle_conv2d_out_size(H, KH, 1, 0), Wc = oracle_conv2d_out_size(W, KW, 1, 0);
    if (Hc < 1 || Wc < 1 || pk < 1 || ps < 1) return ORACLE_EINVAL;
    long Ho = oracle_pool_out_size(Hc, pk, ps, 0, 1), Wo = oracle_pool_out_size(Wc, pk, ps, 0, 1);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
    size_t inter = (size_t)N * Cout * Hc * Wc;
    double *y = (double *)malloc(inter * sizeof(double));
    float *v = (float *)malloc(inter * sizeof(float));
    if (!y || !v) { free(y); free(v); return ORACLE_ENOMEM; }
    oracle_conv2d(x, N, Cin, H, W, w, cb, Cout, KH, KW, 1, 0, y);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (long n = 0; n < N; ++n)
        for (long co = 0; co < Cout; ++co)
            for (long e = 0; e < Hc * Wc; ++e) {
                size_t q = (size_t)(n * Cout + co) * Hc * Wc + e;
                v[q] = tanh_scale_bias((float)y[q], scale, bias[co]);
            }
    oracle_maxpool2d(v, N, Cout, Hc, Wc, pk, ps, 0, 1, out);
    free(y);
    free(v);
    return ORACLE_OK;
}

/* ----------------------------------------------------- conv-transpose ---- */

/* Full ConvTranspose2d in float64, scatter form ([P3] index map): every input
 * tap x[n,ci,ih,iw] adds x * w[ci,co,kh,kw] to y[n,co,ih*s-p+kh, iw*s-p+kw]
 * when that position lies inside the [Ho,Wo] output.  w: [Cin,Cout,K,K]. */
int oracle_convt2d(const float *x, long N, long Cin, long H, long W,
                   const float *w, const float *cb, long Cout, long K,
                   long s, long p, long op, double *y) {
    long Ho = oracle_convt_out_size(H, K, s, p, op), Wo = oracle_convt_out_size(W, K, s, p, op);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (long n = 0; n < N; ++n)
        for (long co = 0; co < Cout; ++co)
            for (long e = 0; e < Ho * Wo; ++e)
                y[(n * Cout + co) * Ho * Wo + e] = cb ? (double)cb[co] : 0.0;
    /* images are independent: each iteration writes only its own y[n] */
#pragma omp parallel for schedule(dynamic)
    for (long n = 0; n < N; ++n)
        for (long ci = 0; ci < Cin; ++ci)
            for (long ih = 0; ih < H; ++ih)
                for (long iw = 0; iw < W; ++iw) {
                    double xv = x[((n * Cin + ci) * H + ih) * W + iw];
                    for (long co = 0; co < Cout; ++co)
                        for (long kh = 0; kh < K; ++kh)
                            for (long kw = 0; kw < K; ++kw) {
                                long oh = ih * s - p + kh, ow = iw * s - p + kw;
                                if (oh < 0 || oh >= Ho || ow < 0 || ow >= Wo) continue;
                                double wv = w[((ci * Cout + co) * K + kh) * K + kw];
                                y[((n * Cout + co) * Ho + oh) * Wo + ow] += xv * wv;
                            }
                }
    return ORACLE_OK;
}

/* One ConvTranspose2d output in float64, gather form: the same sum collected
 * at the output, over the taps with oh = ih*s - p + kh and ow = iw*s - p + kw. */
double oracle_convt2d_one(const float *x, long Cin, long H, long W,
                          const float *w, const float *cb, long Cout, long K,
                          long s, long p, long n, long co, long oh, long ow) {
    double acc = cb ? (double)cb[co] : 0.0;
    for (long ci = 0; ci < Cin; ++ci)
        for (long kh = 0; kh < K; ++kh) {
            long th = oh + p - kh;
            if (th < 0 || th % s != 0 || th / s >= H) continue;
            long ih = th / s;
            for (long kw = 0; kw < K; ++kw) {
                long tw = ow + p - kw;
                if (tw < 0 || tw % s != 0 || tw / s >= W) continue;
                long iw = tw / s;
                acc += (double)x[((n * Cin + ci) * H + ih) * W + iw] *
                       (double)w[((ci * Cout + co) * K + kh) * K + kw];
            }
        }
    return acc;
}

/* Softmax over the C channels of one pixel, rounded to float32:
 *   p[c] = exp(y[c]) / sum_j exp(y[j]),
 * evaluated as exp(y[c] - max_j y[j]) / sum (the same value; no overflow). */
void oracle_softmax_channels(const float *y, long C, double *e_scratch, float *p) {
    double mx = -INFINITY, sum = 0.0;
    for (long c = 0; c < C; ++c) mx = (double)y[c] > mx ? (double)y[c] : mx;
    for (long c = 0; c < C; ++c) { e_scratch[c] = exp((double)y[c] - mx); sum += e_scratch[c]; }
    for (long c = 0; c < C; ++c) p[c] = (float)(e_scratch[c] / sum);
}

/* Softmax over the C channels of one pixel, then +bias[c], *scale, sigmoid
 * ([P3] forward order), each stage rounded to float32.  y: the pixel's C
 * float32 conv-transpose outputs; out: C results (stride 1). */
void oracle_softmax_bias_scale_sigmoid_pixel(const float *y, long C, const float *bias,
                                             float scale, double *e_scratch, float *out) {
    oracle_softmax_channels(y, C, e_scratch, out);
    for (long c = 0; c < C; ++c) {
        float q = (float)((double)out[c] + (double)bias[c]);
        float r = (float)((double)q * (double)scale);
        out[c] = (float)(1.0 / (1.0 + exp(-(double)r)));
    }
}

/* All Cout outputs of [P3]'s model at one pixel (n, oh, ow), conv-transpose by
 * the gather form.  out: Cout values, channel-major (out[c]). */
int oracle_convt_fused_pixel(const float *x, long Cin, long H, long W,
                             const float *w, const float *cb, long Cout, long K,
                             long s, long p, const float *bias, float scale,
                             long n, long oh, long ow, float *out) {
    float *y = (float *)malloc((size_t)Cout * sizeof(float));
    double *e = (double *)malloc((size_t)Cout * sizeof(double));
    if (!y || !e) { free(y); free(e); return ORACLE_ENOMEM; }
    for (long co = 0; co < Cout; ++co)
        y[co] = (float)oracle_convt2d_one(x, Cin, H, W, w, cb, Cout, K, s, p, n, co, oh, ow);
    oracle_softmax_bias_scale_sigmoid_pixel(y, Cout, bias, scale, e, out);
    free(y);
    free(e);
    return ORACLE_OK;
}

/* Full fused model of [P3]: conv-transpose (scatter form, -> float32 tensor),
 * then softmax over dim 1, +bias, *scale, sigmoid.  out: [N,Cout,Ho,Wo]. */
int oracle_convtranspose2d_softmax_bias_scale_sigmoid(const float *x, long N, long Cin, long H, long W,
                                                      const float *w, const float *cb, long Cout,
                                                      long K, long s, long p, long op,
                                                      const float *bias, float scale, float *out) {
    long Ho = oracle_convt_out_size(H, K, s, p, op), Wo = oracle_convt_out_size(W, K, s, p, op);
    if (Ho < 1 || Wo < 1) return ORACLE_EINVAL;
    size_t plane = (size_t)Ho * Wo;
    double *y = (double *)malloc((size_t)N * Cout * plane * sizeof(double));
    if (!y) return ORACLE_ENOMEM;
    oracle_convt2d(x, N, Cin, H, W, w, cb, Cout, K, s, p, op, y);
    int rc = ORACLE_OK;
    /* per-image scratch, so that images are independent */
#pragma omp parallel for schedule(dynamic)
    for (long n = 0; n < N; ++n) {
        float *yc = (float *)malloc((size_t)Cout * sizeof(float));
        float *oc = (float *)malloc((size_t)Cout * sizeof(float));
        double *e = (double *)malloc((size_t)Cout * sizeof(double));
        if (!yc || !oc || !e) {
            rc = ORACLE_ENOMEM;
        } else {
            for (size_t q = 0; q < plane; ++q) {
                for (long c = 0; c < Cout; ++c) yc[c] = (float)y[(n * Cout + c) * plane + q];
                oracle_softmax_bias_scale_sigmoid_pixel(yc, Cout, bias, scale, e, oc);
                for (long c = 0; c < Cout; ++c) out[(n * Cout + c) * plane + q] = oc[c];
            }
        }
        free(yc); free(oc); free(e);
    }
    free(y);
    return rc;
}
