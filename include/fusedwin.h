/*
 * fusedwin.h -- C ABI of libfusedwin: fused 2-D sliding-window operators on
 * dense NCHW float32 tensors, computed by CUDA kernels for sm_103a (GB300).
 *
 * Operators (each one a PyTorch model from the POPCORNBENCH reasoning traces):
 *   fw_conv2d_tanh_scale_bias_maxpool       -- trace "Kimi-K2.6 l2_p82":
 *        Conv2d(k3, stride 1, pad 0) -> tanh -> *scale -> +bias[C,1,1] -> MaxPool2d(k)
 *   fw_maxpool2d                             -- trace "Kimi-K2.6 l1_p42":
 *        MaxPool2d(kernel k, stride s, padding p, dilation d)
 *   fw_convtranspose2d_softmax_bias_scale_sigmoid -- trace "Kimi-K2.6 l2_p91":
 *        ConvTranspose2d(k, s, p, output_padding) -> softmax(dim=1) -> +bias -> *scale -> sigmoid
 *
 * Variants, declared below the call they extend: *_tf32 (conv+pool on plain-TF32
 * tensor cores), *_ffma (conv+pool or conv-transpose on the float32 FMA pipe
 * only), fw_maxpool2d_ex (ceil mode, argmax indices), *_unfused (the two-kernel
 * design, for comparison), *_nhwc (channels last: conv+pool, maxpool, conv-transpose),
 * *_noalloc
 * (conv-transpose without a caller workspace) and *_host (host buffers, copies
 * pipelined with the kernels).
 *
 * Conventions shared by every call:
 *   - Tensors are caller-owned device pointers to dense, contiguous NCHW float32
 *     (row-major, W fastest).  Pointers must be 4-byte aligned; 16-byte aligned
 *     pointers (any cudaMalloc / torch allocation) enable the vectorised paths.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  They do not synchronise and allocate no memory.
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns an error status and launches nothing.  `out` must not overlap any
 *     input (FW_ERR_ALIAS).
 *   - Element counts are limited to 2^62; each dimension to 2^31 - 1.
 *   - Status codes are returned, never aborted on.  Errors raised inside a
 *     kernel (a bounded wait that gave up) are recorded in a device-side error
 *     word and reported by fw_check_device_errors().
 */
#ifndef FUSEDWIN_H
#define FUSEDWIN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fw_status {
    FW_OK = 0,
    FW_ERR_NULL = 1,        /* a required pointer is NULL */
    FW_ERR_SHAPE = 2,       /* a size is < 1, the output would be empty, or too large */
    FW_ERR_PARAM = 3,       /* kernel / stride / padding / dilation / output_padding out of range,
                               or a non-finite scale */
    FW_ERR_ALIAS = 4,       /* out overlaps an input tensor */
    FW_ERR_ALIGN = 5,       /* a tensor pointer is not 4-byte aligned */
    FW_ERR_UNSUPPORTED = 6, /* valid arguments that this library does not implement */
    FW_ERR_LAUNCH = 7,      /* a CUDA call (attribute set-up or kernel launch) failed */
    FW_ERR_TIMEOUT = 8,     /* a bounded wait inside a kernel gave up */
    FW_ERR_INTERNAL = 9     /* a kernel reported an inconsistency */
} fw_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *fw_status_string(fw_status s);

/* Library version as major*10000 + minor*100 + patch. */
int fw_version(void);

/* ------------------------------------------------------------------ shapes */

/* Output size of fw_conv2d_tanh_scale_bias_maxpool.  The conv output is
 * Hc = H - KH + 1 (stride 1, no padding); the pool (no padding, dilation 1,
 * floor mode) gives Ho = floor((Hc - pool_k) / pool_s) + 1, pool_s <= 0 meaning
 * pool_s = pool_k.  For H = 256, KH = 3, pool_k = 4: 254 -> 63
 * (trace "Kimi-K2.6 l2_p82", problem statement). */
fw_status fw_conv2d_pool_out_shape(int H, int W, int KH, int KW, int pool_k, int pool_s,
                                   int *Ho, int *Wo);

/* Output size of fw_maxpool2d: Ho = floor((H + 2p - d(k-1) - 1) / s) + 1
 * (trace "Kimi-K2.6 l1_p42", output-dimension computation: 512 -> 511). */
fw_status fw_maxpool2d_out_shape(int H, int W, int k, int s, int p, int d, int *Ho, int *Wo);

/* Output size of fw_convtranspose2d_softmax_bias_scale_sigmoid:
 * Ho = (H - 1) s - 2p + (k - 1) + op + 1 (trace "Kimi-K2.6 l2_p91",
 * ConvTranspose2d output shape: 64 -> 129). */
fw_status fw_convt_out_shape(int H, int W, int k, int s, int p, int op, int *Ho, int *Wo);

/* --------------------------------------------------------------- operators */

/*
 * Fused conv3x3 -> tanh -> scale -> bias -> MaxPool2d (trace "Kimi-K2.6 l2_p82",
 * the model's forward and the monotone-reorder argument):
 *
 *   y[n,co,h,w]  = conv_b[co] + sum_{ci,i,j} x[n,ci,h+i,w+j] * w[co,ci,i,j]
 *   out[n,co,a,b] = max_{0<=u,v<pool_k} ( bias[co] + scale * tanh(y[n,co,a*pool_s+u, b*pool_s+v]) )
 *
 * x      [N, Cin, H, W]         input
 * w      [Cout, Cin, KH, KW]    conv weight
 * conv_b [Cout] or NULL         conv bias (NULL = zero)
 * bias   [Cout]                 the extra bias of shape [Cout,1,1]
 * scale  finite float           the scalar multiplier
 * pool_k >= 1, pool_s >= 1 (or <= 0 for pool_s = pool_k); no pool padding, dilation 1,
 *        floor mode: conv rows/cols past the last full window are dropped.
 * out    [N, Cout, Ho, Wo]      see fw_conv2d_pool_out_shape
 *
 * The conv intermediate never reaches memory: the window max (min for
 * scale < 0) is taken on y and the elementwise chain is applied once per
 * pooled output, which gives the same value because tanh and the float32
 * rounding of each stage are monotone.  KH = KW = 3 and pool_s = pool_k in
 * {2, 4} with Cin <= 16 take the tiled kernel; other shapes take a direct one.
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool(const float *x, int N, int Cin, int H, int W,
                                            const float *w, const float *conv_b, int Cout,
                                            int KH, int KW, float scale, const float *bias,
                                            int pool_k, int pool_s, float *out, void *stream);

/*
 * The same operator as fw_conv2d_tanh_scale_bias_maxpool (trace "Kimi-K2.6
 * l2_p82", model) with the convolution in plain TF32, the mode the trace
 * "Kimi-K2.6 l2_p91" describes for float32 convolutions on tensor cores (inputs
 * rounded, float32 accumulation); its bound is 5e-3 absolute.  On the tiled
 * tensor-core shapes (Cin = 8, KH = KW = 3, pool_s = pool_k in {2, 4},
 * Cout in {16, 32, 48, 64}) every product of the convolution is taken once in
 * TF32 (both operands rounded to 10 mantissa bits, float32 accumulation) instead
 * of the 3xTF32 split, about 3x less tensor work; on the [128,8,256,256]
 * workload (unit-variance x) the result differs from the 3xTF32 call's (itself
 * within 1e-5 of a float64 evaluation) by at most 1.5e-3.  Other shapes run
 * the float32 FMA kernels of fw_conv2d_tanh_scale_bias_maxpool.  Arguments,
 * statuses, layout and ownership are those of fw_conv2d_tanh_scale_bias_maxpool.
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool_tf32(const float *x, int N, int Cin, int H, int W,
                                                 const float *w, const float *conv_b, int Cout,
                                                 int KH, int KW, float scale, const float *bias,
                                                 int pool_k, int pool_s, float *out, void *stream);

/*
 * Channels-last variant of fw_conv2d_tanh_scale_bias_maxpool (same definition,
 * weights [Cout, Cin, KH, KW], statuses and 3xTF32 tolerance): x [N, H, W, Cin],
 * out [N, Ho, Wo, Cout].  Only the tensor-core shapes (Cin = 8, KH = KW = 3,
 * pool_s = pool_k in {2, 4}, Cout in {16, 32, 48, 64}); other valid arguments
 * return FW_ERR_UNSUPPORTED.  x and out must be 16-byte aligned (FW_ERR_ALIGN
 * otherwise).  A position's 8 input channels are two 16-byte loads that are rows
 * of the MMA's core matrices as they stand, and a pooled pixel's channels are
 * stored as 32 contiguous bytes per thread.  The result equals the NCHW call's
 * bit for bit, transposed.
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool_nhwc(const float *x, int N, int Cin, int H, int W,
                                                 const float *w, const float *conv_b, int Cout,
                                                 int KH, int KW, float scale, const float *bias,
                                                 int pool_k, int pool_s, float *out, void *stream);

/*
 * The same operator as fw_conv2d_tanh_scale_bias_maxpool computed on the float32
 * FMA pipe only (no tensor cores): the implicit GEMM with K = Cin*9 that the trace
 * "Kimi-K2.6 l2_p82" reasons about, float32 products and sums.  KH = KW = 3 and
 * pool_s = pool_k in {2, 4} with Cin <= 16 take the tiled FMA kernel (persistent,
 * 4x4 conv pixels x 4 channels per thread); other shapes take the direct kernel.
 * Within 1e-5 of a float64 evaluation on the tested shapes.  Arguments, statuses,
 * layout and ownership are those of fw_conv2d_tanh_scale_bias_maxpool.
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool_ffma(const float *x, int N, int Cin, int H, int W,
                                                 const float *w, const float *conv_b, int Cout,
                                                 int KH, int KW, float scale, const float *bias,
                                                 int pool_k, int pool_s, float *out, void *stream);

/*
 * MaxPool2d (trace "Kimi-K2.6 l1_p42", problem statement and the -inf padding
 * semantics it quotes):
 *
 *   out[n,c,a,b] = max_{0<=i,j<k} xpad[n,c, a*s - p + i*d, b*s - p + j*d]
 *
 * where taps outside [0,H) x [0,W) are -inf (a window of padding only gives
 * -inf).  Floor mode.  Ties keep the first tap in row-major (i, j) order (so
 * the sign of a zero is that of the first zero of the maximum); a NaN tap makes
 * the output NaN.
 *
 * x   [N, C, H, W];  out [N, C, Ho, Wo] (see fw_maxpool2d_out_shape)
 * k >= 1, s >= 1, p >= 0, d >= 1.
 * Stride 1, dilation 1, k <= 5, p <= min(2, k-1), W a multiple of 4 (16-byte rows)
 * from 32 to 2040 and a 16-byte aligned x take the streaming kernel (rows through
 * the bulk-copy engine); the strided or dilated (k, s, d, p) in {(2,2,1,0|1),
 * (3,2,1,0|1), (4,2,1,1), (5,2,1,2), (3,3,1,0|1), (4,4,1,0), (3,1,2,1|2), (2,1,2,1)}
 * under the same width and alignment conditions take its strided form; other
 * arguments take a direct kernel.
 */
fw_status fw_maxpool2d(const float *x, int N, int C, int H, int W, int k, int s, int p, int d,
                       float *out, void *stream);

/*
 * Channels-last MaxPool2d: x [N, H, W, C] and out [N, Ho, Wo, C] (Ho, Wo from
 * fw_maxpool2d_out_shape), the definition, tie and NaN rules of fw_maxpool2d per
 * channel.  Stride 1, dilation 1, k <= 5, C a multiple of 4 (C <= 1024) and 16-byte
 * aligned x and out take a band kernel: a block's input columns (all channels,
 * contiguous) stream into shared memory by bulk copies, and a thread handles 4
 * adjacent channels of one output column with 16-byte reads and stores (row maxima,
 * then a K-deep ring of rows: the same values as the row-major definition); other
 * arguments take a direct kernel, one output value per thread.  Statuses as
 * fw_maxpool2d.
 */
fw_status fw_maxpool2d_nhwc(const float *x, int N, int H, int W, int C, int k, int s, int p, int d, float *out,
                            void *stream);

/*
 * MaxPool2d with PyTorch's optional extensions (not on the pages: the l1_p42 trace
 * names ceil mode only as the non-default behaviour it does not use; indices are
 * not mentioned).  Same definition, tie and NaN rules as fw_maxpool2d, plus:
 *   ceil_mode != 0: each output size is ceil((H + 2p - d(k-1) - 1)/s) + 1, minus
 *     one when that last window would start at or past H + p (in the right
 *     padding); see fw_maxpool2d_out_shape_ex.  With s = 1 it equals floor mode.
 *   indices (optional, int64 [N, C, Ho, Wo], 8-byte aligned, or NULL): for each
 *     output, the flat index ih*W + iw within its input plane of the tap the value
 *     came from (first maximum in row-major tap order; first NaN if any), or -1
 *     when the window holds no input tap (the value is then -inf).
 * Without indices and with the floor-mode size, the call takes fw_maxpool2d's
 * kernels; otherwise a direct kernel (one thread per output).
 */
fw_status fw_maxpool2d_ex(const float *x, int N, int C, int H, int W, int k, int s, int p, int d,
                          int ceil_mode, float *out, long long *indices, void *stream);
fw_status fw_maxpool2d_out_shape_ex(int H, int W, int k, int s, int p, int d, int ceil_mode, int *Ho, int *Wo);

/*
 * ConvTranspose2d -> softmax over channels -> +bias -> *scale -> sigmoid
 * (trace "Kimi-K2.6 l2_p91", the model and the index map oh = ih*s + kh - p):
 *
 *   y[n,co,oh,ow] = conv_b[co] + sum over ci and (kh,kw) with oh = ih*s - p + kh,
 *                   ow = iw*s - p + kw, 0<=ih<H, 0<=iw<W, of x[n,ci,ih,iw] * w[ci,co,kh,kw]
 *   p[n,c,oh,ow]  = exp(y[n,c,oh,ow]) / sum_j exp(y[n,j,oh,ow])
 *   out           = 1 / (1 + exp(-(p + bias[c]) * scale))
 *
 * x      [N, Cin, H, W]
 * w      [Cin, Cout, k, k]  (ConvTranspose2d weight layout)
 * conv_b [Cout] or NULL;  bias [Cout];  scale finite
 * k >= 1, s >= 1, p >= 0, 0 <= op < s, Cout <= 1024.
 * out    [N, Cout, Ho, Wo] (see fw_convt_out_shape)
 * workspace, workspace_bytes: caller-owned device scratch of at least
 *        fw_convt_workspace_size(Cin, Cout, k, s, p) bytes, 256-byte aligned
 *        (NULL/0 when that size is 0).  The call rewrites the weight into it
 *        (one layout per output parity class); its contents are undefined
 *        afterwards.  Two calls that overlap in time must not share it.
 * k = 4, s = 2, p = 1 and Cout = 128 take the phase-decomposed tiled kernel
 * (each output parity class is a 2x2 convolution); other arguments take a
 * direct one.
 * Precision: with Cin in {8, 16, 32, 64} the tiled kernel runs on the tensor
 * cores in TF32 (both operands rounded to 10 mantissa bits, float32
 * accumulation), the mode the l2_p91 trace describes; its bound is 5e-3
 * absolute.  An error dy in the conv-transpose output moves an output by at
 * most |scale|/2 * p(1-p) * max|dy| (softmax slope p(1-p) per channel, doubled
 * for the normaliser, times the sigmoid slope <= 1/4): on the [128,64,64,64]
 * workload (unit-variance x, weights within +-1/32) the softmax is nearly flat
 * (p ~ 1/128) and the result stays within 1e-5 of a float64 evaluation; inputs
 * that make one channel dominate (x or w several times larger) reach a few
 * 1e-4.  Other Cin take the float32 FMA kernels, as does
 * fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma for every shape.
 */
fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid(const float *x, int N, int Cin, int H, int W,
                                                        const float *w, const float *conv_b,
                                                        int Cout, int k, int s, int p, int op,
                                                        const float *bias, float scale, float *out,
                                                        void *workspace, unsigned long long workspace_bytes,
                                                        void *stream);

/*
 * The same operator as fw_convtranspose2d_softmax_bias_scale_sigmoid (trace
 * "Kimi-K2.6 l2_p91", model) on the float32 FMA pipe only: float32 products
 * and sums, so its error does not grow with a sharp softmax (within 1e-5 of a
 * float64 evaluation on the tested inputs, dominant channels included).
 * k = 4, s = 2, p = 1, Cout = 128 take the tiled FMA kernel, other arguments
 * the direct one.  Arguments, workspace, statuses, layout and ownership are
 * those of fw_convtranspose2d_softmax_bias_scale_sigmoid.
 */
fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b,
                                                             int Cout, int k, int s, int p, int op,
                                                             const float *bias, float scale, float *out,
                                                             void *workspace, unsigned long long workspace_bytes,
                                                             void *stream);

/*
 * Channels-last variant (the l2_p91 trace considers the channels_last memory
 * format for this model): x [N, H, W, Cin] and out [N, Ho, Wo, Cout], same
 * weights, workspace (fw_convt_workspace_size), definition and tolerance.  Only
 * the tensor-core shapes (k = 4, s = 2, p = 1, Cout = 128, Cin in {8, 16, 32, 64});
 * other valid arguments return FW_ERR_UNSUPPORTED.  x must be 16-byte and out
 * 32-byte aligned (FW_ERR_ALIGN otherwise).  A pixel's 128 channels are contiguous
 * in both tensors, so the gather reads 16 bytes per lane and every output store
 * writes whole 32-byte sectors.
 */
fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b, int Cout, int k,
                                                             int s, int p, int op, const float *bias, float scale,
                                                             float *out, void *workspace,
                                                             unsigned long long workspace_bytes, void *stream);

/* Bytes of device workspace fw_convtranspose2d_softmax_bias_scale_sigmoid
 * needs for these arguments (0 when it needs none). */
unsigned long long fw_convt_workspace_size(int Cin, int Cout, int k, int s, int p);

/*
 * Allocation-free variant of fw_convtranspose2d_softmax_bias_scale_sigmoid (no
 * counterpart on the pages: it exists for callers that cannot allocate device
 * memory -- plugins that a host framework hands only input and output buffers
 * because it owns all device memory, real-time loops that may not allocate
 * after start-up, code where an allocation would implicitly synchronise the
 * device).  Same arguments and result, minus the workspace: the weight rewrite
 * goes into a fixed device array of FW_CONVT_STATIC_WS_BYTES inside the library,
 * which every device that loads the library holds until the process exits.
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library routine.
 *   - Returns FW_ERR_UNSUPPORTED, launching nothing, when the rewrite needs more
 *     than FW_CONVT_STATIC_WS_BYTES (fw_convt_workspace_size(Cin, Cout, k, s, p)
 *     bytes; 16*Cin*Cout*4 for the tiled k4 s2 p1 Cout=128 path, so Cin <= 128).
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  A cudaDeviceReset on that device invalidates the cached address:
 *     do not call this entry point on a device after resetting it.
 *   - Every call shares the one array and leaves its contents behind (each call
 *     rewrites all it reads, nothing has to start at zero); calls that overlap on
 *     the GPU -- on different streams, or from different host threads -- race on
 *     it and must be serialised by the caller.
 */
#define FW_CONVT_STATIC_WS_BYTES (1u << 20)
fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc(const float *x, int N, int Cin, int H, int W,
                                                                const float *w, const float *conv_b,
                                                                int Cout, int k, int s, int p, int op,
                                                                const float *bias, float scale, float *out,
                                                                void *stream);

/* ------------------------------------------------------- host-buffer calls */

/*
 * The three operators on tensors in host memory (page-locked for the copies to
 * overlap; pageable memory works, more slowly).  x, w, conv_b, bias and out are
 * HOST pointers with the layouts of the device calls above; `workspace` is
 * caller-owned DEVICE memory of at least the matching *_host_workspace_size
 * bytes, 256-byte aligned, holding the device copies of the inputs and output
 * (and the conv-transpose weight rewrite).  The batch is split into up to 8
 * chunks of images; each chunk's host->device copy, operator launch (on
 * `stream`, through the device entry point above, so the same checks and kernels
 * apply; the conv-transpose's weight rewrite is made once, by the first chunk)
 * and device->host copy are pipelined on two copy streams the library
 * creates once per device, so copies overlap the kernels of neighbouring chunks.
 * The call is ordered after earlier work on `stream`, and later work on `stream`
 * (e.g. a synchronisation) runs after the last output copy: out is complete once
 * `stream` is synchronised.  Calls serialise on a host lock while they enqueue;
 * two calls in flight at once must not share a workspace or host buffers.
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool_host(const float *x, int N, int Cin, int H, int W, const float *w,
                                                 const float *conv_b, int Cout, int KH, int KW, float scale,
                                                 const float *bias, int pool_k, int pool_s, float *out,
                                                 void *workspace, unsigned long long workspace_bytes, void *stream);
unsigned long long fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(int N, int Cin, int H, int W, int Cout,
                                                                         int KH, int KW, int pool_k, int pool_s);
fw_status fw_maxpool2d_host(const float *x, int N, int C, int H, int W, int k, int s, int p, int d, float *out,
                            void *workspace, unsigned long long workspace_bytes, void *stream);
unsigned long long fw_maxpool2d_host_workspace_size(int N, int C, int H, int W, int k, int s, int p, int d);
fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_host(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b, int Cout, int k,
                                                             int s, int p, int op, const float *bias, float scale,
                                                             float *out, void *workspace,
                                                             unsigned long long workspace_bytes, void *stream);
unsigned long long fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(int N, int Cin, int H, int W,
                                                                                     int Cout, int k, int s, int p,
                                                                                     int op);

/* ------------------------------------------------------ unfused comparison */

/*
 * The pages' own design, unfused, built from this library's kernels so that what
 * fusion saves can be measured (trace "Kimi-K2.6 l2_p82": a library convolution
 * writes the whole conv output, then one kernel per pooled output takes the window
 * max and applies tanh, scale and bias; trace "Kimi-K2.6 l2_p91": a library
 * conv-transpose writes its output, then one thread per pixel makes an online
 * pass over the channels for the softmax max and sum and a second pass for the
 * output).  Same arguments, result and tolerance as the fused calls, plus a
 * caller-owned workspace for the intermediate:
 *
 *   conv+pool: y [N, Cout, pool_k*Ho, pool_k*Wo] = conv(x) + conv_b (the conv
 *              outputs the floor-mode pool reads), then out from y.  The result is
 *              bit-identical to fw_conv2d_tanh_scale_bias_maxpool: rounding
 *              y = a + conv_b is monotone in a, so the window maximum of y is the
 *              rounded sum of the window maximum of a and conv_b.
 *   convT:     [rewritten weights | y [N, Cout, Ho, Wo]], then out from y.
 *
 * workspace: at least fw_conv2d_pool_unfused_workspace_size(...) /
 *            fw_convt_unfused_workspace_size(...) bytes, 16-byte aligned, not
 *            overlapping any argument; contents undefined afterwards.
 * Only the shapes the tensor-core kernels take are supported (conv+pool: Cin = 8,
 * 3x3, pool_s = pool_k in {2, 4}, Cout in {16, 32, 48, 64}; convT: k = 4, s = 2,
 * p = 1, Cout = 128, Cin in {8, 16, 32, 64}); other valid arguments return
 * FW_ERR_UNSUPPORTED before any launch.  Two kernels per call (three for convT,
 * counting the weight rewrite).
 */
fw_status fw_conv2d_tanh_scale_bias_maxpool_unfused(const float *x, int N, int Cin, int H, int W,
                                                    const float *w, const float *conv_b, int Cout,
                                                    int KH, int KW, float scale, const float *bias,
                                                    int pool_k, int pool_s, float *out, void *workspace,
                                                    unsigned long long workspace_bytes, void *stream);
unsigned long long fw_conv2d_pool_unfused_workspace_size(int N, int H, int W, int Cout, int KH, int KW,
                                                         int pool_k, int pool_s);

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(const float *x, int N, int Cin, int H, int W,
                                                                const float *w, const float *conv_b,
                                                                int Cout, int k, int s, int p, int op,
                                                                const float *bias, float scale, float *out,
                                                                void *workspace,
                                                                unsigned long long workspace_bytes,
                                                                void *stream);
unsigned long long fw_convt_unfused_workspace_size(int N, int Cin, int H, int W, int Cout, int k, int s, int p,
                                                   int op);

/* ------------------------------------------------------------- diagnostics */

/*
 * Synchronise `stream`, then read and clear the device-side error words the
 * kernels set.  Returns FW_OK, FW_ERR_TIMEOUT (a bounded wait gave up),
 * FW_ERR_INTERNAL, or FW_ERR_LAUNCH if the synchronisation itself failed.
 */
fw_status fw_check_device_errors(void *stream);

/* Number of kernel launches this library has issued in this process (all
 * devices, all calls).  Used to count launches inside a timed region. */
unsigned long long fw_launch_count(void);

/* Diagnostic with no counterpart on the pages: launches one small kernel whose
 * mbarrier wait is never satisfied, so it gives up after limit_us microseconds
 * (1 .. 2,000,000), records a timeout in the device error word and returns --
 * the same bounded-wait path every kernel of the library takes if a stage never
 * arrives.  The next fw_check_device_errors() on that stream then returns
 * FW_ERR_TIMEOUT, and the CUDA context stays usable. */
fw_status fw_selftest_bounded_wait(unsigned int limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FUSEDWIN_H */
