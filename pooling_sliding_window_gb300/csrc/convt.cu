// convt.cu -- ConvTranspose2d -> softmax(dim=1) -> +bias -> *scale -> sigmoid
// (trace "Kimi-K2.6 l2_p91").
//
// Phase decomposition (the page's sub-pixel view): for k = 4, s = 2, p = 1 an
// output pixel (oh, ow) = (2m + py, 2n + px) receives exactly the taps
//   rows: py = 0 -> (kh = 1, ih = m), (kh = 3, ih = m - 1)
//         py = 1 -> (kh = 0, ih = m + 1), (kh = 2, ih = m)
// and the same for columns, so each of the 4 parity classes ("phases") is a
// dense 2x2 convolution: a GEMM with M = pixels of the phase, N = Cout and
// K = 4 * Cin.
//
// Tiled FFMA kernel (k4 s2 p1, Cout = 128):
//   * a prepack kernel rewrites the weight [Cin][Cout][4][4] into the caller's
//     workspace as wp[phase][ci][tap][co], so a CTA streams exactly the weights
//     of its phase with coalesced 16-byte loads;
//   * a CTA owns one phase of an 8 x 16 block of phase-grid pixels (128 output
//     pixels) of one image and all 128 channels; 256 threads, each 8 pixels
//     (one row, 8 consecutive n) x 8 channels ({4g..4g+3} and {64+4g..64+4g+3});
//   * Cin is streamed in chunks of 16: input rows m0-1..m0+8 are staged as three
//     column-shifted copies (dx = -1, 0, +1) so that every tap's 8-pixel row
//     segment is two aligned 16-byte shared loads;
//   * the 16 lanes of a half-warp hold all 128 channels of the same 8 pixels, so
//     the softmax max and sum are 4-step xor-shuffle reductions;
//   * results are transposed through shared memory and stored row by row.
// Direct kernel: one thread per output pixel, two passes over the channels
// (online max/sum, then the outputs), any (k, s, p, op) and Cout <= 1024.
#include <cstdlib>
#include <mutex>

#include "fw_common.cuh"

namespace fw {

// Range violations found by the checked build's kernels in this file.
__device__ unsigned g_err_convt = 0;
#define CHK(p, bytes, base, base_bytes) chk(&g_err_convt, (p), (bytes), (base), (base_bytes))
#define CHKS(p, bytes) chk_smem(&g_err_convt, (p), (bytes))

namespace {

constexpr int T_M = 8, T_N = 16;   // phase-grid pixels per CTA (rows, cols)
constexpr int CK = 16;             // input channels per chunk
constexpr int COUT_T = 128;        // channels of the tiled kernel
constexpr int XS_ROWS = T_M + 2;   // staged input rows m0-1 .. m0+T_M
constexpr int XS_CHUNK = XS_ROWS * 3 * T_N;  // floats per input channel in xs
constexpr int WS_CHUNK = 4 * COUT_T;          // floats per input channel in ws
constexpr int OS_PITCH = COUT_T + 1;          // output transpose pitch (conflict-free reads)

// Tap tables of the k4 s2 p1 phase decomposition: for output parity q and tap
// index t in {0, 1}: kernel index and input offset (ih = m + off).
__host__ __device__ __forceinline__ int tap_k(int q, int t) { return q == 0 ? (t == 0 ? 1 : 3) : (t == 0 ? 0 : 2); }
constexpr float LOG2E_F = 1.4426950408889634f;
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__host__ __device__ __forceinline__ int tap_off(int q, int t) { return q == 0 ? (t == 0 ? 0 : -1) : (t == 0 ? 1 : 0); }

__global__ void convt_prepack_kernel(const float *__restrict__ w, float *__restrict__ wp, int Cin,
                                     int Cout) {
    const long long total = 16LL * Cin * Cout;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int co = (int)(i % Cout);
        long long r = i / Cout;
        const int t = (int)(r % 4);
        r /= 4;
        const int ci = (int)(r % Cin);
        const int ph = (int)(r / Cin);
        const int py = ph >> 1, px = ph & 1;
        const int kh = tap_k(py, t >> 1), kw = tap_k(px, t & 1);
        const float *src = w + (((long long)ci * Cout + co) * 4 + kh) * 4 + kw;
        if (CHK(src, 4, w, 4 * total)) wp[i] = __ldg(src);
    }
}

__global__ void __launch_bounds__(256, 2)
convt_k4s2_ffma_kernel(const float *__restrict__ x, const float *__restrict__ wp,
                       const float *__restrict__ cb, const float *__restrict__ bias, float scale,
                       float *__restrict__ out, int Cin, int H, int W, int Ho, int Wo, int tiles_n) {
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                       // [CK][XS_ROWS][3][T_N]
    float *ws = sm + CK * XS_CHUNK;       // [CK][4][COUT_T]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane & 15, h = lane >> 4;
    const int phase = blockIdx.y, py = phase >> 1, px = phase & 1;
    const int n_img = blockIdx.z;
    const int tm = blockIdx.x / tiles_n, tn = blockIdx.x - tm * tiles_n;
    const int m0 = tm * T_M, n0 = tn * T_N;
    // This phase's grid: rows m with 2m + py < Ho, columns n with 2n + px < Wo.  The launch
    // covers phase 0's (the largest); a tile outside this phase's grid has nothing to do, and
    // a warp whose tile row lies outside it skips the products (its outputs are not stored).
    const int Mp = (Ho - py + 1) / 2, Np = (Wo - px + 1) / 2;
    if (m0 >= Mp || n0 >= Np) return;
    const bool row_live = m0 + warp < Mp;
    const float *xn = x + (long long)n_img * Cin * H * W;
    const float *wph = wp + (long long)phase * Cin * WS_CHUNK;
    // buffer extents for the checked build
    const long long x_bytes = 4LL * gridDim.z * Cin * H * W, wp_bytes = 16LL * 4 * Cin * COUT_T;
    const long long out_bytes = 4LL * gridDim.z * COUT_T * Ho * Wo;

    // shared-memory offset of each tap's 8-pixel row segment (loop-invariant)
    int xoff[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
        xoff[t] = ((warp + tap_off(py, t >> 1) + 1) * 3 + (tap_off(px, t & 1) + 1)) * T_N + 8 * h;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int c0 = 0; c0 < Cin; c0 += CK) {
        const int ck = min(CK, Cin - c0);
        __syncthreads();  // previous chunk fully consumed
        {
            // element e = ((ci * XS_ROWS + r) * 3 + sx) * T_N + c of the chunk; with 256 threads
            // and T_N = 16 a thread's column c stays fixed and each step adds 16 to
            // (ci, r, sx) in mixed radix (16 = 5 * 3 + 1), so no division per element
            static_assert(T_N == 16, "column per thread");
            const int c = tid % T_N;
            int t = tid / T_N, sx = t % 3, r = (t / 3) % XS_ROWS, ci = t / (3 * XS_ROWS);
            for (int e = tid; e < CK * XS_CHUNK; e += 256) {
                const int ih = m0 - 1 + r, iw = n0 + c + sx - 1;
                float v = 0.f;
                if (ci < ck && ih >= 0 && ih < H && iw >= 0 && iw < W) {
                    const float *src = xn + ((long long)(c0 + ci) * H + ih) * W + iw;
                    if (CHK(src, 4, x, x_bytes)) v = __ldg(src);
                }
                if (CHKS(xs + e, 4)) xs[e] = v;
                sx += 1;
                r += 5;
                if (sx >= 3) {
                    sx -= 3;
                    r += 1;
                }
                if (r >= XS_ROWS) {
                    r -= XS_ROWS;
                    ci += 1;
                }
            }
        }
        {
            const float4 *src = reinterpret_cast<const float4 *>(wph + (long long)c0 * WS_CHUNK);
            float4 *dst = reinterpret_cast<float4 *>(ws);
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = tid; e < CK * WS_CHUNK / 4; e += blockDim.x) {
                float4 v = z;
                if (e < ck * WS_CHUNK / 4 && CHK(src + e, 16, wp, wp_bytes)) v = __ldg(src + e);
                if (CHKS(dst + e, 16)) dst[e] = v;
            }
        }
        __syncthreads();
#pragma unroll 2
        for (int ci = 0; ci < (row_live ? ck : 0); ++ci) {
            const float *xc = xs + ci * XS_CHUNK, *wc = ws + ci * WS_CHUNK + 4 * g;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float *xr = xc + xoff[t];
                const float *wr = wc + t * COUT_T;
                if (!(CHKS(xr, 32) && CHKS(wr, 16) && CHKS(wr + 64, 16))) continue;
                const float4 xa = *reinterpret_cast<const float4 *>(xr);
                const float4 xb = *reinterpret_cast<const float4 *>(xr + 4);
                const float4 wa = *reinterpret_cast<const float4 *>(wr);
                const float4 wb = *reinterpret_cast<const float4 *>(wr + 64);
                const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
            }
        }
    }

    // Epilogue: conv bias, softmax over the 128 channels (16 lanes x 8), then
    // +bias, *scale, sigmoid.
    float cbv[8], bv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int co = (j < 4 ? 4 * g + j : 64 + 4 * g + (j - 4));
        cbv[j] = cb ? __ldg(cb + co) : 0.f;
        bv[j] = __ldg(bias + co);
    }
    // Exponentials in base 2 (ex2.approx, relative error ~2^-22) on log2(e)-scaled
    // arguments and one reciprocal of the sum per pixel, as in the tensor-core kernel's
    // epilogue; with float32 products and sums the result stays within 1e-5.
    const float ks = -scale * LOG2E_F;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[i][j] += cbv[j];
            mx = fmaxf(mx, acc[i][j]);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[i][j] = ex2_fast((acc[i][j] - mx) * LOG2E_F);
            sum += acc[i][j];
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float kp = ks / sum;  // 2^(-(p + b) * scale * log2 e) = 2^(e * kp - b * scale * log2 e)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[i][j] = __fdividef(1.f, 1.f + ex2_fast(fmaf(acc[i][j], kp, bv[j] * ks)));
    }

    // Transpose through shared memory, pixel-major with an odd pitch:
    // os[(m_local * T_N + n_local) * OS_PITCH + co].
    __syncthreads();
    float *os = sm;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int co = (j < 4 ? 4 * g + j : 64 + 4 * g + (j - 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float *d = os + (warp * T_N + 8 * h + i) * OS_PITCH + co;
            if (CHKS(d, 4)) *d = acc[i][j];
        }
    }
    __syncthreads();
    float *on = out + (long long)n_img * COUT_T * Ho * Wo;
    for (int e = tid; e < COUT_T * T_M * T_N; e += blockDim.x) {
        const int nl = e % T_N, ml = (e / T_N) % T_M, co = e / (T_N * T_M);
        const int oh = 2 * (m0 + ml) + py, ow = 2 * (n0 + nl) + px;
        float *d = on + ((long long)co * Ho + oh) * Wo + ow;
        const float *sv = os + (ml * T_N + nl) * OS_PITCH + co;
        if (oh < Ho && ow < Wo && CHK(d, 4, out, out_bytes) && CHKS(sv, 4)) *d = *sv;
    }
}

// Gather form of one conv-transpose output (x_bytes, w_bytes: buffer extents for the
// checked build; xn is image n's part of x).
__device__ __forceinline__ float convt_gather(const float *__restrict__ x, long long x_bytes,
                                              const float *__restrict__ xn, const float *__restrict__ w,
                                              float cbv, int Cin, int H, int W, int Cout, int k, int s,
                                              int p, int co, int oh, int ow) {
    const long long w_bytes = 4LL * Cin * Cout * k * k;
    float y = cbv;
    for (int kh = 0; kh < k; ++kh) {
        const int th = oh + p - kh;
        if (th < 0 || th % s) continue;
        const int ih = th / s;
        if (ih >= H) continue;
        for (int kw = 0; kw < k; ++kw) {
            const int tw = ow + p - kw;
            if (tw < 0 || tw % s) continue;
            const int iw = tw / s;
            if (iw >= W) continue;
            for (int ci = 0; ci < Cin; ++ci) {
                const float *xa = xn + ((long long)ci * H + ih) * W + iw;
                const float *wa = w + (((long long)ci * Cout + co) * k + kh) * k + kw;
                if (CHK(xa, 4, x, x_bytes) && CHK(wa, 4, w, w_bytes)) y = fmaf(__ldg(xa), __ldg(wa), y);
            }
        }
    }
    return y;
}

__global__ void convt_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                    const float *__restrict__ cb, const float *__restrict__ bias,
                                    float scale, float *__restrict__ out, int N, int Cin, int H, int W,
                                    int Cout, int k, int s, int p, int Ho, int Wo) {
    const long long total = (long long)N * Ho * Wo;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(idx % Wo);
        const long long t = idx / Wo;
        const int oh = (int)(t % Ho);
        const int n = (int)(t / Ho);
        const float *xn = x + (long long)n * Cin * H * W;
        const long long x_bytes = 4LL * N * Cin * H * W;
        float mx = -INFINITY, sum = 0.f;
        for (int co = 0; co < Cout; ++co) {
            const float y = convt_gather(x, x_bytes, xn, w, cb ? __ldg(cb + co) : 0.f, Cin, H, W, Cout, k, s, p, co,
                                         oh, ow);
            if (y > mx) {
                sum = sum * expf(mx - y) + 1.f;
                mx = y;
            } else {
                sum += expf(y - mx);
            }
        }
        for (int co = 0; co < Cout; ++co) {
            const float y = convt_gather(x, x_bytes, xn, w, cb ? __ldg(cb + co) : 0.f, Cin, H, W, Cout, k, s, p, co,
                                         oh, ow);
            const float pr = __fdiv_rn(expf(y - mx), sum);
            const float r = __fmul_rn(__fadd_rn(pr, __ldg(bias + co)), scale);
            float *d = out + (((long long)n * Cout + co) * Ho + oh) * Wo + ow;
            if (CHK(d, 4, out, 4LL * N * Cout * Ho * Wo)) *d = __fdiv_rn(1.f, 1.f + expf(-r));
        }
    }
}

// FUSEDWIN_CONVT_FFMA=1 in the environment selects the FP32-FMA tiled kernel
// instead of the tensor-core one (used to cross-check the two).
bool force_ffma() {
    static const bool v = [] {
        const char *e = getenv("FUSEDWIN_CONVT_FFMA");
        return e && e[0] == '1';
    }();
    return v;
}

}  // namespace

bool convt_tc_eligible(int Cin, int Cout, int k, int s, int p);
fw_status convt_tc_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                          const float *bias, float scale, float *out, int Ho, int Wo, void *ws, cudaStream_t st,
                          bool prepack);

size_t convt_workspace_bytes(int Cin, int Cout, int k, int s, int p) {
    if (k == 4 && s == 2 && p == 1 && Cout == COUT_T) return (size_t)16 * Cin * Cout * sizeof(float);
    return 0;
}

// ffma = true keeps the call on the FP32-FMA kernels (tiled, else direct).
// weights_ready = true: the workspace already holds the weight rewrite of these
// arguments (written by an earlier call on the same stream), so it is not redone.
fw_status convt_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                       int Cout, int k, int s, int p, int op, const float *bias, float scale, float *out,
                       int Ho, int Wo, void *ws, size_t ws_bytes, bool ffma, bool weights_ready, cudaStream_t st) {
    const size_t need = convt_workspace_bytes(Cin, Cout, k, s, p);
    if (need > 0) {
        if (!ws || ws_bytes < need) return FW_ERR_NULL;
        if (!ffma && convt_tc_eligible(Cin, Cout, k, s, p) && !force_ffma())
            return convt_tc_launch(x, N, Cin, H, W, w, cb, bias, scale, out, Ho, Wo, ws, st, !weights_ready);
        float *wp = static_cast<float *>(ws);
        if (!weights_ready) {
            convt_prepack_kernel<<<(unsigned)min(1024LL, (16LL * Cin * Cout + 255) / 256), 256, 0, st>>>(w, wp, Cin,
                                                                                                         Cout);
            note_launch();
            const fw_status rc = launch_status(cudaGetLastError());
            if (rc != FW_OK) return rc;
        }
        const int Mp = (Ho + 1) / 2, Np = (Wo + 1) / 2;  // phase-grid extent (phase 0)
        const int tiles_m = (Mp + T_M - 1) / T_M, tiles_n = (Np + T_N - 1) / T_N;
        const size_t smem = (size_t)CK * (XS_CHUNK + WS_CHUNK) * sizeof(float);
        const size_t smem_out = (size_t)OS_PITCH * T_M * T_N * sizeof(float);
        const size_t smem_all = smem > smem_out ? smem : smem_out;
        cudaError_t e = cudaFuncSetAttribute(convt_k4s2_ffma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_all);
        if (e != cudaSuccess) return launch_status(e);
        if (N > 65535) return FW_ERR_UNSUPPORTED;
        dim3 grid(tiles_m * tiles_n, 4, N);
        convt_k4s2_ffma_kernel<<<grid, 256, smem_all, st>>>(x, wp, cb, bias, scale, out, Cin, H, W, Ho, Wo,
                                                            tiles_n);
        note_launch();
        return launch_status(cudaGetLastError());
    }
    (void)op;
    const long long total = (long long)N * Ho * Wo;
    const int threads = 128;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    convt_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(x, w, cb, bias, scale, out, N, Cin, H, W, Cout,
                                                              k, s, p, Ho, Wo);
    note_launch();
    return launch_status(cudaGetLastError());
}

unsigned convt_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convt, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convt, &zero, sizeof(zero));
    return v;
}

}  // namespace fw

// ---------------------------------------------------------------------------
// Allocation-free variant of the conv-transpose call.
//
// Some callers cannot call cudaMalloc (or any allocator): plugins that a host
// framework hands only input and output buffers because it owns all device
// memory, real-time loops that may not allocate after start-up, and code where
// an allocation would implicitly synchronise the device.  For them the weight
// rewrite that the tiled kernel needs goes into this fixed array instead of a
// caller workspace.  Every device that loads the library holds it until the
// process exits.
// ---------------------------------------------------------------------------
namespace fw {

static __device__ __align__(256) unsigned char g_convt_static_ws[FW_CONVT_STATIC_WS_BYTES];

namespace {
std::mutex g_static_ws_mu;
void *g_static_ws_ptr[FW_MAX_DEVICES] = {};
}  // namespace

// Device address of g_convt_static_ws on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with cudaGetSymbolAddress (with that device current) and cached.
static fw_status convt_static_workspace(void **ptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FW_ERR_LAUNCH;
    if (dev < 0 || dev >= FW_MAX_DEVICES) return FW_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_ws_mu);
    if (!g_static_ws_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_convt_static_ws) != cudaSuccess || !p) return FW_ERR_LAUNCH;
        g_static_ws_ptr[dev] = p;
    }
    *ptr = g_static_ws_ptr[dev];
    return FW_OK;
}

}  // namespace fw

extern "C" fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_noalloc(
    const float *x, int N, int Cin, int H, int W, const float *w, const float *conv_b, int Cout, int k, int s,
    int p, int op, const float *bias, float scale, float *out, void *stream) {
    const unsigned long long need = fw_convt_workspace_size(Cin, Cout, k, s, p);
    if (need > FW_CONVT_STATIC_WS_BYTES) return FW_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (need > 0) {
        const fw_status rc = fw::convt_static_workspace(&ws);
        if (rc != FW_OK) return rc;
    }
    return fw_convtranspose2d_softmax_bias_scale_sigmoid(x, N, Cin, H, W, w, conv_b, Cout, k, s, p, op, bias,
                                                         scale, out, ws, need > 0 ? FW_CONVT_STATIC_WS_BYTES : 0,
                                                         stream);
}
