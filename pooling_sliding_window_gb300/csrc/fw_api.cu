// fw_api.cu -- the extern "C" entry points of libfusedwin: argument checks on the
// host, then dispatch to the kernels of maxpool.cu, convpool.cu and convt.cu.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "fw_common.cuh"

namespace fw {

fw_status maxpool2d_launch(const float *x, long long NC, int H, int W, int k, int s, int p, int d, int Ho,
                           int Wo, float *out, cudaStream_t st);
fw_status maxpool2d_ex_launch(const float *x, long long NC, int H, int W, int k, int s, int p, int d, int Ho,
                              int Wo, float *out, long long *idx, cudaStream_t st);
fw_status maxpool2d_nhwc_launch(const float *x, int N, int H, int W, int C, int k, int s, int p, int d, int Ho,
                                int Wo, float *out, cudaStream_t st);
unsigned maxpool_read_and_clear_error();
unsigned convt_tc_read_and_clear_error();
unsigned convpool_tc_read_and_clear_error();
unsigned convt_read_and_clear_error();
unsigned convpool_read_and_clear_error();
fw_status convpool_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                          int Cout, int KH, int KW, float scale, const float *bias, int pk, int ps,
                          float *out, int Ho, int Wo, int mode, cudaStream_t st);
fw_status convt_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                       int Cout, int k, int s, int p, int op, const float *bias, float scale, float *out,
                       int Ho, int Wo, void *ws, size_t ws_bytes, bool ffma, bool weights_ready, cudaStream_t st);
size_t convt_workspace_bytes(int Cin, int Cout, int k, int s, int p);
bool convpool_tc_eligible(int Cin, int Cout, int KH, int KW, int pk, int ps);
fw_status convpool_tc_launch_raw(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                                 int pk, float *y, int Ho, int Wo, cudaStream_t st);
fw_status pool_tanh_scale_bias_launch(const float *y, int N, int Cout, const float *bias, float scale, int pk,
                                      float *out, int Ho, int Wo, cudaStream_t st);
bool convt_tc_eligible(int Cin, int Cout, int k, int s, int p);
fw_status convt_tc_launch_raw(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                              float *y, int Ho, int Wo, void *ws, cudaStream_t st);
fw_status softmax_bias_scale_sigmoid_launch(const float *y, int N, int C, int Ho, int Wo, const float *bias,
                                            float scale, float *out, cudaStream_t st);
fw_status convpool_tc_launch_nhwc(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                                  float scale, const float *bias, int pk, float *out, int Ho, int Wo,
                                  cudaStream_t st);
fw_status convt_tc_launch_nhwc(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                               const float *bias, float scale, float *out, int Ho, int Wo, void *ws, cudaStream_t st);

static std::atomic<unsigned long long> g_launches{0};

__device__ unsigned g_err_api = 0;

// Waits on an mbarrier that nothing ever completes; the bounded wait runs out
// after limit_ns and records a timeout in the error word -- the path every
// kernel's waits take when a producer never arrives.
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicOr(&g_err_api, DEVERR_TIMEOUT);
}

unsigned api_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_api, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_api, &zero, sizeof(zero));
    return v;
}

void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

fw_status launch_status(cudaError_t e) { return e == cudaSuccess ? FW_OK : FW_ERR_LAUNCH; }

namespace {

constexpr long long MAX_ELEMS = 1LL << 62;

long long floordiv(long long a, long long b) {
    long long q = a / b;
    if ((a % b != 0) && (a < 0)) --q;
    return q;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) intersect.
bool overlaps(const void *a, long long na, const void *b, long long nb) {
    if (!a || !b || na <= 0 || nb <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)nb && b0 < a0 + (uintptr_t)na;
}

// Product of non-negative sizes, or -1 if it exceeds MAX_ELEMS.
long long prod(std::initializer_list<long long> v) {
    long long r = 1;
    for (long long a : v) {
        if (a < 0) return -1;
        if (a != 0 && r > MAX_ELEMS / a) return -1;
        r *= a;
    }
    return r;
}

fw_status conv_pool_shape(int H, int W, int KH, int KW, int pk, int ps, int *Ho, int *Wo) {
    if (H < 1 || W < 1) return FW_ERR_SHAPE;
    if (KH < 1 || KW < 1 || pk < 1) return FW_ERR_PARAM;
    if (ps <= 0) ps = pk;
    const long long Hc = (long long)H - KH + 1, Wc = (long long)W - KW + 1;
    if (Hc < pk || Wc < pk) return FW_ERR_SHAPE;
    *Ho = (int)((Hc - pk) / ps + 1);
    *Wo = (int)((Wc - pk) / ps + 1);
    return FW_OK;
}

fw_status maxpool_shape(int H, int W, int k, int s, int p, int d, int *Ho, int *Wo) {
    if (H < 1 || W < 1) return FW_ERR_SHAPE;
    if (k < 1 || s < 1 || p < 0 || d < 1) return FW_ERR_PARAM;
    const long long span = (long long)d * (k - 1) + 1;
    const long long ho = floordiv((long long)H + 2LL * p - span, s) + 1;
    const long long wo = floordiv((long long)W + 2LL * p - span, s) + 1;
    if (ho < 1 || wo < 1 || ho > 0x7fffffffLL || wo > 0x7fffffffLL) return FW_ERR_SHAPE;
    *Ho = (int)ho;
    *Wo = (int)wo;
    return FW_OK;
}

// One dimension in ceil mode (PyTorch's MaxPool2d option, not on the pages): the
// size rounds up, and a last window that would start in the right padding is dropped.
long long pool_dim_ceil(long long H, int k, int s, int p, int d) {
    const long long span = H + 2LL * p - (long long)d * (k - 1) - 1;
    long long o = -floordiv(-span, s) + 1;
    if (o >= 1 && (o - 1) * s >= H + p) --o;
    return o;
}

fw_status maxpool_shape_ex(int H, int W, int k, int s, int p, int d, int ceil_mode, int *Ho, int *Wo) {
    if (!ceil_mode) return maxpool_shape(H, W, k, s, p, d, Ho, Wo);
    if (H < 1 || W < 1) return FW_ERR_SHAPE;
    if (k < 1 || s < 1 || p < 0 || d < 1) return FW_ERR_PARAM;
    const long long ho = pool_dim_ceil(H, k, s, p, d), wo = pool_dim_ceil(W, k, s, p, d);
    if (ho < 1 || wo < 1 || ho > 0x7fffffffLL || wo > 0x7fffffffLL) return FW_ERR_SHAPE;
    *Ho = (int)ho;
    *Wo = (int)wo;
    return FW_OK;
}

fw_status convt_shape(int H, int W, int k, int s, int p, int op, int *Ho, int *Wo) {
    if (H < 1 || W < 1) return FW_ERR_SHAPE;
    if (k < 1 || s < 1 || p < 0 || op < 0 || op >= s) return FW_ERR_PARAM;
    const long long ho = ((long long)H - 1) * s - 2LL * p + (k - 1) + op + 1;
    const long long wo = ((long long)W - 1) * s - 2LL * p + (k - 1) + op + 1;
    if (ho < 1 || wo < 1 || ho > 0x7fffffffLL || wo > 0x7fffffffLL) return FW_ERR_SHAPE;
    *Ho = (int)ho;
    *Wo = (int)wo;
    return FW_OK;
}

}  // namespace
}  // namespace fw

using namespace fw;

extern "C" {

const char *fw_status_string(fw_status s) {
    switch (s) {
        case FW_OK: return "FW_OK";
        case FW_ERR_NULL: return "FW_ERR_NULL: a required pointer is NULL";
        case FW_ERR_SHAPE: return "FW_ERR_SHAPE: a size is < 1, the output would be empty, or too large";
        case FW_ERR_PARAM: return "FW_ERR_PARAM: kernel/stride/padding/dilation/output_padding out of range or non-finite scale";
        case FW_ERR_ALIAS: return "FW_ERR_ALIAS: out overlaps an input";
        case FW_ERR_ALIGN: return "FW_ERR_ALIGN: a tensor pointer is misaligned";
        case FW_ERR_UNSUPPORTED: return "FW_ERR_UNSUPPORTED: valid arguments not implemented";
        case FW_ERR_LAUNCH: return "FW_ERR_LAUNCH: a CUDA call failed";
        case FW_ERR_TIMEOUT: return "FW_ERR_TIMEOUT: a bounded wait in a kernel gave up";
        case FW_ERR_INTERNAL: return "FW_ERR_INTERNAL: a kernel reported an inconsistency";
    }
    return "FW_ERR_?: unknown status";
}

int fw_version(void) { return 100; }

unsigned long long fw_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

fw_status fw_conv2d_pool_out_shape(int H, int W, int KH, int KW, int pool_k, int pool_s, int *Ho, int *Wo) {
    if (!Ho || !Wo) return FW_ERR_NULL;
    return conv_pool_shape(H, W, KH, KW, pool_k, pool_s, Ho, Wo);
}

fw_status fw_maxpool2d_out_shape(int H, int W, int k, int s, int p, int d, int *Ho, int *Wo) {
    if (!Ho || !Wo) return FW_ERR_NULL;
    return maxpool_shape(H, W, k, s, p, d, Ho, Wo);
}

fw_status fw_maxpool2d_out_shape_ex(int H, int W, int k, int s, int p, int d, int ceil_mode, int *Ho, int *Wo) {
    if (!Ho || !Wo) return FW_ERR_NULL;
    return maxpool_shape_ex(H, W, k, s, p, d, ceil_mode, Ho, Wo);
}

fw_status fw_convt_out_shape(int H, int W, int k, int s, int p, int op, int *Ho, int *Wo) {
    if (!Ho || !Wo) return FW_ERR_NULL;
    return convt_shape(H, W, k, s, p, op, Ho, Wo);
}

unsigned long long fw_convt_workspace_size(int Cin, int Cout, int k, int s, int p) {
    if (Cin < 1 || Cout < 1) return 0;
    return (unsigned long long)convt_workspace_bytes(Cin, Cout, k, s, p);
}

static fw_status conv_pool_call(const float *x, int N, int Cin, int H, int W, const float *w, const float *conv_b,
                                int Cout, int KH, int KW, float scale, const float *bias, int pool_k, int pool_s,
                                float *out, int mode, void *stream) {
    if (!x || !w || !bias || !out) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = conv_pool_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (pool_s <= 0) pool_s = pool_k;
    if (misaligned(x) || misaligned(w) || misaligned(conv_b) || misaligned(bias) || misaligned(out))
        return FW_ERR_ALIGN;
    const long long nx = prod({N, Cin, H, W}), nw = prod({Cout, Cin, KH, KW}), no = prod({N, Cout, Ho, Wo});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const long long ob = no * 4;
    if (overlaps(out, ob, x, nx * 4) || overlaps(out, ob, w, nw * 4) || overlaps(out, ob, bias, 4LL * Cout) ||
        overlaps(out, ob, conv_b, 4LL * Cout))
        return FW_ERR_ALIAS;
    return convpool_launch(x, N, Cin, H, W, w, conv_b, Cout, KH, KW, scale, bias, pool_k, pool_s, out, Ho, Wo,
                           mode, static_cast<cudaStream_t>(stream));
}

fw_status fw_conv2d_tanh_scale_bias_maxpool(const float *x, int N, int Cin, int H, int W, const float *w,
                                            const float *conv_b, int Cout, int KH, int KW, float scale,
                                            const float *bias, int pool_k, int pool_s, float *out,
                                            void *stream) {
    return conv_pool_call(x, N, Cin, H, W, w, conv_b, Cout, KH, KW, scale, bias, pool_k, pool_s, out, 0, stream);
}

fw_status fw_conv2d_tanh_scale_bias_maxpool_tf32(const float *x, int N, int Cin, int H, int W, const float *w,
                                                 const float *conv_b, int Cout, int KH, int KW, float scale,
                                                 const float *bias, int pool_k, int pool_s, float *out,
                                                 void *stream) {
    return conv_pool_call(x, N, Cin, H, W, w, conv_b, Cout, KH, KW, scale, bias, pool_k, pool_s, out, 1, stream);
}

fw_status fw_conv2d_tanh_scale_bias_maxpool_ffma(const float *x, int N, int Cin, int H, int W, const float *w,
                                                 const float *conv_b, int Cout, int KH, int KW, float scale,
                                                 const float *bias, int pool_k, int pool_s, float *out,
                                                 void *stream) {
    return conv_pool_call(x, N, Cin, H, W, w, conv_b, Cout, KH, KW, scale, bias, pool_k, pool_s, out, 2, stream);
}

fw_status fw_maxpool2d(const float *x, int N, int C, int H, int W, int k, int s, int p, int d, float *out,
                       void *stream) {
    if (!x || !out) return FW_ERR_NULL;
    if (N < 1 || C < 1) return FW_ERR_SHAPE;
    int Ho = 0, Wo = 0;
    fw_status rc = maxpool_shape(H, W, k, s, p, d, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(x) || misaligned(out)) return FW_ERR_ALIGN;
    const long long nx = prod({N, C, H, W}), no = prod({N, C, Ho, Wo});
    if (nx < 0 || no < 0) return FW_ERR_SHAPE;
    if (overlaps(out, no * 4, x, nx * 4)) return FW_ERR_ALIAS;
    return maxpool2d_launch(x, (long long)N * C, H, W, k, s, p, d, Ho, Wo, out,
                            static_cast<cudaStream_t>(stream));
}

fw_status fw_maxpool2d_nhwc(const float *x, int N, int H, int W, int C, int k, int s, int p, int d, float *out,
                            void *stream) {
    if (!x || !out) return FW_ERR_NULL;
    if (N < 1 || C < 1) return FW_ERR_SHAPE;
    int Ho = 0, Wo = 0;
    fw_status rc = maxpool_shape(H, W, k, s, p, d, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(x) || misaligned(out)) return FW_ERR_ALIGN;
    const long long nx = prod({N, H, W, C}), no = prod({N, Ho, Wo, C});
    if (nx < 0 || no < 0) return FW_ERR_SHAPE;
    if (overlaps(out, no * 4, x, nx * 4)) return FW_ERR_ALIAS;
    return maxpool2d_nhwc_launch(x, N, H, W, C, k, s, p, d, Ho, Wo, out, static_cast<cudaStream_t>(stream));
}

fw_status fw_maxpool2d_ex(const float *x, int N, int C, int H, int W, int k, int s, int p, int d, int ceil_mode,
                          float *out, long long *indices, void *stream) {
    if (!x || !out) return FW_ERR_NULL;
    if (N < 1 || C < 1) return FW_ERR_SHAPE;
    int Ho = 0, Wo = 0;
    fw_status rc = maxpool_shape_ex(H, W, k, s, p, d, ceil_mode, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(x) || misaligned(out) || (reinterpret_cast<uintptr_t>(indices) & 7u) != 0) return FW_ERR_ALIGN;
    const long long nx = prod({N, C, H, W}), no = prod({N, C, Ho, Wo});
    if (nx < 0 || no < 0) return FW_ERR_SHAPE;
    if (overlaps(out, no * 4, x, nx * 4) || overlaps(indices, no * 8, x, nx * 4) ||
        overlaps(indices, no * 8, out, no * 4))
        return FW_ERR_ALIAS;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int fHo = 0, fWo = 0;
    if (!indices && maxpool_shape(H, W, k, s, p, d, &fHo, &fWo) == FW_OK && fHo == Ho && fWo == Wo)
        return maxpool2d_launch(x, (long long)N * C, H, W, k, s, p, d, Ho, Wo, out, st);  // same as floor mode
    return maxpool2d_ex_launch(x, (long long)N * C, H, W, k, s, p, d, Ho, Wo, out, indices, st);
}

}  // extern "C"

// The conv-transpose entry points' checks and dispatch.  weights_ready: see
// convt_launch (the host-buffer call sets it for every chunk after the first).
fw_status fw::convt_call(const float *x, int N, int Cin, int H, int W, const float *w, const float *conv_b,
                         int Cout, int k, int s, int p, int op, const float *bias, float scale, float *out,
                         void *workspace, unsigned long long workspace_bytes, bool ffma, bool weights_ready,
                         void *stream) {
    if (!x || !w || !bias || !out) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (Cout > 1024) return FW_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = convt_shape(H, W, k, s, p, op, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(x) || misaligned(w) || misaligned(conv_b) || misaligned(bias) || misaligned(out))
        return FW_ERR_ALIGN;
    const long long nx = prod({N, Cin, H, W}), nw = prod({Cin, Cout, k, k}), no = prod({N, Cout, Ho, Wo});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const unsigned long long need = convt_workspace_bytes(Cin, Cout, k, s, p);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FW_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FW_ERR_ALIGN;
    }
    const long long ob = no * 4;
    if (overlaps(out, ob, x, nx * 4) || overlaps(out, ob, w, nw * 4) || overlaps(out, ob, bias, 4LL * Cout) ||
        overlaps(out, ob, conv_b, 4LL * Cout) || (need && overlaps(out, ob, workspace, (long long)need)))
        return FW_ERR_ALIAS;
    // The weight rewrite into the workspace runs before the main kernel reads any input.
    if (need && (overlaps(workspace, (long long)need, x, nx * 4) || overlaps(workspace, (long long)need, w, nw * 4) ||
                 overlaps(workspace, (long long)need, bias, 4LL * Cout) ||
                 overlaps(workspace, (long long)need, conv_b, 4LL * Cout)))
        return FW_ERR_ALIAS;
    return convt_launch(x, N, Cin, H, W, w, conv_b, Cout, k, s, p, op, bias, scale, out, Ho, Wo, workspace,
                        (size_t)workspace_bytes, ffma, weights_ready, static_cast<cudaStream_t>(stream));
}

extern "C" {

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid(const float *x, int N, int Cin, int H, int W,
                                                        const float *w, const float *conv_b, int Cout,
                                                        int k, int s, int p, int op, const float *bias,
                                                        float scale, float *out, void *workspace,
                                                        unsigned long long workspace_bytes, void *stream) {
    return convt_call(x, N, Cin, H, W, w, conv_b, Cout, k, s, p, op, bias, scale, out, workspace, workspace_bytes,
                      false, false, stream);
}

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_ffma(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b, int Cout,
                                                             int k, int s, int p, int op, const float *bias,
                                                             float scale, float *out, void *workspace,
                                                             unsigned long long workspace_bytes, void *stream) {
    return convt_call(x, N, Cin, H, W, w, conv_b, Cout, k, s, p, op, bias, scale, out, workspace, workspace_bytes,
                      true, false, stream);
}

unsigned long long fw_conv2d_pool_unfused_workspace_size(int N, int H, int W, int Cout, int KH, int KW,
                                                         int pool_k, int pool_s) {
    int Ho = 0, Wo = 0;
    if (N < 1 || Cout < 1 || conv_pool_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo) != FW_OK) return 0;
    const long long n = prod({N, Cout, (long long)pool_k * Ho, (long long)pool_k * Wo});
    return n < 0 ? 0 : 4ULL * (unsigned long long)n;
}

fw_status fw_conv2d_tanh_scale_bias_maxpool_unfused(const float *x, int N, int Cin, int H, int W, const float *w,
                                                    const float *conv_b, int Cout, int KH, int KW, float scale,
                                                    const float *bias, int pool_k, int pool_s, float *out,
                                                    void *workspace, unsigned long long workspace_bytes,
                                                    void *stream) {
    if (!x || !w || !bias || !out || !workspace) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = conv_pool_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (pool_s <= 0) pool_s = pool_k;
    if (misaligned(x) || misaligned(w) || misaligned(conv_b) || misaligned(bias) || misaligned(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return FW_ERR_ALIGN;
    const long long nx = prod({N, Cin, H, W}), nw = prod({Cout, Cin, KH, KW}), no = prod({N, Cout, Ho, Wo});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const unsigned long long need = fw_conv2d_pool_unfused_workspace_size(N, H, W, Cout, KH, KW, pool_k, pool_s);
    if (need == 0) return FW_ERR_SHAPE;
    if (workspace_bytes < need) return FW_ERR_NULL;
    if (!convpool_tc_eligible(Cin, Cout, KH, KW, pool_k, pool_s)) return FW_ERR_UNSUPPORTED;
    const long long ob = no * 4, wb = (long long)need;
    const void *ins[] = {x, w, bias, conv_b};
    const long long insz[] = {nx * 4, nw * 4, 4LL * Cout, 4LL * Cout};
    for (int i = 0; i < 4; ++i)
        if (overlaps(out, ob, ins[i], insz[i]) || overlaps(workspace, wb, ins[i], insz[i])) return FW_ERR_ALIAS;
    if (overlaps(out, ob, workspace, wb)) return FW_ERR_ALIAS;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *y = static_cast<float *>(workspace);
    rc = convpool_tc_launch_raw(x, N, H, W, w, conv_b, Cout, pool_k, y, Ho, Wo, st);
    if (rc != FW_OK) return rc;
    return pool_tanh_scale_bias_launch(y, N, Cout, bias, scale, pool_k, out, Ho, Wo, st);
}

// Workspace of the unfused conv-transpose: the weight rewrite, padded to 256 bytes,
// then the intermediate.
static unsigned long long convt_unfused_weights_bytes(int Cin, int Cout, int k, int s, int p) {
    return ((unsigned long long)convt_workspace_bytes(Cin, Cout, k, s, p) + 255ULL) & ~255ULL;
}

unsigned long long fw_convt_unfused_workspace_size(int N, int Cin, int H, int W, int Cout, int k, int s, int p,
                                                   int op) {
    int Ho = 0, Wo = 0;
    if (N < 1 || Cin < 1 || Cout < 1 || convt_shape(H, W, k, s, p, op, &Ho, &Wo) != FW_OK) return 0;
    const long long n = prod({N, Cout, Ho, Wo});
    return n < 0 ? 0 : convt_unfused_weights_bytes(Cin, Cout, k, s, p) + 4ULL * (unsigned long long)n;
}

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_unfused(const float *x, int N, int Cin, int H, int W,
                                                                const float *w, const float *conv_b, int Cout,
                                                                int k, int s, int p, int op, const float *bias,
                                                                float scale, float *out, void *workspace,
                                                                unsigned long long workspace_bytes,
                                                                void *stream) {
    if (!x || !w || !bias || !out || !workspace) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = convt_shape(H, W, k, s, p, op, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(x) || misaligned(w) || misaligned(conv_b) || misaligned(bias) || misaligned(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return FW_ERR_ALIGN;
    const long long nx = prod({N, Cin, H, W}), nw = prod({Cin, Cout, k, k}), no = prod({N, Cout, Ho, Wo});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const unsigned long long need = fw_convt_unfused_workspace_size(N, Cin, H, W, Cout, k, s, p, op);
    if (need == 0) return FW_ERR_SHAPE;
    if (workspace_bytes < need) return FW_ERR_NULL;
    if (!convt_tc_eligible(Cin, Cout, k, s, p)) return FW_ERR_UNSUPPORTED;
    const long long ob = no * 4, wb = (long long)need;
    const void *ins[] = {x, w, bias, conv_b};
    const long long insz[] = {nx * 4, nw * 4, 4LL * Cout, 4LL * Cout};
    for (int i = 0; i < 4; ++i)
        if (overlaps(out, ob, ins[i], insz[i]) || overlaps(workspace, wb, ins[i], insz[i])) return FW_ERR_ALIAS;
    if (overlaps(out, ob, workspace, wb)) return FW_ERR_ALIAS;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    float *y = reinterpret_cast<float *>(ws + convt_unfused_weights_bytes(Cin, Cout, k, s, p));
    rc = convt_tc_launch_raw(x, N, Cin, H, W, w, conv_b, y, Ho, Wo, ws, st);
    if (rc != FW_OK) return rc;
    return softmax_bias_scale_sigmoid_launch(y, N, Cout, Ho, Wo, bias, scale, out, st);
}

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_nhwc(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b, int Cout, int k,
                                                             int s, int p, int op, const float *bias, float scale,
                                                             float *out, void *workspace,
                                                             unsigned long long workspace_bytes, void *stream) {
    if (!x || !w || !bias || !out) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = convt_shape(H, W, k, s, p, op, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (misaligned(w) || misaligned(conv_b) || misaligned(bias) || (reinterpret_cast<uintptr_t>(x) & 15u) != 0 ||
        (reinterpret_cast<uintptr_t>(out) & 31u) != 0)
        return FW_ERR_ALIGN;
    if (!convt_tc_eligible(Cin, Cout, k, s, p)) return FW_ERR_UNSUPPORTED;
    const long long nx = prod({N, H, W, Cin}), nw = prod({Cin, Cout, k, k}), no = prod({N, Ho, Wo, Cout});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const unsigned long long need = convt_workspace_bytes(Cin, Cout, k, s, p);
    if (!workspace || workspace_bytes < need) return FW_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FW_ERR_ALIGN;
    const long long ob = no * 4, wb = (long long)need;
    const void *ins[] = {x, w, bias, conv_b};
    const long long insz[] = {nx * 4, nw * 4, 4LL * Cout, 4LL * Cout};
    for (int i = 0; i < 4; ++i)
        if (overlaps(out, ob, ins[i], insz[i]) || overlaps(workspace, wb, ins[i], insz[i])) return FW_ERR_ALIAS;
    if (overlaps(out, ob, workspace, wb)) return FW_ERR_ALIAS;
    return convt_tc_launch_nhwc(x, N, Cin, H, W, w, conv_b, bias, scale, out, Ho, Wo, workspace,
                                static_cast<cudaStream_t>(stream));
}

fw_status fw_conv2d_tanh_scale_bias_maxpool_nhwc(const float *x, int N, int Cin, int H, int W, const float *w,
                                                 const float *conv_b, int Cout, int KH, int KW, float scale,
                                                 const float *bias, int pool_k, int pool_s, float *out,
                                                 void *stream) {
    if (!x || !w || !bias || !out) return FW_ERR_NULL;
    if (N < 1 || Cin < 1 || Cout < 1) return FW_ERR_SHAPE;
    if (!std::isfinite(scale)) return FW_ERR_PARAM;
    int Ho = 0, Wo = 0;
    fw_status rc = conv_pool_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo);
    if (rc != FW_OK) return rc;
    if (pool_s <= 0) pool_s = pool_k;
    if (misaligned(w) || misaligned(conv_b) || misaligned(bias) || (reinterpret_cast<uintptr_t>(x) & 15u) != 0 ||
        (reinterpret_cast<uintptr_t>(out) & 15u) != 0)
        return FW_ERR_ALIGN;
    if (!convpool_tc_eligible(Cin, Cout, KH, KW, pool_k, pool_s)) return FW_ERR_UNSUPPORTED;
    const long long nx = prod({N, H, W, Cin}), nw = prod({Cout, Cin, KH, KW}), no = prod({N, Ho, Wo, Cout});
    if (nx < 0 || nw < 0 || no < 0) return FW_ERR_SHAPE;
    const long long ob = no * 4;
    if (overlaps(out, ob, x, nx * 4) || overlaps(out, ob, w, nw * 4) || overlaps(out, ob, bias, 4LL * Cout) ||
        overlaps(out, ob, conv_b, 4LL * Cout))
        return FW_ERR_ALIAS;
    return convpool_tc_launch_nhwc(x, N, H, W, w, conv_b, Cout, scale, bias, pool_k, out, Ho, Wo,
                                   static_cast<cudaStream_t>(stream));
}

fw_status fw_selftest_bounded_wait(unsigned int limit_us, void *stream) {
    if (limit_us == 0 || limit_us > 2000000u) return FW_ERR_PARAM;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * limit_us);
    note_launch();
    return launch_status(cudaGetLastError());
}

fw_status fw_check_device_errors(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FW_ERR_LAUNCH;
    const unsigned e = maxpool_read_and_clear_error() | convt_tc_read_and_clear_error() |
                         convpool_tc_read_and_clear_error() | convt_read_and_clear_error() |
                         convpool_read_and_clear_error() | api_read_and_clear_error();
    if (e & DEVERR_TIMEOUT) return FW_ERR_TIMEOUT;
    if (e) return FW_ERR_INTERNAL;
    return FW_OK;
}

}  // extern "C"
