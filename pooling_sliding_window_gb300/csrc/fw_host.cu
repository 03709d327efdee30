// fw_host.cu -- host-buffer entry points: the three operators on tensors that live in
// (preferably pinned) host memory.  The batch is split into image chunks and the
// chunks are pipelined: host->device copies of chunk i+1 and device->host copies of
// chunk i-1 overlap the kernels of chunk i.  Each chunk runs through the device entry
// points of fw_api.cu, so arguments are validated and dispatched exactly as there.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fw_common.cuh"

extern "C" {
fw_status fw_conv2d_tanh_scale_bias_maxpool(const float *x, int N, int Cin, int H, int W, const float *w,
                                            const float *conv_b, int Cout, int KH, int KW, float scale,
                                            const float *bias, int pool_k, int pool_s, float *out, void *stream);
fw_status fw_maxpool2d(const float *x, int N, int C, int H, int W, int k, int s, int p, int d, float *out,
                       void *stream);
fw_status fw_conv2d_pool_out_shape(int H, int W, int KH, int KW, int pool_k, int pool_s, int *Ho, int *Wo);
fw_status fw_maxpool2d_out_shape(int H, int W, int k, int s, int p, int d, int *Ho, int *Wo);
fw_status fw_convt_out_shape(int H, int W, int k, int s, int p, int op, int *Ho, int *Wo);
unsigned long long fw_convt_workspace_size(int Cin, int Cout, int k, int s, int p);
}

namespace fw {
namespace {

constexpr int MAX_CHUNKS = 8;
constexpr unsigned long long ALIGN = 256;

unsigned long long up(unsigned long long b) { return (b + ALIGN - 1) & ~(ALIGN - 1); }

// Two copy streams and the events of one pipelined call, created once per device.
struct Pipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, in[MAX_CHUNKS] = {}, comp[MAX_CHUNKS] = {};
    bool ok = false;
};
std::mutex g_pipe_mu;
Pipe g_pipes[FW_MAX_DEVICES];

// Returns the device's pipe with g_pipe_mu held by the caller.
Pipe *pipe_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= FW_MAX_DEVICES) return nullptr;
    Pipe &p = g_pipes[dev];
    if (!p.ok) {
        bool good = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; good && i < MAX_CHUNKS; ++i)
            good = cudaEventCreateWithFlags(&p.in[i], cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventCreateWithFlags(&p.comp[i], cudaEventDisableTiming) == cudaSuccess;
        if (!good) return nullptr;
        p.ok = true;
    }
    return &p;
}

// One pipelined call: `small` copies (weights) first, then per chunk of images the
// input copy, the operator (`run`, on the caller's stream) and the output copy.
template <class Run>
fw_status pipelined_enqueue(Pipe *p, cudaStream_t st, int N, size_t in_img_bytes, const void *x_host, void *x_dev,
                            size_t out_img_bytes, void *out_host, const void *out_dev,
                            const void *const *small_src, void *const *small_dst, const size_t *small_bytes,
                            int nsmall, Run run) {
    const int nch = N < MAX_CHUNKS ? N : MAX_CHUNKS;
    const int per = (N + nch - 1) / nch;
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    // device buffers may still be in use by earlier work on the caller's stream
    if (!ck(cudaEventRecord(p->start, st)) || !ck(cudaStreamWaitEvent(p->h2d, p->start, 0)) ||
        !ck(cudaStreamWaitEvent(p->d2h, p->start, 0)))
        return FW_ERR_LAUNCH;
    for (int i = 0; i < nsmall; ++i)
        if (small_bytes[i] &&
            !ck(cudaMemcpyAsync(small_dst[i], small_src[i], small_bytes[i], cudaMemcpyHostToDevice, p->h2d)))
            return FW_ERR_LAUNCH;
    for (int c = 0; c * per < N; ++c) {
        const int i0 = c * per, n = N - i0 < per ? N - i0 : per;
        const size_t ib = in_img_bytes * (size_t)i0, ob = out_img_bytes * (size_t)i0;
        if (!ck(cudaMemcpyAsync(static_cast<char *>(x_dev) + ib, static_cast<const char *>(x_host) + ib,
                                in_img_bytes * (size_t)n, cudaMemcpyHostToDevice, p->h2d)) ||
            !ck(cudaEventRecord(p->in[c], p->h2d)) || !ck(cudaStreamWaitEvent(st, p->in[c], 0)))
            return FW_ERR_LAUNCH;
        const fw_status rc = run(i0, n);
        if (rc != FW_OK) return rc;
        if (!ck(cudaEventRecord(p->comp[c], st)) || !ck(cudaStreamWaitEvent(p->d2h, p->comp[c], 0)) ||
            !ck(cudaMemcpyAsync(static_cast<char *>(out_host) + ob, static_cast<const char *>(out_dev) + ob,
                                out_img_bytes * (size_t)n, cudaMemcpyDeviceToHost, p->d2h)))
            return FW_ERR_LAUNCH;
    }
    // the caller's stream continues after the last output copy
    if (!ck(cudaEventRecord(p->done, p->d2h)) || !ck(cudaStreamWaitEvent(st, p->done, 0))) return FW_ERR_LAUNCH;
    return FW_OK;
}

template <class Run>
fw_status pipelined(cudaStream_t st, int N, size_t in_img_bytes, const void *x_host, void *x_dev,
                    size_t out_img_bytes, void *out_host, const void *out_dev,
                    const void *const *small_src, void *const *small_dst, const size_t *small_bytes, int nsmall,
                    Run run) {
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    Pipe *p = pipe_for_current_device();
    if (!p) return FW_ERR_LAUNCH;
    const fw_status rc = pipelined_enqueue(p, st, N, in_img_bytes, x_host, x_dev, out_img_bytes, out_host, out_dev,
                                           small_src, small_dst, small_bytes, nsmall, run);
    if (rc != FW_OK) {
        // A failed call returns only once no copy it enqueued is still in flight, so
        // the caller may free or reuse the workspace and the host buffers at once.
        cudaStreamSynchronize(p->h2d);
        cudaStreamSynchronize(p->d2h);
    }
    return rc;
}

bool valid_sizes(int N, int a, int b) { return N >= 1 && a >= 1 && b >= 1; }

}  // namespace
}  // namespace fw

using namespace fw;

extern "C" {

unsigned long long fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(int N, int Cin, int H, int W, int Cout,
                                                                         int KH, int KW, int pool_k, int pool_s) {
    int Ho = 0, Wo = 0;
    if (!valid_sizes(N, Cin, Cout) || fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo) != FW_OK)
        return 0;
    const unsigned long long f = 4;
    return up(f * N * Cin * H * W) + up(f * Cout * Cin * KH * KW) + 2 * up(f * Cout) + up(f * N * Cout * Ho * Wo);
}

fw_status fw_conv2d_tanh_scale_bias_maxpool_host(const float *x, int N, int Cin, int H, int W, const float *w,
                                                 const float *conv_b, int Cout, int KH, int KW, float scale,
                                                 const float *bias, int pool_k, int pool_s, float *out,
                                                 void *workspace, unsigned long long workspace_bytes, void *stream) {
    if (!x || !w || !bias || !out || !workspace) return FW_ERR_NULL;
    const unsigned long long need =
        fw_conv2d_tanh_scale_bias_maxpool_host_workspace_size(N, Cin, H, W, Cout, KH, KW, pool_k, pool_s);
    if (need == 0) return FW_ERR_SHAPE;
    if (workspace_bytes < need) return FW_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % ALIGN) return FW_ERR_ALIGN;
    int Ho = 0, Wo = 0;
    fw_conv2d_pool_out_shape(H, W, KH, KW, pool_k, pool_s, &Ho, &Wo);
    char *ws = static_cast<char *>(workspace);
    const size_t xb = 4ull * N * Cin * H * W, wb = 4ull * Cout * Cin * KH * KW, cbb = 4ull * Cout;
    float *xd = reinterpret_cast<float *>(ws);
    float *wd = reinterpret_cast<float *>(ws + up(xb));
    float *cbd = reinterpret_cast<float *>(ws + up(xb) + up(wb));
    float *bd = reinterpret_cast<float *>(ws + up(xb) + up(wb) + up(cbb));
    float *od = reinterpret_cast<float *>(ws + up(xb) + up(wb) + 2 * up(cbb));
    const void *src[] = {w, conv_b, bias};
    void *dst[] = {wd, cbd, bd};
    const size_t bytes[] = {wb, conv_b ? cbb : 0, cbb};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t in_img = 4ull * Cin * H * W, out_img = 4ull * Cout * Ho * Wo;
    return pipelined(st, N, in_img, x, xd, out_img, out, od, src, dst, bytes, 3, [&](int i0, int n) {
        return fw_conv2d_tanh_scale_bias_maxpool(xd + (size_t)i0 * Cin * H * W, n, Cin, H, W, wd,
                                                 conv_b ? cbd : nullptr, Cout, KH, KW, scale, bd, pool_k, pool_s,
                                                 od + (size_t)i0 * Cout * Ho * Wo, stream);
    });
}

unsigned long long fw_maxpool2d_host_workspace_size(int N, int C, int H, int W, int k, int s, int p, int d) {
    int Ho = 0, Wo = 0;
    if (!valid_sizes(N, C, 1) || fw_maxpool2d_out_shape(H, W, k, s, p, d, &Ho, &Wo) != FW_OK) return 0;
    return up(4ull * N * C * H * W) + up(4ull * N * C * Ho * Wo);
}

fw_status fw_maxpool2d_host(const float *x, int N, int C, int H, int W, int k, int s, int p, int d, float *out,
                            void *workspace, unsigned long long workspace_bytes, void *stream) {
    if (!x || !out || !workspace) return FW_ERR_NULL;
    const unsigned long long need = fw_maxpool2d_host_workspace_size(N, C, H, W, k, s, p, d);
    if (need == 0) return FW_ERR_SHAPE;
    if (workspace_bytes < need) return FW_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % ALIGN) return FW_ERR_ALIGN;
    int Ho = 0, Wo = 0;
    fw_maxpool2d_out_shape(H, W, k, s, p, d, &Ho, &Wo);
    char *ws = static_cast<char *>(workspace);
    float *xd = reinterpret_cast<float *>(ws);
    float *od = reinterpret_cast<float *>(ws + up(4ull * N * C * H * W));
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return pipelined(st, N, 4ull * C * H * W, x, xd, 4ull * C * Ho * Wo, out, od, nullptr, nullptr, nullptr, 0,
                     [&](int i0, int n) {
                         return fw_maxpool2d(xd + (size_t)i0 * C * H * W, n, C, H, W, k, s, p, d,
                                             od + (size_t)i0 * C * Ho * Wo, stream);
                     });
}

unsigned long long fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(int N, int Cin, int H, int W,
                                                                                     int Cout, int k, int s, int p,
                                                                                     int op) {
    int Ho = 0, Wo = 0;
    if (!valid_sizes(N, Cin, Cout) || fw_convt_out_shape(H, W, k, s, p, op, &Ho, &Wo) != FW_OK) return 0;
    const unsigned long long f = 4;
    return up(f * N * Cin * H * W) + up(f * Cin * Cout * k * k) + 2 * up(f * Cout) + up(f * N * Cout * Ho * Wo) +
           up(fw_convt_workspace_size(Cin, Cout, k, s, p));
}

fw_status fw_convtranspose2d_softmax_bias_scale_sigmoid_host(const float *x, int N, int Cin, int H, int W,
                                                             const float *w, const float *conv_b, int Cout, int k,
                                                             int s, int p, int op, const float *bias, float scale,
                                                             float *out, void *workspace,
                                                             unsigned long long workspace_bytes, void *stream) {
    if (!x || !w || !bias || !out || !workspace) return FW_ERR_NULL;
    const unsigned long long need =
        fw_convtranspose2d_softmax_bias_scale_sigmoid_host_workspace_size(N, Cin, H, W, Cout, k, s, p, op);
    if (need == 0) return FW_ERR_SHAPE;
    if (workspace_bytes < need) return FW_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % ALIGN) return FW_ERR_ALIGN;
    int Ho = 0, Wo = 0;
    fw_convt_out_shape(H, W, k, s, p, op, &Ho, &Wo);
    char *ws = static_cast<char *>(workspace);
    const size_t xb = 4ull * N * Cin * H * W, wb = 4ull * Cin * Cout * k * k, cbb = 4ull * Cout,
                 ob = 4ull * N * Cout * Ho * Wo;
    float *xd = reinterpret_cast<float *>(ws);
    float *wd = reinterpret_cast<float *>(ws + up(xb));
    float *cbd = reinterpret_cast<float *>(ws + up(xb) + up(wb));
    float *bd = reinterpret_cast<float *>(ws + up(xb) + up(wb) + up(cbb));
    float *od = reinterpret_cast<float *>(ws + up(xb) + up(wb) + 2 * up(cbb));
    char *tws = ws + up(xb) + up(wb) + 2 * up(cbb) + up(ob);
    const unsigned long long tws_bytes = fw_convt_workspace_size(Cin, Cout, k, s, p);
    const void *src[] = {w, conv_b, bias};
    void *dst[] = {wd, cbd, bd};
    const size_t bytes[] = {wb, conv_b ? cbb : 0, cbb};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t in_img = 4ull * Cin * H * W, out_img = 4ull * Cout * Ho * Wo;
    // the weight rewrite into `tws` is made by the first chunk only: the chunks run in
    // order on `stream`, so the later ones find it in place
    return pipelined(st, N, in_img, x, xd, out_img, out, od, src, dst, bytes, 3, [&](int i0, int n) {
        return convt_call(xd + (size_t)i0 * Cin * H * W, n, Cin, H, W, wd, conv_b ? cbd : nullptr, Cout, k, s, p,
                          op, bd, scale, od + (size_t)i0 * Cout * Ho * Wo, tws_bytes ? tws : nullptr, tws_bytes,
                          false, i0 > 0, stream);
    });
}

}  // extern "C"
