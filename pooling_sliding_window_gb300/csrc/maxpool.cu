// maxpool.cu -- MaxPool2d kernels (trace "Kimi-K2.6 l1_p42": MaxPool2d(k=4, s=1,
// p=1, d=1) on [32,64,512,512], -inf padding, output 511x511).
//
// Streaming kernel (stride 1, dilation 1, W % 4 == 0):
//   * one CTA per (plane, band of output rows); thread t owns input and output
//     columns [4t, 4t+4) (threads past the row read -inf guard columns);
//   * input rows of the band stream HBM -> shared memory through the TMA bulk-copy
//     engine (one cp.async.bulk per row) into a ring of NSTAGE slots, each slot
//     holding `rps` rows; an mbarrier per slot completes on the copied bytes;
//   * each row is read once from shared memory (float4 + edge scalars from -inf
//     guard columns, which realise the padding), reduced horizontally (a pairwise
//     tree for k = 4), and kept in a K-deep register ring; every new row
//     completes one output row, reduced vertically (separable max: the page's
//     row-max-then-column-max decomposition, exact for max).  The reductions use
//     the single-instruction max.NaN (NaN propagates); a zero maximum, whose sign
//     the definition fixes by tap order, is recomputed tap by tap;
//   * output rows (W odd in general, so not 16-byte aligned) are transposed
//     through a per-warp shared buffer so that each store instruction writes 32
//     consecutive floats.
// Direct kernel: one thread per output, taps read through the read-only cache;
// covers every other (k, s, p, d, W).
#include "fw_common.cuh"

namespace fw {

__device__ unsigned g_err_maxpool = 0;
#define CHK(p, bytes, base, base_bytes) chk(&g_err_maxpool, (p), (bytes), (base), (base_bytes))
#define CHKS(p, bytes) chk_smem(&g_err_maxpool, (p), (bytes))

namespace {

constexpr int NSTAGE = 2;   // ring slots (two large stages measured faster than 3-8 small ones)
constexpr int GUARD = 4;    // -inf columns on each side of a shared-memory row

// max.NaN: the larger value, or a canonical NaN when either input is NaN.
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// The definition's window maximum for one output (taps in row-major order,
// -inf padding, first of equal values kept), read from global memory.  Inlined,
// with the tap loops rolled for K >= 4: as a called function it made the kernels
// keep registers in local memory (spills), and fully unrolled at K = 4 the rarely
// taken branch cost the hot loop 14 % more instructions (measured: 0.654 ms called,
// 0.695 ms unrolled, 0.644 ms rolled on the full workload).
template <int K, int P>
__device__ __forceinline__ float window_max_exact(const float *__restrict__ plane, int H, int W, int oh, int ow,
                                                  const float *x, long long x_bytes) {
    constexpr int UNROLL = K <= 3 ? K : 1;
    float m = -INFINITY;
#pragma unroll UNROLL
    for (int i = 0; i < K; ++i) {
        const int ih = oh - P + i;
#pragma unroll UNROLL
        for (int j = 0; j < K; ++j) {
            const int iw = ow - P + j;
            const float *a = plane + (long long)ih * W + iw;
            const float v = (ih >= 0 && ih < H && iw >= 0 && iw < W && CHK(a, 4, x, x_bytes)) ? __ldg(a) : -INFINITY;
            m = max_update(m, v);
        }
    }
    return m;
}

// Shared-memory row pitch (floats): GUARD -inf columns, the W data columns, and
// -inf columns up to and past the last column any thread of the block reads.
__host__ __device__ inline int stream_pitch(int threads) { return 4 * threads + 4 * GUARD; }

template <int K, int P>
__global__ void __launch_bounds__(512) maxpool_s1_stream_kernel(const float *__restrict__ x,
                                                                 float *__restrict__ out, int H, int W,
                                                                 int Ho, int Wo, int band, int nbands,
                                                                 int rps) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);
    const int pitch = stream_pitch(blockDim.x);           // floats per shared row
    float *ring = reinterpret_cast<float *>(smem_raw + 64);  // NSTAGE * rps rows
    float *ostage = ring + (size_t)NSTAGE * rps * pitch;  // 128 floats per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long plane = blockIdx.x / nbands;
    const int b = blockIdx.x - (int)(plane * nbands);
    const int r0 = b * band, r1 = min(Ho, r0 + band);       // output rows [r0, r1)
    const int la = max(0, r0 - P), lb = min(H, r1 - 1 - P + K);  // input rows [la, lb)
    const int nrows = max(0, lb - la);
    const int nst = (nrows + rps - 1) / rps;               // stages of this band
    const float *src = x + plane * (long long)H * W;
    float *dst = out + plane * (long long)Ho * Wo;
    // buffer extents for the checked build (gridDim.x = planes x bands)
    const long long NCp = gridDim.x / nbands;
    const long long x_bytes = 4LL * NCp * H * W, out_bytes = 4LL * NCp * Ho * Wo;

    // -inf guard columns of every slot row (never touched by the bulk copies).
    const int nguard = pitch - W;
    for (int i = tid; i < NSTAGE * rps * nguard; i += blockDim.x) {
        const int row = i / nguard, g = i % nguard;
        float *gp = ring + (size_t)row * pitch + (g < GUARD ? g : W + g);
        if (CHKS(gp, 4)) *gp = -INFINITY;
    }
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int st) {  // thread 0 only: copy stage `st` into its slot
        const int slot = st % NSTAGE;
        const int row0 = la + st * rps, cnt = min(rps, lb - row0);
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t row_bytes = (uint32_t)W * 4u;
        // checked build: rows outside x or the ring are not copied (nor expected)
        int ok_rows = 0;
        for (int r = 0; r < cnt; ++r)
            ok_rows += CHK(src + (long long)(row0 + r) * W, row_bytes, x, x_bytes) &&
                       CHKS(ring + ((size_t)slot * rps + r) * pitch + GUARD, row_bytes);
        mbar_arrive_expect_tx(bar, row_bytes * ok_rows);
        for (int r = 0; r < cnt; ++r)
            if (!FW_CHECKED || (CHK(src + (long long)(row0 + r) * W, row_bytes, x, x_bytes) &&
                                CHKS(ring + ((size_t)slot * rps + r) * pitch + GUARD, row_bytes)))
                bulk_g2s(smem_u32(ring + ((size_t)slot * rps + r) * pitch + GUARD),
                         src + (long long)(row0 + r) * W, row_bytes, bar);
    };
    if (tid == 0) {
        fence_proxy_async_smem();
        for (int st = 0; st < min(NSTAGE, nst); ++st) issue(st);
    }

    // Register ring of the last K horizontal-max rows (4 columns each); row ir
    // lives in hist[(ir - ir_begin) % K], so the unrolled loop below indexes it
    // statically.
    float4 hist[K];
#pragma unroll
    for (int i = 0; i < K; ++i) hist[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);

    const int c0 = 4 * tid + GUARD;  // this thread's first column in a shared row
    const float *xplane = src;
    bool err = false, any_err = false;
    int st = 0, r_in_st = 0, st_rows = min(rps, lb - la);
    // Walk input rows ir = r0-P .. r1-2-P+K (rows outside [0,H) are all -inf).
    const int ir_begin = r0 - P, ir_end = r1 - 1 - P + K;
    for (int base = ir_begin; base < ir_end && !any_err; base += K) {
#pragma unroll
        for (int u = 0; u < K; ++u) {
            const int ir = base + u;
            if (ir >= ir_end) break;
            float4 h = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (ir >= la && ir < lb) {
                const int slot = st % NSTAGE;
                if (r_in_st == 0 && !mbar_wait_bounded(smem_u32(&bars[slot]), (uint32_t)(st / NSTAGE) & 1u))
                    err = true;
                const float *row = ring + ((size_t)slot * rps + r_in_st) * pitch;
                // window of 3+K values: columns 4t-P .. 4t+2-P+K
                float v[K + 3];
                const bool row_ok = CHKS(row + c0 - P, (K + 3) * 4);
                const float4 mid = row_ok ? *reinterpret_cast<const float4 *>(row + c0)
                                          : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
                for (int i = 0; i < K + 3; ++i) {
                    const int c = i - P;  // offset from 4t
                    if (c == 0) v[i] = mid.x;
                    else if (c == 1) v[i] = mid.y;
                    else if (c == 2) v[i] = mid.z;
                    else if (c == 3) v[i] = mid.w;
                    else v[i] = row_ok ? row[c0 + c] : -INFINITY;
                }
                float hv[4];
                if (K == 4) {  // pairwise tree: 10 max for 4 outputs
                    float a[6];
#pragma unroll
                    for (int i = 0; i < 6; ++i) a[i] = max_nan(v[i], v[i + 1]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) hv[j] = max_nan(a[j], a[j + 2]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float m = v[j];
#pragma unroll
                        for (int kw = 1; kw < K; ++kw) m = max_nan(m, v[j + kw]);
                        hv[j] = m;
                    }
                }
                h = make_float4(hv[0], hv[1], hv[2], hv[3]);
                if (++r_in_st == st_rows) {  // stage consumed: release the slot, refill it
                    if (__syncthreads_or(err)) {
                        if (tid == 0) atomicOr(&g_err_maxpool, DEVERR_TIMEOUT);
                        any_err = true;
                        break;
                    }
                    if (tid == 0 && st + NSTAGE < nst) {
                        fence_proxy_async_smem();
                        issue(st + NSTAGE);
                    }
                    ++st;
                    r_in_st = 0;
                    st_rows = min(rps, lb - (la + st * rps));
                }
            }
            hist[u] = h;
            const int oh = ir + P - (K - 1);  // output row whose last window row is ir
            if (oh >= r0) {
                float4 m = hist[(u + 1) % K];
#pragma unroll
                for (int i = 2; i <= K; ++i) {
                    const float4 g = hist[(u + i) % K];
                    m.x = max_nan(m.x, g.x);
                    m.y = max_nan(m.y, g.y);
                    m.z = max_nan(m.z, g.z);
                    m.w = max_nan(m.w, g.w);
                }
                // max.NaN leaves the sign of a zero maximum to the hardware; the
                // definition keeps the first zero of the window, so a zero result
                // is recomputed tap by tap (rare).
                if (m.x == 0.f || m.y == 0.f || m.z == 0.f || m.w == 0.f) {
                    if (m.x == 0.f) m.x = window_max_exact<K, P>(xplane, H, W, oh, 4 * tid, x, x_bytes);
                    if (m.y == 0.f) m.y = window_max_exact<K, P>(xplane, H, W, oh, 4 * tid + 1, x, x_bytes);
                    if (m.z == 0.f) m.z = window_max_exact<K, P>(xplane, H, W, oh, 4 * tid + 2, x, x_bytes);
                    if (m.w == 0.f) m.w = window_max_exact<K, P>(xplane, H, W, oh, 4 * tid + 3, x, x_bytes);
                }
                float *os = ostage + warp * 128;
                const bool os_ok = CHKS(os, 512);
                __syncwarp();
                if (os_ok) *reinterpret_cast<float4 *>(os + lane * 4) = m;
                __syncwarp();
                float *orow = dst + (long long)oh * Wo + warp * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = q * 32 + lane;
                    if (warp * 128 + c < Wo && os_ok && CHK(orow + c, 4, out, out_bytes)) orow[c] = os[c];
                }
            }
        }
    }
    if (any_err && tid == 0) {
        // Drain copies still in flight into this CTA's shared memory (bounded).
        for (int s2 = st; s2 < min(nst, st + NSTAGE); ++s2)
            mbar_wait_bounded(smem_u32(&bars[s2 % NSTAGE]), (uint32_t)(s2 / NSTAGE) & 1u);
    }
}

__global__ void maxpool_direct_kernel(const float *__restrict__ x, float *__restrict__ out,
                                      long long NC, int H, int W, int Ho, int Wo, int k, int s, int p,
                                      int d) {
    const long long total = NC * Ho * Wo;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(idx % Wo);
        const long long t = idx / Wo;
        const int oh = (int)(t % Ho);
        const long long nc = t / Ho;
        const float *plane = x + nc * (long long)H * W;
        float m = -INFINITY;
        for (int i = 0; i < k; ++i) {
            const int ih = oh * s - p + i * d;
            const bool rin = ih >= 0 && ih < H;
            for (int j = 0; j < k; ++j) {
                const int iw = ow * s - p + j * d;
                const float *a = plane + (long long)ih * W + iw;
                const float v = (rin && iw >= 0 && iw < W && CHK(a, 4, x, 4LL * NC * H * W)) ? __ldg(a) : -INFINITY;
                m = max_update(m, v);
            }
        }
        if (CHK(out + idx, 4, out, 4 * total)) out[idx] = m;
    }
}

// Generic MaxPool2d with the optional PyTorch extensions (not on the pages): any
// (k, s, p, d), an output size from floor or ceil mode (given), and optional argmax
// indices.  One thread per output; the first in-bounds tap initialises the
// running (value, index), later taps replace it by the running-max rule (a larger
// value, or a NaN when the current value is not NaN), so values equal the other
// kernels' and an index is the flat ih*W + iw of the tap the value came from (-1
// when the window has no input tap; the value is then -inf).
__global__ void __launch_bounds__(256) maxpool_direct_ex_kernel(const float *__restrict__ x, float *__restrict__ out,
                                                                long long *__restrict__ idx, long long NC, int H,
                                                                int W, int Ho, int Wo, int k, int s, int p, int d) {
    const long long total = NC * Ho * Wo;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(o % Wo);
        const long long t = o / Wo;
        const int oh = (int)(t % Ho);
        const long long nc = t / Ho;
        const float *plane = x + nc * (long long)H * W;
        float m = -INFINITY;
        long long at = -1;
        for (int i = 0; i < k; ++i) {
            const int ih = oh * s - p + i * d;
            if (ih < 0 || ih >= H) continue;
            for (int j = 0; j < k; ++j) {
                const int iw = ow * s - p + j * d;
                if (iw < 0 || iw >= W || !CHK(plane + (long long)ih * W + iw, 4, x, 4LL * NC * H * W)) continue;
                const float v = __ldg(plane + (long long)ih * W + iw);
                if (at < 0 || (m == m && (v != v || v > m))) {
                    m = v;
                    at = (long long)ih * W + iw;
                }
            }
        }
        if (CHK(out + o, 4, out, 4 * total)) out[o] = m;
        if (idx && CHK(idx + o, 8, idx, 8 * total)) idx[o] = at;
    }
}

// The definition's window maximum for one output with any stride and dilation
// (inlined, loops rolled for K >= 4, like window_max_exact).
template <int K>
__device__ __forceinline__ float window_max_exact_sd(const float *__restrict__ plane, int H, int W, int s, int p,
                                                     int d, int oh, int ow, const float *x, long long x_bytes) {
    constexpr int UNROLL = K <= 3 ? K : 1;
    float m = -INFINITY;
#pragma unroll UNROLL
    for (int i = 0; i < K; ++i) {
        const int ih = oh * s - p + i * d;
#pragma unroll UNROLL
        for (int j = 0; j < K; ++j) {
            const int iw = ow * s - p + j * d;
            const float *a = plane + (long long)ih * W + iw;
            const float v = (ih >= 0 && ih < H && iw >= 0 && iw < W && CHK(a, 4, x, x_bytes)) ? __ldg(a) : -INFINITY;
            m = max_update(m, v);
        }
    }
    return m;
}

// Streaming kernel for stride S and dilation D (S > 1 or D > 1): the same bulk-copy
// row ring and -inf guards as the stride-1 kernel.  Thread t owns output columns
// [4t, 4t+4), whose taps span the SPAN input columns from 4tS - P; it reads them
// with aligned float4 loads and takes the horizontal maxima (taps D apart, outputs
// S apart).  The last R = (K-1)D + 1 row maxima stay in a register ring; input row
// ir completes output row oh when ir = oh*S - P + (K-1)D.
template <int K, int S, int D, int P>
__global__ void __launch_bounds__(512) maxpool_stream_sd_kernel(const float *__restrict__ x, float *__restrict__ out,
                                                                int H, int W, int Ho, int Wo, int band, int nbands,
                                                                int rps, int pitch) {
    constexpr int SPAN = 3 * S + (K - 1) * D + 1;    // input columns of 4 outputs
    constexpr int R = (K - 1) * D + 1;               // rows a window spans
    constexpr int OFF = (4 - P % 4) % 4;             // span start - aligned load start
    constexpr int NQ = (OFF + SPAN + 3) / 4;         // float4 loads per row
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);
    float *ring = reinterpret_cast<float *>(smem_raw + 64);  // NSTAGE * rps rows
    float *ostage = ring + (size_t)NSTAGE * rps * pitch;    // 128 floats per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long plane = blockIdx.x / nbands;
    const int b = blockIdx.x - (int)(plane * nbands);
    const int r0 = b * band, r1 = min(Ho, r0 + band);                    // output rows [r0, r1)
    const int ir_begin = r0 * S - P, ir_end = (r1 - 1) * S - P + (K - 1) * D;  // input rows [.., ir_end]
    const int la = max(0, ir_begin), lb = min(H, ir_end + 1);            // of them, inside the plane
    const int nrows = max(0, lb - la);
    const int nst = (nrows + rps - 1) / rps;
    const float *src = x + plane * (long long)H * W;
    float *dst = out + plane * (long long)Ho * Wo;
    // buffer extents for the checked build (gridDim.x = planes x bands)
    const long long NCp = gridDim.x / nbands;
    const long long x_bytes = 4LL * NCp * H * W, out_bytes = 4LL * NCp * Ho * Wo;

    const int nguard = pitch - W;
    for (int i = tid; i < NSTAGE * rps * nguard; i += blockDim.x) {
        const int row = i / nguard, g = i % nguard;
        float *gp = ring + (size_t)row * pitch + (g < GUARD ? g : W + g);
        if (CHKS(gp, 4)) *gp = -INFINITY;
    }
    if (tid == 0) {
        for (int st = 0; st < NSTAGE; ++st) mbar_init(smem_u32(&bars[st]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int st) {  // thread 0 only: copy stage `st` into its slot
        const int slot = st % NSTAGE;
        const int row0 = la + st * rps, cnt = min(rps, lb - row0);
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t row_bytes = (uint32_t)W * 4u;
        // checked build: rows outside x or the ring are not copied (nor expected)
        int ok_rows = 0;
        for (int r = 0; r < cnt; ++r)
            ok_rows += CHK(src + (long long)(row0 + r) * W, row_bytes, x, x_bytes) &&
                       CHKS(ring + ((size_t)slot * rps + r) * pitch + GUARD, row_bytes);
        mbar_arrive_expect_tx(bar, row_bytes * ok_rows);
        for (int r = 0; r < cnt; ++r)
            if (!FW_CHECKED || (CHK(src + (long long)(row0 + r) * W, row_bytes, x, x_bytes) &&
                                CHKS(ring + ((size_t)slot * rps + r) * pitch + GUARD, row_bytes)))
                bulk_g2s(smem_u32(ring + ((size_t)slot * rps + r) * pitch + GUARD), src + (long long)(row0 + r) * W,
                         row_bytes, bar);
    };
    if (tid == 0) {
        fence_proxy_async_smem();
        for (int st = 0; st < min(NSTAGE, nst); ++st) issue(st);
    }

    float4 hist[R];
#pragma unroll
    for (int i = 0; i < R; ++i) hist[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const int a0 = GUARD + 4 * tid * S - P - OFF;  // aligned first column this thread loads
    bool err = false, any_err = false;
    int st = 0, r_in_st = 0, st_rows = min(rps, lb - la);
    for (int base = ir_begin; base <= ir_end && !any_err; base += R) {
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int ir = base + u;
            if (ir > ir_end) break;
            float4 h = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (ir >= la && ir < lb) {
                const int slot = st % NSTAGE;
                if (r_in_st == 0 && !mbar_wait_bounded(smem_u32(&bars[slot]), (uint32_t)(st / NSTAGE) & 1u))
                    err = true;
                const float *row = ring + ((size_t)slot * rps + r_in_st) * pitch + a0;
                const bool row_ok = CHKS(row, 16 * NQ);
                float v[4 * NQ];
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const float4 f = row_ok ? *reinterpret_cast<const float4 *>(row + 4 * q)
                                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    v[4 * q] = f.x;
                    v[4 * q + 1] = f.y;
                    v[4 * q + 2] = f.z;
                    v[4 * q + 3] = f.w;
                }
                float hv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float m = v[OFF + j * S];
#pragma unroll
                    for (int i = 1; i < K; ++i) m = max_nan(m, v[OFF + j * S + i * D]);
                    hv[j] = m;
                }
                h = make_float4(hv[0], hv[1], hv[2], hv[3]);
                if (++r_in_st == st_rows) {  // stage consumed: release the slot, refill it
                    if (__syncthreads_or(err)) {
                        if (tid == 0) atomicOr(&g_err_maxpool, DEVERR_TIMEOUT);
                        any_err = true;
                        break;
                    }
                    if (tid == 0 && st + NSTAGE < nst) {
                        fence_proxy_async_smem();
                        issue(st + NSTAGE);
                    }
                    ++st;
                    r_in_st = 0;
                    st_rows = min(rps, lb - (la + st * rps));
                }
            }
            hist[u] = h;
            const int t = ir - ir_begin - (K - 1) * D;  // = (oh - r0) * S when this row completes output row oh
            if (t >= 0 && t % S == 0) {
                const int oh = r0 + t / S;
                if (oh < r1) {
                    float4 m = hist[((u - (K - 1) * D) % R + R) % R];
#pragma unroll
                    for (int i = 1; i < K; ++i) {
                        const float4 g = hist[((u - (K - 1 - i) * D) % R + R) % R];
                        m.x = max_nan(m.x, g.x);
                        m.y = max_nan(m.y, g.y);
                        m.z = max_nan(m.z, g.z);
                        m.w = max_nan(m.w, g.w);
                    }
                    // a zero maximum: the sign is the first zero's by the definition
                    if (m.x == 0.f || m.y == 0.f || m.z == 0.f || m.w == 0.f) {
                        if (m.x == 0.f) m.x = window_max_exact_sd<K>(src, H, W, S, P, D, oh, 4 * tid, x, x_bytes);
                        if (m.y == 0.f) m.y = window_max_exact_sd<K>(src, H, W, S, P, D, oh, 4 * tid + 1, x, x_bytes);
                        if (m.z == 0.f) m.z = window_max_exact_sd<K>(src, H, W, S, P, D, oh, 4 * tid + 2, x, x_bytes);
                        if (m.w == 0.f) m.w = window_max_exact_sd<K>(src, H, W, S, P, D, oh, 4 * tid + 3, x, x_bytes);
                    }
                    float *os = ostage + warp * 128;
                    const bool os_ok = CHKS(os, 512);
                    __syncwarp();
                    if (os_ok) *reinterpret_cast<float4 *>(os + lane * 4) = m;
                    __syncwarp();
                    float *orow = dst + (long long)oh * Wo + warp * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int c = q * 32 + lane;
                        if (warp * 128 + c < Wo && os_ok && CHK(orow + c, 4, out, out_bytes)) orow[c] = os[c];
                    }
                }
            }
        }
    }
    if (any_err && tid == 0) {
        for (int s2 = st; s2 < min(nst, st + NSTAGE); ++s2)
            mbar_wait_bounded(smem_u32(&bars[s2 % NSTAGE]), (uint32_t)(s2 / NSTAGE) & 1u);
    }
}

template <int K, int S, int D, int P>
fw_status launch_stream_sd(const float *x, float *out, long long NC, int H, int W, int Ho, int Wo, cudaStream_t st) {
    const int threads = ((Wo + 3) / 4 + 31) / 32 * 32;
    if (threads > 512) return FW_ERR_UNSUPPORTED;
    // every column a thread may load: up to 4*threads*S + SPAN past the guard
    const int pitch = (GUARD + 4 * threads * S + 3 * S + (K - 1) * D + 1 + 8 + 3) / 4 * 4;
    if (pitch - W < GUARD) return FW_ERR_UNSUPPORTED;
    const int row_bytes = W * 4;
    // Stages of ~96 bytes per thread (12 KB at 128 threads): a block of few threads
    // (large strides: Wo/4 columns) takes smaller stages, so more blocks fit an SM and
    // more copies are in flight (x [32,64,512,512]: k3 s3 0.51 -> 0.37 ms, k4 s4 0.38 ->
    // 0.36 ms; 12 KB stages stay best for the 128-thread k3 s1 d2 blocks).
    const int rps = max(1, min(8, 96 * threads / row_bytes));
    const size_t smem = 64 + (size_t)NSTAGE * rps * pitch * 4 + (size_t)(threads / 32) * 128 * 4;
    const int band = Ho <= 64 ? Ho : 64;
    const int nbands = (Ho + band - 1) / band;
    const long long blocks = NC * nbands;
    if (blocks > 0x7fffffffLL) return FW_ERR_SHAPE;
    cudaError_t e = cudaFuncSetAttribute(maxpool_stream_sd_kernel<K, S, D, P>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    maxpool_stream_sd_kernel<K, S, D, P><<<(unsigned)blocks, threads, smem, st>>>(x, out, H, W, Ho, Wo, band, nbands,
                                                                                 rps, pitch);
    note_launch();
    return launch_status(cudaGetLastError());
}

template <int K, int P>
fw_status launch_stream(const float *x, float *out, long long NC, int H, int W, int Ho, int Wo,
                        cudaStream_t st) {
    // Threads cover every output column group; those past W/4 read -inf guards.
    const int threads = ((max(W, Wo) + 3) / 4 + 31) / 32 * 32;
    if (threads > 512) return FW_ERR_UNSUPPORTED;
    const int pitch = stream_pitch(threads);
    const int row_bytes = W * 4;
    // About 12 KB per bulk-copy stage: a small shared-memory footprint keeps 8 CTAs
    // per SM (the register limit) with few, large copies in flight per CTA.
    const int rps = max(1, min(8, 12288 / row_bytes));
    const size_t smem = 64 + (size_t)NSTAGE * rps * pitch * 4 + (size_t)(threads / 32) * 128 * 4;
    // Bands of output rows: long enough that the K-1 halo rows re-read per band
    // (from L2: neighbouring bands run at the same time) stay a few percent of the
    // band, short enough for many CTAs per plane (64 rows measured fastest).
    const int band = Ho <= 64 ? Ho : 64;
    const int nbands = (Ho + band - 1) / band;
    const long long blocks = NC * nbands;
    if (blocks > 0x7fffffffLL) return FW_ERR_SHAPE;
    cudaError_t e = cudaFuncSetAttribute(maxpool_s1_stream_kernel<K, P>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    maxpool_s1_stream_kernel<K, P><<<(unsigned)blocks, threads, smem, st>>>(x, out, H, W, Ho, Wo, band,
                                                                           nbands, rps);
    note_launch();
    return launch_status(cudaGetLastError());
}

using StreamFn = fw_status (*)(const float *, float *, long long, int, int, int, int, cudaStream_t);

StreamFn stream_fn(int k, int p) {
#define FW_MP_CASE(KK, PP) \
    if (k == KK && p == PP) return launch_stream<KK, PP>;
    FW_MP_CASE(1, 0) FW_MP_CASE(2, 0) FW_MP_CASE(2, 1) FW_MP_CASE(3, 0) FW_MP_CASE(3, 1)
    FW_MP_CASE(4, 0) FW_MP_CASE(4, 1) FW_MP_CASE(4, 2) FW_MP_CASE(5, 0) FW_MP_CASE(5, 1) FW_MP_CASE(5, 2)
#undef FW_MP_CASE
    return nullptr;
}

StreamFn stream_sd_fn(int k, int s, int d, int p) {
#define FW_MP_SD(KK, SS, DD, PP) \
    if (k == KK && s == SS && d == DD && p == PP) return launch_stream_sd<KK, SS, DD, PP>;
    FW_MP_SD(2, 2, 1, 0) FW_MP_SD(2, 2, 1, 1) FW_MP_SD(3, 2, 1, 0) FW_MP_SD(3, 2, 1, 1) FW_MP_SD(4, 2, 1, 1)
    FW_MP_SD(5, 2, 1, 2) FW_MP_SD(3, 3, 1, 0) FW_MP_SD(3, 3, 1, 1) FW_MP_SD(4, 4, 1, 0) FW_MP_SD(3, 1, 2, 1)
    FW_MP_SD(3, 1, 2, 2) FW_MP_SD(2, 1, 2, 1)
#undef FW_MP_SD
    return nullptr;
}

}  // namespace

fw_status maxpool2d_launch(const float *x, long long NC, int H, int W, int k, int s, int p, int d,
                           int Ho, int Wo, float *out, cudaStream_t st) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0);
    if (s == 1 && d == 1 && aligned && W % 4 == 0 && W >= 32 && W <= 2040) {
        if (StreamFn f = stream_fn(k, p)) return f(x, out, NC, H, W, Ho, Wo, st);
    }
    if ((s > 1 || d > 1) && aligned && W % 4 == 0 && W >= 32 && W <= 2040) {
        if (StreamFn f = stream_sd_fn(k, s, d, p)) {
            const fw_status rc = f(x, out, NC, H, W, Ho, Wo, st);
            if (rc != FW_ERR_UNSUPPORTED) return rc;
        }
    }
    const long long total = NC * Ho * Wo;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    maxpool_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(x, out, NC, H, W, Ho, Wo, k, s, p, d);
    note_launch();
    return launch_status(cudaGetLastError());
}

// ------------------------------------------------------------ channels last --
// x [N, H, W, C], out [N, Ho, Wo, C]: the same definition, tie and NaN rules as the
// NCHW kernels, applied per channel (the channel axis is the innermost, so a thread
// handles 4 adjacent channels of one output column with 16-byte loads and stores).

namespace {

// The definition's window maximum of one channel-last output value (taps in row-major
// order, -inf padding, first of equal values kept), read from global memory: the rare
// recompute of a zero maximum, whose sign the definition fixes by tap order.  Inlined,
// with the tap loops rolled for K >= 4 as in the NCHW kernels: as a called function it
// kept the stride-1 kernel at 96 registers (2 CTAs per SM, 0.77 ms on the full workload
// against 0.65 ms inlined at 64).
template <int K>
__device__ __forceinline__ float window_max_exact_nhwc(const float *__restrict__ img, int H, int W, int C, int oh,
                                                       int ow, int P, const float *x, long long x_bytes) {
    constexpr int UNROLL = K <= 3 ? K : 1;
    float m = -INFINITY;
#pragma unroll UNROLL
    for (int i = 0; i < K; ++i) {
        const int ih = oh - P + i;
#pragma unroll UNROLL
        for (int j = 0; j < K; ++j) {
            const int iw = ow - P + j;
            const float *a = img + ((long long)ih * W + iw) * C;
            const float v = (ih >= 0 && ih < H && iw >= 0 && iw < W && CHK(a, 4, x, x_bytes)) ? __ldg(a) : -INFINITY;
            m = max_update(m, v);
        }
    }
    return m;
}

// Stride 1, dilation 1, C % 4 == 0, 16-byte aligned x and out.  A block covers `cols`
// = 256 / (C/4) output columns of one band of output rows of one image; thread =
// (output column, channels 4c4..4c4+3).  The block's input columns ow0 - P ..
// ow0 - P + cols + K - 2 of a row are contiguous in memory (all channels), so they
// stream into shared memory as one bulk copy per row (TMA engine), rps rows per stage
// in a ring of NSTAGE stages; columns outside the image are -inf columns of the slot,
// written once.  Each thread takes the row's maximum over its K columns (16-byte
// shared-memory reads, consecutive threads on consecutive channels) and keeps the last
// K row maxima in a register ring, so output row oh is the maximum of the rows oh - P ..
// oh - P + K - 1 (separable max; rows outside the input are -inf).  The reductions use
// max.NaN (a NaN propagates); a zero maximum is recomputed tap by tap with the
// definition's rule, which fixes its sign.
template <int K>
__global__ void __launch_bounds__(256) maxpool_nhwc_s1_kernel(const float *__restrict__ x, float *__restrict__ out,
                                                              int H, int W, int C4, int Ho, int Wo, int P, int band,
                                                              int nbands, int owb, int rps) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);
    float4 *ring = reinterpret_cast<float4 *>(smem_raw + 64);  // NSTAGE * rps slot rows
    const int tid = threadIdx.x;
    const int cols = 256 / C4;            // output columns per block (C4 <= 256)
    const int seg = cols + K - 1;         // input columns per slot row
    const int pitch = seg * C4;           // float4 per slot row
    const long long blk = blockIdx.x;
    const int cw = (int)(blk % owb);      // block of output columns
    const long long t1 = blk / owb;
    const int b = (int)(t1 % nbands);
    const long long n = t1 / nbands;
    const bool active = tid < cols * C4;
    const int oc = active ? tid / C4 : 0, c4 = tid % C4;  // idle threads read slot column 0
    const int ow = cw * cols + oc;
    const bool store = active && ow < Wo;
    const int r0 = b * band, r1 = min(Ho, r0 + band);       // output rows [r0, r1)
    const int la = max(0, r0 - P), lb = min(H, r1 - 1 - P + K);  // input rows [la, lb)
    const int nrows = max(0, lb - la);
    const int nst = (nrows + rps - 1) / rps;                // stages of this band
    const int col0 = cw * cols - P;                          // input column of slot column 0
    const int ca = max(0, col0), cb = min(W, col0 + seg);   // input columns inside the image
    const long long row_pitch = (long long)W * C4;          // float4 per input row
    const long long N = (long long)gridDim.x / ((long long)nbands * owb);
    const float4 *xn = reinterpret_cast<const float4 *>(x) + n * H * row_pitch;
    float4 *on = reinterpret_cast<float4 *>(out) + n * (long long)Ho * Wo * C4 + c4;
    const long long x_bytes = 16 * N * H * row_pitch, out_bytes = 16 * N * Ho * Wo * C4;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);

    // -inf columns (outside the image) of every slot row; the copies never touch them
    const int nleft = (ca - col0) * C4, nright = (col0 + seg - max(cb, ca)) * C4;
    for (int i = tid; i < NSTAGE * rps * (nleft + nright); i += 256) {
        const int row = i / (nleft + nright), g = i % (nleft + nright);
        float4 *gp = ring + (size_t)row * pitch + (g < nleft ? g : pitch - nright + (g - nleft));
        if (CHKS(gp, 16)) *gp = ninf;
    }
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t row_bytes = cb > ca ? (uint32_t)(cb - ca) * (uint32_t)C4 * 16u : 0u;
    auto issue = [&](int st) {  // thread 0 only: copy stage `st` into its slot
        const int slot = st % NSTAGE;
        const int row0 = la + st * rps, cnt = min(rps, lb - row0);
        const uint32_t bar = smem_u32(&bars[slot]);
        auto src_of = [&](int r) { return xn + (long long)(row0 + r) * row_pitch + (long long)ca * C4; };
        auto dst_of = [&](int r) { return ring + ((size_t)slot * rps + r) * pitch + (size_t)(ca - col0) * C4; };
        // checked build: rows outside x or the ring are not copied (nor expected)
        int ok_rows = 0;
        for (int r = 0; r < cnt; ++r) ok_rows += CHK(src_of(r), row_bytes, x, x_bytes) && CHKS(dst_of(r), row_bytes);
        mbar_arrive_expect_tx(bar, row_bytes * ok_rows);
        for (int r = 0; r < cnt; ++r)
            if (row_bytes > 0 && (!FW_CHECKED || (CHK(src_of(r), row_bytes, x, x_bytes) && CHKS(dst_of(r), row_bytes))))
                bulk_g2s(smem_u32(dst_of(r)), src_of(r), row_bytes, bar);
    };
    if (tid == 0) {
        fence_proxy_async_smem();
        for (int st = 0; st < min(NSTAGE, nst); ++st) issue(st);
    }

    auto upd4 = [](float4 &m, const float4 &v) {
        m.x = max_nan(m.x, v.x);
        m.y = max_nan(m.y, v.y);
        m.z = max_nan(m.z, v.z);
        m.w = max_nan(m.w, v.w);
    };
    // Register ring of the last K row maxima; row ir lives in hist[(ir - ir_begin) % K],
    // so the unrolled loop below indexes it statically.
    float4 hist[K];
#pragma unroll
    for (int i = 0; i < K; ++i) hist[i] = ninf;
    bool err = false, any_err = false;
    int st = 0, r_in_st = 0, st_rows = min(rps, nrows);
    const int ir_begin = r0 - P, ir_end = r1 - 1 - P + K;  // input rows the band's outputs read
    for (int base = ir_begin; base < ir_end && !any_err; base += K) {
#pragma unroll
        for (int u = 0; u < K; ++u) {
            const int ir = base + u;
            if (ir >= ir_end) break;
            float4 h = ninf;
            if (ir >= la && ir < lb) {
                const int slot = st % NSTAGE;
                if (r_in_st == 0 && !mbar_wait_bounded(smem_u32(&bars[slot]), (uint32_t)(st / NSTAGE) & 1u))
                    err = true;
                const float4 *row = ring + ((size_t)slot * rps + r_in_st) * pitch + (size_t)oc * C4 + c4;
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (CHKS(row + j * C4, 16)) upd4(h, row[j * C4]);
                if (++r_in_st == st_rows) {  // stage consumed: release the slot, refill it
                    if (__syncthreads_or(err)) {
                        if (tid == 0) atomicOr(&g_err_maxpool, DEVERR_TIMEOUT);
                        any_err = true;
                        break;
                    }
                    if (tid == 0 && st + NSTAGE < nst) {
                        fence_proxy_async_smem();
                        issue(st + NSTAGE);
                    }
                    ++st;
                    r_in_st = 0;
                    st_rows = min(rps, lb - (la + st * rps));
                }
            }
            hist[u] = h;
            const int oh = ir + P - (K - 1);  // output row whose last window row is ir
            if (oh >= r0 && store) {
                float4 m = hist[(u + 1) % K];
#pragma unroll
                for (int i = 2; i <= K; ++i) upd4(m, hist[(u + i) % K]);
                if (m.x == 0.f || m.y == 0.f || m.z == 0.f || m.w == 0.f) {
                    const float *img = x + n * H * (long long)W * (4 * C4) + 4 * c4;
                    if (m.x == 0.f) m.x = window_max_exact_nhwc<K>(img, H, W, 4 * C4, oh, ow, P, x, x_bytes);
                    if (m.y == 0.f) m.y = window_max_exact_nhwc<K>(img + 1, H, W, 4 * C4, oh, ow, P, x, x_bytes);
                    if (m.z == 0.f) m.z = window_max_exact_nhwc<K>(img + 2, H, W, 4 * C4, oh, ow, P, x, x_bytes);
                    if (m.w == 0.f) m.w = window_max_exact_nhwc<K>(img + 3, H, W, 4 * C4, oh, ow, P, x, x_bytes);
                }
                float4 *o = on + ((long long)oh * Wo + ow) * C4;
                if (CHK(o, 16, out, out_bytes)) *o = m;
            }
        }
    }
    if (any_err && tid == 0) {
        // Drain copies still in flight into this CTA's shared memory (bounded).
        for (int s2 = st; s2 < min(nst, st + NSTAGE); ++s2)
            mbar_wait_bounded(smem_u32(&bars[s2 % NSTAGE]), (uint32_t)(s2 / NSTAGE) & 1u);
    }
}

// Any (k, s, p, d) and C: one thread per output value, taps in row-major order.
__global__ void maxpool_nhwc_direct_kernel(const float *__restrict__ x, float *__restrict__ out, long long total,
                                           int H, int W, int C, int Ho, int Wo, int k, int s, int p, int d) {
    const long long x_elems = total / ((long long)Ho * Wo) * H * W;  // N * C * H * W
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % C);
        long long t = idx / C;
        const int ow = (int)(t % Wo);
        t /= Wo;
        const int oh = (int)(t % Ho);
        const long long n = t / Ho;
        const float *img = x + n * H * (long long)W * C + c;
        float m = -INFINITY;
        for (int i = 0; i < k; ++i) {
            const int ih = oh * s - p + i * d;
            const bool rin = ih >= 0 && ih < H;
            for (int j = 0; j < k; ++j) {
                const int iw = ow * s - p + j * d;
                const float *a = img + ((long long)ih * W + iw) * C;
                const float v = (rin && iw >= 0 && iw < W && CHK(a, 4, x, 4 * x_elems)) ? __ldg(a) : -INFINITY;
                m = max_update(m, v);
            }
        }
        if (CHK(out + idx, 4, out, 4 * total)) out[idx] = m;
    }
}

template <int K>
fw_status launch_nhwc_s1(const float *x, float *out, int N, int H, int W, int C, int Ho, int Wo, int p,
                         cudaStream_t st) {
    const int C4 = C / 4;
    const int cols = 256 / C4;  // output columns per block
    const int band = Ho <= 64 ? Ho : 64;
    const int nbands = (Ho + band - 1) / band;
    const int owb = (Wo + cols - 1) / cols;
    const long long blocks = (long long)N * nbands * owb;
    if (blocks > 0x7fffffffLL) return FW_ERR_SHAPE;
    // About 24 KB per bulk-copy stage (two stages: ~48 KB of shared memory, 4 CTAs per SM
    // at 64 registers); 12 KB stages measured 0.88 ms against 0.65 ms, 48 KB ones 0.75 ms
    const int slot_row_bytes = (cols + K - 1) * C4 * 16;
    const int rps = max(1, min(8, 24576 / slot_row_bytes));
    const size_t smem = 64 + (size_t)NSTAGE * rps * slot_row_bytes;
    cudaError_t e = cudaFuncSetAttribute(maxpool_nhwc_s1_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    maxpool_nhwc_s1_kernel<K><<<(unsigned)blocks, 256, smem, st>>>(x, out, H, W, C4, Ho, Wo, p, band, nbands, owb,
                                                                   rps);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace

fw_status maxpool2d_nhwc_launch(const float *x, int N, int H, int W, int C, int k, int s, int p, int d, int Ho,
                                int Wo, float *out, cudaStream_t st) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
    if (s == 1 && d == 1 && aligned && C % 4 == 0 && C <= 1024) {
        switch (k) {
            case 1: return launch_nhwc_s1<1>(x, out, N, H, W, C, Ho, Wo, p, st);
            case 2: return launch_nhwc_s1<2>(x, out, N, H, W, C, Ho, Wo, p, st);
            case 3: return launch_nhwc_s1<3>(x, out, N, H, W, C, Ho, Wo, p, st);
            case 4: return launch_nhwc_s1<4>(x, out, N, H, W, C, Ho, Wo, p, st);
            case 5: return launch_nhwc_s1<5>(x, out, N, H, W, C, Ho, Wo, p, st);
        }
    }
    const long long total = (long long)N * Ho * Wo * C;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    maxpool_nhwc_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(x, out, total, H, W, C, Ho, Wo, k, s, p, d);
    note_launch();
    return launch_status(cudaGetLastError());
}

unsigned maxpool_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_maxpool, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_maxpool, &zero, sizeof(zero));
    return v;
}

fw_status maxpool2d_ex_launch(const float *x, long long NC, int H, int W, int k, int s, int p, int d, int Ho,
                              int Wo, float *out, long long *idx, cudaStream_t st) {
    const long long total = NC * Ho * Wo;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    maxpool_direct_ex_kernel<<<(unsigned)blocks, threads, 0, st>>>(x, out, idx, NC, H, W, Ho, Wo, k, s, p, d);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace fw
