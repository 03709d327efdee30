// convpool.cu -- fused Conv2d(3x3, stride 1, no padding) -> tanh -> *scale ->
// +bias -> MaxPool2d(k, stride k) (trace "Kimi-K2.6 l2_p82").
//
// The page reasons that max over a window of scale*tanh(y)+b equals
// scale*tanh(max y)+b because tanh is increasing (the monotone-reorder
// argument); with pool stride = pool kernel, every conv output feeds exactly one
// pooled output, so the conv, the window max and the epilogue fuse into one
// kernel without recomputation and the conv intermediate never leaves registers.
//
// Tiled FFMA kernel (KH = KW = 3, pool_s = pool_k in {2, 4}, Cin <= 16):
//   * a work item is a 16 x 32 block of conv pixels (4x8 pooled outputs for pool 4,
//     8x16 for pool 2) of one image and a block of up to 32 output channels; CTAs
//     are persistent over items;
//   * the input tile (16+2) x (32+2) x Cin with its 3x3 halo and the block's
//     weights are staged in shared memory by cp.async, two buffers deep: the next
//     item's copies are in flight while the current item is computed (rows padded
//     to 36 floats so every thread's 6-wide row segment is one 16-byte + one 8-byte
//     load);
//   * each thread accumulates a 4 x 4 conv-pixel block for 4 output channels
//     (64 FP32 accumulators) -- an implicit GEMM with K = Cin*9 on the FMA pipe;
//     a warp shares its 4 channels, so weight reads are shared-memory broadcasts;
//   * the window max (min when scale < 0; max.NaN / min.NaN) is taken in registers,
//     the conv bias is added, and tanh / scale / bias run once per pooled output.
// Direct kernel: one thread per pooled output, every other shape.
#include <cstdlib>

#include "fw_common.cuh"

namespace fw {

// Range violations found by the checked build's kernels in this file.
__device__ unsigned g_err_convpool = 0;
#define CHK(p, bytes, base, base_bytes) chk(&g_err_convpool, (p), (bytes), (base), (base_bytes))
#define CHKS(p, bytes) chk_smem(&g_err_convpool, (p), (bytes))

namespace {

constexpr int TILE_R = 16, TILE_C = 32;          // conv pixels per CTA
constexpr int XR = TILE_R + 2, XC = TILE_C + 2;  // staged input rows / cols
constexpr int XP = 36;                            // shared row pitch (floats)
constexpr int MAX_CIN = 16;
constexpr int MAX_COB = 32;                       // output channels per CTA

__device__ __forceinline__ float epilogue(float m, float cbv, float scale, float b) {
    const float t = tanh_fast(m + cbv);
    return __fadd_rn(__fmul_rn(t, scale), b);
}

template <int POOL>
__global__ void __launch_bounds__(256, 2)
convpool3x3_ffma_kernel(const float *__restrict__ x, const float *__restrict__ w,
                        const float *__restrict__ cb, const float *__restrict__ bias, float scale,
                        float *__restrict__ out, int N, int Cin, int H, int W, int Cout, int Ho, int Wo,
                        int tiles_w, int tiles, int ncob, int cob, bool vec) {
    extern __shared__ __align__(16) float sm[];
    // The weights [Cin][9][cob] of this CTA's channel block (resident), then two input
    // buffers [Cin][XR][XP].  CTA b serves channel block b % ncob; its items are the
    // (image, tile) pairs j = b / ncob, b / ncob + gridDim.x / ncob, ...
    const int XS = Cin * XR * XP, WSZ = Cin * 9 * cob;
    float *ws = sm, *xbuf = sm + WSZ;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int co0 = (int)(blockIdx.x % ncob) * cob;
    const long long per_block = (long long)N * tiles;
    const int gstride = gridDim.x / ncob;
    // buffer extents for the checked build
    const long long x_bytes = 4LL * N * Cin * H * W, w_bytes = 4LL * Cout * Cin * 9;
    const long long out_bytes = 4LL * N * Cout * Ho * Wo;
    for (int e = tid; e < WSZ; e += blockDim.x) {
        const int j = e % cob, u = e / cob, tap = u % 9, ci = u / 9;
        const int co = co0 + j;
        const bool ok = co < Cout;
        const float *src = ok ? w + ((long long)co * Cin + ci) * 9 + tap : w;
        if (CHK(src, 4, w, w_bytes) && CHKS(ws + e, 4)) cp_async4(smem_u32(ws + e), src, ok ? 4u : 0u);
    }
    // copies of item j's input tile into buffer b, zero-filled outside x: per staged row, eight
    // 16-byte copies and two 4-byte ones when x rows are 16-byte aligned, else 34 4-byte ones
    auto stage = [&](long long j, int b) {
        const long long n = j / tiles;
        const int tile = (int)(j - n * tiles);
        const int tr = tile / tiles_w, tcl = tile - tr * tiles_w;
        const int row0 = tr * TILE_R, col0 = tcl * TILE_C;
        const float *xn = x + n * Cin * H * W;
        float *xsb = xbuf + b * XS;
        if (vec) {
            for (int e = tid; e < Cin * XR * 10; e += blockDim.x) {
                const int row = e / 10, k = e - row * 10, ci = row / XR, r = row - ci * XR;
                const int ih = row0 + r;
                const int c = k < 8 ? 4 * k : 24 + k;  // k = 8, 9: columns 32, 33
                const bool ok = ih < H && col0 + c < W;  // W % 4 == 0: a 16-byte piece is all in or out
                const float *src = ok ? xn + ((long long)ci * H + ih) * W + col0 + c : x;
                const int nb = k < 8 ? 16 : 4;
                if (!(CHK(src, ok ? nb : 0, x, x_bytes) && CHKS(xsb + row * XP + c, nb))) continue;
                if (k < 8)
                    cp_async16(smem_u32(xsb + row * XP + c), src, ok ? 16u : 0u);
                else
                    cp_async4(smem_u32(xsb + row * XP + c), src, ok ? 4u : 0u);
            }
        } else {
            for (int e = tid; e < Cin * XR * XC; e += blockDim.x) {
                const int c = e % XC, u = e / XC, r = u % XR, ci = u / XR;
                const int ih = row0 + r, iw = col0 + c;
                const bool ok = ih < H && iw < W;
                const float *src = ok ? xn + ((long long)ci * H + ih) * W + iw : x;
                if (CHK(src, ok ? 4 : 0, x, x_bytes) && CHKS(xsb + (ci * XR + r) * XP + c, 4))
                    cp_async4(smem_u32(xsb + (ci * XR + r) * XP + c), src, ok ? 4u : 0u);
            }
        }
        cp_async_commit();
    };
    const long long j0 = blockIdx.x / ncob;
    if (j0 < per_block)
        stage(j0, 0);  // (the weights' copies join this group)
    else
        cp_async_commit();
    int it = 0;
    for (long long j = j0; j < per_block; j += gstride, ++it) {
        const int b = it & 1;
        if (j + gstride < per_block)
            stage(j + gstride, b ^ 1);
        else
            cp_async_commit();  // an empty group keeps the wait count uniform
        cp_async_wait<1>();     // this item's copies (of every thread, after the barrier) have landed
        __syncthreads();
        const float *xs = xbuf + b * XS;
        const long long n = j / tiles;
        const int tile = (int)(j - n * tiles);
        const int tr = tile / tiles_w, tcl = tile - tr * tiles_w;
        const int row0 = tr * TILE_R, col0 = tcl * TILE_C;

        const int pr = lane >> 3, pc = lane & 7;  // 4x4 conv-pixel block (pr, pc)
        const int cw = warp * 4;                  // this warp's channels [cw, cw+4) of the block
        float acc[4][4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[r][c][j] = 0.f;

#pragma unroll 2
        for (int ci = 0; ci < Cin; ++ci) {
            float xv[6][6];
            const float *xr = xs + (ci * XR + 4 * pr) * XP + 4 * pc;
            const float *wr = ws + ci * 9 * cob + cw;
            if (!(CHKS(xr, (5 * XP + 6) * 4) && CHKS(wr, (8 * cob + 4) * 4))) continue;
#pragma unroll
            for (int r = 0; r < 6; ++r) {
                const float4 a = *reinterpret_cast<const float4 *>(xr + r * XP);
                const float2 b = *reinterpret_cast<const float2 *>(xr + r * XP + 4);
                xv[r][0] = a.x; xv[r][1] = a.y; xv[r][2] = a.z; xv[r][3] = a.w;
                xv[r][4] = b.x; xv[r][5] = b.y;
            }
#pragma unroll
            for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                for (int kw = 0; kw < 3; ++kw) {
                    const float4 wv = *reinterpret_cast<const float4 *>(wr + (kh * 3 + kw) * cob);
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float xx = xv[r + kh][c + kw];
                            acc[r][c][0] = fmaf(xx, wv.x, acc[r][c][0]);
                            acc[r][c][1] = fmaf(xx, wv.y, acc[r][c][1]);
                            acc[r][c][2] = fmaf(xx, wv.z, acc[r][c][2]);
                            acc[r][c][3] = fmaf(xx, wv.w, acc[r][c][3]);
                        }
                }
        }

        // Window reduction + epilogue.  Pool windows tile the 4x4 block exactly; the window
        // extreme is max.NaN (min.NaN when scale < 0), one instruction per value.
        constexpr int NW = 4 / POOL;  // windows per block side
        float mw[4][NW][NW];
        auto reduce = [&](auto ext) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int wr_ = 0; wr_ < NW; ++wr_)
#pragma unroll
                    for (int wc = 0; wc < NW; ++wc) {
                        float m = acc[wr_ * POOL][wc * POOL][j];
#pragma unroll
                        for (int u = 0; u < POOL; ++u)
#pragma unroll
                            for (int v = 0; v < POOL; ++v)
                                if (u != 0 || v != 0) m = ext(m, acc[wr_ * POOL + u][wc * POOL + v][j]);
                        mw[j][wr_][wc] = m;
                    }
        };
        if (scale < 0.f)
            reduce([](float a, float b) { return min_nan(a, b); });
        else
            reduce([](float a, float b) { return max_nan(a, b); });
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int co = co0 + cw + j;
            if (co >= Cout) continue;
            const float cbv = cb ? __ldg(cb + co) : 0.f;
            const float bv = __ldg(bias + co);
            float *oc = out + ((long long)n * Cout + co) * Ho * Wo;
#pragma unroll
            for (int wr_ = 0; wr_ < NW; ++wr_)
#pragma unroll
                for (int wc = 0; wc < NW; ++wc) {
                    const int ph = (row0 + 4 * pr) / POOL + wr_;
                    const int pw = (col0 + 4 * pc) / POOL + wc;
                    if (ph < Ho && pw < Wo && CHK(oc + (long long)ph * Wo + pw, 4, out, out_bytes))
                        oc[(long long)ph * Wo + pw] = epilogue(mw[j][wr_][wc], cbv, scale, bv);
                }
        }
        __syncthreads();  // buffer b is free for the item after next
    }
    cp_async_wait<0>();
}

// One thread per pooled output: the window's conv values computed directly.
__global__ void convpool_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                       const float *__restrict__ cb, const float *__restrict__ bias,
                                       float scale, float *__restrict__ out, int N, int Cin, int H,
                                       int W, int Cout, int KH, int KW, int pk, int ps, int Ho,
                                       int Wo) {
    const long long total = (long long)N * Cout * Ho * Wo;
    const bool use_min = scale < 0.f;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int pw = (int)(idx % Wo);
        long long t = idx / Wo;
        const int ph = (int)(t % Ho);
        t /= Ho;
        const int co = (int)(t % Cout);
        const int n = (int)(t / Cout);
        float m = 0.f;
        for (int u = 0; u < pk; ++u)
            for (int v = 0; v < pk; ++v) {
                const int oh = ph * ps + u, ow = pw * ps + v;
                float y = 0.f;
                for (int ci = 0; ci < Cin; ++ci) {
                    const float *xp = x + (((long long)n * Cin + ci) * H + oh) * W + ow;
                    const float *wp = w + ((long long)co * Cin + ci) * KH * KW;
                    for (int i = 0; i < KH; ++i)
                        for (int j = 0; j < KW; ++j) {
                            const float *xa = xp + (long long)i * W + j, *wa = wp + i * KW + j;
                            if (CHK(xa, 4, x, 4LL * N * Cin * H * W) && CHK(wa, 4, w, 4LL * Cout * Cin * KH * KW))
                                y = fmaf(__ldg(xa), __ldg(wa), y);
                        }
                }
                if (u == 0 && v == 0) m = y;
                else m = use_min ? min_update(m, y) : max_update(m, y);
            }
        if (CHK(out + idx, 4, out, 4 * total)) out[idx] = epilogue(m, cb ? __ldg(cb + co) : 0.f, scale, __ldg(bias + co));
    }
}

template <int POOL>
fw_status launch_tiled(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                       int Cout, float scale, const float *bias, float *out, int Ho, int Wo,
                       cudaStream_t st) {
    const int tiles_h = (Ho * POOL + TILE_R - 1) / TILE_R;
    const int tiles_w = (Wo * POOL + TILE_C - 1) / TILE_C;
    const int cob = min(MAX_COB, (Cout + 3) / 4 * 4);
    const int threads = cob / 4 * 32;
    const size_t smem = (size_t)Cin * (2 * XR * XP + 9 * cob) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(convpool3x3_ffma_kernel<POOL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, convpool3x3_ffma_kernel<POOL>, threads, smem) !=
            cudaSuccess)
        return FW_ERR_LAUNCH;
    const int tiles = tiles_h * tiles_w, ncob = (Cout + cob - 1) / cob;
    const long long per_block = (long long)N * tiles;
    long long per_cob = (long long)sms * (per_sm > 0 ? per_sm : 1) / ncob;  // persistent: one wave
    if (per_cob < 1) per_cob = 1;
    if (per_cob > per_block) per_cob = per_block;
    const int grid = (int)(per_cob * ncob);
    const bool vec = W % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    convpool3x3_ffma_kernel<POOL><<<grid, threads, smem, st>>>(x, w, cb, bias, scale, out, N, Cin, H, W, Cout, Ho,
                                                              Wo, tiles_w, tiles, ncob, cob, vec);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace

bool convpool_tc_eligible(int Cin, int Cout, int KH, int KW, int pk, int ps);
fw_status convpool_tc_launch(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                             float scale, const float *bias, int pk, float *out, int Ho, int Wo, bool x3,
                             cudaStream_t st);

// FUSEDWIN_CONVPOOL_FFMA=1 in the environment selects the FP32-FMA tiled kernel
// instead of the tensor-core one (used to cross-check the two).
static bool convpool_force_ffma() {
    static const bool v = [] {
        const char *e = getenv("FUSEDWIN_CONVPOOL_FFMA");
        return e && e[0] == '1';
    }();
    return v;
}

// mode 0: the tensor-core kernel with the 3xTF32 split where it applies; 1: the same
// with one TF32 product per K step; 2: float32 FMA kernels only.
fw_status convpool_launch(const float *x, int N, int Cin, int H, int W, const float *w,
                          const float *cb, int Cout, int KH, int KW, float scale, const float *bias,
                          int pk, int ps, float *out, int Ho, int Wo, int mode, cudaStream_t st) {
    if (mode != 2 && convpool_tc_eligible(Cin, Cout, KH, KW, pk, ps) && !convpool_force_ffma())
        return convpool_tc_launch(x, N, H, W, w, cb, Cout, scale, bias, pk, out, Ho, Wo, mode == 0, st);
    if (KH == 3 && KW == 3 && pk == ps && Cin <= MAX_CIN && (pk == 4 || pk == 2)) {
        if (pk == 4) return launch_tiled<4>(x, N, Cin, H, W, w, cb, Cout, scale, bias, out, Ho, Wo, st);
        return launch_tiled<2>(x, N, Cin, H, W, w, cb, Cout, scale, bias, out, Ho, Wo, st);
    }
    const long long total = (long long)N * Cout * Ho * Wo;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    convpool_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(x, w, cb, bias, scale, out, N, Cin, H,
                                                                 W, Cout, KH, KW, pk, ps, Ho, Wo);
    note_launch();
    return launch_status(cudaGetLastError());
}

unsigned convpool_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convpool, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convpool, &zero, sizeof(zero));
    return v;
}

}  // namespace fw
