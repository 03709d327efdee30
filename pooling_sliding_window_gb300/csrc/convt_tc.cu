// convt_tc.cu -- ConvTranspose2d(k4, s2, p1) -> softmax(dim 1) -> +bias -> *scale ->
// sigmoid on the 5th-generation tensor cores (tcgen05.mma kind::tf32, accumulators
// in TMEM) for Cout = 128 (trace "Kimi-K2.6 l2_p91": the model, its 4-phase
// sub-pixel decomposition and the per-pixel channel softmax).
//
// Each output parity class (py, px) -- a "phase" -- is the GEMM
//   D[pixel][co] = sum_{taps (dy,dx) of the phase} sum_ci x[ci][m+dy][n+dx] * W_tap[ci][co]
// with M = pixels, N = 128 channels, K = 4 taps x Cin.
//
// Layout that turns every tap into a shared-memory address offset:
//   * the batch is read as one sequence of "positions": images stacked
//     vertically, each row W+1 wide (the extra column reads as zero) and one zero
//     row above every image, so position q = R*(W+1) + c with R = n*(H+1) + row + 1;
//   * output pixel (n, m, nn) of a phase is "anchor" a = (n*(H+1)+m)*(W+1)+nn and
//     reads position a + (W+1) + dy*(W+1) + dx for tap (dy, dx); the shared zero
//     row/column supply exactly the out-of-range taps, including the extra output
//     row/column that output_padding adds;
//   * the operand A of a 128-anchor tile is thus 128 consecutive positions.  Staged
//     in shared memory as planes of 4 channels (16 bytes per position: K-major core
//     matrices whose 8-row groups are 128 bytes apart), a horizontal tap is a start
//     address 16 bytes further on and a vertical tap a second "slab".
//
// CTA roles (288 threads, one CTA per SM, persistent over the tiles of one phase):
//   warps 0-3  producers: gather the 129 positions x Cin channels a slab needs from
//              NCHW x, round to TF32, write the planar shared layout (2 stages);
//   warp  8    allocates TMEM; one lane issues the MMAs: per tile 2 slabs (vertical
//              taps) x 2 horizontal taps x Cin/8 K-steps into one of two 128-column
//              accumulators;
//   warps 4-7  epilogue: each thread owns one pixel (a TMEM lane), reads its 128
//              channel sums, adds the conv bias, takes the softmax in registers and
//              writes sigmoid((p + bias) * scale).
// The phase's weights (TF32, 2*Cin KB) stay resident in shared memory; they are
// rewritten into the caller's workspace by convt_tc_prepack_kernel.
// TF32 operands (10-bit mantissa) are enough here: the channel softmax scales an
// error dy in the conv-transpose output by p(1-p) <= 1/4 and then by the sigmoid
// slope times the scale, so the result stays within 1e-5 of the float64 oracle.
#include "fw_common.cuh"

namespace fw {

__device__ unsigned g_err_convt_tc = 0;

namespace {

constexpr int COUT = 128;
constexpr int MT = 128;            // anchors per tile
constexpr int SLAB_POS = MT + 1;   // positions per slab (two horizontal taps)
constexpr int NSTAGE = 2;          // slab stages
constexpr int NTHREADS = 288;
constexpr int MMA_WARP = 8;
constexpr uint32_t IDESC = tc::idesc_tf32(128, COUT);
constexpr size_t MIN_SMEM = 116 * 1024;  // > half an SM: one CTA per SM

// Tap tables of the k4 s2 p1 decomposition (output parity q, tap index t in {0,1}):
// kernel index and input offset (input row = m + offset).
__host__ __device__ __forceinline__ int tap_k(int q, int t) { return q == 0 ? (t == 0 ? 1 : 3) : (t == 0 ? 0 : 2); }
__host__ __device__ __forceinline__ int tap_off(int q, int t) { return q == 0 ? (t == 0 ? 0 : -1) : (t == 0 ? 1 : 0); }

// wtc[phase][t = 2*ty + tx][g][co][c4] = tf32(w[4g + c4][co][kh(py,ty)][kw(px,tx)])
__global__ void convt_tc_prepack_kernel(const float *__restrict__ w, float *__restrict__ wtc, int Cin) {
    const int G = Cin / 4;
    const long long total = 16LL * Cin * COUT;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c4 = (int)(i & 3);
        long long r = i >> 2;
        const int co = (int)(r % COUT);
        r /= COUT;
        const int g = (int)(r % G);
        r /= G;
        const int t = (int)(r & 3), phase = (int)(r >> 2);
        const int py = phase >> 1, px = phase & 1;
        const int kh = tap_k(py, t >> 1), kw = tap_k(px, t & 1);
        wtc[i] = tc::to_tf32(__ldg(w + (((long long)(4 * g + c4) * COUT + co) * 4 + kh) * 4 + kw));
    }
}

struct Bars {
    uint64_t b_full;
    uint64_t slab_full[NSTAGE];
    uint64_t slab_empty[NSTAGE];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
};

template <int G>  // input channels / 4
__global__ void __launch_bounds__(NTHREADS, 1)
convt_k4s2_tc_kernel(const float *__restrict__ x, const float *__restrict__ wtc, const float *__restrict__ cb,
                     const float *__restrict__ bias, float scale, float *__restrict__ out, int N, int H, int W,
                     int Ho, int Wo) {
    constexpr int CIN = 4 * G;
    constexpr int B_BYTES = 4 * G * COUT * 16;  // 4 taps x G planes x 128 co x 16 B
    constexpr int SLAB_PLANE = SLAB_POS * 16;   // bytes per plane in a slab
    constexpr int SLAB_BYTES = G * SLAB_PLANE;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *sB = smem;
    unsigned char *sSlab = smem + B_BYTES;
    float *sCb = reinterpret_cast<float *>(sSlab + NSTAGE * SLAB_BYTES);
    float *sBias = sCb + COUT;
    Bars &bars = *reinterpret_cast<Bars *>(sBias + COUT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int phase = blockIdx.x & 3, py = phase >> 1, px = phase & 1;
    const int rank = blockIdx.x >> 2, nct = gridDim.x >> 2;
    const int BW = W + 1, BH = H + 1;
    const long long n_anchor = (long long)N * BH * BW;
    const long long n_pos = ((long long)N * BH + 1) * BW;
    const int n_tiles = (int)((n_anchor + MT - 1) / MT);
    const int dx0 = px == 0 ? -1 : 0;  // smaller horizontal tap offset of the phase

    for (int i = tid; i < COUT; i += NTHREADS) {
        sCb[i] = cb ? __ldg(cb + i) : 0.f;
        sBias[i] = __ldg(bias + i);
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bars.b_full), 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(smem_u32(&bars.slab_full[s]), 4);
            mbar_init(smem_u32(&bars.slab_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars.acc_full[b]), 1);
            mbar_init(smem_u32(&bars.acc_empty[b]), 4);
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) tc::alloc(smem_u32(&bars.tmem_base), 256);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    volatile int *abort_flag = &bars.abort;

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_err_convt_tc, DEVERR_TIMEOUT);
    };

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        const long long plane_stride = (long long)H * W;
        int k = 0;
        for (int tile = rank; tile < n_tiles && !*abort_flag; tile += nct) {
            for (int s = 0; s < 2; ++s, ++k) {
                const int stage = k & 1, use = k >> 1;
                if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) {
                    fail();
                    break;
                }
                const int dy = tap_off(py, s);
                const long long pbase = (long long)tile * MT + BW + (long long)dy * BW + dx0;
                unsigned char *slab = sSlab + stage * SLAB_BYTES;
                for (int pos = tid; pos < SLAB_POS; pos += 128) {
                    const long long q = pbase + pos;
                    const float *src = nullptr;
                    if (q >= 0 && q < n_pos) {
                        const long long R = q / BW;
                        const int c = (int)(q - R * BW);
                        if (c < W && R > 0) {
                            const long long n = (R - 1) / BH;
                            const int row = (int)(R - 1 - n * BH);
                            if (row < H) src = x + ((n * CIN) * H + row) * (long long)W + c;
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (src) {
                            v.x = tc::to_tf32(__ldg(src + (4 * g + 0) * plane_stride));
                            v.y = tc::to_tf32(__ldg(src + (4 * g + 1) * plane_stride));
                            v.z = tc::to_tf32(__ldg(src + (4 * g + 2) * plane_stride));
                            v.w = tc::to_tf32(__ldg(src + (4 * g + 3) * plane_stride));
                        }
                        *reinterpret_cast<float4 *>(slab + g * SLAB_PLANE + pos * 16) = v;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t bfull = smem_u32(&bars.b_full);
            mbar_arrive_expect_tx(bfull, B_BYTES);
            const unsigned char *src = reinterpret_cast<const unsigned char *>(wtc) + (size_t)phase * B_BYTES;
            for (int off = 0; off < B_BYTES; off += 32768)
                bulk_g2s(smem_u32(sB + off), src + off, (uint32_t)min(32768, B_BYTES - off), bfull);
            bool ok = mbar_wait_bounded(bfull, 0);
            if (!ok) fail();
            tc::fence_after_sync();
            const uint32_t sB_addr = smem_u32(sB), sSlab_addr = smem_u32(sSlab);
            int k = 0, u = 0;
            for (int tile = rank; ok && tile < n_tiles && !*abort_flag; tile += nct, ++u) {
                const int b = u & 1, ause = u >> 1;
                if (ause > 0 && !mbar_wait_bounded(smem_u32(&bars.acc_empty[b]), (ause - 1) & 1)) {
                    fail();
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * COUT);
                for (int s = 0; s < 2; ++s, ++k) {
                    const int stage = k & 1, use = k >> 1;
                    if (!mbar_wait_bounded(smem_u32(&bars.slab_full[stage]), use & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t slab = sSlab_addr + stage * SLAB_BYTES;
#pragma unroll
                    for (int tx = 0; tx < 2; ++tx) {
                        const int o = tap_off(px, tx) - dx0;  // 0 or 1 position
                        const int tap = 2 * s + tx;
#pragma unroll
                        for (int j = 0; j < G / 2; ++j) {
                            const uint64_t ad = tc::smem_desc(slab + (2 * j * SLAB_POS + o) * 16, SLAB_PLANE, 128);
                            const uint64_t bd =
                                tc::smem_desc(sB_addr + (tap * G + 2 * j) * (COUT * 16), COUT * 16, 128);
                            tc::mma_tf32(d, ad, bd, IDESC, (s | tx | j) != 0);
                        }
                    }
                    tc::commit(smem_u32(&bars.slab_empty[stage]));
                }
                if (!ok) break;
                tc::commit(smem_u32(&bars.acc_full[b]));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const long long img_anchors = (long long)BH * BW;
        const long long plane_out = (long long)Ho * Wo;
        int u = 0;
        for (int tile = rank; tile < n_tiles && !*abort_flag; tile += nct, ++u) {
            const int b = u & 1;
            if (!mbar_wait_bounded(smem_u32(&bars.acc_full[b]), (u >> 1) & 1)) {
                fail();
                break;
            }
            tc::fence_after_sync();
            float v[COUT];
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * COUT);
#pragma unroll
            for (int c = 0; c < COUT / 32; ++c) tc::ld32(taddr + 32 * c, v + 32 * c);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[b]));

            const long long a = (long long)tile * MT + 32 * q + lane;
            const long long n = a / img_anchors;
            const int rem = (int)(a - n * img_anchors);
            const int m = rem / BW, nn = rem - m * BW;
            const int oh = 2 * m + py, ow = 2 * nn + px;
            const bool valid = a < n_anchor && oh < Ho && ow < Wo;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < COUT; ++c) {
                v[c] += sCb[c];
                mx = fmaxf(mx, v[c]);
            }
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < COUT; ++c) {
                v[c] = __expf(v[c] - mx);
                sum += v[c];
            }
            const float inv = __frcp_rn(sum);
            if (valid) {
                float *o = out + (n * COUT) * plane_out + (long long)oh * Wo + ow;
#pragma unroll
                for (int c = 0; c < COUT; ++c) {
                    const float r = __fmul_rn(__fadd_rn(v[c] * inv, sBias[c]), scale);
                    o[c * plane_out] = __frcp_rn(1.f + __expf(-r));
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after_sync();
        tc::dealloc(tmem, 256);
    }
}

template <int G>
fw_status launch_g(const float *x, int N, int H, int W, const float *wtc, const float *cb, const float *bias,
                   float scale, float *out, int Ho, int Wo, cudaStream_t st) {
    constexpr int B_BYTES = 4 * G * COUT * 16;
    constexpr int SLAB_BYTES = G * SLAB_POS * 16;
    size_t smem = (size_t)B_BYTES + NSTAGE * SLAB_BYTES + 2 * COUT * 4 + sizeof(Bars);
    if (smem < MIN_SMEM) smem = MIN_SMEM;
    cudaError_t e = cudaFuncSetAttribute(convt_k4s2_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FW_ERR_LAUNCH;
    const long long tiles = ((long long)N * (H + 1) * (W + 1) + MT - 1) / MT;
    int per_phase = sms / 4 > 0 ? sms / 4 : 1;
    if (per_phase > tiles) per_phase = (int)tiles;
    convt_k4s2_tc_kernel<G><<<4 * per_phase, NTHREADS, smem, st>>>(x, wtc, cb, bias, scale, out, N, H, W, Ho, Wo);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace

bool convt_tc_eligible(int Cin, int Cout, int k, int s, int p) {
    return k == 4 && s == 2 && p == 1 && Cout == COUT && (Cin == 8 || Cin == 16 || Cin == 32 || Cin == 64);
}

fw_status convt_tc_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                          const float *bias, float scale, float *out, int Ho, int Wo, void *ws, cudaStream_t st) {
    float *wtc = static_cast<float *>(ws);
    const long long total = 16LL * Cin * COUT;
    convt_tc_prepack_kernel<<<(unsigned)min(1024LL, (total + 255) / 256), 256, 0, st>>>(w, wtc, Cin);
    note_launch();
    fw_status rc = launch_status(cudaGetLastError());
    if (rc != FW_OK) return rc;
    switch (Cin) {
        case 8: return launch_g<2>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 16: return launch_g<4>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 32: return launch_g<8>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 64: return launch_g<16>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
    }
    return FW_ERR_UNSUPPORTED;
}

unsigned convt_tc_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convt_tc, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convt_tc, &zero, sizeof(zero));
    return v;
}

}  // namespace fw
