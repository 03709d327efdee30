// convpool_tc.cu -- fused Conv2d(3x3, stride 1, no padding) -> tanh -> *scale ->
// +bias -> MaxPool2d(P, stride P) on the 5th-generation tensor cores (tcgen05.mma
// kind::tf32 with accumulators in TMEM), trace "Kimi-K2.6 l2_p82": the model and
// its monotone-reorder argument (the window max commutes with the increasing
// map y -> scale*tanh(y)+b, so tanh runs once per pooled output).
//
// Precision: a single TF32 product keeps 11 significant bits, about 1e-3 of
// error after tanh -- too coarse for a 1e-5 bound.  Each operand is split as
// v = hi + lo with hi = tf32(v) and lo = tf32(v - hi), and the product is
// accumulated as hi*hi + lo*hi + hi*lo (the lo*lo term, ~2^-22 relative, is
// dropped): three MMAs per K step, float32 accumulation in TMEM.
//
// Work item = one pooled output row of one image and a block of 128 conv columns:
//   * the P conv rows of the pooled row are P GEMMs, M = 128 columns, N = Cout,
//     K = 9 taps x 8 channels, each into its own TMEM accumulator;
//   * the input the item reads -- P+2 rows x 130 columns x 8 channels -- is staged
//     as hi and lo planes of 4 channels (16 bytes per position, row pitch 130
//     positions), so tap (kh, kw) of conv row j is the start address of the MMA's
//     A operand moved by (j+kh)*130 + kw positions;
//   * the weights, split into hi/lo in the CTA prologue, stay resident.
// CTA roles (416 threads, one CTA per SM, persistent over items):
//   warps 0-3   producers: load and split a slab (two stages);
//   warp  12    allocates TMEM; one lane issues 3 x 9 x P MMAs per item into one of
//               two accumulator sets;
//   warps 4-11  epilogue, every warp on every item (warps 4-7 and 8-11 take
//              alternate 16-channel chunks): a thread owns one conv column (TMEM
//              lane) of one TMEM lane quarter; the max over
//              the P rows is taken in registers, the max over the P columns of a
//              window by a butterfly over lanes that halves the channels each lane
//              keeps at every step, then out = bias + scale*tanh(m + conv_b).
// Scale < 0 takes the window minimum instead (the map is then decreasing).
#include "fw_common.cuh"

namespace fw {

__device__ unsigned g_err_convpool_tc = 0;

namespace {

constexpr int MT = 128;       // conv columns per item (MMA M)
constexpr int SW = MT + 2;    // slab row pitch in positions
constexpr int NSTAGE = 2;
constexpr int EPI_WARP0 = 4;     // warps 4-11: epilogue
constexpr int MMA_WARP = 12;
constexpr int NTHREADS = (MMA_WARP + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int ACC_STRIDE = 256;  // TMEM columns between the two accumulator sets

struct Bars {
    uint64_t slab_full[NSTAGE];
    uint64_t slab_empty[NSTAGE];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
};

template <int G, int P, int N>
struct Cfg {
    static constexpr int CIN = 4 * G;
    static constexpr int ROWS = P + 2;
    static constexpr int PLANE = ROWS * SW * 16;      // bytes per 4-channel plane
    static constexpr int SPLIT = G * PLANE;           // hi (or lo) half of a slab
    static constexpr int SLAB = 2 * SPLIT;
    static constexpr int BPLANE = N * 16;             // bytes per (split, tap, plane) of B
    static constexpr int B_BYTES = 2 * 9 * G * BPLANE;
    static constexpr int NITER = (ROWS * SW + 127) / 128;
    static constexpr size_t SMEM = (size_t)B_BYTES + NSTAGE * SLAB + 2 * N * 4 + sizeof(Bars);
};

__device__ __forceinline__ float upd(float m, float v, bool use_min) {
    return use_min ? min_update(m, v) : max_update(m, v);
}

// tanh(z) = 1 - 2 / (1 + e^(2z)) with a base-2 exponential and a fast reciprocal:
// absolute error a few 1e-7 over all z (e^(2z) overflows to inf for large z and
// gives exactly 1; underflows to 0 for very negative z and gives exactly -1).
__device__ __forceinline__ float tanh_fast(float z) {
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * (2.f * LOG2E)));
    return 1.f - __fdividef(2.f, 1.f + e);
}

template <int G, int P, int N>
__global__ void __launch_bounds__(NTHREADS, 1)
convpool_tc_kernel(const float *__restrict__ x, const float *__restrict__ w, const float *__restrict__ cb,
                   const float *__restrict__ bias, float scale, float *__restrict__ out, int Nimg, int H, int W,
                   int Ho, int Wo, int ncb) {
    using C = Cfg<G, P, N>;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *sB = smem;
    unsigned char *sSlab = smem + C::B_BYTES;
    float *sCb = reinterpret_cast<float *>(sSlab + NSTAGE * C::SLAB);
    float *sBias = sCb + N;
    Bars &bars = *reinterpret_cast<Bars *>(sBias + N);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long n_items = (long long)Nimg * Ho * ncb;
    const bool use_min = scale < 0.f;

    for (int i = tid; i < N; i += NTHREADS) {
        sCb[i] = cb ? __ldg(cb + i) : 0.f;
        sBias[i] = __ldg(bias + i);
    }
    // Weights split into TF32 hi/lo: B[split][tap][plane][co][c4].
    for (int e = tid; e < 9 * C::CIN * N; e += NTHREADS) {
        const int co = e % N, t = e / N, ci = t % C::CIN, tap = t / C::CIN;
        const float v = __ldg(w + ((long long)co * C::CIN + ci) * 9 + tap);
        const float hi = tc::to_tf32(v), lo = tc::to_tf32(v - hi);
        const int off = ((tap * G + ci / 4) * N + co) * 16 + (ci % 4) * 4;
        *reinterpret_cast<float *>(sB + off) = hi;
        *reinterpret_cast<float *>(sB + 9 * G * C::BPLANE + off) = lo;
    }
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(smem_u32(&bars.slab_full[s]), 4);
            mbar_init(smem_u32(&bars.slab_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars.acc_full[b]), 1);
            mbar_init(smem_u32(&bars.acc_empty[b]), 8);  // the 8 epilogue warps
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) tc::alloc(smem_u32(&bars.tmem_base), 512);
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    volatile int *abort_flag = &bars.abort;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_err_convpool_tc, DEVERR_TIMEOUT);
    };

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        const long long plane_stride = (long long)H * W;
        int k = 0;
        for (long long item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++k) {
            const int stage = k & 1, use = k >> 1;
            const int cblk = (int)(item % ncb);
            const long long t = item / ncb;
            const int pr = (int)(t % Ho);
            const long long n = t / Ho;
            const int row0 = pr * P, col0 = cblk * MT;
            const float *xn = x + n * C::CIN * plane_stride;
            float r[C::NITER][C::CIN];
#pragma unroll
            for (int it = 0; it < C::NITER; ++it) {
                const int pos = tid + it * 128;
                const int rr = pos / SW, cc = pos - (pos / SW) * SW;
                const int row = row0 + rr, col = col0 + cc;
                const bool ok = pos < C::ROWS * SW && row < H && col < W;
                const float *src = xn + (long long)row * W + col;
#pragma unroll
                for (int ci = 0; ci < C::CIN; ++ci) r[it][ci] = ok ? __ldg(src + ci * plane_stride) : 0.f;
            }
            if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
            unsigned char *slab = sSlab + stage * C::SLAB;
#pragma unroll
            for (int it = 0; it < C::NITER; ++it) {
                const int pos = tid + it * 128;
                if (pos < C::ROWS * SW) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float hi[4], lo[4];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            hi[c4] = tc::to_tf32(r[it][4 * g + c4]);
                            lo[c4] = tc::to_tf32(r[it][4 * g + c4] - hi[c4]);
                        }
                        *reinterpret_cast<float4 *>(slab + g * C::PLANE + pos * 16) =
                            make_float4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<float4 *>(slab + C::SPLIT + g * C::PLANE + pos * 16) =
                            make_float4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t IDESC = tc::idesc_tf32(128, N);
            const uint32_t sB_addr = smem_u32(sB), sSlab_addr = smem_u32(sSlab);
            int k = 0;
            for (long long item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++k) {
                const int stage = k & 1, use = k >> 1, buf = k & 1;
                if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.acc_empty[buf]), (use - 1) & 1)) {
                    fail();
                    break;
                }
                if (!mbar_wait_bounded(smem_u32(&bars.slab_full[stage]), use & 1)) {
                    fail();
                    break;
                }
                tc::fence_after_sync();
                // Base descriptors; every tap / K step / split only moves the start
                // address, i.e. adds (bytes >> 4) to the low field (no carry: shared
                // addresses stay below 2^18).
                const uint64_t a0 = tc::smem_desc(sSlab_addr + stage * C::SLAB, C::PLANE, 128);
                const uint64_t b0 = tc::smem_desc(sB_addr, C::BPLANE, 128);
#pragma unroll
                for (int j = 0; j < P; ++j) {
                    const uint32_t d = tmem + (uint32_t)(buf * ACC_STRIDE + j * N);
                    uint32_t acc = 0;
#pragma unroll
                    for (int tap = 0; tap < 9; ++tap) {
                        const int off = ((j + tap / 3) * SW + tap % 3) * 16;
#pragma unroll
                        for (int s = 0; s < G / 2; ++s) {
                            const uint64_t ah = a0 + (uint64_t)((2 * s * C::PLANE + off) >> 4);
                            const uint64_t al = ah + (uint64_t)(C::SPLIT >> 4);
                            const uint64_t bh = b0 + (uint64_t)(((tap * G + 2 * s) * C::BPLANE) >> 4);
                            const uint64_t bl = bh + (uint64_t)((9 * G * C::BPLANE) >> 4);
                            tc::mma_tf32(d, al, bh, IDESC, acc);
                            tc::mma_tf32(d, ah, bl, IDESC, 1);
                            tc::mma_tf32(d, ah, bh, IDESC, 1);
                            acc = 1;
                        }
                    }
                }
                tc::commit(smem_u32(&bars.slab_empty[stage]));
                tc::commit(smem_u32(&bars.acc_full[buf]));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // All 8 epilogue warps serve every item: warp w reads TMEM lane quarter w % 4
        // and the 16-channel chunks c with c % 2 == (w - 4) / 4.
        const int q = warp & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        int k = 0;
        for (long long item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++k) {
            const int buf = k & 1;
            if (!mbar_wait_bounded(smem_u32(&bars.acc_full[buf]), (k >> 1) & 1)) {
                fail();
                break;
            }
            tc::fence_after_sync();
            const int cblk = (int)(item % ncb);
            const long long t = item / ncb;
            const int pr = (int)(t % Ho);
            const long long n = t / Ho;
            const int col = cblk * MT + 32 * q + lane;
            const int pw = col / P;
            const bool valid = pw < Wo;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * ACC_STRIDE);
#pragma unroll
            for (int c0 = 16 * half; c0 < N; c0 += 32) {
                float v[P][16];
#pragma unroll
                for (int j = 0; j < P; ++j) tc::ld16(taddr + j * N + c0, v[j]);
                tc::wait_ld();
                float m[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    m[i] = v[0][i];
#pragma unroll
                    for (int j = 1; j < P; ++j) m[i] = upd(m[i], v[j][i], use_min);
                }
                // butterfly over the P lanes of a window: keep half the channels per step
                const int b0 = lane & 1;
                float h[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float give = b0 ? m[i] : m[8 + i];
                    const float keep = b0 ? m[8 + i] : m[i];
                    h[i] = upd(keep, __shfl_xor_sync(0xffffffffu, give, 1), use_min);
                }
                int cbase = c0 + 8 * b0;
                float res[8];
                int nres = 8;
                if (P == 4) {
                    const int b1 = (lane >> 1) & 1;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float give = b1 ? h[i] : h[4 + i];
                        const float keep = b1 ? h[4 + i] : h[i];
                        res[i] = upd(keep, __shfl_xor_sync(0xffffffffu, give, 2), use_min);
                    }
                    cbase += 4 * b1;
                    nres = 4;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) res[i] = h[i];
                }
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (i < nres) {
                            const int co = cbase + i;
                            const float tv = tanh_fast(res[i] + sCb[co]);
                            out[((n * N + co) * Ho + pr) * (long long)Wo + pw] = __fadd_rn(__fmul_rn(tv, scale), sBias[co]);
                        }
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[buf]));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after_sync();
        tc::dealloc(tmem, 512);
    }
}

template <int P, int N>
fw_status launch_pn(const float *x, int Nimg, int H, int W, const float *w, const float *cb, const float *bias,
                    float scale, float *out, int Ho, int Wo, cudaStream_t st) {
    using C = Cfg<2, P, N>;
    size_t smem = C::SMEM < 116 * 1024 ? 116 * 1024 : C::SMEM;  // one CTA per SM
    cudaError_t e = cudaFuncSetAttribute(convpool_tc_kernel<2, P, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FW_ERR_LAUNCH;
    const int ncb = (Wo * P + MT - 1) / MT;
    const long long items = (long long)Nimg * Ho * ncb;
    const int grid = (int)(items < sms ? items : sms);
    convpool_tc_kernel<2, P, N><<<grid, NTHREADS, smem, st>>>(x, w, cb, bias, scale, out, Nimg, H, W, Ho, Wo, ncb);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace

bool convpool_tc_eligible(int Cin, int Cout, int KH, int KW, int pk, int ps) {
    return Cin == 8 && KH == 3 && KW == 3 && pk == ps && (pk == 2 || pk == 4) &&
           (Cout == 16 || Cout == 32 || Cout == 48 || Cout == 64);
}

fw_status convpool_tc_launch(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                             float scale, const float *bias, int pk, float *out, int Ho, int Wo, cudaStream_t st) {
#define FW_CP_CASE(PP, NN) \
    if (pk == PP && Cout == NN) return launch_pn<PP, NN>(x, N, H, W, w, cb, bias, scale, out, Ho, Wo, st);
    FW_CP_CASE(4, 64) FW_CP_CASE(4, 48) FW_CP_CASE(4, 32) FW_CP_CASE(4, 16)
    FW_CP_CASE(2, 64) FW_CP_CASE(2, 48) FW_CP_CASE(2, 32) FW_CP_CASE(2, 16)
#undef FW_CP_CASE
    return FW_ERR_UNSUPPORTED;
}

unsigned convpool_tc_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convpool_tc, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convpool_tc, &zero, sizeof(zero));
    return v;
}

}  // namespace fw
