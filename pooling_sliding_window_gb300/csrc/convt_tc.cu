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
// CTA roles (640 threads, one CTA per SM, persistent over the tiles of one phase):
//   warps 0-6   producers: gather the positions x Cin channels a slab needs from
//               NCHW x (all channel loads of a position in flight at once), round
//               to TF32, write the planar shared layout (2 stages); a slab covers
//               both vertical taps of the tile when it fits, else one each;
//   warp  19    allocates TMEM; one lane issues the MMAs: 4 taps x Cin/8 K-steps
//               per tile, accumulating into one of three 128-column accumulators
//               (round robin) that already hold the conv bias;
//   warps 7-18  epilogue, three groups of 4 warps, group g serving accumulator g:
//               each thread owns one pixel (a TMEM lane) and walks its 128 channel
//               sums three times in 32-column chunks: the max, then 2^(z - max)
//               written back to TMEM with the running sum, then
//               sigmoid((p + bias) * scale) to global memory, after which the chunk
//               is reset to the conv bias for the accumulator's next tile.
// Exponentials run in base 2: the weights are prescaled by log2(e) when they are
// rewritten (TF32) into the caller's workspace by convt_tc_prepack_kernel, and the
// bias of the accumulators is conv_b * log2(e), so an accumulator holds
// z = (conv-transpose + conv_b) * log2(e) directly.  The phase's weights (2*Cin KB)
// stay resident in shared memory.
// TF32 operands (10-bit mantissa), float32 accumulation: an error dy in the
// conv-transpose output moves out_c by at most sigma' * |scale| * |dp_c| with
// |dp_c| = p_c |dy_c - sum_j p_j dy_j| <= 2 p_c (1 - p_c) max|dy| and sigma' <= 1/4,
// i.e. by |scale|/2 * p_c(1-p_c) * max|dy|.  With unit-variance x and weights within
// +-1/32 (the l2_p91 workload) the softmax is nearly flat (p ~ 1/128) and the result
// stays within 1e-5 of the float64 oracle; logits a few times larger, or one
// dominant channel, give errors of a few 1e-4, inside the 5e-3 bound of the TF32
// path.  The float32 FMA kernels (convt.cu) keep 1e-5 for any softmax.
#include <cstdlib>

#include "fw_common.cuh"

namespace fw {

__device__ unsigned g_err_convt_tc = 0;

namespace {

constexpr int COUT = 128;
constexpr int MT = 128;            // anchors per tile
constexpr int NSTAGE = 2;          // slab stages

// Warp roles.  Gathering kernel: warps 0-6 gather slabs, three epilogue groups of 4
// warps (each covering TMEM lane quarters 0-3) serve three accumulators, the last
// warp issues the MMAs.  Staged kernel (slabs moved by the bulk-copy engine from a
// pre-staged copy of x): one lane of warp 0 issues the copies, four epilogue groups
// serve four accumulators (all 512 TMEM columns).
template <bool STAGED>
struct Roles {
    static constexpr int PROD_WARPS = STAGED ? 1 : 7;
    static constexpr int EPI_WARP0 = PROD_WARPS;
    static constexpr int NACC = STAGED ? 4 : 3;  // TMEM accumulators of 128 columns, one epilogue group each
    static constexpr int MMA_WARP = EPI_WARP0 + 4 * NACC;
    static constexpr int NTHREADS = (MMA_WARP + 1) * 32;
};
constexpr int NACC_MAX = 4;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr uint32_t IDESC = tc::idesc_tf32(128, COUT);
constexpr size_t MIN_SMEM = 116 * 1024;  // > half an SM: one CTA per SM
constexpr size_t SMEM_LIMIT = 232448;    // 227 KB of dynamic shared memory per CTA

// Tap tables of the k4 s2 p1 decomposition (output parity q, tap index t in {0,1}):
// kernel index and input offset (input row = m + offset).
__host__ __device__ __forceinline__ int tap_k(int q, int t) { return q == 0 ? (t == 0 ? 1 : 3) : (t == 0 ? 0 : 2); }
__host__ __device__ __forceinline__ int tap_off(int q, int t) { return q == 0 ? (t == 0 ? 0 : -1) : (t == 0 ? 1 : 0); }

// wtc[phase][t = 2*ty + tx][g][co][c4] = tf32(log2(e) * w[4g + c4][co][kh(py,ty)][kw(px,tx)])
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
        wtc[i] = tc::to_tf32(__ldg(w + (((long long)(4 * g + c4) * COUT + co) * 4 + kh) * 4 + kw) * LOG2E);
    }
}

// Staged copy of x for the staged kernel: per plane of 4 input channels, the
// stacked position sequence (see the top of this file) as TF32 float4s, preceded by
// XS_FRONT zero positions (a slab of tile 0 starts at position -1) and padded with
// zeros past the last position any slab reads.
constexpr int XS_FRONT = 8;

__host__ __device__ inline long long xs_plane_positions(int N, int H, int W) {
    const long long BW = W + 1, n_anchor = (long long)N * (H + 1) * BW;
    const long long n_tiles = (n_anchor + MT - 1) / MT;
    // a slab reads positions up to n_tiles * MT + 2 * BW
    return (XS_FRONT + n_tiles * MT + 2 * BW + 1 + 7) / 8 * 8;
}

// xs[g][XS_FRONT + q] = tf32(x[n][4g .. 4g+3][row][c]) for position q = R*(W+1) + c,
// R = n*(H+1) + row + 1 (zero for the extra column, the zero rows and the padding).
__global__ void __launch_bounds__(256) convt_stage_x_kernel(const float *__restrict__ x, float4 *__restrict__ xs,
                                                            int N, int Cin, int H, int W, long long xs_plane) {
    const long long total = (long long)(Cin / 4) * xs_plane;
    const int BW = W + 1, BH = H + 1;
    const long long n_pos = ((long long)N * BH + 1) * BW;
    const long long plane = (long long)H * W;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long g = i / xs_plane;
        const long long q = i - g * xs_plane - XS_FRONT;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q >= 0 && q < n_pos) {
            const long long R = q / BW;
            const int c = (int)(q - R * BW);
            if (c < W && R > 0) {
                const long long n = (R - 1) / BH;
                const int row = (int)(R - 1 - n * BH);
                if (row < H) {
                    const float *src = x + ((n * Cin + 4 * g) * H + row) * (long long)W + c;
                    v = make_float4(tc::to_tf32(__ldg(src)), tc::to_tf32(__ldg(src + plane)),
                                    tc::to_tf32(__ldg(src + 2 * plane)), tc::to_tf32(__ldg(src + 3 * plane)));
                }
            }
        }
        xs[i] = v;
    }
}

struct Bars {
    uint64_t b_full;
    uint64_t slab_full[NSTAGE];
    uint64_t slab_empty[NSTAGE];
    uint64_t acc_full[NACC_MAX];
    uint64_t acc_empty[NACC_MAX];
    uint32_t tmem_base;
    int abort;
};

// Shared memory of one CTA: resident weights, NSTAGE slabs of G planes x L
// positions x 16 B, two per-channel constant vectors, barriers.
__host__ __device__ inline size_t tc_smem_bytes(int G, int L) {
    return (size_t)4 * G * COUT * 16 + (size_t)NSTAGE * G * L * 16 + 2 * COUT * 4 + sizeof(Bars);
}

// One 256-bit store (8 floats, 32-byte aligned address): a whole L2 sector.
__device__ __forceinline__ void st_global_v8(float *p, const float *v) {
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]),
                 "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A slab holds the positions one tile reads for the vertical taps it covers:
// nslab == 1 -> both vertical taps (L = 129 + (W+1) positions), nslab == 2 ->
// one vertical tap per slab (L = 129).
// RAW = false: the fused operator.  RAW = true: the first kernel of the unfused
// comparison path -- `out` receives the conv-transpose output y (+ conv_b) for every
// output pixel and channel; scale and bias are unused.
// NHWC = true: x is [N, H, W, Cin] and out [N, Ho, Wo, Cout] (channels last); the
// gather then loads 4 channels per lane with one 16-byte load, and each epilogue
// thread writes its pixel's 128 channels as 256-bit stores (whole 32-byte sectors).
// STAGED = true: x has been rewritten by convt_stage_x_kernel into `xs` (TF32, the
// planar stacked-position layout of the slabs, xs_plane positions per plane), so a
// slab is G contiguous runs that one lane moves with the bulk-copy engine.
template <int G, bool RAW, bool NHWC = false, bool STAGED = false>  // G = input channels / 4
__global__ void __launch_bounds__(Roles<STAGED>::NTHREADS, 1)
convt_k4s2_tc_kernel(const float *__restrict__ x, const float *__restrict__ wtc, const float *__restrict__ cb,
                     const float *__restrict__ bias, float scale, float *__restrict__ out, int N, int H, int W,
                     int Ho, int Wo, int nslab, int L, const float4 *__restrict__ xs, long long xs_plane) {
    constexpr int PROD_WARPS = Roles<STAGED>::PROD_WARPS, EPI_WARP0 = Roles<STAGED>::EPI_WARP0;
    constexpr int NACC = Roles<STAGED>::NACC, MMA_WARP = Roles<STAGED>::MMA_WARP;
    constexpr int NTHREADS = Roles<STAGED>::NTHREADS;
    static_assert(!(STAGED && (RAW || NHWC)), "the staged kernel serves the fused NCHW operator");
    constexpr int CIN = 4 * G;
    constexpr int B_BYTES = 4 * G * COUT * 16;  // 4 taps x G planes x 128 co x 16 B
    extern __shared__ __align__(1024) unsigned char smem[];
    const int slab_plane = L * 16;  // bytes per plane in a slab
    const int slab_bytes = G * slab_plane;
    unsigned char *sB = smem;
    unsigned char *sSlab = smem + B_BYTES;
    float *sCb = reinterpret_cast<float *>(sSlab + NSTAGE * slab_bytes);  // conv_b * log2(e)
    float *sKb = sCb + COUT;                                              // -bias * scale * log2(e)
    Bars &bars = *reinterpret_cast<Bars *>(sKb + COUT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int phase = blockIdx.x & 3, py = phase >> 1, px = phase & 1;
    const int rank = blockIdx.x >> 2, nct = gridDim.x >> 2;
    const int BW = W + 1, BH = H + 1;
    const long long n_anchor = (long long)N * BH * BW;
    const long long n_pos = ((long long)N * BH + 1) * BW;
    const int n_tiles = (int)((n_anchor + MT - 1) / MT);
    const int dx0 = px == 0 ? -1 : 0;  // smaller horizontal tap offset of the phase
    const int dy0 = py == 0 ? -1 : 0;  // smaller vertical tap offset of the phase

    for (int i = tid; i < COUT; i += NTHREADS) {
        sCb[i] = cb ? __ldg(cb + i) * LOG2E : 0.f;
        sKb[i] = bias ? -__ldg(bias + i) * scale * LOG2E : 0.f;
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bars.b_full), 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(smem_u32(&bars.slab_full[s]), STAGED ? 1 : PROD_WARPS);
            mbar_init(smem_u32(&bars.slab_empty[s]), 1);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(smem_u32(&bars.acc_full[b]), 1);
            mbar_init(smem_u32(&bars.acc_empty[b]), 4);
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) tc::alloc(smem_u32(&bars.tmem_base), 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    volatile int *abort_flag = &bars.abort;

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_err_convt_tc, DEVERR_TIMEOUT);
    };

    if (STAGED && warp < PROD_WARPS) {
        // ------------------------------------------- slabs by the bulk-copy engine
        // One lane: per slab, G copies of L positions (one per plane of 4 channels),
        // completing on the stage's full barrier.
        if (lane == 0) {
            int k = 0;
            bool ok = true;
            int last_use[NSTAGE] = {-1, -1};  // last use of each stage a copy was issued for
            for (int tile = rank; ok && tile < n_tiles && !*abort_flag; tile += nct) {
                for (int s = 0; s < nslab; ++s, ++k) {
                    const int stage = k & 1, use = k >> 1;
                    if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    last_use[stage] = use;
                    const int dy_lo = nslab == 1 ? dy0 : tap_off(py, s);
                    const long long pbase = (long long)tile * MT + BW + (long long)dy_lo * BW + dx0;
                    const uint32_t bar = smem_u32(&bars.slab_full[stage]);
                    mbar_arrive_expect_tx(bar, (uint32_t)slab_bytes);
                    const uint32_t dst = smem_u32(sSlab + stage * slab_bytes);
                    const float4 *src = xs + XS_FRONT + pbase;
                    for (int g = 0; g < G; ++g)
                        bulk_g2s(dst + (uint32_t)(g * slab_plane), src + g * xs_plane, (uint32_t)slab_plane, bar);
                }
            }
            // No copy may still be landing in shared memory when the CTA exits: wait
            // (bounded) for the last copy issued into each stage (already complete
            // unless the pipeline was aborted).
            for (int st = 0; st < NSTAGE; ++st)
                if (last_use[st] >= 0) mbar_wait_bounded(smem_u32(&bars.slab_full[st]), last_use[st] & 1);
        }
        __syncwarp();
    } else if (!STAGED && warp < PROD_WARPS) {
        // ------------------------------------------------------------ producers
        // Each thread owns at most one position of a slab (L <= 224 when one slab
        // covers both vertical taps; two positions otherwise).  Its channel loads
        // are issued before the wait for the stage to be free, so their latency
        // overlaps the tensor cores still reading that stage.
        const long long plane_stride = (long long)H * W;
        // x address of position q of the stacked sequence (nullptr: a zero position)
        auto pos_src = [&](long long q) -> const float * {
            if (q < 0 || q >= n_pos) return nullptr;
            int R, c;
            if (n_pos < 0x7fffffffLL) {
                R = (int)q / BW;
                c = (int)q - R * BW;
            } else {
                R = (int)(q / BW);
                c = (int)(q - (long long)R * BW);
            }
            if (c >= W || R <= 0) return nullptr;
            const int n = (R - 1) / BH;
            const int row = R - 1 - n * BH;
            return row < H ? x + (((long long)n * CIN) * H + row) * (long long)W + c : nullptr;
        };
        if (!NHWC && L <= PROD_WARPS * 32) {
            // One position per thread and slab, software-pipelined: converting and storing
            // channels 4g..4g+3 of this slab frees their registers, which then load the same
            // channels of the thread's position in the next slab, so the next slab's loads
            // are in flight while this one is stored.
            auto slab_src = [&](int tile, int s) -> const float * {
                const int dy_lo = nslab == 1 ? dy0 : tap_off(py, s);
                const long long pbase = (long long)tile * MT + BW + (long long)dy_lo * BW + dx0;
                return tid < L ? pos_src(pbase + tid) : nullptr;
            };
            float r[CIN];
            {
                const float *src = rank < n_tiles ? slab_src(rank, 0) : nullptr;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) r[ci] = src ? __ldg(src + ci * plane_stride) : 0.f;
            }
            int k = 0;
            for (int tile = rank; tile < n_tiles && !*abort_flag; tile += nct) {
                for (int s = 0; s < nslab; ++s, ++k) {
                    const int stage = k & 1, use = k >> 1;
                    int ntile = tile, ns = s + 1;
                    if (ns == nslab) {
                        ns = 0;
                        ntile += nct;
                    }
                    const float *nsrc = ntile < n_tiles ? slab_src(ntile, ns) : nullptr;
                    if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                    unsigned char *slab = sSlab + stage * slab_bytes;
                    if (tid < L) {
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            *reinterpret_cast<float4 *>(slab + g * slab_plane + tid * 16) =
                                make_float4(tc::to_tf32(r[4 * g]), tc::to_tf32(r[4 * g + 1]),
                                            tc::to_tf32(r[4 * g + 2]), tc::to_tf32(r[4 * g + 3]));
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                r[4 * g + j] = nsrc ? __ldg(nsrc + (4 * g + j) * plane_stride) : 0.f;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
                    if (*abort_flag) break;
                }
            }
        }
        int k = 0;
        for (int tile = rank; tile < n_tiles && !*abort_flag && (NHWC || L > PROD_WARPS * 32); tile += nct) {
            for (int s = 0; s < nslab; ++s, ++k) {
                const int stage = k & 1, use = k >> 1;
                const int dy_lo = nslab == 1 ? dy0 : tap_off(py, s);
                const long long pbase = (long long)tile * MT + BW + (long long)dy_lo * BW + dx0;
                unsigned char *slab = sSlab + stage * slab_bytes;
                bool waited = use == 0;
                if constexpr (NHWC) {
                    // G lanes per position, lane g loading channels 4g..4g+3 (16 bytes);
                    // PPP positions per pass, NB passes in flight per batch.
                    constexpr int PPP = PROD_WARPS * 32 / G, NB = 14;
                    const int g = tid % G, pslot = tid / G;
                    for (int b0 = 0; b0 < L; b0 += PPP * NB) {
                        float4 r[NB];
                        // decode the batch's first position once, then step PPP positions
                        // at a time (row / image carries instead of divisions)
                        long long q = pbase + b0 + pslot;
                        int R, c;
                        if (n_pos < 0x7fffffffLL) {
                            R = (int)q / BW;
                            c = (int)q - R * BW;
                        } else {
                            R = (int)(q / BW);
                            c = (int)(q - (long long)R * BW);
                        }
                        int n = R > 0 ? (R - 1) / BH : 0;
                        int row = R > 0 ? R - 1 - n * BH : -1;  // -1: the zero row above image 0
#pragma unroll
                        for (int j = 0; j < NB; ++j) {
                            const int pos = b0 + pslot + PPP * j;
                            r[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (pos < L && q >= 0 && q < n_pos && c >= 0 && c < W && row >= 0 && row < H)
                                r[j] = __ldg(reinterpret_cast<const float4 *>(
                                    x + (((long long)n * H + row) * W + c) * CIN + 4 * g));
                            q += PPP;
                            c += PPP;
                            while (c >= BW) {
                                c -= BW;
                                if (++row == BH) {
                                    row = 0;
                                    ++n;
                                }
                            }
                        }
                        if (!waited) {
                            if (!mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                            waited = true;
                        }
#pragma unroll
                        for (int j = 0; j < NB; ++j) {
                            const int pos = b0 + pslot + PPP * j;
                            if (pos < L)
                                *reinterpret_cast<float4 *>(slab + g * slab_plane + pos * 16) =
                                    make_float4(tc::to_tf32(r[j].x), tc::to_tf32(r[j].y), tc::to_tf32(r[j].z),
                                                tc::to_tf32(r[j].w));
                        }
                    }
                }
                for (int pos = NHWC ? L : tid; pos < L; pos += PROD_WARPS * 32) {
                    const long long q = pbase + pos;
                    const float *src = nullptr;
                    if (q >= 0 && q < n_pos) {
                        int R, c;
                        if (n_pos < 0x7fffffffLL) {
                            R = (int)q / BW;
                            c = (int)q - R * BW;
                        } else {
                            R = (int)(q / BW);
                            c = (int)(q - (long long)R * BW);
                        }
                        if (c < W && R > 0) {
                            const int n = (R - 1) / BH;
                            const int row = R - 1 - n * BH;
                            if (row < H) src = x + (((long long)n * CIN) * H + row) * (long long)W + c;
                        }
                    }
                    float r[CIN];
#pragma unroll
                    for (int ci = 0; ci < CIN; ++ci) r[ci] = src ? __ldg(src + ci * plane_stride) : 0.f;
                    if (!waited) {
                        if (!mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                        waited = true;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float4 v = make_float4(tc::to_tf32(r[4 * g]), tc::to_tf32(r[4 * g + 1]),
                                                     tc::to_tf32(r[4 * g + 2]), tc::to_tf32(r[4 * g + 3]));
                        *reinterpret_cast<float4 *>(slab + g * slab_plane + pos * 16) = v;
                    }
                }
                // threads without a position still wait, so the whole warp arrives in order
                if (!waited && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
                if (*abort_flag) break;
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
                const int b = u % NACC, ause = u / NACC;
                // phase 0 of acc_empty completes when the epilogue has written the bias
                if (!mbar_wait_bounded(smem_u32(&bars.acc_empty[b]), ause & 1)) {
                    fail();
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * COUT);
                const uint32_t acc = 1;  // accumulate onto the conv bias
                for (int s = 0; s < nslab; ++s, ++k) {
                    const int stage = k & 1, use = k >> 1;
                    if (!mbar_wait_bounded(smem_u32(&bars.slab_full[stage]), use & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t slab = sSlab_addr + stage * slab_bytes;
                    const int dy_lo = nslab == 1 ? dy0 : tap_off(py, s);
                    for (int ty = (nslab == 1 ? 0 : s); ty <= (nslab == 1 ? 1 : s); ++ty) {
#pragma unroll
                        for (int tx = 0; tx < 2; ++tx) {
                            const int o = (tap_off(py, ty) - dy_lo) * BW + (tap_off(px, tx) - dx0);
                            const int tap = 2 * ty + tx;
#pragma unroll
                            for (int j = 0; j < G / 2; ++j) {
                                const uint64_t ad =
                                    tc::smem_desc(slab + (2 * j * L + o) * 16, (uint32_t)slab_plane, 128);
                                const uint64_t bd =
                                    tc::smem_desc(sB_addr + (tap * G + 2 * j) * (COUT * 16), COUT * 16, 128);
                                tc::mma_tf32(d, ad, bd, IDESC, acc);
                            }
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
        // Group eg handles the tiles u = eg, eg + NACC, ... of this CTA (accumulator eg).
        const int q = warp & 3;                     // TMEM lane quarter of this warp
        const int eg = (warp - EPI_WARP0) >> 2;     // epilogue group = accumulator buffer
        const long long img_anchors = (long long)BH * BW;
        const long long plane_out = (long long)Ho * Wo;
        const float ks = -scale * LOG2E;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(eg * COUT);
        const float4 *cb4 = reinterpret_cast<const float4 *>(sCb);
        const float4 *kb4 = reinterpret_cast<const float4 *>(sKb);
        float v[32];
        // the 32 columns of chunk c <- conv_b * log2(e) (v is scratch)
        auto reset_chunk = [&](int c) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 t = cb4[8 * c + i];
                v[4 * i] = t.x;
                v[4 * i + 1] = t.y;
                v[4 * i + 2] = t.z;
                v[4 * i + 3] = t.w;
            }
            tc::st32(taddr + 32 * c, v);
        };
#pragma unroll 1
        for (int c = 0; c < COUT / 32; ++c) reset_chunk(c);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[eg]));

        int u = eg;
        for (int tile = rank + eg * nct; tile < n_tiles && !*abort_flag; tile += NACC * nct, u += NACC) {
            if (!mbar_wait_bounded(smem_u32(&bars.acc_full[eg]), (u / NACC) & 1)) {
                fail();
                break;
            }
            tc::fence_after_sync();
            const long long a = (long long)tile * MT + 32 * q + lane;
            const long long n = a / img_anchors;
            const int rem = (int)(a - n * img_anchors);
            const int m = rem / BW, nn = rem - m * BW;
            const int oh = 2 * m + py, ow = 2 * nn + px;
            const bool valid = a < n_anchor && oh < Ho && ow < Wo;
            float *o = NHWC ? out + ((n * Ho + oh) * (long long)Wo + ow) * COUT
                            : out + (n * COUT) * plane_out + (long long)oh * Wo + ow;
            if constexpr (RAW) {
                // y = z * ln(2): the accumulator holds (conv-transpose + conv_b) * log2(e)
#pragma unroll 2
                for (int c = 0; c < COUT / 32; ++c) {
                    tc::ld32(taddr + 32 * c, v);
                    tc::wait_ld();
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[(32 * c + i) * plane_out] = v[i] * LN2;
                    }
                    reset_chunk(c);
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[eg]));
                continue;
            }
            // The chunk loops are unrolled only twice: fully unrolled, the three
            // passes no longer fit the instruction caches next to the producer and
            // MMA code (measured 12 % slower).
            // pass 1: max over channels of z
            float mx = -INFINITY;
#pragma unroll 2
            for (int c = 0; c < COUT / 32; ++c) {
                tc::ld32(taddr + 32 * c, v);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
            }
            // pass 2: e = 2^(z - max) written back to TMEM, and their sum
            float sum = 0.f;
#pragma unroll 2
            for (int c = 0; c < COUT / 32; ++c) {
                tc::ld32(taddr + 32 * c, v);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = ex2_approx(v[i] - mx);
                    sum += v[i];
                }
                tc::st32(taddr + 32 * c, v);
            }
            tc::wait_st();
            // softmax p = e / sum; out = 1 / (1 + 2^(-(p + bias) * scale * log2(e)))
            const float kp = ks / sum;
#pragma unroll 2
            for (int c = 0; c < COUT / 32; ++c) {
                tc::ld32(taddr + 32 * c, v);
                tc::wait_ld();
                if (valid) {
                    if constexpr (NHWC) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 kb = kb4[8 * c + i / 4];
                            v[i] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i], kp, kb.x)));
                            v[i + 1] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 1], kp, kb.y)));
                            v[i + 2] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 2], kp, kb.z)));
                            v[i + 3] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 3], kp, kb.w)));
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 8) st_global_v8(o + 32 * c + i, v + i);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 kb = kb4[8 * c + i / 4];
                            float *oc = o + (32 * c + i) * plane_out;
                            oc[0] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i], kp, kb.x)));
                            oc[plane_out] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 1], kp, kb.y)));
                            oc[2 * plane_out] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 2], kp, kb.z)));
                            oc[3 * plane_out] = __fdividef(1.f, 1.f + ex2_approx(fmaf(v[i + 3], kp, kb.w)));
                        }
                    }
                }
                reset_chunk(c);
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[eg]));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after_sync();
        tc::dealloc(tmem, 512);
    }
}

template <int G, bool RAW, bool NHWC, bool STAGED = false>
fw_status launch_g(const float *x, int N, int H, int W, const float *wtc, const float *cb, const float *bias,
                   float scale, float *out, int Ho, int Wo, cudaStream_t st, const float4 *xs = nullptr,
                   long long xs_plane = 0) {
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return FW_ERR_LAUNCH;
    const size_t limit = (size_t)optin < SMEM_LIMIT ? (size_t)optin : SMEM_LIMIT;
    int nslab = 1, L = MT + 1 + (W + 1);
    if (NHWC) L |= 1;  // an odd plane stride (in 16-byte units) spreads the gather's stores over the banks
    size_t smem = tc_smem_bytes(G, L);
    if (smem > limit) {
        nslab = 2;
        L = MT + 1;
        smem = tc_smem_bytes(G, L);
    }
    if (smem > limit) return FW_ERR_UNSUPPORTED;
    if (smem < MIN_SMEM) smem = MIN_SMEM;
    cudaError_t e = cudaFuncSetAttribute(convt_k4s2_tc_kernel<G, RAW, NHWC, STAGED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    const long long tiles = ((long long)N * (H + 1) * (W + 1) + MT - 1) / MT;
    int per_phase = sms / 4 > 0 ? sms / 4 : 1;
    if (per_phase > tiles) per_phase = (int)tiles;
    convt_k4s2_tc_kernel<G, RAW, NHWC, STAGED><<<4 * per_phase, Roles<STAGED>::NTHREADS, smem, st>>>(
        x, wtc, cb, bias, scale, out, N, H, W, Ho, Wo, nslab, L, xs, xs_plane);
    note_launch();
    return launch_status(cudaGetLastError());
}

// Workspace of the staged kernel: the weight rewrite (rounded up to 256 bytes), then
// the staged copy of x.
size_t wtc_bytes_aligned(int Cin) { return ((size_t)16 * Cin * COUT * 4 + 255) & ~(size_t)255; }

// FUSEDWIN_CONVT_GATHER=1 in the environment keeps the gathering kernel even when the
// workspace would hold the staged copy (used to cross-check the two kernels).
bool force_gather() {
    static const bool v = [] {
        const char *e = getenv("FUSEDWIN_CONVT_GATHER");
        return e && e[0] == '1';
    }();
    return v;
}

}  // namespace

bool convt_tc_eligible(int Cin, int Cout, int k, int s, int p) {
    return k == 4 && s == 2 && p == 1 && Cout == COUT && (Cin == 8 || Cin == 16 || Cin == 32 || Cin == 64);
}

// Workspace bytes with which the fused NCHW call takes the staged kernel.
size_t convt_tc_staged_bytes(int N, int Cin, int H, int W) {
    return wtc_bytes_aligned(Cin) + (size_t)(Cin / 4) * (size_t)xs_plane_positions(N, H, W) * 16;
}

namespace {

// prepack = false: the workspace already holds this call's weight rewrite (an earlier
// launch on the same stream wrote it), so only the main kernel runs.
// ws_bytes >= convt_tc_staged_bytes(N, Cin, H, W) (fused NCHW operator only): x is
// first rewritten into the workspace by convt_stage_x_kernel and the staged kernel
// moves its slabs with the bulk-copy engine; otherwise the producers gather them.
template <bool RAW, bool NHWC = false>
fw_status tc_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                    const float *bias, float scale, float *out, int Ho, int Wo, void *ws, cudaStream_t st,
                    bool prepack = true, size_t ws_bytes = 0) {
    float *wtc = static_cast<float *>(ws);
    if (prepack) {
        const long long total = 16LL * Cin * COUT;
        convt_tc_prepack_kernel<<<(unsigned)min(1024LL, (total + 255) / 256), 256, 0, st>>>(w, wtc, Cin);
        note_launch();
        const fw_status rc = launch_status(cudaGetLastError());
        if (rc != FW_OK) return rc;
    }
    if (!RAW && !NHWC && ws_bytes >= convt_tc_staged_bytes(N, Cin, H, W) && !force_gather()) {
        const long long xs_plane = xs_plane_positions(N, H, W);
        float4 *xs = reinterpret_cast<float4 *>(static_cast<unsigned char *>(ws) + wtc_bytes_aligned(Cin));
        const long long total = (long long)(Cin / 4) * xs_plane;
        convt_stage_x_kernel<<<(unsigned)min(152LL * 8, (total + 255) / 256), 256, 0, st>>>(x, xs, N, Cin, H, W,
                                                                                           xs_plane);
        note_launch();
        const fw_status rc = launch_status(cudaGetLastError());
        if (rc != FW_OK) return rc;
        switch (Cin) {
            case 8: return launch_g<2, false, false, true>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st, xs, xs_plane);
            case 16: return launch_g<4, false, false, true>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st, xs, xs_plane);
            case 32: return launch_g<8, false, false, true>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st, xs, xs_plane);
            case 64: return launch_g<16, false, false, true>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st, xs, xs_plane);
        }
        return FW_ERR_UNSUPPORTED;
    }
    switch (Cin) {
        case 8: return launch_g<2, RAW, NHWC>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 16: return launch_g<4, RAW, NHWC>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 32: return launch_g<8, RAW, NHWC>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
        case 64: return launch_g<16, RAW, NHWC>(x, N, H, W, wtc, cb, bias, scale, out, Ho, Wo, st);
    }
    return FW_ERR_UNSUPPORTED;
}

// Stage 2 of the unfused path, one thread per output pixel: an online pass over the
// channels for the softmax max and sum (the sum rescaled whenever the max grows),
// then a second pass for sigmoid((p + bias) * scale).
__global__ void __launch_bounds__(256) softmax_bias_scale_sigmoid_kernel(const float *__restrict__ y,
                                                                         const float *__restrict__ bias,
                                                                         float scale, float *__restrict__ out,
                                                                         long long npix, int C, long long plane) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < npix;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long n = idx / plane, hw = idx - n * plane;
        const float *yb = y + n * C * plane + hw;
        float mx = -INFINITY, sum = 0.f;
        for (int c = 0; c < C; ++c) {
            const float z = __ldg(yb + c * plane) * LOG2E;
            if (z > mx) {
                sum *= ex2_approx(mx - z);
                mx = z;
            }
            sum += ex2_approx(z - mx);
        }
        const float kp = -scale * LOG2E / sum;
        float *ob = out + n * C * plane + hw;
        for (int c = 0; c < C; ++c) {
            const float e = ex2_approx(__ldg(yb + c * plane) * LOG2E - mx);
            const float kb = -__ldg(bias + c) * scale * LOG2E;
            ob[c * plane] = __fdividef(1.f, 1.f + ex2_approx(fmaf(e, kp, kb)));
        }
    }
}

}  // namespace

fw_status convt_tc_launch(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                          const float *bias, float scale, float *out, int Ho, int Wo, void *ws, size_t ws_bytes,
                          cudaStream_t st, bool prepack) {
    return tc_launch<false>(x, N, Cin, H, W, w, cb, bias, scale, out, Ho, Wo, ws, st, prepack, ws_bytes);
}

// Channels-last: x [N, H, W, Cin], out [N, Ho, Wo, 128] (out 32-byte aligned).
fw_status convt_tc_launch_nhwc(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                               const float *bias, float scale, float *out, int Ho, int Wo, void *ws, cudaStream_t st) {
    return tc_launch<false, true>(x, N, Cin, H, W, w, cb, bias, scale, out, Ho, Wo, ws, st);
}

// Stage 1 of the unfused path: y [N, 128, Ho, Wo] = conv-transpose(x) + conv_b.
fw_status convt_tc_launch_raw(const float *x, int N, int Cin, int H, int W, const float *w, const float *cb,
                              float *y, int Ho, int Wo, void *ws, cudaStream_t st) {
    return tc_launch<true>(x, N, Cin, H, W, w, cb, nullptr, 0.f, y, Ho, Wo, ws, st);
}

fw_status softmax_bias_scale_sigmoid_launch(const float *y, int N, int C, int Ho, int Wo, const float *bias,
                                            float scale, float *out, cudaStream_t st) {
    const long long plane = (long long)Ho * Wo, npix = (long long)N * plane;
    const long long want = (npix + 255) / 256;
    const unsigned blocks = (unsigned)(want < 152LL * 64 ? want : 152LL * 64);
    softmax_bias_scale_sigmoid_kernel<<<blocks, 256, 0, st>>>(y, bias, scale, out, npix, C, plane);
    note_launch();
    return launch_status(cudaGetLastError());
}

unsigned convt_tc_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convt_tc, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convt_tc, &zero, sizeof(zero));
    return v;
}

}  // namespace fw
