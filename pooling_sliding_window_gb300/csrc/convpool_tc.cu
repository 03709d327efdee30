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
// dropped): three MMAs per K step, float32 accumulation in TMEM.  X3 = false
// is the plain TF32 variant (one product, hi*hi, per K step, bounded at 5e-3: the
// float32-on-TF32 mode the trace "Kimi-K2.6 l2_p91" describes for convolutions):
// no lo planes are staged, and at N = 64 the three kh taps of a kw are stacked
// along N so that one MMA of an input row feeds up to three conv rows.
//
// Work item = one pooled output row of one image and a block of 128 conv columns:
//   * the P conv rows of the pooled row are P GEMMs, M = 128 columns, K = 9 taps x
//     8 channels, each into one slot of a 4-slot TMEM accumulator ring;
//   * the weights are stacked along N as [w_hi | w_lo] (N = 2*Cout), so one MMA
//     gives x_hi*w_hi and x_hi*w_lo side by side and a second, N = Cout, adds
//     x_lo*w_hi onto the first half: two MMAs per tap instead of three;
//   * the input the item reads -- P+2 rows x 130 columns x 8 channels -- is staged
//     per input row in "column-interleaved" core matrices: core i (i < 18) holds
//     columns i, i+16, ..., i+112 as its 8 rows, both 4-channel planes side by
//     side (256 bytes).  MMA row m = 8*i + r is then conv column i + 16*r, and
//     tap (kh, kw) of conv row j is the start address moved by input row j+kh and
//     kw whole core matrices: every operand start stays 256-byte aligned and the
//     operands keep the compact K-major layout (K-adjacent core matrices 128 B
//     apart, M-adjacent ones 256 B apart) that the tensor cores read at full rate.
//     Columns 16..17 + 16k appear twice (as rows 0/1 of core 16/17 too);
//   * the weights, split into hi/lo in the CTA prologue, stay resident.
// CTA roles (512 threads -- 768 for the plain TF32 variant -- one CTA per SM,
// persistent over items):
//   warps 1-3 and the last three  producers: load and split a slab (two stages);
//   warp  0     allocates TMEM; one lane issues 2 x 9 MMAs per conv row;
//   warps 4-11  epilogue (4-19: two groups of eight taking the items in turn in the
//               plain TF32 variant), every warp of a group on every conv row of
//               its items: warp w reads TMEM lane
//               quarter w % 4 and half the channels; the max over the P rows of a
//               window is kept in registers while the rows arrive, the max over
//               its P columns (lanes 8 apart) by a butterfly that halves the
//               channels each lane keeps at every step; out = bias +
//               scale*tanh(m + conv_b) goes through shared memory so that the
//               global stores are row-contiguous.
// Scale < 0 takes the window minimum instead (the map is then decreasing).
#include "fw_common.cuh"

namespace fw {

__device__ unsigned g_err_convpool_tc = 0;
#define CHK(p, bytes, base, base_bytes) chk(&g_err_convpool_tc, (p), (bytes), (base), (base_bytes))
#define CHKS(p, bytes) chk_smem(&g_err_convpool_tc, (p), (bytes))

namespace {

constexpr int MT = 128;          // conv columns per item (MMA M)
constexpr int NCORE = MT / 8 + 2;  // core matrices per staged input row
constexpr int CORE = 256;        // bytes of one core index: 2 planes x 8 rows x 16 B
constexpr int RB = NCORE * CORE;   // bytes of one staged input row (per split)
constexpr int MAX_STAGE = 4;  // slab ring depth bound (Cfg::NST stages are used)
// Warp roles.  A warp runs on SM sub-partition warp % 4 and reads TMEM lane quarter
// warp % 4, so every sub-partition hosts epilogue warps; the MMA issuer (warp 0)
// shares sub-partition 0 only with the quarter-0 epilogue warps (two; four in the
// plain-TF32 variant) and the idle warp: busy warps on the issuer's sub-partition
// slow MMA issue (measured: 2.3x with two FMA-bound warps there, none with the same
// warps on the other three), so the producers run on sub-partitions 1-3.
constexpr int MMA_WARP = 0;
constexpr int EPI_WARP0 = 4;     // warps 4 .. 4 + NEPI - 1: epilogue
constexpr int NPROD = 6;         // warps 1-3 and the last three: producers (the one before idles)
// nw warps in the CTA (a multiple of 4): producer number 0..5 of a warp, or -1
__device__ __forceinline__ int producer_index(int warp, int nw) {
    return (warp >= 1 && warp <= 3) ? warp - 1 : (warp >= nw - 3 ? warp - (nw - 6) : -1);
}
constexpr int TMEM_COLS = 512;   // all of the SM's tensor memory (one CTA per SM)
constexpr int MAX_SLOT = 8;

struct Bars {
    uint64_t slab_full[MAX_STAGE];
    uint64_t slab_empty[MAX_STAGE];
    uint64_t slot_full[MAX_SLOT];
    uint64_t slot_empty[MAX_SLOT];
    uint64_t stg_full[4];  // [group][buffer]
    uint64_t raw_full[2];  // raw mode: a conv row staged by all epilogue warps
    uint32_t tmem_base;
    int abort;
};

template <int P, int N, bool RAW, bool X3>
struct Cfg {
    static constexpr int ROWS = P + 2;
    static constexpr int SPLIT = ROWS * RB;           // hi (or lo) half of a slab
    static constexpr int SLAB = (X3 ? 2 : 1) * SPLIT;
    static constexpr int NST = 2;                     // slab ring stages
    // TMEM accumulator ring, one conv row per slot: [x*w_hi (+ x_lo*w_hi) | x_hi*w_lo]
    static constexpr int SLOT_COLS = X3 ? 128 : 64;
    // Plain TF32 at N = 64: the three kh taps of a kw are stacked along N, so one
    // MMA of an input row feeds up to three conv rows (adjacent slots) at once.
    static constexpr bool STACK = !X3 && !RAW && N == SLOT_COLS;
    static constexpr int NSLOT = TMEM_COLS / SLOT_COLS;
    static_assert((X3 ? 2 : 1) * N <= SLOT_COLS && NSLOT <= MAX_SLOT, "slots");
    static constexpr int BTAP = ((X3 ? 2 : 1) * N / 8) * CORE;  // one tap of [w_hi | w_lo] (or w_hi)
    static constexpr int B_BYTES = 9 * BTAP;
    static constexpr int PW = MT / P;                 // pooled columns per item
    // floats of one staging buffer: a pooled row, or (raw mode) one conv row of the block
    static constexpr int STG = RAW ? N * MT : N * PW;
    // Epilogue: NGRP groups of 8 warps; a group reads every conv row of its items
    // (warp w: lane quarter w % 4, half the channels) and the groups take the items
    // in turn, so one group's pooling tail overlaps the next group's TMEM rows.  Two
    // groups where the tensor work per item is short (plain TF32), one otherwise.
    static constexpr int NGRP = (!RAW && !X3) ? 2 : 1;
    static constexpr int NEPI = 8 * NGRP;
    static constexpr int NTHREADS = (8 + NEPI) * 32;  // + MMA warp, 6 producers, 1 idle
    static constexpr int NH = N / 2;                  // channels per epilogue warp
    static constexpr int LDC = NGRP > 1 && NH % 16 == 0 ? 16 : NH;  // TMEM columns per load round
    // Each group's items must map to slots of their own (item k -> slots (k*P .. k*P+P-1) % NSLOT):
    // with shared slots a group one item ahead would wait on a slot barrier of the other group's
    // phase and read its parity as complete.
    static_assert(NGRP == 1 || NSLOT % (NGRP * P) == 0, "epilogue groups need disjoint TMEM slots");
    static constexpr size_t SMEM =
        (size_t)B_BYTES + NST * SLAB + 2 * NGRP * STG * 4 + 2 * N * 4 + sizeof(Bars);
    static_assert(NST <= MAX_STAGE, "slab ring");
};

// Item index -> (image n, pooled row pr, column block cblk), item = (n*Ho + pr)*ncb + cblk,
// advanced by the grid stride without a division per item (one at the start).
struct ItemCursor {
    long long n, dn;
    int pr, cblk, dp, dc;
    __device__ ItemCursor(long long item, long long stride, int Ho, int ncb) {
        cblk = (int)(item % ncb);
        const long long t = item / ncb;
        pr = (int)(t % Ho);
        n = t / Ho;
        dc = (int)(stride % ncb);
        const long long ts = stride / ncb;
        dp = (int)(ts % Ho);
        dn = ts / Ho;
    }
    __device__ __forceinline__ void advance(int Ho, int ncb) {
        cblk += dc;
        int carry = cblk >= ncb;
        cblk -= carry ? ncb : 0;
        pr += dp + carry;
        carry = pr >= Ho;
        pr -= carry ? Ho : 0;
        n += dn + carry;
    }
};

__device__ __forceinline__ float upd(float m, float v, bool use_min) {
    return use_min ? min_nan(m, v) : max_nan(m, v);
}


// RAW = false: the fused operator.  RAW = true: the first kernel of the unfused
// comparison path -- `out` receives y = conv(x) + conv_b for the P*Ho x P*Wo conv
// outputs the pool reads ([Nimg, N, P*Ho, P*Wo]); scale and bias are unused.
// X3 selects the 3xTF32 split (true) or a single TF32 product (false).
// NHWC = true (3xTF32 fused operator only): x is [Nimg, H, W, 8] and out [Nimg, Ho, Wo, N]
// (channels last); a producer loads a position's 4 channels of a K plane as one 16-byte
// load, which is one row of a core matrix as it stands, and each pooled row (its pixels'
// channels contiguous) is stored as 16-byte runs.
template <int P, int N, bool RAW, bool X3, bool NHWC = false>
__global__ void __launch_bounds__(Cfg<P, N, RAW, X3>::NTHREADS, 1)
convpool_tc_kernel(const float *__restrict__ x, const float *__restrict__ w, const float *__restrict__ cb,
                   const float *__restrict__ bias, float scale, float *__restrict__ out, int Nimg, int H, int W,
                   int Ho, int Wo, int ncb, bool vec) {
    using C = Cfg<P, N, RAW, X3>;
    constexpr int CIN = 8, NEPI = C::NEPI, NTHREADS = C::NTHREADS, NW = NTHREADS / 32;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *sB = smem;
    unsigned char *sSlab = smem + C::B_BYTES;
    float *sStg = reinterpret_cast<float *>(sSlab + C::NST * C::SLAB);  // 2 staging buffers per group
    float *sCb = sStg + 2 * C::NGRP * C::STG;
    float *sBias = sCb + N;
    Bars &bars = *reinterpret_cast<Bars *>(sBias + N);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long n_items = (long long)Nimg * Ho * ncb;
    const bool use_min = scale < 0.f;
    // buffer extents for the checked build
    const long long x_bytes = 4LL * Nimg * CIN * H * W;
    const long long out_bytes = RAW ? 4LL * Nimg * N * (P * Ho) * (P * Wo) : 4LL * Nimg * N * Ho * Wo;

    for (int i = tid; i < N; i += NTHREADS) {
        sCb[i] = cb ? __ldg(cb + i) : 0.f;
        sBias[i] = bias ? __ldg(bias + i) : 0.f;  // raw mode passes no bias
    }
    // Weights split into TF32 hi/lo: B[tap][co' / 8][plane][co' % 8][c4] with
    // co' = co for w_hi and N + co for w_lo.  Stacked form: B[kw][n' / 8][plane][n' % 8][c4]
    // with n' = (2 - kh) * N + co (the kh blocks in descending order).
    for (int e = tid; e < 9 * CIN * N; e += NTHREADS) {
        const int co = e % N, t = e / N, ci = t % CIN, tap = t / CIN;
        const float v = __ldg(w + ((long long)co * CIN + ci) * 9 + tap);
        const float hi = tc::to_tf32(v), lo = tc::to_tf32(v - hi);
        if constexpr (C::STACK) {
            const int np = (2 - tap / 3) * N + co;
            float *d = reinterpret_cast<float *>(sB + (tap % 3) * 3 * C::BTAP + (np / 8) * CORE + (ci / 4) * 128 +
                                                 (np % 8) * 16 + (ci % 4) * 4);
            if (CHKS(d, 4)) *d = hi;
            continue;
        }
        const int base = tap * C::BTAP + (ci / 4) * 128 + (ci % 4) * 4;
        float *dh = reinterpret_cast<float *>(sB + base + (co / 8) * CORE + (co % 8) * 16);
        if (CHKS(dh, 4)) *dh = hi;
        if constexpr (X3) {
            float *dl = reinterpret_cast<float *>(sB + base + ((N + co) / 8) * CORE + ((N + co) % 8) * 16);
            if (CHKS(dl, 4)) *dl = lo;
        }
    }
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(smem_u32(&bars.slab_full[s]), NPROD);
            mbar_init(smem_u32(&bars.slab_empty[s]), 1);
        }
        for (int b = 0; b < C::NSLOT; ++b) {
            mbar_init(smem_u32(&bars.slot_full[b]), 1);
            mbar_init(smem_u32(&bars.slot_empty[b]), 8);  // one group reads a row
        }
        for (int b = 0; b < 2 * C::NGRP; ++b) mbar_init(smem_u32(&bars.stg_full[b]), 8);
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&bars.raw_full[b]), NEPI);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) tc::alloc(smem_u32(&bars.tmem_base), TMEM_COLS);
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

    if (producer_index(warp, NW) >= 0) {
        // ------------------------------------------------------------ producers
        // Main task (row rr, group a, r): the 4 input columns 4a + 16r .. +3 of the
        // block, i.e. row r of cores 4a .. 4a+3.  Lane r + 8a of a warp, so a warp's
        // loads cover 512 contiguous bytes (one float4 per channel when x rows are
        // 16-byte aligned) and its shared-memory stores hit 8 distinct 16-byte bank
        // groups per 8 lanes.  Tail task (row rr, r, t): row r of core 16 + t,
        // input column 16 + t + 16r (a second copy of a main-task column, or
        // column 128 / 129 for r = 7).
        // Software-pipelined over items: in the plain-TF32 variant, storing channels 4g..4g+3
        // of this item's tasks frees their registers, which then load the same channels of the
        // next item, so the next item's loads are in flight while this one is stored (0.206 ->
        // 0.193 ms at full size).  The 3xTF32 kernel, bound by its MMAs and near its register
        // limit, issues all of the next item's loads after its stores (interleaving: +1 %).
        constexpr int NPT = NPROD * 32;  // producer threads
        constexpr int MTASK = C::ROWS * 32, TTASK = C::ROWS * 16;
        static_assert(MTASK <= NPT && TTASK <= NPT, "one main and one tail task per producer thread");
        const int ptid = producer_index(warp, NW) * 32 + lane;
        const long long plane_stride = (long long)H * W;
        const int mr = ptid >> 5, ma = (ptid >> 3) & 3, mrr = ptid & 7;  // main task: row, group a, core row r
        const int tr = ptid >> 4, tu = ptid & 15;                         // tail task (ptid < TTASK)
        // x addresses of the thread's tasks in the item at `c`; ok = false: zeros, nothing read
        auto main_src = [&](const ItemCursor &c, int &col, bool &ok) {
            const int row = c.pr * P + mr;
            col = c.cblk * MT + 4 * ma + 16 * mrr;
            ok = ptid < MTASK && row < H;
            return x + (c.n * CIN * plane_stride + (long long)row * W + col);
        };
        auto tail_src = [&](const ItemCursor &c, bool &ok) {
            const int row = c.pr * P + tr, col = c.cblk * MT + 16 + (tu >> 3) + 16 * (tu & 7);
            ok = ptid < TTASK && row < H && col < W;
            return x + (c.n * CIN * plane_stride + (long long)row * W + col);
        };
        auto load_main = [&](const float *src, int col, bool ok, int ci) {
            const float *sp = src + ci * plane_stride;
            if (vec)  // W % 4 == 0: the 4 columns are all in or all out
                return ok && col < W && CHK(sp, 16, x, x_bytes) ? __ldg(reinterpret_cast<const float4 *>(sp))
                                                                : make_float4(0.f, 0.f, 0.f, 0.f);
            const int nv = ok ? min(4, max(0, W - col)) : 0;  // columns inside the row
            if (nv > 0 && !CHK(sp, 4 * nv, x, x_bytes)) return make_float4(0.f, 0.f, 0.f, 0.f);
            return make_float4(ok && col < W ? __ldg(sp) : 0.f, ok && col + 1 < W ? __ldg(sp + 1) : 0.f,
                               ok && col + 2 < W ? __ldg(sp + 2) : 0.f, ok && col + 3 < W ? __ldg(sp + 3) : 0.f);
        };
        auto load_tail = [&](const float *src, bool ok, int ci) {
            const float *sp = src + ci * plane_stride;
            return ok && CHK(sp, 4, x, x_bytes) ? __ldg(sp) : 0.f;
        };
        // channels last: x + ((n*H + row)*W + col)*8 + 4g holds channels 4g..4g+3 of a position
        auto nhwc_src = [&](const ItemCursor &c, int row, int col) {
            return x + ((((long long)c.n * H + row) * W + col) * CIN);
        };
        auto load4 = [&](const float *sp, bool ok) {
            return ok && CHK(sp, 16, x, x_bytes) ? __ldg(reinterpret_cast<const float4 *>(sp))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        if constexpr (NHWC) {
            static_assert(!NHWC || (X3 && !RAW), "channels last serves the fused 3xTF32 operator");
            // the same tasks: main = 4 columns x 2 planes, tail = 1 column x 2 planes
            float4 vm4[8], vt4[2];
            ItemCursor cur(blockIdx.x, gridDim.x, Ho, ncb), nxt = cur;
            auto load_item = [&](const ItemCursor &c, bool has) {
                const int mrow = c.pr * P + mr, mcol = c.cblk * MT + 4 * ma + 16 * mrr;
                const bool mok = has && ptid < MTASK && mrow < H;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int g = 0; g < 2; ++g)
                        vm4[2 * j + g] = load4(nhwc_src(c, mrow, mcol + j) + 4 * g, mok && mcol + j < W);
                const int trow = c.pr * P + tr, tcol = c.cblk * MT + 16 + (tu >> 3) + 16 * (tu & 7);
                const bool tok = has && ptid < TTASK && trow < H && tcol < W;
#pragma unroll
                for (int g = 0; g < 2; ++g) vt4[g] = load4(nhwc_src(c, trow, tcol) + 4 * g, tok);
            };
            load_item(cur, blockIdx.x < n_items);
            int k = 0;
            for (long long item = blockIdx.x; item < n_items && !*abort_flag;
                 item += gridDim.x, ++k, cur.advance(Ho, ncb)) {
                const int stage = k % C::NST, use = k / C::NST;
                nxt.advance(Ho, ncb);
                if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                unsigned char *slab = sSlab + stage * C::SLAB;
                auto put4 = [&](unsigned char *dst, float4 v) {  // hi/lo split into the two halves
                    const float h0 = tc::to_tf32(v.x), h1 = tc::to_tf32(v.y), h2 = tc::to_tf32(v.z),
                                h3 = tc::to_tf32(v.w);
                    if (CHKS(dst, 16)) *reinterpret_cast<float4 *>(dst) = make_float4(h0, h1, h2, h3);
                    if (CHKS(dst + C::SPLIT, 16))
                        *reinterpret_cast<float4 *>(dst + C::SPLIT) = make_float4(
                            tc::to_tf32(v.x - h0), tc::to_tf32(v.y - h1), tc::to_tf32(v.z - h2), tc::to_tf32(v.w - h3));
                };
                if (ptid < MTASK) {
                    unsigned char *dst = slab + mr * RB + 4 * ma * CORE + mrr * 16;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int g = 0; g < 2; ++g) put4(dst + j * CORE + g * 128, vm4[2 * j + g]);
                }
                if (ptid < TTASK) {
                    unsigned char *dst = slab + tr * RB + (16 + (tu >> 3)) * CORE + (tu & 7) * 16;
                    put4(dst, vt4[0]);
                    put4(dst + 128, vt4[1]);
                }
                // the next item's loads after this item's stores (as the NCHW 3xTF32 producers)
                load_item(nxt, item + gridDim.x < n_items);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
            }
        } else {
            float4 vm[CIN];
            float vt[CIN];
            ItemCursor cur(blockIdx.x, gridDim.x, Ho, ncb), nxt = cur;
            {
                int col;
                bool ok, tok;
                const float *ms = main_src(cur, col, ok), *ts = tail_src(cur, tok);
                ok = ok && blockIdx.x < n_items;
                tok = tok && blockIdx.x < n_items;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) {
                    vm[ci] = load_main(ms, col, ok, ci);
                    vt[ci] = load_tail(ts, tok, ci);
                }
            }
            int k = 0;
            for (long long item = blockIdx.x; item < n_items && !*abort_flag;
                 item += gridDim.x, ++k, cur.advance(Ho, ncb)) {
                const int stage = k % C::NST, use = k / C::NST;
                nxt.advance(Ho, ncb);
                const bool has_next = item + gridDim.x < n_items;
                int ncol;
                bool nok, ntok;
                const float *nms = main_src(nxt, ncol, nok), *nts = tail_src(nxt, ntok);
                nok = nok && has_next;
                ntok = ntok && has_next;
                if (use > 0 && !mbar_wait_bounded(smem_u32(&bars.slab_empty[stage]), (use - 1) & 1)) fail();
                unsigned char *slab = sSlab + stage * C::SLAB;
                // hi/lo split of 4 channels of one position into the two halves of the slab
                auto put = [&](unsigned char *dst, float c0, float c1, float c2, float c3) {
                    const float h0 = tc::to_tf32(c0), h1 = tc::to_tf32(c1), h2 = tc::to_tf32(c2), h3 = tc::to_tf32(c3);
                    if (CHKS(dst, 16)) *reinterpret_cast<float4 *>(dst) = make_float4(h0, h1, h2, h3);
                    if constexpr (X3)
                        if (CHKS(dst + C::SPLIT, 16))
                            *reinterpret_cast<float4 *>(dst + C::SPLIT) = make_float4(
                                tc::to_tf32(c0 - h0), tc::to_tf32(c1 - h1), tc::to_tf32(c2 - h2), tc::to_tf32(c3 - h3));
                };
                if (ptid < MTASK) {
                    unsigned char *dst = slab + mr * RB + 4 * ma * CORE + mrr * 16;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const float4 *v = &vm[4 * g];
                        put(dst + g * 128, v[0].x, v[1].x, v[2].x, v[3].x);
                        put(dst + CORE + g * 128, v[0].y, v[1].y, v[2].y, v[3].y);
                        put(dst + 2 * CORE + g * 128, v[0].z, v[1].z, v[2].z, v[3].z);
                        put(dst + 3 * CORE + g * 128, v[0].w, v[1].w, v[2].w, v[3].w);
                        if constexpr (!X3) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) vm[4 * g + j] = load_main(nms, ncol, nok, 4 * g + j);
                        }
                    }
                    if constexpr (X3) {
#pragma unroll
                        for (int ci = 0; ci < CIN; ++ci) vm[ci] = load_main(nms, ncol, nok, ci);
                    }
                }
                if (ptid < TTASK) {
                    unsigned char *dst = slab + tr * RB + (16 + (tu >> 3)) * CORE + (tu & 7) * 16;
                    put(dst, vt[0], vt[1], vt[2], vt[3]);
                    put(dst + 128, vt[4], vt[5], vt[6], vt[7]);
#pragma unroll
                    for (int ci = 0; ci < CIN; ++ci) vt[ci] = load_tail(nts, ntok, ci);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.slab_full[stage]));
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t IDESC_HH_HL = tc::idesc_tf32(128, (X3 ? 2 : 1) * N);
            constexpr uint32_t IDESC_LH = tc::idesc_tf32(128, N);
            const uint32_t sB_addr = smem_u32(sB), sSlab_addr = smem_u32(sSlab);
            // checked build: the shared-memory bytes an MMA reads -- A: 16 core groups
            // CORE apart plus the second K core 128 B on; B: n rows, 8 per CORE
            auto mma_ok = [&](uint32_t a_addr, uint32_t b_addr, int n) {
                return CHKS(a_addr, 15 * CORE + 256) && CHKS(b_addr, (uint32_t)((n / 8 - 1) * CORE + 256));
            };
            int k = 0, rowc = 0;
            bool ok = true;
            for (long long item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x, ++k) {
                const int stage = k % C::NST, use = k / C::NST;
                if (!mbar_wait_bounded(smem_u32(&bars.slab_full[stage]), use & 1)) {
                    fail();
                    break;
                }
                tc::fence_after_sync();
                // Base descriptors; every row / tap / split only moves the start
                // address, i.e. adds (bytes >> 4) to the low field (no carry: shared
                // addresses stay below 2^18).
                const uint64_t a0 = tc::smem_desc(sSlab_addr + stage * C::SLAB, 128, CORE);
                const uint64_t b0 = tc::smem_desc(sB_addr, 128, CORE);
                if constexpr (C::STACK) {
                    // Input row i feeds conv rows jlo..jhi (tap kh = i - j).  Conv row i
                    // starts with its own kh = 0, kw = 0 MMA (accumulate off); the rows
                    // before it take the stacked blocks kh = i - jlo .. 1 (kw = 0) or
                    // .. i - jhi (kw = 1, 2) in one MMA, N = 64 per row.  Row i - 2 is
                    // complete after input row i.
                    constexpr int BKW = 3 * C::BTAP;          // one kw of the stacked weights
#pragma unroll
                    for (int i = 0; i < P + 2; ++i) {
                        const int jlo = i < 2 ? 0 : i - 2, jhi = i < P - 1 ? i : P - 1;
                        const bool fresh = i < P;
                        if (fresh) {
                            const int rc = rowc + i, slot = rc % C::NSLOT, sus = rc / C::NSLOT;
                            if (sus > 0 && !mbar_wait_bounded(smem_u32(&bars.slot_empty[slot]), (sus - 1) & 1)) {
                                fail();
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                        }
                        const uint32_t dlo = tmem + (uint32_t)(((rowc + jlo) % C::NSLOT) * C::SLOT_COLS);
#pragma unroll
                        for (int kw = 0; kw < 3; ++kw) {
                            const uint64_t a = a0 + (uint64_t)((i * RB + kw * CORE) >> 4);
                            const uint32_t a_addr = sSlab_addr + stage * C::SLAB + i * RB + kw * CORE;
                            const int top = fresh && kw == 0 ? i - 1 : jhi;  // last row of the stacked MMA
                            if (fresh && kw == 0 && mma_ok(a_addr, sB_addr + kw * BKW + 2 * C::BTAP, N))
                                tc::mma_tf32(tmem + (uint32_t)(((rowc + i) % C::NSLOT) * C::SLOT_COLS), a,
                                             b0 + (uint64_t)((kw * BKW + 2 * C::BTAP) >> 4),
                                             tc::idesc_tf32(128, N), 0u);
                            if (top >= jlo &&
                                mma_ok(a_addr, sB_addr + kw * BKW + (2 - (i - jlo)) * C::BTAP, (top - jlo + 1) * N))
                                tc::mma_tf32(dlo, a, b0 + (uint64_t)((kw * BKW + (2 - (i - jlo)) * C::BTAP) >> 4),
                                             tc::idesc_tf32(128, (top - jlo + 1) * N), 1u);
                        }
                        if (i >= 2) tc::commit(smem_u32(&bars.slot_full[(rowc + i - 2) % C::NSLOT]));
                    }
                    rowc += P;
                } else {
#pragma unroll
                for (int j = 0; j < P; ++j, ++rowc) {
                    const int slot = rowc % C::NSLOT, sus = rowc / C::NSLOT;
                    if (sus > 0 && !mbar_wait_bounded(smem_u32(&bars.slot_empty[slot]), (sus - 1) & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t d = tmem + (uint32_t)(slot * C::SLOT_COLS);
#pragma unroll
                    for (int tap = 0; tap < 9; ++tap) {
                        const uint64_t ah = a0 + (uint64_t)((((j + tap / 3) * RB) + (tap % 3) * CORE) >> 4);
                        const uint64_t al = ah + (uint64_t)(C::SPLIT >> 4);
                        const uint64_t bd = b0 + (uint64_t)((tap * C::BTAP) >> 4);
                        const uint32_t ah_addr =
                            sSlab_addr + stage * C::SLAB + (j + tap / 3) * RB + (tap % 3) * CORE;
                        if (mma_ok(ah_addr, sB_addr + tap * C::BTAP, (X3 ? 2 : 1) * N))
                            tc::mma_tf32(d, ah, bd, IDESC_HH_HL, tap > 0 ? 1u : 0u);
                        if constexpr (X3)
                            if (mma_ok(ah_addr + C::SPLIT, sB_addr + tap * C::BTAP, N))
                                tc::mma_tf32(d, al, bd, IDESC_LH, 1u);
                    }
                    tc::commit(smem_u32(&bars.slot_full[slot]));
                }
                }
                tc::commit(smem_u32(&bars.slab_empty[stage]));
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NEPI) {
        // ------------------------------------------------------------ epilogue
        // Warp w: TMEM lane quarter q = w % 4, channels [h*NH, (h+1)*NH).  Lane l of
        // quarter q is MMA row m = 32q + l = 8*i + r with i = 4q + l/8, r = l % 8:
        // conv column i + 16r.  The P columns of a pooling window are lanes l ^ 8
        // (and l ^ 16 for P = 4) of the same warp.
        constexpr int NH = C::NH, NG = C::NGRP;
        const int ew = warp - EPI_WARP0, grp = ew >> 3, gw = ew & 7;  // group, warp within the group
        const int q = warp & 3;
        const int h = gw >> 2;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * NH);
        bool ok = true;
        // this group's items: the CTA's item sequence numbers k = grp, grp + NG, ...
        ItemCursor cur(blockIdx.x + (long long)grp * gridDim.x, (long long)NG * gridDim.x, Ho, ncb);
        int k = grp, kk = 0;
        for (long long item = blockIdx.x + (long long)grp * gridDim.x; ok && item < n_items && !*abort_flag;
             item += (long long)NG * gridDim.x, k += NG, ++kk, cur.advance(Ho, ncb)) {
            float m[NH];
#pragma unroll
            for (int c = 0; c < NH; ++c) m[c] = use_min ? INFINITY : -INFINITY;
#pragma unroll 1
            for (int j = 0; j < P; ++j) {
                const int rowc = k * P + j;  // conv rows in MMA order
                const int slot = rowc % C::NSLOT, sus = rowc / C::NSLOT;
                // one outcome for the whole warp: the TMEM loads below are warp-collective
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars.slot_full[slot]), sus & 1))) {
                    fail();
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t ts = tq + (uint32_t)(slot * C::SLOT_COLS);
                // NH channels in rounds of C::LDC TMEM columns (fewer live registers)
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += C::LDC) {
                    float a[C::LDC], b[C::LDC];
#pragma unroll
                    for (int c = 0; c < C::LDC; c += 8) {
                        tc::ld8(ts + c0 + c, a + c);                   // x_hi*w_hi + x_lo*w_hi
                        if constexpr (X3) tc::ld8(ts + N + c0 + c, b + c);  // x_hi*w_lo
                    }
                    tc::wait_ld();
                    if (c0 + C::LDC == NH) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&bars.slot_empty[slot]));
                    }
                    if constexpr (RAW) {
                    // Stage the row as [channel][position]; conv column i + 16r sits at
                    // 8i + (r ^ 2(i/4)), so both the writes here and the column-order
                    // reads below hit 32 distinct banks.
                    float *rs = sStg + (rowc & 1) * C::STG;
                    const int i = 4 * q + (lane >> 3), r = lane & 7;
                    const int pos = 8 * i + (r ^ (2 * (i >> 2)));
#pragma unroll
                    for (int c = 0; c < C::LDC; ++c)
                        if (CHKS(rs + (h * NH + c0 + c) * MT + pos, 4))
                            rs[(h * NH + c0 + c) * MT + pos] = (a[c] + b[c]) + sCb[h * NH + c0 + c];
                    if (c0 + C::LDC < NH) continue;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars.raw_full[rowc & 1]));
                    if (!mbar_wait_bounded(smem_u32(&bars.raw_full[rowc & 1]), (rowc >> 1) & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    const int HI = P * Ho, WI = P * Wo;
                    const int row = cur.pr * P + j, col0 = cur.cblk * MT;
                    float *yrow = out + cur.n * (long long)N * HI * WI + (long long)row * WI + col0;
                    for (int e = tid - EPI_WARP0 * 32; e < N * MT; e += NEPI * 32) {
                        const int co = e / MT, cc = e - co * MT;
                        const int ci = cc & 15, cr = cc >> 4;
                        float *d = yrow + (long long)co * HI * WI + cc;
                        const float *sv = rs + co * MT + 8 * ci + (cr ^ (2 * (ci >> 2)));
                        if (col0 + cc < WI && CHK(d, 4, out, out_bytes) && CHKS(sv, 4)) *d = *sv;
                    }
                    } else if (use_min) {  // warp-uniform: one instruction per conv value
#pragma unroll
                        for (int c = 0; c < C::LDC; ++c) m[c0 + c] = min_nan(m[c0 + c], X3 ? a[c] + b[c] : a[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < C::LDC; ++c) m[c0 + c] = max_nan(m[c0 + c], X3 ? a[c] + b[c] : a[c]);
                    }
                }
                if (!ok) break;
            }
            if (!ok) break;
            if constexpr (RAW) continue;
            // butterfly over the P lanes of a window: keep half the channels per step
            const int b3 = (lane >> 3) & 1;
            float hbuf[NH / 2];
#pragma unroll
            for (int i = 0; i < NH / 2; ++i) {
                const float give = b3 ? m[i] : m[NH / 2 + i];
                const float keep = b3 ? m[NH / 2 + i] : m[i];
                hbuf[i] = upd(keep, __shfl_xor_sync(0xffffffffu, give, 8), use_min);
            }
            int cbase = h * NH + b3 * (NH / 2);
            constexpr int NRES = P == 4 ? NH / 4 : NH / 2;
            float res[NRES];
            int pwl;
            if constexpr (P == 4) {
                const int b4 = (lane >> 4) & 1;
#pragma unroll
                for (int i = 0; i < NH / 4; ++i) {
                    const float give = b4 ? hbuf[i] : hbuf[NH / 4 + i];
                    const float keep = b4 ? hbuf[NH / 4 + i] : hbuf[i];
                    res[i] = upd(keep, __shfl_xor_sync(0xffffffffu, give, 16), use_min);
                }
                cbase += b4 * (NH / 4);
                pwl = q + 4 * (lane & 7);  // window base column 4q + 16r
            } else {
#pragma unroll
                for (int i = 0; i < NH / 2; ++i) res[i] = hbuf[i];
                pwl = 2 * q + ((lane >> 4) & 1) + 8 * (lane & 7);  // base column 4q + 2*(l/16) + 16r
            }
            const int sb = grp * 2 + (kk & 1);  // this group's staging buffer for the item
            // A pooled row is staged [channel][column] with the column rotated by rot(co): the lanes
            // that hold the same window column for different channels (lane bits 3 and 4) then
            // write different banks, and the row-order reads below stay conflict-free.
            auto rot = [](int co) { return P == 4 ? (co / (NH / 4)) & 3 : 2 * ((co / (NH / 2)) & 1); };
            float *stg = sStg + sb * C::STG;
#pragma unroll
            for (int i = 0; i < NRES; ++i) {
                const int co = cbase + i;
                const float tv = tanh_fast(res[i] + sCb[co]);
                float *d = stg + co * C::PW + ((pwl + rot(co)) & (C::PW - 1));
                if (CHKS(d, 4)) *d = __fadd_rn(__fmul_rn(tv, scale), sBias[co]);
            }
            // the group's eight warps have staged this item (its other buffer is still
            // being read only by warps that have not reached this point)
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.stg_full[sb]));
            if (!mbar_wait_bounded(smem_u32(&bars.stg_full[sb]), (kk >> 1) & 1)) {
                fail();
                break;
            }
            const int et = gw * 32 + lane, pw0 = cur.cblk * C::PW;
            if constexpr (NHWC) {
                // channels last: thread et stores channels 8o..8o+7 (32 bytes) of pixel px; a
                // warp takes 32 adjacent pixels of one channel octet, so each staged read hits
                // 32 distinct banks
                float *orow = out + (((long long)cur.n * Ho + cur.pr) * Wo + pw0) * N;
                for (int f = et; f < C::PW * (N / 8); f += 256) {
                    const int px = f % C::PW, o8 = f / C::PW;
                    if (pw0 + px >= Wo) continue;
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int co = 8 * o8 + j;
                        const float *sv = stg + co * C::PW + ((px + rot(co)) & (C::PW - 1));
                        v[j] = CHKS(sv, 4) ? *sv : 0.f;
                    }
                    float *d = orow + (long long)px * N + 8 * o8;
                    if (CHK(d, 32, out, out_bytes)) {
                        *reinterpret_cast<float4 *>(d) = make_float4(v[0], v[1], v[2], v[3]);
                        *reinterpret_cast<float4 *>(d + 4) = make_float4(v[4], v[5], v[6], v[7]);
                    }
                }
                continue;
            }
            // thread et stores column pw of channels co0, co0 + CSTEP, ...: row-contiguous
            // warps, a pointer stride per store
            constexpr int CSTEP = 8 * 32 / C::PW;
            const int pw = et % C::PW, co0 = et / C::PW;
            if (pw0 + pw < Wo) {
                const long long cstride = (long long)Ho * Wo;
                float *op = out + ((cur.n * N + co0) * Ho + cur.pr) * (long long)Wo + pw0 + pw;
                static_assert(N % CSTEP == 0, "store passes");
#pragma unroll
                for (int i = 0; i < N / CSTEP; ++i, op += CSTEP * cstride) {
                    const int co = co0 + i * CSTEP;
                    const float *sv = stg + co * C::PW + ((pw + rot(co)) & (C::PW - 1));
                    if (CHK(op, 4, out, out_bytes) && CHKS(sv, 4)) *op = *sv;
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after_sync();
        tc::dealloc(tmem, TMEM_COLS);
    }
}

template <int P, int N, bool RAW, bool X3, bool NHWC = false>
fw_status launch_pn(const float *x, int Nimg, int H, int W, const float *w, const float *cb, const float *bias,
                    float scale, float *out, int Ho, int Wo, cudaStream_t st) {
    using C = Cfg<P, N, RAW, X3>;
    size_t smem = C::SMEM < 116 * 1024 ? 116 * 1024 : C::SMEM;  // one CTA per SM
    cudaError_t e = cudaFuncSetAttribute(convpool_tc_kernel<P, N, RAW, X3, NHWC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return launch_status(e);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FW_ERR_LAUNCH;
    const int ncb = (Wo * P + MT - 1) / MT;
    const long long items = (long long)Nimg * Ho * ncb;
    const int grid = (int)(items < sms ? items : sms);
    const bool vec = W % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;  // float4 input rows
    convpool_tc_kernel<P, N, RAW, X3, NHWC><<<grid, C::NTHREADS, smem, st>>>(x, w, cb, bias, scale, out, Nimg, H, W,
                                                                          Ho, Wo, ncb, vec);
    note_launch();
    return launch_status(cudaGetLastError());
}

}  // namespace

bool convpool_tc_eligible(int Cin, int Cout, int KH, int KW, int pk, int ps) {
    return Cin == 8 && KH == 3 && KW == 3 && pk == ps && (pk == 2 || pk == 4) &&
           (Cout == 16 || Cout == 32 || Cout == 48 || Cout == 64);
}

// x3 = true: 3xTF32 split (float32-level accuracy); false: one TF32 product per K step.
fw_status convpool_tc_launch(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                             float scale, const float *bias, int pk, float *out, int Ho, int Wo, bool x3,
                             cudaStream_t st) {
#define FW_CP_CASE(PP, NN)                                                                                      \
    if (pk == PP && Cout == NN)                                                                                 \
        return x3 ? launch_pn<PP, NN, false, true>(x, N, H, W, w, cb, bias, scale, out, Ho, Wo, st)             \
                  : launch_pn<PP, NN, false, false>(x, N, H, W, w, cb, bias, scale, out, Ho, Wo, st);
    FW_CP_CASE(4, 64) FW_CP_CASE(4, 48) FW_CP_CASE(4, 32) FW_CP_CASE(4, 16)
    FW_CP_CASE(2, 64) FW_CP_CASE(2, 48) FW_CP_CASE(2, 32) FW_CP_CASE(2, 16)
#undef FW_CP_CASE
    return FW_ERR_UNSUPPORTED;
}

// Channels last (3xTF32 only): x [N, H, W, 8], out [N, Ho, Wo, Cout], both 16-byte aligned.
fw_status convpool_tc_launch_nhwc(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                                  float scale, const float *bias, int pk, float *out, int Ho, int Wo,
                                  cudaStream_t st) {
#define FW_CP_CASE(PP, NN) \
    if (pk == PP && Cout == NN) return launch_pn<PP, NN, false, true, true>(x, N, H, W, w, cb, bias, scale, out, Ho, Wo, st);
    FW_CP_CASE(4, 64) FW_CP_CASE(4, 48) FW_CP_CASE(4, 32) FW_CP_CASE(4, 16)
    FW_CP_CASE(2, 64) FW_CP_CASE(2, 48) FW_CP_CASE(2, 32) FW_CP_CASE(2, 16)
#undef FW_CP_CASE
    return FW_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- unfused path
// The pages' own (unfused) design, built from this library's kernels for comparison:
// the convolution writes its output to memory, then a second kernel pools it and
// applies tanh, scale and bias.

namespace {

// One thread per pooled output: max (min for scale < 0) over the P x P window of
// y = conv + conv_b, then bias + scale * tanh(m), rounded as in the fused kernel.
template <int P>
__global__ void __launch_bounds__(256) pool_tanh_scale_bias_kernel(const float *__restrict__ y,
                                                                   const float *__restrict__ bias, float scale,
                                                                   float *__restrict__ out, long long total, int C,
                                                                   int Ho, int Wo) {
    const bool use_min = scale < 0.f;
    const int WI = P * Wo;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int pw = (int)(idx % Wo);
        const long long t = idx / Wo;
        const int pr = (int)(t % Ho);
        const long long nc = t / Ho;
        const float *base = y + (nc * (long long)(P * Ho) + (long long)pr * P) * WI + (long long)pw * P;
        float m = use_min ? INFINITY : -INFINITY;
        const long long y_bytes = 4 * total * P * P;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            if (!CHK(base + (long long)r * WI, 4 * P, y, y_bytes)) continue;
            if constexpr (P == 4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(base + (long long)r * WI));
                m = upd(upd(upd(upd(m, v.x, use_min), v.y, use_min), v.z, use_min), v.w, use_min);
            } else {
                const float2 v = __ldg(reinterpret_cast<const float2 *>(base + (long long)r * WI));
                m = upd(upd(m, v.x, use_min), v.y, use_min);
            }
        }
        const int co = (int)(nc % C);
        if (CHK(out + idx, 4, out, 4 * total)) out[idx] = __fadd_rn(__fmul_rn(tanh_fast(m), scale), __ldg(bias + co));
    }
}

}  // namespace

// Stage 1 of the unfused path: y [N, Cout, pk*Ho, pk*Wo] = conv(x) + conv_b.
fw_status convpool_tc_launch_raw(const float *x, int N, int H, int W, const float *w, const float *cb, int Cout,
                                 int pk, float *y, int Ho, int Wo, cudaStream_t st) {
#define FW_CP_CASE(PP, NN) \
    if (pk == PP && Cout == NN) return launch_pn<PP, NN, true, true>(x, N, H, W, w, cb, nullptr, 0.f, y, Ho, Wo, st);
    FW_CP_CASE(4, 64) FW_CP_CASE(4, 48) FW_CP_CASE(4, 32) FW_CP_CASE(4, 16)
    FW_CP_CASE(2, 64) FW_CP_CASE(2, 48) FW_CP_CASE(2, 32) FW_CP_CASE(2, 16)
#undef FW_CP_CASE
    return FW_ERR_UNSUPPORTED;
}

// Stage 2 of the unfused path (y 16-byte aligned for pk = 4, 8-byte for pk = 2).
fw_status pool_tanh_scale_bias_launch(const float *y, int N, int Cout, const float *bias, float scale, int pk,
                                      float *out, int Ho, int Wo, cudaStream_t st) {
    const long long total = (long long)N * Cout * Ho * Wo;
    const long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)(want < 152LL * 64 ? want : 152LL * 64);
    if (pk == 4)
        pool_tanh_scale_bias_kernel<4><<<blocks, 256, 0, st>>>(y, bias, scale, out, total, Cout, Ho, Wo);
    else if (pk == 2)
        pool_tanh_scale_bias_kernel<2><<<blocks, 256, 0, st>>>(y, bias, scale, out, total, Cout, Ho, Wo);
    else
        return FW_ERR_UNSUPPORTED;
    note_launch();
    return launch_status(cudaGetLastError());
}

unsigned convpool_tc_read_and_clear_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_convpool_tc, sizeof(v)) != cudaSuccess) return DEVERR_INTERNAL;
    if (v) cudaMemcpyToSymbol(g_err_convpool_tc, &zero, sizeof(zero));
    return v;
}

}  // namespace fw
