// fw_common.cuh -- internal helpers shared by the libfusedwin translation units.
// Not part of the public ABI (include/fusedwin.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fusedwin.h"

namespace fw {

// Device-side error bits, OR-ed into a per-translation-unit error word.
enum : unsigned {
    DEVERR_TIMEOUT = 1u,   // a bounded mbarrier wait gave up
    DEVERR_INTERNAL = 2u,  // an internal consistency check failed
};

// Devices for which per-device state is cached.
constexpr int FW_MAX_DEVICES = 64;

// Wall-clock limit of a bounded wait inside a kernel.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// Launch bookkeeping (host side, fw_api.cu).
void note_launch(int n = 1);
fw_status launch_status(cudaError_t e);

// Checks and dispatch of the conv-transpose entry points (fw_api.cu).
fw_status convt_call(const float *x, int N, int Cin, int H, int W, const float *w, const float *conv_b, int Cout,
                     int k, int s, int p, int op, const float *bias, float scale, float *out, void *workspace,
                     unsigned long long workspace_bytes, bool ffma, bool weights_ready, void *stream);

// ---------------------------------------------------------- checked build --
// Built with -DFW_CHECKED=1 (build.py, checked=True), every kernel tests the
// address range of each memory access -- or of each run of accesses made from one
// computed address -- against the buffer it belongs to before making it.  An access
// outside its buffer is skipped and DEVERR_INTERNAL is recorded in the translation
// unit's error word, which fw_check_device_errors reports as FW_ERR_INTERNAL; no
// kernel traps.  In the default build every check is the constant `true`.
#ifndef FW_CHECKED
#define FW_CHECKED 0
#endif

// ---------------------------------------------------------------- device --

// [p, p + bytes) inside [base, base + base_bytes)?  Checked build only; else true.
__device__ __forceinline__ bool chk(unsigned *err, const void *p, long long bytes, const void *base,
                                    long long base_bytes) {
    if (!FW_CHECKED) return true;
    const unsigned long long a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    const bool ok = base != nullptr && bytes >= 0 && a >= b && a + (unsigned long long)bytes <= b + (unsigned long long)base_bytes;
    if (!ok) atomicOr(err, 2u);  // DEVERR_INTERNAL
    return ok;
}

#if FW_CHECKED
// The block's dynamic shared memory (every kernel's extern __shared__ array starts here).
extern __shared__ __align__(1024) unsigned char fw_dyn_smem[];
#endif

// Shared-memory address range [addr, addr + bytes) inside the dynamic shared memory?
__device__ __forceinline__ bool chk_smem(unsigned *err, uint32_t addr, uint32_t bytes) {
#if FW_CHECKED
    uint32_t size;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(fw_dyn_smem));
    const bool ok = addr >= base && (unsigned long long)addr + bytes <= (unsigned long long)base + size;
    if (!ok) atomicOr(err, 2u);
    return ok;
#else
    (void)err, (void)addr, (void)bytes;
    return true;
#endif
}
__device__ __forceinline__ bool chk_smem(unsigned *err, const void *p, uint32_t bytes) {
    return chk_smem(err, static_cast<uint32_t>(__cvta_generic_to_shared(p)), bytes);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Running max of the MaxPool2d definition: a larger value or a NaN replaces the
// current value unless that is already NaN; ties keep the current (earlier) tap.
__device__ __forceinline__ float max_update(float m, float v) {
    return (m == m && !(v <= m)) ? v : m;
}
// Mirror rule for a running minimum (used when the scale is negative).
__device__ __forceinline__ float min_update(float m, float v) {
    return (m == m && !(v >= m)) ? v : m;
}
// One-instruction window extreme for the conv+pool epilogues: max.NaN / min.NaN (a NaN
// propagates).  The sign of a zero extreme is left to the hardware, which that
// operator's absolute-error bound cannot see (+0 and -0 differ by 0).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float min_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// tanh(z) = 1 - 2 / (1 + e^(2z)) with a base-2 exponential and a fast reciprocal:
// absolute error a few 1e-7 over all z (e^(2z) overflows to inf for large z and
// gives exactly 1; underflows to 0 for very negative z and gives exactly -1).
__device__ __forceinline__ float tanh_fast(float z) {
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * 2.8853900817779268f));  // 2 log2(e)
    return 1.f - __fdividef(2.f, 1.f + e);
}

// ------------------------------------------------------------- mbarriers --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns` (default
// WAIT_LIMIT_NS).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- clusters --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address), with
// release semantics at cluster scope: the caller's earlier memory operations are
// visible to a thread that then observes the phase with acquire at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrive on an mbarrier of any CTA of the cluster with the default (CTA-scope release)
// semantics: no memory fence at cluster scope, so a thread with loads or stores in
// flight does not wait for them.  Enough where what the arrival publishes is the
// arriving CTA's own shared memory (fenced to the async proxy) or its TMEM, read by
// the peer's tensor-core operations.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for a phase completed by arrivals from other CTAs of the cluster.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}
// Every thread of every CTA of the cluster (unbounded: only where all of them arrive
// unconditionally).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Asynchronous 4-byte global -> shared copy (cp.async): `valid` (4 or 0) bytes are read
// from src and the rest of the destination is zero-filled (valid = 0 reads nothing; src
// must still be a valid global address).  A thread sees its own copies once
// cp_async_wait<n> has left at most n of its committed groups pending.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid) : "memory");
}
// 16-byte variant: both addresses 16-byte aligned, `valid` 16 or 0.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace fw

// ------------------------------------------------ tcgen05 (5th-gen tensor cores) --
namespace fw {
namespace tc {

// Shared-memory matrix descriptor for tcgen05.mma, K-major operand without
// swizzle.  The operand is stored as 8-row x 16-byte core matrices (rows 16 B
// apart); `lbo` = byte distance between core matrices adjacent along K, `sbo` =
// byte distance between 8-row groups adjacent along M (or N).  Bits: start
// address >> 4 in [0,14), LBO >> 4 in [16,30), SBO >> 4 in [32,46), descriptor
// version 1 in [46,48), base offset 0, layout type 0 (no swizzle) in [61,64).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of tcgen05.mma.kind::tf32: F32 accumulator (bits 4-5 =
// 1), A and B TF32 (bits 7-9, 10-12 = 2), both K-major, N >> 3 at bit 17, M >> 4
// at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// CTA pair (cluster of two, .cta_group::2): M = 256 with rows 0..127 from the even
// CTA's shared memory and 128..255 from the odd CTA's (same offsets), the N rows of B
// split likewise (first half from the even CTA), D written to both CTAs' TMEM at the
// same address.  Issued by one thread of the even CTA.
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive once on the mbarrier at offset `bar` in both CTAs of the pair when every
// tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}
// Collective TMEM allocation / release of a CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive once on an mbarrier when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole-warp TMEM allocation of `ncols` columns (power of two >= 32); the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Wait until this thread's earlier tcgen05.ld have written their registers.
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// TMEM loads whose completion wait sits in the same asm statement: the destination
// registers are written asynchronously until tcgen05.wait::ld, so nothing the compiler
// schedules (a spill, a copy, a reuse of the register) may come between the load and
// the wait.  The outputs are early-clobber ("=&r"): a register of the first load's
// destination must not also carry the second load's address.  32 columns of this
// thread's lane:
__device__ __forceinline__ void ld32_wait(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=&r"(r[0]), "=&r"(r[1]), "=&r"(r[2]), "=&r"(r[3]), "=&r"(r[4]), "=&r"(r[5]), "=&r"(r[6]), "=&r"(r[7]),
          "=&r"(r[8]), "=&r"(r[9]), "=&r"(r[10]), "=&r"(r[11]), "=&r"(r[12]), "=&r"(r[13]), "=&r"(r[14]), "=&r"(r[15]),
          "=&r"(r[16]), "=&r"(r[17]), "=&r"(r[18]), "=&r"(r[19]), "=&r"(r[20]), "=&r"(r[21]), "=&r"(r[22]), "=&r"(r[23]),
          "=&r"(r[24]), "=&r"(r[25]), "=&r"(r[26]), "=&r"(r[27]), "=&r"(r[28]), "=&r"(r[29]), "=&r"(r[30]), "=&r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 columns at each of two TMEM addresses of this thread's lane (both in flight together).
__device__ __forceinline__ void ld32x2_wait(uint32_t ta, uint32_t tb, float *va, float *vb) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=&r"(r[0]), "=&r"(r[1]), "=&r"(r[2]), "=&r"(r[3]), "=&r"(r[4]), "=&r"(r[5]), "=&r"(r[6]), "=&r"(r[7]),
          "=&r"(r[8]), "=&r"(r[9]), "=&r"(r[10]), "=&r"(r[11]), "=&r"(r[12]), "=&r"(r[13]), "=&r"(r[14]), "=&r"(r[15]),
          "=&r"(r[16]), "=&r"(r[17]), "=&r"(r[18]), "=&r"(r[19]), "=&r"(r[20]), "=&r"(r[21]), "=&r"(r[22]), "=&r"(r[23]),
          "=&r"(r[24]), "=&r"(r[25]), "=&r"(r[26]), "=&r"(r[27]), "=&r"(r[28]), "=&r"(r[29]), "=&r"(r[30]), "=&r"(r[31]),
          "=&r"(r[32]), "=&r"(r[33]), "=&r"(r[34]), "=&r"(r[35]), "=&r"(r[36]), "=&r"(r[37]), "=&r"(r[38]), "=&r"(r[39]),
          "=&r"(r[40]), "=&r"(r[41]), "=&r"(r[42]), "=&r"(r[43]), "=&r"(r[44]), "=&r"(r[45]), "=&r"(r[46]), "=&r"(r[47]),
          "=&r"(r[48]), "=&r"(r[49]), "=&r"(r[50]), "=&r"(r[51]), "=&r"(r[52]), "=&r"(r[53]), "=&r"(r[54]), "=&r"(r[55]),
          "=&r"(r[56]), "=&r"(r[57]), "=&r"(r[58]), "=&r"(r[59]), "=&r"(r[60]), "=&r"(r[61]), "=&r"(r[62]), "=&r"(r[63])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[32 + i]);
    }
}

// 8 consecutive 32-bit columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. +31), written asynchronously: call wait_ld() before using the values.
__device__ __forceinline__ void ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 32 consecutive 32-bit columns of this thread's TMEM lane; call wait_st()
// before reading them back.
__device__ __forceinline__ void st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Round-to-nearest (ties away) float32 -> TF32, returned as a float32 bit pattern.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

}  // namespace tc
}  // namespace fw
