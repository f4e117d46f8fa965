// PTX helpers shared by the FFN kernels (sm_103a): shared-memory addresses,
// mbarriers with bounded waits, TMA and bulk copies, E2M1/E8M0 conversions and
// power-of-two prescales.  Every wait ends by a deadline; a wait that runs out
// sets MOE_ERR_TIMEOUT and records where it gave up.
#pragma once

#include "internal.cuh"

namespace moe {
namespace {

constexpr unsigned long long kTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Waits until the grid this one was launched behind (programmatic dependent
// launch) has completed and its writes are visible; returns at once otherwise.
// Every kernel launched with launch_pdl calls it before it reads the previous
// kernel's outputs and before any of its CTAs can exit, so that a kernel's
// completion implies its predecessors'.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the barrier phase with the given parity; false when the deadline
// passed (status set, abort raised, the place recorded in diag) or another warp
// raised abort.  where: 1 = stage full (consumer), 2 = stage empty (producer).
__device__ __noinline__ bool mbar_wait(uint64_t* bar, unsigned parity, volatile int* abort, int* status, int* diag,
                                       int where, int slot, int stage, int extra) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kTimeoutNs) {
                *abort = 1;
                if (diag && atomicCAS(diag, 0, 1) == 0) {
                    diag[1] = blockIdx.x;
                    diag[2] = (int)(threadIdx.x >> 5);
                    diag[3] = where;
                    diag[4] = slot;
                    diag[5] = (int)parity;
                    diag[6] = stage;
                    diag[7] = extra;
                    diag[8] = mbar_try_wait(bar, parity ^ 1u) ? 1 : 0;
                    __threadfence();
                }
                set_status(status, MOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// mbar_wait with its first poll inline: the call is made only when the phase is
// not complete yet.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, unsigned parity, volatile int* abort, int* status,
                                               int* diag, int where, int slot, int stage, int extra) {
    return mbar_try_wait(bar, parity) || mbar_wait(bar, parity, abort, status, diag, where, slot, stage, extra);
}

// Bounded wait used when draining copies in flight before exit (ignores abort).
__device__ __noinline__ void mbar_drain(uint64_t* bar, unsigned parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kTimeoutNs) return;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// tma_load_2d with an L2 cache policy (from l2_policy_evict_first / _last).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// The same for a converged warp: one elected lane issues.
__device__ __forceinline__ void tma_load_2d_hint_elect(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                       uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;\n\t}" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// mbarrier.arrive.expect_tx by one elected lane of a converged warp.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, unsigned bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// L2 policies: data read once (streamed weights) goes first when L2 needs room;
// data read many times (activations) stays.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Generic-proxy writes to shared memory by this thread are ordered before later
// async-proxy accesses (TMA, bulk copies) to the same bytes once a barrier follows.
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16-byte read of pinned, device-mapped host memory (or any global memory),
// bypassing L1.
// 16-byte load from pinned host memory (mapped): a plain global load.  Over the
// GB300's host link it streams faster than the read-only (.nc) or no-L1-allocate
// forms (measured: 199 against 191-193 GB/s for the same copy).
__device__ __forceinline__ uint4 ld_host_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) {
    uint32_t v;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Four E8M0 exponent bytes (byte j = block j) -> 2^(e_j - 127) as fp32, exactly
// (e = 0 gives the subnormal 2^-127, e = 255 gives NaN): two ue8m0x2 -> bf16x2
// conversions, then the bf16 halves are widened to fp32.
__device__ __forceinline__ void e8m0x4_to_f32(uint32_t w, float (&s)[4]) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "mov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.bf16x2.ue8m0x2 %0, h0;\n\t"
        "cvt.rn.bf16x2.ue8m0x2 %1, h1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
    s[0] = __uint_as_float(lo << 16);
    s[1] = __uint_as_float(lo & 0xffff0000u);
    s[2] = __uint_as_float(hi << 16);
    s[3] = __uint_as_float(hi & 0xffff0000u);
}

// 8 E2M1 nibbles (byte b holds elements 2b, 2b+1) -> 4 f16x2 (r[b] = {elem 2b, elem 2b+1}).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(w));
}

// 2^p for p in [-126, 127].
__device__ __forceinline__ float pow2i(int p) { return __uint_as_float((uint32_t)(p + 127) << 23); }

// Power-of-two prescale exponent so that amax * 2^-p lies in [2^14, 2^15).
__device__ __forceinline__ int prescale_exp(float amax) {
    uint32_t b = __float_as_uint(amax) & 0x7fffffffu;
    if (b == 0u) return 0;
    int e = (int)(b >> 23);
    if (e == 255) return 0;
    int p = (e == 0 ? -126 : e - 127) - 14;
    return p < -126 ? -126 : (p > 126 ? 126 : p);
}


// ---- tensor memory and tensor-core helpers shared by the tcgen05 kernels ----

// Shared-memory matrix descriptor of a K-major operand with the 128-byte swizzle:
// 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// tc_commit for a converged warp: one elected lane commits.
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's lane, waited for in the same asm.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads (gate and up accumulators) with one wait.
__device__ __forceinline__ void tc_ld16x2(uint32_t ta, uint32_t tb, float (&va)[16], float (&vb)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

// A wait taken by a whole warp: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity, const FfnArgs& a, volatile int* abort,
                                          int where, int slot, int stage, int extra) {
    const bool w = mbar_wait_fast(bar, parity, abort, a.status, a.diag, where, slot, stage, extra);
    return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ void advance(int& slot, unsigned& phase, int n) {
    if (++slot == n) {
        slot = 0;
        phase ^= 1u;
    }
}

}  // namespace
}  // namespace moe
