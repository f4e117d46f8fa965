// Dense block-scaled FP4 tensor-core rate of this GPU, the denominator the
// prefill path's tensor fraction is reported against: one CTA per SM issues
// back-to-back tcgen05 kind::mxf4 MMAs of M = 128, N = 256, K = 64 (4.19 MFLOP
// each) on operands resident in shared memory, with unit scale factors in tensor
// memory, accumulating into tensor memory.  Nothing is read from or written to
// global memory except the status word, so the launch's duration is the tensor
// pipe's.  The single wait is bounded; if it runs out the kernel sets
// MOE_ERR_TIMEOUT and returns after freeing tensor memory.
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPkN = 256;
constexpr int kPkASmem = 128 * 128;  // A: 128 rows x 128 bytes (256 E2M1 per row)
constexpr int kPkBSmem = kPkN * 128;
constexpr size_t kPkSmem = 1024 + kPkASmem + kPkBSmem + 64;

__global__ void __launch_bounds__(128, 1) mxf4_peak_kernel(int iters, int* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = base;
    uint8_t* sB = base + kPkASmem;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sB + kPkBSmem);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // operands: E2M1 codes 1.0 and 0.5 alternating (every product finite)
    for (int i = threadIdx.x; i < (kPkASmem + kPkBSmem) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(base)[i] = make_uint4(0x12121212u, 0x21212121u, 0x12121212u, 0x21212121u);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tbase))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    {
        // unit scale factors (E8M0 127) in columns [256, 272) of every lane
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0x7f7f7f7fu;
        const uint32_t a = tm + ((uint32_t)(warp * 32) << 16) + 256u;
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                a),
            "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
            "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
            : "memory");
        tc_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint64_t ad = sw128_desc(smem_u32(sA)), bd = sw128_desc(smem_u32(sB));
        // kind::mxf4, E2M1 x E2M1, K-major, UE8M0 scales, M = 128, N = 256
        const uint32_t id = (1u << 7) | (1u << 10) | ((uint32_t)(kPkN >> 3) << 17) | (1u << 23) | (8u << 24);
        for (int i = 0; i < iters; ++i) {
            const uint32_t kk = (uint32_t)(i & 3);
            const uint32_t sf = (kk & 1u) * 2u;
            const uint32_t idk = id | (sf << 4) | (sf << 29);
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                    tm),
                "l"(ad + 2 * kk), "l"(bd + 2 * kk), "r"(idk), "r"(tm + 256u), "r"(tm + 264u), "r"(i > 0 ? 1u : 0u)
                : "memory");
        }
        tc_commit(bar);
    }
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar, 0u)) {
            if (globaltimer() - t0 > kTimeoutNs) {
                set_status(status, MOE_ERR_TIMEOUT);
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm) : "memory");
    }
}

}  // namespace
}  // namespace moe

extern "C" int moe_mxf4_peak_probe(int iters, int ctas, int* status_dev, void* stream) {
    if (iters < 1 || iters > (1 << 20) || ctas < 0 || !status_dev) return MOE_ERR_INVALID_ARG;
    if (ctas == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    static std::atomic<uint64_t> configured{0};
    if (moe::ensure_smem_limit((const void*)moe::mxf4_peak_kernel, (int)moe::kPkSmem, configured) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe::mxf4_peak_kernel<<<ctas, 128, moe::kPkSmem, static_cast<cudaStream_t>(stream)>>>(iters, status_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
