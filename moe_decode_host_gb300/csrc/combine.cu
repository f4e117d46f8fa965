// Combine and residency byte swap.
//
// Combine: "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 4 --
// the experts' contributions are summed with the router weights; the summation
// order only moves the last decimal places.  Here the order is fixed: pick 0..k-1.
//
// Swap: same page, section 1 -- between steps the residency manager moves
// often-picked experts into HBM and quiet ones out.  A promotion and its paired
// demotion exchange bytes in place: every thread reads its 16-byte chunk of both
// the HBM slot and the host blob, then writes each into the other, so no staging
// buffer is needed and both link directions run at once.
#include "internal.cuh"

namespace moe {
namespace {

template <bool F32>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ w, int T,
                                                      int k, int H, void* __restrict__ out) {
    // launched behind the FFN (programmatic dependent launch): y is complete after this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int t = blockIdx.y;
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;  // index of 4 consecutive columns
    if (c4 * 4 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const float wj = __ldg(w + (size_t)t * k + j);
        const float4 v = __ldg(reinterpret_cast<const float4*>(y + ((size_t)t * k + j) * H) + c4);
        acc.x = fmaf(wj, v.x, acc.x);
        acc.y = fmaf(wj, v.y, acc.y);
        acc.z = fmaf(wj, v.z, acc.z);
        acc.w = fmaf(wj, v.w, acc.w);
    }
    if (F32) {
        reinterpret_cast<float4*>(static_cast<float*>(out) + (size_t)t * H)[c4] = acc;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&lo);
        o.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + (size_t)t * H)[c4] = o;
    }
}

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(kSwapThreads) swap_kernel(SwapList s, size_t blob_bytes, int seg) {
    const size_t chunks = blob_bytes / 16;
    const int items = s.n * seg;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int i = it / seg, part = it % seg;
        uint4* a = reinterpret_cast<uint4*>(s.hot[i]);
        uint4* b = reinterpret_cast<uint4*>(s.host[i]);
        const size_t c0 = chunks * (size_t)part / (size_t)seg;
        const size_t c1 = chunks * (size_t)(part + 1) / (size_t)seg;
        const size_t stride = (size_t)kSwapThreads * kSwapUnroll;
        for (size_t base = c0 + threadIdx.x; base < c1; base += stride) {
            uint4 va[kSwapUnroll], vb[kSwapUnroll];
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const size_t ci = base + (size_t)u * kSwapThreads;
                if (ci < c1) {
                    va[u] = a[ci];
                    vb[u] = b[ci];
                }
            }
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const size_t ci = base + (size_t)u * kSwapThreads;
                if (ci < c1) {
                    a[ci] = vb[u];
                    b[ci] = va[u];
                }
            }
        }
    }
}

// dst[i] <- src[i] (blob_bytes each) for every pair; s.hot holds dst, s.host src.
__global__ void __launch_bounds__(kSwapThreads) copy_list_kernel(SwapList s, size_t blob_bytes, int seg) {
    const size_t chunks = blob_bytes / 16;
    const int items = s.n * seg;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int i = it / seg, part = it % seg;
        uint4* a = reinterpret_cast<uint4*>(s.hot[i]);
        const uint4* b = reinterpret_cast<const uint4*>(s.host[i]);
        const size_t c0 = chunks * (size_t)part / (size_t)seg;
        const size_t c1 = chunks * (size_t)(part + 1) / (size_t)seg;
        const size_t stride = (size_t)kSwapThreads * kSwapUnroll;
        for (size_t base = c0 + threadIdx.x; base < c1; base += stride) {
            uint4 vb[kSwapUnroll];
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const size_t ci = base + (size_t)u * kSwapThreads;
                if (ci < c1) vb[u] = b[ci];
            }
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const size_t ci = base + (size_t)u * kSwapThreads;
                if (ci < c1) a[ci] = vb[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* w, int T, int k, int H, void* out, int out_fp32,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    dim3 grid((H / 4 + 255) / 256, T);
    if (out_fp32) return launch_pdl(combine_kernel<true>, grid, dim3(256), 0, st, y, w, T, k, H, out);
    return launch_pdl(combine_kernel<false>, grid, dim3(256), 0, st, y, w, T, k, H, out);
}

cudaError_t launch_swap(const SwapList& s, size_t blob_bytes, int ctas, cudaStream_t st) {
    if (s.n == 0) return cudaSuccess;
    if (ctas < 1) ctas = 1;
    int seg = ctas / s.n;
    if (seg < 1) seg = 1;
    swap_kernel<<<ctas, kSwapThreads, 0, st>>>(s, blob_bytes, seg);
    return cudaGetLastError();
}

cudaError_t launch_copy_list(const SwapList& s, size_t blob_bytes, int ctas, cudaStream_t st) {
    if (s.n <= 0) return cudaSuccess;
    if (ctas < 1) ctas = 1;
    int seg = ctas / s.n;
    if (seg < 1) seg = 1;
    copy_list_kernel<<<ctas, kSwapThreads, 0, st>>>(s, blob_bytes, seg);
    return cudaGetLastError();
}

}  // namespace moe
