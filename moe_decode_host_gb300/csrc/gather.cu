// Cold dedupe, id remap and gather.
//
// "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1 (The
// idea): cold experts sit in pinned host memory that the GPU reads directly; one
// small kernel per layer looks at the router's picks and copies just the cold
// ones among them into their scratch slots.  Section 3 measured that copy at
// 2.60 ms of a 10.49 ms step, so the copy is the host-link-bound part of the path.
//
// A one-CTA remap kernel marks the picked cold slots in shared memory and lists
// them in ascending order with warp ballots; a copy kernel, running concurrently,
// derives the same list per CTA and streams the listed host blobs into their
// slots with 16-byte zero-copy loads, several in flight per thread to cover the
// link latency.
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 8;          // 16-byte loads in flight per thread
constexpr int kMaxColdSlots = 4096;  // n_cold bound checked at layer creation


// Copies chunk range [c0, c1) (16-byte chunks) from src to dst with the whole CTA:
// each warp streams its own contiguous eighth of the range, kUnroll 16-byte loads
// in flight per lane including the ragged last round.  Contiguous runs per warp
// read the host link faster than a CTA-wide stride (measured: 203 against 199
// GB/s).
__device__ __forceinline__ void copy_range(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t c0,
                                           size_t c1) {
    constexpr int kWarps = kGatherThreads / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t n = c1 - c0;
    const size_t w0 = c0 + n * (size_t)warp / kWarps, w1 = c0 + n * (size_t)(warp + 1) / kWarps;
    for (size_t base = w0 + lane; base < w1; base += 32 * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t i = base + (size_t)u * 32;
            if (i < w1) v[u] = ld_host_v4(src + i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t i = base + (size_t)u * 32;
            if (i < w1) dst[i] = v[u];
        }
    }
}

// Distinct picked cold slots (ascending) and the physical id of every pick.  One
// CTA of 1024 threads; each thread takes four picks at a time so that their id and
// placement loads overlap.
constexpr int kRemapThreads = 1024;
__global__ void __launch_bounds__(kRemapThreads) cold_remap_kernel(
    const int32_t* __restrict__ ids, int n_picks, const int32_t* __restrict__ loc, int E, int n_hot, int n_cold,
    int32_t* __restrict__ phys, int32_t* __restrict__ cold_list, int32_t* __restrict__ n_picked, int* status) {
    __shared__ unsigned char flag[kMaxColdSlots];
    for (int c = threadIdx.x; c < n_cold; c += blockDim.x) flag[c] = 0;
    __syncthreads();
    for (int base = 0; base < n_picks; base += 4 * kRemapThreads) {
        int id[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * kRemapThreads + threadIdx.x;
            id[u] = i < n_picks ? __ldg(ids + i) : 0;
        }
        int p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) p[u] = (id[u] >= 0 && id[u] < E) ? __ldg(loc + id[u]) : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * kRemapThreads + threadIdx.x;
            if (i >= n_picks) continue;
            if (p[u] < 0) set_status(status, MOE_ERR_BAD_EXPERT);
            else if (p[u] >= n_hot) flag[p[u] - n_hot] = 1;
            phys[i] = p[u];
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int cnt = 0;
        for (int base = 0; base < n_cold; base += 32) {
            int c = base + lane;
            bool f = (c < n_cold) && flag[c];
            unsigned m = __ballot_sync(0xffffffffu, f);
            if (f) cold_list[cnt + __popc(m & ((1u << lane) - 1u))] = c;
            cnt += __popc(m);
        }
        if (lane == 0) *n_picked = cnt;
    }
}

// Streams every picked cold expert's host blob into its scratch slot.  Each CTA
// derives the ascending list of picked cold slots from the picks itself (the same
// marking and ballot compaction as the remap kernel), so the copy needs nothing
// from the remap kernel and the two run concurrently.  A launch copies bytes
// [part_lo, part_hi) of every picked blob (a call copies a blob in two launches:
// the gate/up planes, then the down planes), each picked slot's range cut into
// `seg` contiguous pieces spread over the grid.  CTA 0 also marks every
// picked slot with the copying layer's id (slot_tag), which tells the residency
// manager which slots hold this layer's copy of their expert.
__global__ void __launch_bounds__(kGatherThreads) cold_copy_kernel(
    const int32_t* __restrict__ ids, int n_picks, const int32_t* __restrict__ loc, int E, int n_hot, int n_cold,
    const uint8_t* const* __restrict__ cold_src, uint8_t* __restrict__ slot_base, size_t blob_bytes,
    size_t part_lo, size_t part_hi, int32_t* __restrict__ slot_tag, int uid) {
    __shared__ unsigned char flag[kMaxColdSlots];
    __shared__ int32_t list[kMaxColdSlots];
    __shared__ int s_cnt;
    for (int c = threadIdx.x; c < n_cold; c += blockDim.x) flag[c] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n_picks; i += blockDim.x) {
        const int id = __ldg(ids + i);
        if (id >= 0 && id < E) {
            const int p = __ldg(loc + id);
            if (p >= n_hot) flag[p - n_hot] = 1;
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int cnt = 0;
        for (int base = 0; base < n_cold; base += 32) {
            const int c = base + lane;
            const bool f = (c < n_cold) && flag[c];
            const unsigned m = __ballot_sync(0xffffffffu, f);
            if (f) list[cnt + __popc(m & ((1u << lane) - 1u))] = c;
            cnt += __popc(m);
        }
        if (lane == 0) s_cnt = cnt;
    }
    __syncthreads();
    const int cnt = s_cnt;
    if (cnt <= 0) return;
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < cnt; i += blockDim.x) slot_tag[list[i]] = uid;
    const size_t first = part_lo / 16, chunks = (part_hi - part_lo) / 16;
    int seg = (int)gridDim.x / cnt;
    if (seg < 1) seg = 1;
    const int items = cnt * seg;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int c = list[it / seg];
        const int s = it % seg;
        const size_t c0 = first + chunks * (size_t)s / (size_t)seg;
        const size_t c1 = first + chunks * (size_t)(s + 1) / (size_t)seg;
        copy_range(reinterpret_cast<const uint4*>(cold_src[c]),
                   reinterpret_cast<uint4*>(slot_base + (size_t)c * blob_bytes), c0, c1);
    }
}

__global__ void __launch_bounds__(kGatherThreads) link_probe_kernel(const uint8_t* __restrict__ src,
                                                                    uint8_t* __restrict__ dst, size_t bytes) {
    const size_t chunks = bytes / 16;
    const size_t c0 = chunks * (size_t)blockIdx.x / gridDim.x;
    const size_t c1 = chunks * (size_t)(blockIdx.x + 1) / gridDim.x;
    copy_range(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), c0, c1);
}

}  // namespace

cudaError_t launch_cold_remap(const int32_t* ids, int n_picks, const int32_t* loc, int E, int n_hot, int n_cold,
                              int32_t* phys, int32_t* cold_list, int32_t* n_picked, int* status, cudaStream_t st) {
    if (n_cold > kMaxColdSlots) return cudaErrorInvalidValue;
    cold_remap_kernel<<<1, kRemapThreads, 0, st>>>(ids, n_picks, loc, E, n_hot, n_cold, phys, cold_list, n_picked,
                                                    status);
    return cudaGetLastError();
}

cudaError_t launch_cold_copy(const int32_t* ids, int n_picks, const int32_t* loc, int E, int n_hot, int n_cold,
                             const uint8_t* const* cold_src, uint8_t* slot_base, size_t blob_bytes, size_t part_lo,
                             size_t part_hi, int32_t* slot_tag, int uid, int ctas, cudaStream_t st) {
    if (n_cold > kMaxColdSlots || part_lo % 16 || part_hi % 16 || part_lo > part_hi || part_hi > blob_bytes)
        return cudaErrorInvalidValue;
    cold_copy_kernel<<<ctas, kGatherThreads, 0, st>>>(ids, n_picks, loc, E, n_hot, n_cold, cold_src, slot_base,
                                                      blob_bytes, part_lo, part_hi, slot_tag, uid);
    return cudaGetLastError();
}

cudaError_t launch_link_probe(const uint8_t* src, uint8_t* dst, size_t bytes, int ctas, cudaStream_t st) {
    link_probe_kernel<<<ctas, kGatherThreads, 0, st>>>(src, dst, bytes);
    return cudaGetLastError();
}

}  // namespace moe
