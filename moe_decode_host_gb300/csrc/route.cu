// Router: top-k selection, softmax weights and token-to-expert bucketing.
//
// "Milo and James Try Inference Engineering", the mixture-of-experts paragraph:
// a router picks 6 of 384 experts per token.  Selection compares the fp32 logits
// (descending, ties to the lower expert index); weights are softmax
// probabilities over all E experts.  Bucketing lists pick ids t*k+j grouped by
// expert, ascending, computed with warp ballots so the result never depends on
// atomic ordering.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kMaxV = 32;  // logits per lane: E <= 1024


// One warp routes one token.  Lane l holds experts l, l+32, ...
template <int V>
__device__ __forceinline__ void route_token(const float* __restrict__ lrow, int E, int k, int renorm,
                                            int32_t* __restrict__ ids_out, float* __restrict__ w_out,
                                            int32_t* smem_ids, int* status) {
    const int lane = threadIdx.x & 31;
    float v[V];
    bool finite = true;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(lrow + e) : -INFINITY;
        if (e < E && !isfinite(v[i])) finite = false;
    }
    const bool all_finite = __all_sync(0xffffffffu, finite);
    if (!all_finite) {
        if (lane < k) {
            ids_out[lane] = lane;
            w_out[lane] = 0.0f;
            if (smem_ids) smem_ids[lane] = lane;
        }
        if (lane == 0) set_status(status, MOE_ERR_NONFINITE);
        return;
    }
    uint32_t taken = 0;
    float mx = 0.f;
    int my_id = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (v[i] > bv || be == 0x7fffffff)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (j == 0) mx = bv;
        if (lane == j) {
            my_id = be;
            my_v = bv;
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        int e = lane + 32 * i;
        if (e < E) s += expf(v[i] - mx);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    float p = (lane < k) ? expf(my_v - mx) / s : 0.f;
    if (renorm) {
        float ps = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        p = p / ps;
    }
    if (lane < k) {
        ids_out[lane] = my_id;
        w_out[lane] = p;
        if (smem_ids) smem_ids[lane] = my_id;
    }
}

__device__ __forceinline__ void route_any(const float* lrow, int E, int k, int renorm, int32_t* ids, float* w,
                                          int32_t* sids, int* status) {
    const int nv = (E + 31) / 32;
    if (nv <= 1) route_token<1>(lrow, E, k, renorm, ids, w, sids, status);
    else if (nv <= 2) route_token<2>(lrow, E, k, renorm, ids, w, sids, status);
    else if (nv <= 4) route_token<4>(lrow, E, k, renorm, ids, w, sids, status);
    else if (nv <= 8) route_token<8>(lrow, E, k, renorm, ids, w, sids, status);
    else if (nv <= 12) route_token<12>(lrow, E, k, renorm, ids, w, sids, status);
    else if (nv <= 16) route_token<16>(lrow, E, k, renorm, ids, w, sids, status);
    else route_token<kMaxV>(lrow, E, k, renorm, ids, w, sids, status);
}

// Bucketing of expert e over n pick ids (any memory space), one warp.
__device__ __forceinline__ void bucket_expert(const int32_t* ids, int n, int e, int E, int32_t* counts,
                                              int32_t* offsets, int32_t* entries, int32_t* window) {
    const int lane = threadIdx.x & 31;
    int c_lt = 0, c_eq = 0;
    for (int base = 0; base < n; base += 32) {
        int i = base + lane;
        int id = (i < n) ? ids[i] : 0x7fffffff;
        c_lt += __popc(__ballot_sync(0xffffffffu, id < e));
        c_eq += __popc(__ballot_sync(0xffffffffu, id == e));
    }
    int pos = c_lt;
    if (c_eq > 0) {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = 0; base < n; base += 32) {
            int i = base + lane;
            int id = (i < n) ? ids[i] : 0x7fffffff;
            unsigned m = __ballot_sync(0xffffffffu, id == e);
            if (id == e) entries[pos + __popc(m & lt_mask)] = i;
            pos += __popc(m);
        }
    }
    if (lane == 0) {
        counts[e] = c_eq;
        offsets[e] = c_lt;
        if (e == E - 1) offsets[E] = c_lt + c_eq;
        if (c_eq > 0 && window) atomicAdd(window + e, c_eq);
    }
}

// Small batches: one CTA routes every token, then buckets from shared memory with
// one thread per expert (count, block-wide exclusive scan, ordered placement).
constexpr int kSmallThreads = 512;
constexpr int kSmallMaxPicks = 2048;
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(const float* __restrict__ logits, int T, int E,
                                                                    int k, int renorm, int32_t* ids, float* w,
                                                                    int32_t* counts, int32_t* offsets,
                                                                    int32_t* entries, int32_t* window,
                                                                    int* status) {
    __shared__ int32_t sids[kSmallMaxPicks];
    __shared__ int32_t scnt[kMaxE];
    __shared__ int32_t wsum[kSmallThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int t = warp; t < T; t += nwarps)
        route_any(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k, sids + t * k,
                  status);
    __syncthreads();
    const int n = T * k;
    // counts: one thread per expert scans the pick list (a broadcast read per step)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int i = 0; i < n; ++i) c += (sids[i] == e);
        scnt[e] = c;
        counts[e] = c;
        if (c > 0 && window) atomicAdd(window + e, c);
    }
    __syncthreads();
    // exclusive scan of scnt over E (E <= 1024): each thread owns up to 2 entries
    const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
    const int v0 = e0 < E ? scnt[e0] : 0, v1 = e1 < E ? scnt[e1] : 0;
    int incl = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w2 = 0; w2 < warp; ++w2) base += wsum[w2];
    const int ex0 = base + incl - v0 - v1;
    __syncthreads();
    if (e0 < E) scnt[e0] = ex0;
    if (e1 < E) scnt[e1] = ex0 + v0;
    if (threadIdx.x == 0) offsets[E] = n;
    __syncthreads();
    // placement: picks of expert e in ascending pick order
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int start = scnt[e];
        offsets[e] = start;
        const int end = (e + 1 < E) ? scnt[e + 1] : n;
        if (end > start) {
            int pos = start;
            for (int i = 0; i < n && pos < end; ++i)
                if (sids[i] == e) entries[pos++] = i;
        }
    }
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int renorm, int32_t* ids, float* w, int* status) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    route_any(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k, nullptr, status);
}

__global__ void __launch_bounds__(256) route_bucket_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                           int32_t* counts, int32_t* offsets, int32_t* entries,
                                                           int32_t* window) {
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (e >= E) return;
    bucket_expert(ids, n, e, E, counts, offsets, entries, window);
}

// Large batches: one CTA per expert, its 8 warps each scanning one eighth of the
// picks (counts first, then placement from each warp's exclusive start), so every
// SM shares the scans; the entries keep ascending pick order.
constexpr int kSplitWarps = 8;
__global__ void __launch_bounds__(32 * kSplitWarps) route_bucket_split_kernel(const int32_t* __restrict__ ids, int n,
                                                                              int E, int32_t* counts, int32_t* offsets,
                                                                              int32_t* entries, int32_t* window) {
    __shared__ int s_lt[kSplitWarps], s_eq[kSplitWarps];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = ((n + kSplitWarps - 1) / kSplitWarps + 31) & ~31;  // picks per warp, a multiple of 32
    const int beg = min(n, warp * per), end = min(n, beg + per);
    int c_lt = 0, c_eq = 0;
    for (int base = beg; base < end; base += 32) {
        const int i = base + lane;
        const int id = (i < end) ? __ldg(ids + i) : 0x7fffffff;
        c_lt += __popc(__ballot_sync(0xffffffffu, id < e));
        c_eq += __popc(__ballot_sync(0xffffffffu, id == e));
    }
    if (lane == 0) {
        s_lt[warp] = c_lt;
        s_eq[warp] = c_eq;
    }
    __syncthreads();
    int lt = 0, eq = 0, pos = 0;
#pragma unroll
    for (int w = 0; w < kSplitWarps; ++w) {
        lt += s_lt[w];
        eq += s_eq[w];
        if (w < warp) pos += s_eq[w];
    }
    pos += lt;  // this warp's first entry
    if (c_eq > 0) {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = beg; base < end; base += 32) {
            const int i = base + lane;
            const int id = (i < end) ? __ldg(ids + i) : 0x7fffffff;
            const unsigned m = __ballot_sync(0xffffffffu, id == e);
            if (id == e) entries[pos + __popc(m & lt_mask)] = i;
            pos += __popc(m);
        }
    }
    if (threadIdx.x == 0) {
        counts[e] = eq;
        offsets[e] = lt;
        if (e == E - 1) offsets[E] = lt + eq;
        if (eq > 0 && window) atomicAdd(window + e, eq);
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids, float* w,
                         int32_t* counts, int32_t* offsets, int32_t* entries, int32_t* window, int* status,
                         cudaStream_t st) {
    if (T <= 64 && T * k <= kSmallMaxPicks) {
        route_small_kernel<<<1, kSmallThreads, 0, st>>>(logits, T, E, k, renorm, ids, w, counts, offsets, entries,
                                                       window, status);
        return cudaGetLastError();
    }
    route_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, E, k, renorm, ids, w, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (T * k >= 4096)
        route_bucket_split_kernel<<<E, 32 * kSplitWarps, 0, st>>>(ids, T * k, E, counts, offsets, entries, window);
    else
        route_bucket_kernel<<<(E + 7) / 8, 256, 0, st>>>(ids, T * k, E, counts, offsets, entries, window);
    return cudaGetLastError();
}

}  // namespace moe
