// Grouped SwiGLU expert FFN for prefill-sized buckets (more than 64 tokens per
// expert) on the 5th-generation tensor cores.
//
// "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1: the layer
// runs all experts in one call.  When an expert receives many tokens its weights
// are reused across them and the work is a dense contraction, so it runs as a
// GEMM: D[128 weight rows x N tokens] += W[128 x K] * X[N x K]^T with
// tcgen05.mma (kind::f16, f16 operands, fp32 accumulators in tensor memory).
//
// Warp roles of one persistent CTA per SM:
//   warp 0      TMA of the raw MXFP4 weight slices (128 rows x 64 elements) into a
//               ring of raw stages;
//   warp 1      owns tensor memory and issues the MMAs (one thread), committing
//               each stage back to its producers and each tile to the epilogue;
//   warp 2      TMA of the activation tiles (64 tokens x 64 elements, f16,
//               128-byte swizzle), gathered per expert beforehand;
//   warps 4-7   converters: one weight row per thread, E2M1 -> f16 with the row's
//               E8M0 block scales rebased to 2^12 below the row's largest scale,
//               so that every block whose scale is within 2^35 of the largest is
//               exact in f16 (smaller blocks lose low bits), written in the
//               128-byte-swizzled K-major layout the MMA reads;
//   warps 8-11  epilogue: tensor memory -> registers -> h (gate/up phase, SiLU
//               gate times up) or y (down phase), undoing the power-of-two
//               rebasing of weights and activations.
// Every wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT, and the CTA
// drains its copies and MMAs before it frees tensor memory and returns.
#include <cuda.h>

#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;        // weight rows per tile = tensor-memory lanes
constexpr int kBK = 64;         // K elements per stage (128 bytes of f16 per row)
constexpr int kNMax = 192;      // token columns per pass
constexpr int kRawStages = 8;
constexpr int kABStages = 2;
constexpr int kThreadsTC = 384;
constexpr int kRawBytes = 2 * kBM * 32;            // gate + up raw slices (phase 1 uses half)
constexpr int kATile = kBM * 128;                  // f16 tile, 16 KB
constexpr int kBTile = kNMax * 128;                // activation tile, 24 KB
constexpr int kABBytes = 2 * kATile + kBTile;      // 56 KB
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;

struct alignas(16) TcHead {
    uint64_t raw_full[kRawStages];
    uint64_t raw_empty[kRawStages];
    uint64_t a_full[kABStages];
    uint64_t b_full[kABStages];
    uint64_t ab_empty[kABStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint32_t tmem_base;
    int abort;
    int D;
    int list[kMaxE];
};

constexpr size_t kTcSmem = 1024 + (size_t)kRawStages * kRawBytes + (size_t)kABStages * kABBytes + sizeof(TcHead);

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    // K-major operand, 128-byte swizzle: 8-row core groups 1024 bytes apart
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Largest E8M0 exponent of a scale row (n bytes, n a multiple of 4).
__device__ __forceinline__ int row_max_exp(const uint8_t* srow, int n) {
    uint32_t m = 0;
    for (int i = 0; i < n; i += 4) m = __vmaxu4(m, ld_u32(srow + i));
    const uint32_t a = max(m & 0xffu, (m >> 8) & 0xffu), b = max((m >> 16) & 0xffu, m >> 24);
    return (int)max(a, b);
}

// f16 bits of 2^m (0 when below the smallest subnormal).
__device__ __forceinline__ uint32_t f16_pow2(int m) {
    if (m >= -14) return (uint32_t)(m + 15) << 10;
    if (m >= -24) return 1u << (m + 24);
    return 0u;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

struct TcTask {
    int e, rb, cnt, off, phys;
    bool valid;
};

__device__ __forceinline__ TcTask tc_task(const FfnArgs& a, const TcHead& hd, int task, int tiles) {
    TcTask t;
    t.e = hd.list[task / tiles];
    t.rb = task % tiles;
    t.cnt = __ldg(a.counts + t.e);
    t.off = __ldg(a.offsets + t.e);
    t.phys = __ldg(a.phys_ids + __ldg(a.entries + t.off));
    t.valid = t.phys >= 0 && t.phys < a.n_phys;
    return t;
}

__device__ __forceinline__ int ncols_pad(int nb) { return nb <= 64 ? 64 : (nb <= 128 ? 128 : 192); }

template <int P>
__global__ void __launch_bounds__(kThreadsTC, 1) ffn_tc_kernel(FfnArgs a, const __grid_constant__ CUtensorMap act_map,
                                                               int lo, int sel) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw = base;                                  // [kRawStages][kRawBytes]
    uint8_t* ab = base + (size_t)kRawStages * kRawBytes;  // [kABStages][kABBytes]
    TcHead& hd = *reinterpret_cast<TcHead*>(ab + (size_t)kABStages * kABBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I;
    const int K = P == 0 ? H : I;
    const int nks = K / kBK;
    const int tiles = (P == 0 ? I : H) / kBM;
    volatile int* abort = &hd.abort;

    if (warp == 0) {
        int cnt = 0;
        for (int base_e = 0; base_e < a.E; base_e += 32) {
            const int e = base_e + lane;
            bool act = false;
            if (e < a.E) {
                act = __ldg(a.counts + e) > lo;
                if (act && sel != 0) {
                    const bool hot = __ldg(a.loc + e) < a.n_hot;
                    act = (sel == 1) ? hot : !hot;
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, act);
            if (act) hd.list[cnt + __popc(m & ((1u << lane) - 1u))] = e;
            cnt += __popc(m);
        }
        if (lane == 0) {
            hd.D = cnt;
            hd.abort = 0;
            for (int s = 0; s < kRawStages; ++s) {
                mbar_init(&hd.raw_full[s], 1);
                mbar_init(&hd.raw_empty[s], 4);
            }
            for (int s = 0; s < kABStages; ++s) {
                mbar_init(&hd.a_full[s], 4);
                mbar_init(&hd.b_full[s], 1);
                mbar_init(&hd.ab_empty[s], 1);
            }
            mbar_init(&hd.acc_full, 1);
            mbar_init(&hd.acc_empty, 4);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&hd.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hd.tmem_base;
    const int ntask = hd.D * tiles;

    if (warp == 0 && lane == 0) {
        // ---------------- raw weight producer ----------------
        int rs = 0;
        unsigned rph = 0;
        bool ok = true;
        for (int task = blockIdx.x; task < ntask && ok; task += gridDim.x) {
            const TcTask t = tc_task(a, hd, task, tiles);
            if (!t.valid) continue;
            const CUtensorMap* map = P == 0 ? &a.tmaps[t.phys].w13r : &a.tmaps[t.phys].w2r;
            asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
            const int r0 = t.rb * kBM;
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                for (int s = 0; s < nks; ++s) {
                    if (!mbar_wait(&hd.raw_empty[rs], rph ^ 1u, abort, a.status, a.diag, 12, rs, s, task)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = raw + (size_t)rs * kRawBytes;
                    mbar_arrive_expect_tx(&hd.raw_full[rs], P == 0 ? 2 * kBM * 32 : kBM * 32);
                    tma_load_2d(dst, map, s * 32, r0, &hd.raw_full[rs]);
                    if (P == 0) tma_load_2d(dst + kBM * 32, map, s * 32, I + r0, &hd.raw_full[rs]);
                    if (++rs == kRawStages) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
            }
        }
        for (int s = 0; s < kRawStages; ++s) mbar_drain(&hd.raw_full[s], (s < rs) ? rph : (rph ^ 1u));
    } else if (warp == 2 && lane == 0) {
        // ---------------- activation producer ----------------
        int bs = 0;
        unsigned bph = 0;
        bool ok = true;
        for (int task = blockIdx.x; task < ntask && ok; task += gridDim.x) {
            const TcTask t = tc_task(a, hd, task, tiles);
            if (!t.valid) continue;
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                const int N = ncols_pad(min(kNMax, t.cnt - tb));
                for (int s = 0; s < nks; ++s) {
                    if (!mbar_wait(&hd.ab_empty[bs], bph ^ 1u, abort, a.status, a.diag, 13, bs, s, task)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ab + (size_t)bs * kABBytes + 2 * kATile;
                    mbar_arrive_expect_tx(&hd.b_full[bs], (unsigned)N * 128u);
                    for (int c = 0; c < N / 64; ++c)
                        tma_load_2d(dst + c * 64 * 128, &act_map, s * kBK, t.off + tb + 64 * c, &hd.b_full[bs]);
                    if (++bs == kABStages) {
                        bs = 0;
                        bph ^= 1u;
                    }
                }
            }
        }
        for (int s = 0; s < kABStages; ++s) mbar_drain(&hd.b_full[s], (s < bs) ? bph : (bph ^ 1u));
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int bs = 0;
        unsigned bph = 0;
        unsigned aph = 0;  // acc_empty parity
        bool ok = true;
        int issued = 0;    // commits to ab_empty / acc_full not yet known complete
        for (int task = blockIdx.x; task < ntask && ok; task += gridDim.x) {
            const TcTask t = tc_task(a, hd, task, tiles);
            if (!t.valid) continue;
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                const int N = ncols_pad(min(kNMax, t.cnt - tb));
                const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
                if (!mbar_wait(&hd.acc_empty, aph ^ 1u, abort, a.status, a.diag, 14, 0, 0, task)) {
                    ok = false;
                    break;
                }
                aph ^= 1u;
                tc_fence_after();
                for (int s = 0; s < nks; ++s) {
                    if (!mbar_wait(&hd.a_full[bs], bph, abort, a.status, a.diag, 15, bs, s, task) ||
                        !mbar_wait(&hd.b_full[bs], bph, abort, a.status, a.diag, 16, bs, s, task)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(ab + (size_t)bs * kABBytes);
                    const uint32_t sb = sa + 2 * kATile;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t bdesc = sw128_desc(sb + kk * 32);
                        const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
                        tc_mma_f16(tmem, sw128_desc(sa + kk * 32), bdesc, idesc, acc);
                        if (P == 0) tc_mma_f16(tmem + kNMax, sw128_desc(sa + kATile + kk * 32), bdesc, idesc, acc);
                    }
                    tc_commit(&hd.ab_empty[bs]);
                    ++issued;
                    if (++bs == kABStages) {
                        bs = 0;
                        bph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&hd.acc_full);
            }
        }
        // drain: wait for the last commit on each stage (bounded) so no MMA is in flight
        for (int s = 0; s < kABStages; ++s) mbar_drain(&hd.ab_empty[s], (s < bs) ? bph : (bph ^ 1u));
        (void)issued;
    } else if (warp >= 4 && warp < 8) {
        // ---------------- converters ----------------
        const int t_row = (warp - 4) * 32 + lane;  // weight row within the tile
        int rs = 0, bs = 0;
        unsigned rph = 0, bph = 0;
        bool ok = true;
        for (int task = blockIdx.x; task < ntask && ok; task += gridDim.x) {
            const TcTask t = tc_task(a, hd, task, tiles);
            if (!t.valid) continue;
            const uint8_t* blob = a.ptr[t.phys];
            const int r0 = t.rb * kBM;
            const int srl = K / 32;  // scale bytes per row
            const uint8_t* sc0 = blob + (P == 0 ? a.w13s : a.w2s) + (size_t)(r0 + t_row) * srl;
            const uint8_t* sc1 = P == 0 ? blob + a.w13s + (size_t)(I + r0 + t_row) * srl : sc0;
            const int c0 = row_max_exp(sc0, srl) - 12;
            const int c1 = P == 0 ? row_max_exp(sc1, srl) - 12 : c0;
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                for (int s = 0; s < nks; ++s) {
                    // scale bytes of blocks 2s, 2s+1 (read before the waits)
                    const uint32_t e0 = *reinterpret_cast<const uint16_t*>(sc0 + 2 * s);
                    const uint32_t e1 = P == 0 ? *reinterpret_cast<const uint16_t*>(sc1 + 2 * s) : e0;
                    bool w = mbar_wait(&hd.raw_full[rs], rph, abort, a.status, a.diag, 17, rs, s, task) &&
                             mbar_wait(&hd.ab_empty[bs], bph ^ 1u, abort, a.status, a.diag, 18, bs, s, task);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* rsrc = raw + (size_t)rs * kRawBytes;
                    uint8_t* adst = ab + (size_t)bs * kABBytes;
#pragma unroll
                    for (int ti = 0; ti < (P == 0 ? 2 : 1); ++ti) {
                        const uint4* rp = reinterpret_cast<const uint4*>(rsrc + ti * kBM * 32 + t_row * 32);
                        const uint4 w0 = rp[0], w1 = rp[1];
                        const uint32_t ew = ti == 0 ? e0 : e1;
                        const int cb = ti == 0 ? c0 : c1;
                        const uint32_t m0 = f16_pow2((int)(ew & 0xffu) - cb);
                        const uint32_t m1 = f16_pow2((int)(ew >> 8) - cb);
                        const uint32_t mm0 = m0 | (m0 << 16), mm1 = m1 | (m1 << 16);
                        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        uint8_t* arow = adst + ti * kATile + t_row * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c = elements 8c..8c+7
                            uint32_t h4[4];
                            e2m1x8_to_f16x2(words[c], h4);
                            const uint32_t mm = c < 4 ? mm0 : mm1;
                            uint4 o;
                            o.x = hmul2(h4[0], mm);
                            o.y = hmul2(h4[1], mm);
                            o.z = hmul2(h4[2], mm);
                            o.w = hmul2(h4[3], mm);
                            *reinterpret_cast<uint4*>(arow + ((c ^ (t_row & 7)) * 16)) = o;
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&hd.a_full[bs]);
                        mbar_arrive(&hd.raw_empty[rs]);
                    }
                    if (++rs == kRawStages) {
                        rs = 0;
                        rph ^= 1u;
                    }
                    if (++bs == kABStages) {
                        bs = 0;
                        bph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= 8) {
        // ---------------- epilogue ----------------
        const int q4 = warp - 8;                // tensor-memory lane quarter
        const int t_row = q4 * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        unsigned fph = 0;
        bool ok = true;
        for (int task = blockIdx.x; task < ntask && ok; task += gridDim.x) {
            const TcTask t = tc_task(a, hd, task, tiles);
            if (!t.valid) {
                // zero outputs for an expert whose physical id is out of range
                if (t.rb == 0 && threadIdx.x == 8 * 32) set_status(a.status, MOE_ERR_BAD_EXPERT);
                const int r0 = t.rb * kBM;
                for (int c = 0; c < t.cnt; ++c) {
                    const int pick = __ldg(a.entries + t.off + c);
                    if (P == 0) a.h[(size_t)pick * I + r0 + t_row] = 0.f;
                    else a.y[(size_t)pick * H + r0 + t_row] = 0.f;
                }
                continue;
            }
            const uint8_t* blob = a.ptr[t.phys];
            const int r0 = t.rb * kBM;
            const int srl = K / 32;
            const int c0 = row_max_exp(blob + (P == 0 ? a.w13s : a.w2s) + (size_t)(r0 + t_row) * srl, srl) - 12;
            const int c1 = P == 0 ? row_max_exp(blob + a.w13s + (size_t)(I + r0 + t_row) * srl, srl) - 12 : c0;
            const float s0 = pow2i(max(-126, min(127, c0 - 127)));
            const float s1 = pow2i(max(-126, min(127, c1 - 127)));
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                const int nb = min(kNMax, t.cnt - tb);
                const bool w = mbar_wait(&hd.acc_full, fph, abort, a.status, a.diag, 19, 0, tb, task);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                fph ^= 1u;
                tc_fence_after();
                for (int cb = 0; cb < nb; cb += 16) {
                    float v0[16], v1[16];
                    tc_ld16(lane_addr + cb, v0);
                    if (P == 0) tc_ld16(lane_addr + kNMax + cb, v1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = cb + i;
                        if (n >= nb) break;
                        const int pick = __ldg(a.entries + t.off + tb + n);
                        if constexpr (P == 0) {
                            const float sx = pow2i(__ldg(a.xexp + pick / a.k));
                            const float gv = v0[i] * s0 * sx;
                            const float uv = v1[i] * s1 * sx;
                            const float hv = gv / (1.0f + expf(-gv)) * uv;
                            a.h[(size_t)pick * I + r0 + t_row] = hv;
                            const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
                            if (lane == 0) atomicMax(a.hamax + pick, m);
                        } else {
                            a.y[(size_t)pick * H + r0 + t_row] = v0[i] * s0 * pow2i(__ldg(a.hexp + pick));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hd.acc_empty);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// dst[i][:] = src[row(i)][:] for every bucketed pick i; row = token (mode 0) or pick (mode 1).
__global__ void __launch_bounds__(256) gather_rows_kernel(const __half* __restrict__ src, int len,
                                                          const int32_t* __restrict__ entries, int n, int k, int mode,
                                                          __half* __restrict__ dst) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const int pick = __ldg(entries + i);
    const int row = mode == 0 ? pick / k : pick;
    const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)row * len);
    uint4* d = reinterpret_cast<uint4*>(dst + (size_t)i * len);
    for (int c = threadIdx.x; c < len / 8; c += blockDim.x) d[c] = __ldg(s + c);
}

}  // namespace

size_t ffn_tc_smem_bytes() { return kTcSmem; }

cudaError_t launch_ffn_tc(const FfnArgs& a, int phase, int sel, int lo, int sm_count, cudaStream_t st) {
    const int K = phase == 0 ? a.H : a.I;
    const int n = a.T * a.k;
    __half* g = a.g;
    if (!g) return cudaErrorInvalidValue;
    gather_rows_kernel<<<n, 256, 0, st>>>(phase == 0 ? a.x16 : a.h16, K, a.entries, n, a.k, phase, g);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    CUtensorMap map;
    if (!encode_tmap_2d(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g, (uint64_t)K, (uint64_t)n, (uint64_t)K * 2, 64, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const long dmax = (long)(a.E < n / (lo + 1) + 1 ? a.E : n / (lo + 1) + 1);
    const long tasks = dmax * ((phase == 0 ? a.I : a.H) / kBM);
    const int grid = (int)(tasks < sm_count ? tasks : sm_count);
    if (grid <= 0) return cudaSuccess;
    static bool configured[2] = {false, false};
    if (!configured[phase]) {
        err = phase == 0 ? cudaFuncSetAttribute(ffn_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kTcSmem)
                         : cudaFuncSetAttribute(ffn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kTcSmem);
        if (err != cudaSuccess) return err;
        configured[phase] = true;
    }
    if (phase == 0) ffn_tc_kernel<0><<<grid, kThreadsTC, kTcSmem, st>>>(a, map, lo, sel);
    else ffn_tc_kernel<1><<<grid, kThreadsTC, kTcSmem, st>>>(a, map, lo, sel);
    return cudaGetLastError();
}

}  // namespace moe
