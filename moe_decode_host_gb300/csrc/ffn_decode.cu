// Grouped SwiGLU expert FFN, decode path (tokens per expert handled 8, 16 or 32
// at a time).
//
// "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1: after the
// cold copy, the layer runs all experts in one call, as if they were resident.
// At decode sizes each distinct expert's MXFP4 weights (about 20 MB at H=4096,
// I=3072) are streamed once from HBM (or from its scratch slot) and applied to
// the few tokens routed to it, so the kernel is bound by HBM bandwidth.
//
// Structure (one persistent CTA per SM):
//  - two producer threads (one per producer warp, taking alternate stages) stream
//    128-byte-wide slices of the weight rows of each task (an expert and 32 or 64
//    output rows) into a ring of shared-memory stages with 2D TMA loads (128-byte
//    swizzle), and with them the stage's slice of the bucket-ordered activation
//    rows of the expert's tokens (one 2D TMA load), signalling mbarriers;
//  - sixteen consumer warps dequantise the E2M1 nibbles in registers (one
//    e2m1x2 -> f16x2 conversion per byte) and feed mma.sync m16n8k16 as an exact
//    f16 x f16 -> fp32 dot-product engine; each 32-element block's E8M0 scale is
//    applied in fp32 to that block's partial sums.  Eight warps share each stage
//    (one 16-row tile and one 128-element half each) and the two groups of eight
//    take alternate stages; at the end of a task the partial sums meet in shared
//    memory and the first two or four warps add them in a fixed order.
// Each lane of a quad reads 8 elements of each 32-element block from the staged
// K-major rows, so every mma step sees a single block.  Activations are staged as f16 with an exact
// power-of-two prescale per row, in bucket order (row i belongs to entries[i]), so
// that an expert's tokens are consecutive rows.  Every wait is bounded by a deadline; a wait
// that runs out sets MOE_ERR_TIMEOUT in the status word and the CTA drains its
// copies and returns.
#include <cuda.h>

#include "ptx.cuh"

namespace moe {
namespace {

// Consumer warps: 16, in two groups of 8 that take the even and the odd stages.
// Within a group each warp handles one 16-row tile of the stage's 64 weight rows and
// one of its two 128-element groups, so every stage is worked on by 8 warps at once
// and two stages are in flight.
constexpr int kConsumers = 16;
constexpr int kPerStage = 8;    // consumer warps that read each stage
constexpr int kProducers = 2;   // producer warps; producer p fills the stages g with g % 2 == p
constexpr int kThreads = 32 * (kConsumers + kProducers);
constexpr int kMaxE = 1024;
constexpr int kSliceBytes = 128;  // bytes of one row per stage (256 elements)
constexpr int kStageRows = 64;    // weight rows per stage (both phases)

// Output rows per task: gate/up phase 32 (32 gate + 32 up weight rows per stage),
// down phase 64.
template <int P>
struct Cfg {
    static constexpr int kTaskRows = P == 0 ? 32 : 64;
};
constexpr int kActRow = 512;  // bytes of one activation row's slice in a stage (256 f16)
constexpr int kTaskQ = 4;     // depth of the CTA's task queue

struct alignas(16) SmemHead {
    uint64_t full[64];
    uint64_t empty[64];
    // tasks come from a launch-wide counter: producer 0 takes the next index and
    // publishes it in slot k % kTaskQ for the other producer and the consumer warps
    uint64_t tq_full[kTaskQ];
    uint64_t tq_empty[kTaskQ];
    int tq[kTaskQ];
    int D;
    int abort;
    int pad[2];
    int e[kMaxE];     // experts of this launch, ascending
    int cnt[kMaxE];   // and for each: its picks,
    int off[kMaxE];   // its first bucket entry,
    int phys[kMaxE];  // its physical id,
    const uint8_t* blob[kMaxE];  // and the base of its blob (null when phys is invalid)
};

template <int P, int NT>
struct Layout {
    static constexpr int kWBytes = kStageRows * 128;
    static constexpr int kABytes = 8 * NT * kActRow;
    // the stage rows' scale bytes (16 per row: this stage's 8 blocks and its
    // neighbour's), by TMA where the scale plane allows it
    static constexpr int kSBytes = kStageRows * 16;
    static constexpr int kStageBytes = ((kWBytes + kABytes + kSBytes) + 1023) & ~1023;
    // one partial-sum fragment per consumer warp, reduced once per task
    static constexpr int kFrag = NT * 4 * 32;
    static constexpr int kRedBytes = (int)sizeof(float) * kConsumers * kFrag;
    static constexpr int kBudget = 232448 - 1024 - (int)sizeof(SmemHead) - kRedBytes;
    // an even number of slots, so that each producer owns the slots of its parity
    static constexpr int kStages = ((kBudget / kStageBytes) < 64 ? (kBudget / kStageBytes) : 64) & ~1;
    static_assert(kStages >= 4, "ring too shallow");
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// Fragment row g (0..7) of an m16 tile is weight row perm8(g) (and +8): with the
// 128-byte swizzle this keeps the two rows a quarter-warp reads in disjoint banks.
__device__ __forceinline__ int perm8(int g) { return (g >> 1) | ((g & 1) << 2); }

// B operand from the stage's activation slices: column n (bucket row off + tb + n)
// of the stage lives at act + n * kActRow, 256 prescaled f16 values.  Columns past
// the expert's tokens hold other rows (or the zero fill past the tensor's end); an
// mma output column depends only on its own B column, and those columns are never
// stored, so every column is read unconditionally.
template <int NT>
struct SmemB {
    const uint8_t* col[NT];  // this lane's column in each n-tile
    __device__ __forceinline__ uint4 load(int nt, int byte_off) const {
        return *reinterpret_cast<const uint4*>(col[nt] + byte_off);
    }
};

// One warp's slice of a stage: acc[nt] += W[rows g, g+8 of the warp's 16-row tile,
// 128-element group gl] x B.  srow[r]: the two shared-memory rows of this lane;
// sc[r]: their 4 scale bytes for the group (byte j = 32-element block j).
template <int NT>
__device__ __forceinline__ void slice_mma(const uint8_t* stage, const int (&srow)[2], const uint32_t (&sc)[2],
                                          int gl, const SmemB<NT>& bl, float (&acc)[NT][4]) {
    const int q = threadIdx.x & 3;
    // word j of this lane: elements 8q..8q+7 of block j of the group (16-byte chunk
    // gl*4+j of the swizzled row); the 8 rows of a quarter-warp have distinct row%8,
    // so the 32 lanes hit 32 distinct banks
    uint32_t wv[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = srow[r];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int chunk = (gl * 4 + j) ^ (row & 7);
            wv[r][j] = *reinterpret_cast<const uint32_t*>(stage + row * kSliceBytes + chunk * 16 + q * 4);
        }
    }
    float scf[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) e8m0x4_to_f32(sc[r], scf[r]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t af[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) e2m1x8_to_f16x2(wv[r][j], af[r]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4 bv = bl.load(nt, gl * 256 + 64 * j + 16 * q);
            float d[4];
            mma_f16(d, af[0][0], af[1][0], af[0][1], af[1][1], bv.x, bv.y, 0.f, 0.f, 0.f, 0.f);
            mma_f16(d, af[0][2], af[1][2], af[0][3], af[1][3], bv.z, bv.w, d[0], d[1], d[2], d[3]);
            acc[nt][0] = fmaf(scf[0][j], d[0], acc[nt][0]);
            acc[nt][1] = fmaf(scf[0][j], d[1], acc[nt][1]);
            acc[nt][2] = fmaf(scf[1][j], d[2], acc[nt][2]);
            acc[nt][3] = fmaf(scf[1][j], d[3], acc[nt][3]);
        }
    }
}

// Task t of this CTA: listed expert t / tiles, row tile t % tiles.
struct TaskInfo {
    int rt, cnt, off, phys;
    bool valid;
    const uint8_t* blob;
};

__device__ __forceinline__ TaskInfo task_info(const FfnArgs& a, const SmemHead& hd, int task, int tiles) {
    TaskInfo ti;
    const int i = task / tiles;
    ti.rt = task % tiles;
    ti.cnt = hd.cnt[i];
    ti.off = hd.off[i];
    ti.phys = hd.phys[i];
    ti.valid = ti.phys >= 0 && ti.phys < a.n_phys;
    ti.blob = hd.blob[i];
    return ti;
}

// ZC (zero copy): the listed experts are cold and their weights are read in place
// from pinned host memory: the producer warps load each stage's 64 rows x 128 bytes
// with 16-byte loads over the host link and store them in the layout the TMA gives
// (128-byte swizzle); the activation slice still comes by TMA.
template <int P, int NT, bool ZC>
__global__ void __launch_bounds__(kThreads, 1) ffn_tma_kernel(FfnArgs a, const __grid_constant__ CUtensorMap act_map,
                                                                int lo, int hi, int sel, int ctr) {
    using C = Cfg<P>;
    using L = Layout<P, NT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    SmemHead& hd = *reinterpret_cast<SmemHead*>(stages + L::kStages * L::kStageBytes);
    float* red = reinterpret_cast<float*>(&hd + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I;
    const int K = P == 0 ? H : I;
    const int ngroups = K / 128;
    const int nst = (ngroups + 1) / 2;
    const int tiles = (P == 0 ? I : H) / C::kTaskRows;
    // scale words reach the stage by TMA (copy path, scale rows a whole number of
    // 16-byte units), else the consumers read them from the blob
    const bool smem_sc = !ZC && mx_scale_maps(K);

    // active experts in this launch's token-count range and placement class: every
    // thread takes some experts and, for the active ones, follows the chain to the
    // blob at once (picks, first entry and placement are independent loads, then the
    // entry's physical id and the blob pointer), keeping per-expert values in the
    // stage ring (unused until the producers start); then warp 0 compacts the flags
    // into an ascending list and every thread copies the listed experts' values
    struct PerExpert {
        const uint8_t* blob;
        int cnt, off, phys, act;
    };
    PerExpert* pe = reinterpret_cast<PerExpert*>(stages);
    static_assert(sizeof(PerExpert) * kMaxE <= 2 * L::kStageBytes, "per-expert scratch fits two stages");
#pragma unroll 1
    for (int e = threadIdx.x; e < a.E; e += kThreads) {
        const int c = __ldg(a.counts + e);
        const int off = __ldg(a.offsets + e);
        const int le = sel != 0 ? __ldg(a.loc + e) : 0;
        bool act_e = c > lo && c <= hi;
        if (act_e && sel != 0) act_e = (sel == 1) ? (le < a.n_hot) : (le >= a.n_hot);
        PerExpert v;
        v.act = act_e;
        v.cnt = c;
        v.off = off;
        v.phys = -1;
        v.blob = nullptr;
        if (act_e) {
            v.phys = __ldg(a.phys_ids + __ldg(a.entries + off));
            v.blob = (v.phys >= 0 && v.phys < a.n_phys)
                         ? ((ZC && v.phys >= a.n_hot) ? a.cold_host[v.phys - a.n_hot] : a.ptr[v.phys])
                         : nullptr;
        }
        pe[e] = v;
    }
    __syncthreads();
    if (warp == 0) {
        int cnt = 0;
        for (int base = 0; base < a.E; base += 32) {
            const int e = base + lane;
            const bool act_e = e < a.E && pe[e].act != 0;
            const unsigned m = __ballot_sync(0xffffffffu, act_e);
            if (act_e) hd.e[cnt + __popc(m & ((1u << lane) - 1u))] = e;
            cnt += __popc(m);
        }
        if (lane == 0) {
            hd.D = cnt;
            hd.abort = 0;
            for (int s = 0; s < L::kStages; ++s) {
                // zero copy: the activation TMA's arrival and the producer warp's, after its stores
                mbar_init(&hd.full[s], ZC ? 2 : 1);
                mbar_init(&hd.empty[s], kPerStage);
            }
            for (int j = 0; j < kTaskQ; ++j) {
                mbar_init(&hd.tq_full[j], 1);
                mbar_init(&hd.tq_empty[j], 1 + kConsumers);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < hd.D; i += kThreads) {
        const PerExpert v = pe[hd.e[i]];
        hd.cnt[i] = v.cnt;
        hd.off[i] = v.off;
        hd.phys[i] = v.phys;
        hd.blob[i] = v.blob;
    }
    // the ring is rewritten by the async proxy (TMA) from here on
    fence_proxy_async_shared();
    __syncthreads();
    // the activations, their prescales and the outputs belong to the previous kernel
    // until it completes; the work above only read routing results
    grid_dep_wait();
    const int ntask = hd.D * tiles;
    volatile int* abort = &hd.abort;

    if (warp >= kConsumers) {
        if constexpr (ZC) {
            // ---------------- producers, zero copy (whole producer warp) ----------------
            const unsigned pp = (unsigned)(warp - kConsumers);
            const int rowb = K / 2;  // bytes of one weight row
            int slot = 0;
            unsigned phase = 0;
            int gstage = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int j = k % kTaskQ;
                const unsigned qpar = (unsigned)(k / kTaskQ) & 1u;
                int task = -1;
                bool got = true;
                if (lane == 0) {
                    if (pp == 0) {
                        got = mbar_wait_fast(&hd.tq_empty[j], qpar ^ 1u, abort, a.status, a.diag, 4, j, k, 0);
                        if (got) {
                            task = atomicAdd(a.task_ctr + ctr, 1);
                            if (task >= ntask) task = -1;
                            *reinterpret_cast<volatile int*>(&hd.tq[j]) = task;
                            mbar_arrive(&hd.tq_full[j]);
                        }
                    } else {
                        got = mbar_wait_fast(&hd.tq_full[j], qpar, abort, a.status, a.diag, 5, j, k, 0);
                        if (got) {
                            task = *reinterpret_cast<volatile int*>(&hd.tq[j]);
                            mbar_arrive(&hd.tq_empty[j]);
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, got, 0)) break;
                task = __shfl_sync(0xffffffffu, task, 0);
                if (task < 0) break;
                const TaskInfo ti = task_info(a, hd, task, tiles);
                if (!ti.valid) continue;
                const uint8_t* wbase = ti.blob + (P == 0 ? 0 : a.w2n);
                const int r0 = ti.rt * C::kTaskRows;
                for (int tb = 0; tb < ti.cnt && ok; tb += 8 * NT) {
                    for (int s = 0; s < nst && ok; ++s) {
                        if (((unsigned)gstage & 1u) == pp) {
                            // this lane's 16 of the stage's 512 16-byte chunks (64 rows x 128
                            // bytes; the gate/up phase: 32 gate rows, then 32 up rows), loaded
                            // before the slot is free so the host latency overlaps the wait;
                            // chunks past the row's end (an odd K tail) read as zero
                            uint4 v[16];
#pragma unroll
                            for (int i2 = 0; i2 < 16; ++i2) {
                                const int idx = lane + 32 * i2;
                                const int lr = idx >> 3, ch = idx & 7;
                                const int grow = P == 0 ? (lr < 32 ? r0 + lr : I + r0 + lr - 32) : r0 + lr;
                                const int col = s * kSliceBytes + ch * 16;
                                v[i2] = col < rowb ? ld_host_v4(wbase + (size_t)grow * rowb + col)
                                                   : make_uint4(0u, 0u, 0u, 0u);
                            }
                            bool w = true;
                            if (lane == 0)
                                w = mbar_wait_fast(&hd.empty[slot], phase ^ 1u, abort, a.status, a.diag, 2, slot, s,
                                                   (task << 8) | min(8 * NT, ti.cnt - tb));
                            if (!__shfl_sync(0xffffffffu, w, 0)) {
                                ok = false;
                                break;
                            }
                            uint8_t* dst = stages + slot * L::kStageBytes;
                            if (lane == 0) {
                                mbar_arrive_expect_tx(&hd.full[slot], (unsigned)L::kABytes);
                                tma_load_2d(dst + L::kWBytes, &act_map, s * 256, ti.off + tb, &hd.full[slot]);
                            }
#pragma unroll
                            for (int i2 = 0; i2 < 16; ++i2) {
                                const int idx = lane + 32 * i2;
                                const int lr = idx >> 3, ch = idx & 7;
                                *reinterpret_cast<uint4*>(dst + lr * kSliceBytes + ((ch ^ (lr & 7)) << 4)) = v[i2];
                            }
                            __syncwarp();  // the lanes' stores come before lane 0's arrival
                            if (lane == 0) mbar_arrive(&hd.full[slot]);
                        }
                        ++gstage;
                        if (++slot == L::kStages) {
                            slot = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // drain: every activation copy this producer issued has landed
            if (lane == 0)
                for (int s = (int)pp; s < L::kStages; s += kProducers) {
                    if (s >= gstage) break;
                    const int g_last = s + L::kStages * ((gstage - 1 - s) / L::kStages);
                    mbar_drain(&hd.full[s], (unsigned)(g_last / L::kStages) & 1u);
                }
            return;
        }
        // ---------------- producers (lane 0 of each producer warp) ----------------
        if (lane == 0) {
            const unsigned pp = (unsigned)(warp - kConsumers);
            int slot = 0;
            unsigned phase = 0;
            int gstage = 0;  // global stage number in this CTA's stream
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int j = k % kTaskQ;
                const unsigned qpar = (unsigned)(k / kTaskQ) & 1u;
                int task;
                if (pp == 0) {
                    if (!mbar_wait_fast(&hd.tq_empty[j], qpar ^ 1u, abort, a.status, a.diag, 4, j, k, 0)) break;
                    task = atomicAdd(a.task_ctr + ctr, 1);
                    if (task >= ntask) task = -1;
                    *reinterpret_cast<volatile int*>(&hd.tq[j]) = task;
                    mbar_arrive(&hd.tq_full[j]);
                } else {
                    if (!mbar_wait_fast(&hd.tq_full[j], qpar, abort, a.status, a.diag, 5, j, k, 0)) break;
                    task = *reinterpret_cast<volatile int*>(&hd.tq[j]);
                    mbar_arrive(&hd.tq_empty[j]);
                }
                if (task < 0) break;
                const TaskInfo ti = task_info(a, hd, task, tiles);
                if (!ti.valid) continue;
                const CUtensorMap* map = P == 0 ? &a.tmaps[ti.phys].w13n : &a.tmaps[ti.phys].w2n;
                const CUtensorMap* smap = P == 0 ? &a.tmaps[ti.phys].w13s : &a.tmaps[ti.phys].w2s;
                // descriptors live in global memory and a layer's table may reuse the
                // address of a destroyed one: acquire the current contents for the async proxy
                asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
                if (smem_sc) asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(smap) : "memory");
                const int r0 = ti.rt * C::kTaskRows;
                for (int tb = 0; tb < ti.cnt && ok; tb += 8 * NT) {
                    for (int s = 0; s < nst; ++s) {
                        if (((unsigned)gstage & 1u) == pp) {
                            if (!mbar_wait_fast(&hd.empty[slot], phase ^ 1u, abort, a.status, a.diag, 2, slot, s,
                                                (task << 8) | min(8 * NT, ti.cnt - tb))) {
                                ok = false;
                                break;
                            }
                            uint8_t* dst = stages + slot * L::kStageBytes;
                            // full boxes land even past the tensor's edge (zero filled)
                            mbar_arrive_expect_tx(&hd.full[slot],
                                                  (unsigned)(L::kWBytes + L::kABytes + (smem_sc ? L::kSBytes : 0)));
                            if (P == 0) {
                                tma_load_2d(dst, map, s * kSliceBytes, r0, &hd.full[slot]);
                                tma_load_2d(dst + C::kTaskRows * kSliceBytes, map, s * kSliceBytes, I + r0,
                                            &hd.full[slot]);
                            } else {
                                tma_load_2d(dst, map, s * kSliceBytes, r0, &hd.full[slot]);
                            }
                            if (smem_sc) {
                                // 16 scale bytes per row (this stage's 8 blocks and the neighbour
                                // stage's), 32 rows per box: gate then up rows, or two w2 boxes
                                uint8_t* sdst = dst + L::kWBytes + L::kABytes;
                                tma_load_2d(sdst, smap, 16 * (s >> 1), r0, &hd.full[slot]);
                                tma_load_2d(sdst + 32 * 16, smap, 16 * (s >> 1), P == 0 ? I + r0 : r0 + 32,
                                            &hd.full[slot]);
                            }
                            tma_load_2d(dst + L::kWBytes, &act_map, s * 256, ti.off + tb, &hd.full[slot]);
                        }
                        ++gstage;
                        if (++slot == L::kStages) {
                            slot = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // drain: every copy this producer issued has landed before the CTA may exit.
            // Slot s (of this producer's parity) last held stage s + S * ((G - 1 - s) / S)
            // of the G stages counted, if s < G.
            for (int s = (int)pp; s < L::kStages; s += kProducers) {
                if (s >= gstage) break;
                const int g_last = s + L::kStages * ((gstage - 1 - s) / L::kStages);
                mbar_drain(&hd.full[s], (unsigned)(g_last / L::kStages) & 1u);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    // warp = sp * 8 + (tile << 2 | rt << 1 | gl) in the gate/up phase (tile 0 gate, 1 up;
    // rt = 16-row tile of the 32 output rows), sp * 8 + (rt << 1 | gl) in the down
    // phase (rt = 16-row tile of 64); sp = parity of the stages this warp reads, gl =
    // its 128-element group of each stage
    const int sp = warp >> 3;
    const int gl = warp & 1;
    const int tile = P == 0 ? ((warp >> 2) & 1) : 0;
    const int rt = P == 0 ? ((warp >> 1) & 1) : ((warp >> 1) & 3);
    const int g = lane >> 2, q = lane & 3;
    const int pg = perm8(g);
    const size_t srs = (size_t)K / 32;  // scale bytes per row
    // epilogue warps: the first 2 (gate/up phase) or 4 (down phase) consumer warps,
    // one per 16 output rows
    constexpr int kEpi = P == 0 ? 2 : 4;
    int gstage = 0;
    bool done = false;
    for (int k = 0;; ++k) {
        const int j = k % kTaskQ;
        const unsigned qpar = (unsigned)(k / kTaskQ) & 1u;
        const bool got = __all_sync(0xffffffffu, mbar_wait_fast(&hd.tq_full[j], qpar, abort, a.status, a.diag, 5, j,
                                                                k, 1));
        // all consumer warps must take the same task or stop together (they meet at
        // named barriers inside a task)
        unsigned qstop;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.eq.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(qstop)
            : "r"((unsigned)got), "n"(32 * kConsumers)
            : "memory");
        const int task = qstop ? -1 : *reinterpret_cast<volatile int*>(&hd.tq[j]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd.tq_empty[j]);
        if (task < 0) break;
        const TaskInfo ti = task_info(a, hd, task, tiles);
        const int r0 = ti.rt * C::kTaskRows;
        if (!ti.valid) {
            // zero outputs for an expert whose physical id is out of range
            if (ti.rt == 0 && threadIdx.x == 0) set_status(a.status, MOE_ERR_BAD_EXPERT);
            for (int c = threadIdx.x; c < ti.cnt * C::kTaskRows; c += 32 * kConsumers) {
                const int pos = ti.off + c / C::kTaskRows;
                const int row = r0 + c % C::kTaskRows;
                if (P == 0) a.h[(size_t)pos * I + row] = 0.f;
                else a.y[(size_t)__ldg(a.entries + pos) * H + row] = 0.f;
            }
            continue;
        }
        const uint8_t* sb = ti.blob + (P == 0 ? a.w13s : a.w2s);
        // this lane's two weight rows: within the stage and in the plane
        int srow[2], grow[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int lr = 16 * rt + pg + 8 * r;
            srow[r] = (P == 0 ? tile * C::kTaskRows : 0) + lr;
            grow[r] = (P == 0 && tile == 1 ? I : 0) + r0 + lr;
        }
        for (int tb = 0; tb < ti.cnt; tb += 8 * NT) {
            const int ncols = min(8 * NT, ti.cnt - tb);
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
            // this warp reads every other stage; the 4 scale bytes of its group for its
            // two rows sit in two register pairs used alternately, each refilled right
            // after use for the stage two own stages later
            uint32_t scA[2], scB[2];
            auto load_sc = [&](int s, uint32_t(&dst)[2]) {
                if (smem_sc) return;  // read from the stage once it has landed
                const int grp = 2 * s + gl;
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    dst[r] = grp < ngroups ? ld_u32(sb + (size_t)grow[r] * srs + (size_t)grp * 4) : 0u;
            };
            // own stages: those whose global number gstage + s has parity sp (a pass can
            // have an odd number of stages, so the first one depends on gstage)
            const int sf = (sp ^ gstage) & 1;
            if (sf < nst) load_sc(sf, scA);
            if (sf + 2 < nst) load_sc(sf + 2, scB);
            bool ok = true;
            // The parity wait below cannot match a phase one lap old: slots have the parity
            // of their stages (kStages is even), so this warp's group reads every stage
            // ever put in slot sl, and it waited for the previous one (gs - kStages)
            // before this; every warp of the group waits on every stage of its parity,
            // even where its group is past the K tail.
            auto own_stage = [&](int s, uint32_t(&sc)[2]) -> bool {
                const int gs = gstage + s;
                const int sl = gs % L::kStages;
                const unsigned ph = (unsigned)(gs / L::kStages) & 1u;
                if (!mbar_wait_fast(&hd.full[sl], ph, abort, a.status, a.diag, 1, sl, s, (task << 8) | ncols))
                    return false;
                if (2 * s + gl < ngroups) {  // (an odd K tail leaves group 1 of the last stage empty)
                    const uint8_t* stage = stages + sl * L::kStageBytes;
                    if (smem_sc) {
                        // word gl of the stage's 8 blocks in each of this lane's two rows
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            sc[r] = *reinterpret_cast<const uint32_t*>(stage + L::kWBytes + L::kABytes + srow[r] * 16 +
                                                                       8 * (s & 1) + 4 * gl);
                    }
                    SmemB<NT> bl;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int n = nt * 8 + g;
                        bl.col[nt] = stage + L::kWBytes + n * kActRow;
                    }
                    slice_mma<NT>(stage, srow, sc, gl, bl, acc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hd.empty[sl]);
                if (s + 4 < nst) load_sc(s + 4, sc);
                return true;
            };
            for (int s = sf; s < nst && ok; s += 4) {
                ok = own_stage(s, scA);
                if (ok && s + 2 < nst) ok = own_stage(s + 2, scB);
            }
            gstage += nst;
            // all consumer warps take the same decision to stop (a timed-out wait anywhere)
            unsigned stop;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, 1, %2, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(stop)
                : "r"((unsigned)(!ok || *abort)), "n"(32 * kConsumers)
                : "memory");
            if (stop) {
                done = true;
                break;
            }
            // partial sums meet in shared memory; the epilogue warps add them in a fixed
            // order (stage parity, then group)
            float* mine = red + (size_t)warp * L::kFrag;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) mine[(nt * 4 + c) * 32 + lane] = acc[nt][c];
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers));
            if (warp < kEpi) {
                const int ert = warp;  // output row tile of this epilogue warp
                // this lane's output columns: prescale exponent (and for the down phase
                // the pick), loaded first so that the partial-sum reads hide their latency
                int cexp[NT][2], cpick[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int col = nt * 8 + 2 * q + c2;
                        const int pos = ti.off + tb + col;
                        cexp[nt][c2] = col < ncols ? __ldg(a.gexp + pos) : 0;
                        cpick[nt][c2] = (P == 1 && col < ncols) ? __ldg(a.entries + pos) : 0;
                    }
                float v0[NT][4], v1[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) v0[nt][c] = v1[nt][c] = 0.f;
#pragma unroll
                for (int sp2 = 0; sp2 < 2; ++sp2)
#pragma unroll
                    for (int gl2 = 0; gl2 < 2; ++gl2) {
                        const int w0 = sp2 * 8 + (ert << 1) + gl2;             // gate (or w2) rows
                        const int w1 = sp2 * 8 + (1 << 2) + (ert << 1) + gl2;  // up rows
                        const float* p0 = red + (size_t)w0 * L::kFrag;
                        const float* p1 = red + (size_t)w1 * L::kFrag;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                v0[nt][c] += p0[(nt * 4 + c) * 32 + lane];
                                if (P == 0) v1[nt][c] += p1[(nt * 4 + c) * 32 + lane];
                            }
                    }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int col = nt * 8 + 2 * q + (c & 1);
                        if (col >= ncols) continue;
                        const int pos = ti.off + tb + col;
                        const float sx = pow2i(cexp[nt][c & 1]);
                        const int orow = r0 + 16 * ert + pg + ((c >> 1) << 3);  // output row
                        if constexpr (P == 0) {
                            const float gv = v0[nt][c] * sx;
                            const float uv = v1[nt][c] * sx;
                            a.h[(size_t)pos * I + orow] = gv / (1.0f + expf(-gv)) * uv;
                        } else {
                            a.y[(size_t)cpick[nt][c & 1] * H + orow] = v0[nt][c] * sx;
                        }
                    }
            }
            // (the next writes to the partial sums come after the next task's first
            // barrier, which the epilogue warps reach only when done)
        }
        if (done) break;
    }
}

// Row of `rows` fp32 or bf16 values -> f16 with a power-of-two prescale that puts
// the row's amax in [2^14, 2^15) (exact up to the f16 rounding of each value).  One
// CTA of 256 threads; up to 4 chunks of 8 values per thread stay in registers.
template <bool BF16>
__device__ __forceinline__ void prescale_row(const void* src_row, int len, __half* dst_row, int32_t* exp_out) {
    __shared__ float wmax[8];
    const int nch = len / 8;
    constexpr int kPer = 4;
    float v[kPer][8];
    float amax = 0.f;
    auto load = [&](int c, float (&f)[8]) {
        if constexpr (BF16) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(src_row) + c);
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 t = __bfloat1622float2(p[i]);
                f[2 * i] = t.x;
                f[2 * i + 1] = t.y;
            }
        } else {
            const float4 a0 = __ldcg(reinterpret_cast<const float4*>(src_row) + 2 * c);
            const float4 a1 = __ldcg(reinterpret_cast<const float4*>(src_row) + 2 * c + 1);
            f[0] = a0.x, f[1] = a0.y, f[2] = a0.z, f[3] = a0.w;
            f[4] = a1.x, f[5] = a1.y, f[6] = a1.z, f[7] = a1.w;
        }
    };
    auto upd = [&](const float (&f)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    };
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int c = threadIdx.x + u * 256;
        if (c < nch) {
            load(c, v[u]);
            upd(v[u]);
        }
    }
    for (int c = threadIdx.x + kPer * 256; c < nch; c += 256) {
        float f[8];
        load(c, f);
        upd(f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = wmax[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
    const int p = prescale_exp(amax);
    const float sc = pow2i(-p);
    auto store = [&](int c, const float (&f)[8]) {
        uint4 o;
        __half2* po = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) po[i] = __floats2half2_rn(f[2 * i] * sc, f[2 * i + 1] * sc);
        reinterpret_cast<uint4*>(dst_row)[c] = o;
    };
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int c = threadIdx.x + u * 256;
        if (c < nch) store(c, v[u]);
    }
    for (int c = threadIdx.x + kPer * 256; c < nch; c += 256) {
        float f[8];
        load(c, f);
        store(c, f);
    }
    if (threadIdx.x == 0) *exp_out = p;
}

// One CTA per bucket row i: x of token entries[i] / k, prescaled, into g row i.
__global__ void __launch_bounds__(256) xprep_kernel(const __nv_bfloat16* __restrict__ x, int H, int k,
                                                    const int32_t* __restrict__ entries, int gstride,
                                                    __half* __restrict__ g, int32_t* __restrict__ gexp,
                                                    int32_t* __restrict__ task_ctr) {
    const int i = blockIdx.x;
    if (i == 0 && threadIdx.x < kTaskCounters) task_ctr[threadIdx.x] = 0;
    const int t = __ldg(entries + i) / k;
    prescale_row<true>(x + (size_t)t * H, H, g + (size_t)i * gstride, gexp + i);
}

// One CTA per bucket row i of the selected class: h row i, prescaled, into g row i.
__global__ void __launch_bounds__(256) hprep_kernel(const float* __restrict__ h, const int32_t* __restrict__ entries,
                                                    const int32_t* __restrict__ phys_ids, int n_hot, int n_phys,
                                                    int sel, int I, int gstride, __half* __restrict__ g,
                                                    int32_t* __restrict__ gexp) {
    grid_dep_wait();
    const int i = blockIdx.x;
    const int ph = __ldg(phys_ids + __ldg(entries + i));
    const bool hot = ph >= 0 && ph < n_hot;
    const bool valid = ph >= 0 && ph < n_phys;
    if (sel == 1 && !hot) return;
    if (sel == 2 && (hot || !valid)) return;
    prescale_row<false>(h + (size_t)i * I, I, g + (size_t)i * gstride, gexp + i);
}

__global__ void debug_e2m1_kernel(uint32_t* out) {
    const int b = threadIdx.x;
    uint32_t r[4];
    e2m1x8_to_f16x2((uint32_t)b, r);
    out[b] = r[0];
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct WsLayout {
    size_t ctr, g, gexp, h, total;
};

WsLayout ws_layout(int T, int k, int H, int I) {
    WsLayout w;
    const size_t n = (size_t)T * k;
    size_t o = 0;
    w.ctr = o;
    o = align256(o + kTaskCounters * sizeof(int32_t));
    w.g = o;
    o = align256(o + n * (H > I ? H : I) * sizeof(__half));
    w.gexp = o;
    o = align256(o + n * sizeof(int32_t));
    w.h = o;
    o = align256(o + n * I * sizeof(float));
    w.total = o;
    return w;
}

template <int P, int NT>
size_t smem_bytes() {
    using L = Layout<P, NT>;
    return 1024 + (size_t)L::kStages * L::kStageBytes + sizeof(SmemHead) + (size_t)L::kRedBytes;
}

template <int P, int NT, bool ZC>
cudaError_t launch_phase(const FfnArgs& a, int lo, int hi, int sel, int ctr, int grid, cudaStream_t st) {
    static std::atomic<uint64_t> configured{0};
    const size_t sm = smem_bytes<P, NT>();
    const cudaError_t e = ensure_smem_limit((const void*)ffn_tma_kernel<P, NT, ZC>, (int)sm, configured);
    if (e != cudaSuccess) return e;
    // the stage's activation slice: 256 elements of 8 * NT consecutive bucket rows
    CUtensorMap act_map;
    if (!encode_act_map(&act_map, a, P, 256, 8 * NT, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    return launch_pdl(ffn_tma_kernel<P, NT, ZC>, dim3(grid), dim3(kThreads), sm, st, a, act_map, lo, hi, sel, ctr);
}

}  // namespace

size_t ffn_decode_workspace(int T, int k, int H, int I) { return ws_layout(T, k, H, I).total; }

bool encode_act_map(CUtensorMap* m, const FfnArgs& a, int phase, uint32_t box_inner, uint32_t box_rows,
                    CUtensorMapSwizzle sw) {
    const uint64_t stride = (uint64_t)(a.H > a.I ? a.H : a.I) * sizeof(__half);
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.g, (uint64_t)(phase == 0 ? a.H : a.I),
                          (uint64_t)a.T * a.k, stride, box_inner, box_rows, sw);
}

cudaError_t launch_ffn_prep(FfnArgs& a, void* workspace, cudaStream_t st) {
    const WsLayout w = ws_layout(a.T, a.k, a.H, a.I);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.task_ctr = reinterpret_cast<int32_t*>(ws + w.ctr);
    a.g = reinterpret_cast<__half*>(ws + w.g);
    a.gexp = reinterpret_cast<int32_t*>(ws + w.gexp);
    a.h = reinterpret_cast<float*>(ws + w.h);
    if (a.T == 0) return cudaSuccess;
    xprep_kernel<<<a.T * a.k, 256, 0, st>>>(a.x, a.H, a.k, a.entries, a.H > a.I ? a.H : a.I, a.g, a.gexp,
                                            a.task_ctr);
    return cudaGetLastError();
}

cudaError_t launch_ffn_phase(const FfnArgs& a, int phase, int sel, int sm_count, cudaStream_t st, bool zc) {
    if (a.T == 0) return cudaSuccess;
    // token-count ranges per kernel (a bound on the largest bucket is T); buckets
    // above kTcMinTokens go to the tensor-core kernel
    struct Range {
        int nt, lo, hi;
    };
    const Range ranges[3] = {{1, 0, 8}, {2, 8, 16}, {4, 16, kTcMinTokens}};
    const long dmax = (long)(a.E < a.T * a.k ? a.E : a.T * a.k);
    const long tasks = dmax * (phase == 0 ? a.I / Cfg<0>::kTaskRows : a.H / Cfg<1>::kTaskRows);
    if (phase == 1) {
        cudaError_t e = launch_pdl(hprep_kernel, dim3(a.T * a.k), dim3(256), 0, st, (const float*)a.h,
                                   (const int32_t*)a.entries, (const int32_t*)a.phys_ids, a.n_hot, a.n_phys, sel, a.I,
                                   a.H > a.I ? a.H : a.I, a.g, a.gexp);
        if (e != cudaSuccess) return e;
    }
    const int grid = (int)(tasks < sm_count ? tasks : sm_count);
    for (int ri = 0; ri < 3; ++ri) {
        const Range& r = ranges[ri];
        if (a.T <= r.lo) break;
        // each launch of the call takes tasks from its own counter (zeroed by xprep)
        const int ctr = ((sel == 2 ? 2 : 0) + phase) * 3 + ri;
        cudaError_t err;
        if (zc) {
            if (phase == 0) {
                err = r.nt == 1 ? launch_phase<0, 1, true>(a, r.lo, r.hi, sel, ctr, grid, st)
                    : r.nt == 2 ? launch_phase<0, 2, true>(a, r.lo, r.hi, sel, ctr, grid, st)
                                : launch_phase<0, 4, true>(a, r.lo, r.hi, sel, ctr, grid, st);
            } else {
                err = r.nt == 1 ? launch_phase<1, 1, true>(a, r.lo, r.hi, sel, ctr, grid, st)
                    : r.nt == 2 ? launch_phase<1, 2, true>(a, r.lo, r.hi, sel, ctr, grid, st)
                                : launch_phase<1, 4, true>(a, r.lo, r.hi, sel, ctr, grid, st);
            }
        } else if (phase == 0) {
            err = r.nt == 1 ? launch_phase<0, 1, false>(a, r.lo, r.hi, sel, ctr, grid, st)
                : r.nt == 2 ? launch_phase<0, 2, false>(a, r.lo, r.hi, sel, ctr, grid, st)
                            : launch_phase<0, 4, false>(a, r.lo, r.hi, sel, ctr, grid, st);
        } else {
            err = r.nt == 1 ? launch_phase<1, 1, false>(a, r.lo, r.hi, sel, ctr, grid, st)
                : r.nt == 2 ? launch_phase<1, 2, false>(a, r.lo, r.hi, sel, ctr, grid, st)
                            : launch_phase<1, 4, false>(a, r.lo, r.hi, sel, ctr, grid, st);
        }
        if (err != cudaSuccess) return err;
    }
    if (a.T > kTcMinTokens) {
        if (zc) return cudaErrorInvalidValue;  // the tensor-core kernel reads the scratch copies
        return launch_ffn_tc(a, phase, sel, kTcMinTokens, sm_count, st);
    }
    return cudaSuccess;
}

cudaError_t launch_debug_e2m1(uint32_t* out, cudaStream_t st) {
    debug_e2m1_kernel<<<1, 256, 0, st>>>(out);
    return cudaGetLastError();
}

}  // namespace moe
