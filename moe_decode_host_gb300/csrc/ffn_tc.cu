// Grouped SwiGLU expert FFN for prefill-sized buckets (more than 64 tokens per
// expert) on the 5th-generation tensor cores.
//
// "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1: the layer
// runs all experts in one call.  When an expert receives many tokens its weights
// are reused across them and the work is a dense contraction, so it runs as a
// GEMM: D[128 weight rows x N tokens] += W[128 x K] * X[N x K]^T with
// tcgen05.mma (kind::f16, f16 operands, fp32 accumulators in tensor memory).
//
// A column pass covers up to 160 of an expert's tokens, so at about 128 tokens per
// expert every expert's weights are expanded once. Its K dimension runs in chunks
// of 128 elements; in the gate/up phase each chunk is two stages, one for the tile's
// 128 gate rows and one for its 128 up rows, in the down phase one stage.
//
// Warp roles of one persistent CTA per SM (16 warps):
//   warp 0       takes tasks (an expert and a 128-row tile) from a launch-wide
//                counter, experts with the most tokens first, and publishes them in
//                a small shared-memory queue; TMA of the raw MXFP4 slice of each
//                stage (one matrix's 128 rows x 128 elements, 64-byte swizzle)
//                into a ring of raw stages;
//   warps 1, 3   own tensor memory (warp 1) and issue the MMAs, one thread each:
//                in the gate/up phase warp 1 the gate stages into the gate
//                accumulator and warp 3 the up stages into the up accumulator (a
//                thread issues a tcgen05 MMA about every 45 cycles, so each issuer
//                has the other matrix's MMA time as slack); the down phase has one
//                issuer and two accumulator buffers, so a tile's epilogue overlaps
//                the next tile's main loop;
//   warp 2       TMA of the activation chunks (up to 160 bucket rows x 128
//                elements, f16, as two 64-element atoms with 128-byte swizzle; the
//                prescale kernels write the activations in bucket order, so an
//                expert's tokens are consecutive rows), into a ring of its own;
//   warps 4-11   converters: E2M1 -> f16 for one half of a weight row's stage per
//                thread, each E8M0 block scale rebased to 2^12 below the row's
//                largest scale, so that every block whose scale is within 2^35 of
//                the largest is exact in f16 (smaller blocks lose low bits); the f16
//                tiles go to tensor memory (tcgen05.st: one weight row per lane,
//                consecutive K elements packed two per column) in a ring of three
//                64-column slots, where the MMA reads its A operand, so shared
//                memory carries only raw weights and activations;
//   warps 12-15  epilogue: tensor memory -> registers -> h (gate/up phase, SiLU
//                gate times up, full 16-token chunks through shared memory and bulk
//                tensor stores) or y (down phase), undoing the power-of-two
//                rebasing of weights and activations.
// Every wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT, and the CTA
// drains its copies and MMAs before it frees tensor memory and returns.
#include <cuda.h>

#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;    // weight rows per tile = tensor-memory lanes
constexpr int kBK = 128;    // K elements per stage (two 128-byte swizzle atoms of f16 per row)
constexpr int kNMax = 160;  // token columns per pass (a multiple of 32)
constexpr int kRawStages = 8;  // raw E2M1 slices of one matrix: 128 rows x 128 elements, 8 KB each
constexpr int kAStages = 3;    // f16 weight stages in tensor memory, 64 columns each
constexpr int kBStages = 3;    // activation tiles, one per 128-element chunk of K
constexpr int kFirstConv = 4;   // first converter warp
constexpr int kConvWarps = 8;
constexpr int kFirstEpi = 12;   // first epilogue warp (warp % 4 = lane quarter)
constexpr int kThreadsTC = 512;
constexpr int kRawRow = kBK / 2;             // E2M1 bytes of one row per stage
constexpr int kRawBytes = kBM * kRawRow;     // 8 KB
constexpr int kActBoxRows = 32;              // activation rows per TMA box
constexpr int kBAtom = kNMax * 128;          // 64 elements of K of the activation tile, 20 KB
constexpr int kBStageBytes = 2 * kBAtom;     // activation tile, 40 KB
// Tensor memory (512 columns): accumulators in [0, 320) -- gate and up (160 columns
// each) in the gate/up phase, two 160-column buffers in the down phase -- and the
// f16 weight stages in [320, 512), 64 columns each (one matrix, 128 elements of K,
// two f16 per column).
constexpr uint32_t kAccCols = 160;           // columns per accumulator (N <= 160)
constexpr uint32_t kACol0 = 320;             // first column of the weight stages
constexpr uint32_t kAStageCols = 64;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr int kTaskQ = 4;  // depth of the CTA's task queue
// Gate/up phase: a pass runs its K chunks as stages that alternate between the gate
// rows and the up rows of the tile (stage 2c: gate rows of chunk c, 2c+1: up rows),
// so one weight stage holds one matrix and the pass needs no second column pass up
// to 160 tokens. Warp 1 issues the gate MMAs into the gate accumulator and warp 3
// the up MMAs (a thread issues a tcgen05 MMA about every 45 cycles, so each issuer
// gets a stage's worth of slack while the other matrix's MMAs run). Down phase:
// one stage per chunk, one issuer.
template <int P>
__host__ __device__ constexpr int issuers() { return P == 0 ? 2 : 1; }
template <int P>
__host__ __device__ constexpr int mats() { return P == 0 ? 2 : 1; }  // weight matrices per chunk
// roles that take each task from the queue: activation producer, MMA issuers,
// converter warps, epilogue warps (the raw weight producer fetches them)
template <int P>
__host__ __device__ constexpr int task_takers() { return 1 + issuers<P>() + kConvWarps + 4; }

// One task: a listed expert (picks, first bucket entry, physical id, blob) and a
// 128-row tile.
struct TcTask {
    const uint8_t* blob;
    int e, rb, cnt, off, phys;
    bool valid;
};

struct alignas(16) TcHead {
    uint64_t raw_full[kRawStages];
    uint64_t raw_empty[kRawStages];
    // weight stage g of the CTA's stream lives in tensor-memory slot g % kAStages:
    // a_full when the converters have written it, a_empty when its MMAs are done
    uint64_t a_full[kAStages];
    uint64_t a_empty[kAStages];
    // activation chunk c of the stream in slot c % kBStages: b_full when it has
    // landed, b_empty when every issuer's MMAs on it are done
    uint64_t b_full[kBStages];
    uint64_t b_empty[kBStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    // tasks are taken from a global counter by the raw weight producer, which
    // publishes task k in slot k % kTaskQ for the other roles (-1: no more) with
    // its expert's routing values
    uint64_t tq_full[kTaskQ];
    uint64_t tq_empty[kTaskQ];
    int tq[kTaskQ];
    TcTask tqt[kTaskQ];
    uint32_t tmem_base;
    int abort;
    int D;
    alignas(16) int key[kMaxE];  // tokens of each active expert, -1 when inactive
    int list[kMaxE];             // active experts, most tokens first
    alignas(16) int col_pick[4][kNMax];     // per epilogue warp: output row of each column of the pass
    alignas(16) float col_scale[4][kNMax];  // and its activation prescale 2^p
};

constexpr int kEpiChunk = 16;  // token columns per epilogue chunk
constexpr size_t kEpiBufBytes = (size_t)kEpiChunk * 32 * sizeof(float);  // one warp's [16 tokens][32 rows] of h

constexpr size_t kRawOff = 0;
constexpr size_t kBOff = kRawOff + (size_t)kRawStages * kRawBytes;
constexpr size_t kEpiOff = kBOff + (size_t)kBStages * kBStageBytes;  // 2 staging buffers per epilogue warp
constexpr size_t kHeadOff = kEpiOff + 4 * 2 * kEpiBufBytes;
constexpr size_t kTcSmem = 1024 + kHeadOff + sizeof(TcHead);
static_assert(kTcSmem <= 232448, "shared memory budget of one CTA");

// D[tmem] (+)= A[tmem] * B[smem]: A is 128 lanes x 16 f16 (8 columns) at a_tmem.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// This thread's lane of tensor memory, 16 or 32 consecutive columns from taddr.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Bulk tensor store of a [box rows][box inner] tile from shared memory, and the
// bulk async-group bookkeeping of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk stores of all but the newest group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every bulk store of this thread is complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// SiLU(x) = x * sigmoid(x) with sigmoid(x) = (1 + tanh(x / 2)) / 2: one
// special-function operation per element (hardware tanh, relative error about
// 2^-11, absolute error of sigmoid about 2^-12).
__device__ __forceinline__ float silu_tanh(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return x * fmaf(0.5f, t, 0.5f);
}
// Largest E8M0 exponent of a scale row (n bytes, n a multiple of 4). A 16-byte
// aligned row is read eight 16-byte words at a time, all in flight together.
__device__ __forceinline__ int row_max_exp(const uint8_t* srow, int n) {
    uint32_t m = 0;
    if (((n | (int)reinterpret_cast<uintptr_t>(srow)) & 15) == 0) {
        for (int i = 0; i < n; i += 128) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int o = min(i + 16 * j, n - 16);  // past the row: reread its last word
                v[j] = __ldg(reinterpret_cast<const uint4*>(srow + o));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) m = __vmaxu4(m, __vmaxu4(__vmaxu4(v[j].x, v[j].y), __vmaxu4(v[j].z, v[j].w)));
        }
    } else {
        for (int i = 0; i < n; i += 4) m = __vmaxu4(m, ld_u32(srow + i));
    }
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

// 8 E2M1 values (one 32-bit word) times the f16x2 multiplier mm -> one 16-byte chunk.
__device__ __forceinline__ uint4 convert_chunk(uint32_t word, uint32_t mm) {
    uint32_t h4[4];
    e2m1x8_to_f16x2(word, h4);
    uint4 o;
    o.x = hmul2(h4[0], mm);
    o.y = hmul2(h4[1], mm);
    o.z = hmul2(h4[2], mm);
    o.w = hmul2(h4[3], mm);
    return o;
}

__device__ __forceinline__ TcTask tc_task(const FfnArgs& a, const TcHead& hd, int task, int tiles) {
    TcTask t;
    t.e = hd.list[task / tiles];
    t.rb = task % tiles;
    t.cnt = __ldg(a.counts + t.e);
    t.off = __ldg(a.offsets + t.e);
    t.phys = __ldg(a.phys_ids + __ldg(a.entries + t.off));
    t.valid = t.phys >= 0 && t.phys < a.n_phys;
    t.blob = t.valid ? a.ptr[t.phys] : nullptr;
    return t;
}

// MMA width of a pass over nb tokens: a multiple of 16 (the M = 128 shape's step).
__device__ __forceinline__ int ncols16(int nb) { return (nb + 15) & ~15; }

// Task k of this CTA from the queue (-1: no more tasks, or a wait ran out), taken
// by one thread.
__device__ __forceinline__ int take_task(TcHead& hd, int k, const FfnArgs& a, volatile int* abort, int who,
                                         TcTask& t) {
    const int j = k % kTaskQ;
    if (!mbar_wait_fast(&hd.tq_full[j], (unsigned)(k / kTaskQ) & 1u, abort, a.status, a.diag, 20, j, k, who))
        return -1;
    const int task = *reinterpret_cast<volatile int*>(&hd.tq[j]);
    t = hd.tqt[j];
    mbar_arrive(&hd.tq_empty[j]);
    return task;
}

// The same, taken by a whole warp (every lane returns the same task).
__device__ __forceinline__ int warp_take_task(TcHead& hd, int k, const FfnArgs& a, volatile int* abort, int who,
                                              TcTask& t) {
    const int j = k % kTaskQ;
    if (!warp_wait(&hd.tq_full[j], (unsigned)(k / kTaskQ) & 1u, a, abort, 20, j, k, who)) return -1;
    const int task = *reinterpret_cast<volatile int*>(&hd.tq[j]);
    t = hd.tqt[j];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&hd.tq_empty[j]);
    return task;
}

template <int P>
__global__ void __launch_bounds__(kThreadsTC, 1) ffn_tc_kernel(FfnArgs a, const __grid_constant__ CUtensorMap act_map,
                                                               const __grid_constant__ CUtensorMap h_map, int lo,
                                                               int sel, int ctr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw = base + kRawOff;
    uint8_t* sb = base + kBOff;
    TcHead& hd = *reinterpret_cast<TcHead*>(base + kHeadOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I;
    const int K = P == 0 ? H : I;
    const int nks = K / kBK;  // K is a multiple of 128
    const int tiles = (P == 0 ? I : H) / kBM;
    volatile int* abort = &hd.abort;

    // active experts (more than lo tokens, in the selected placement class), listed
    // with the most tokens first (ties by id) so that the largest tasks start first
    // and the CTAs' last tasks are short: every thread keys some experts (one round
    // of independent loads), then ranks its experts against all keys
    for (int e = threadIdx.x; e < a.E; e += kThreadsTC) {
        const int c = __ldg(a.counts + e);
        bool act = c > lo;
        if (act && sel != 0) {
            const bool hot = __ldg(a.loc + e) < a.n_hot;
            act = (sel == 1) ? hot : !hot;
        }
        hd.key[e] = act ? c : -1;
    }
    for (int e = a.E + threadIdx.x; e < ((a.E + 3) & ~3); e += kThreadsTC) hd.key[e] = -1;  // pad to 4
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += kThreadsTC) {
        const int ke = hd.key[e];
        if (ke < 0) continue;
        int r = 0;
        for (int f = 0; f < a.E; f += 4) {
            const int4 k4 = *reinterpret_cast<const int4*>(&hd.key[f]);
            r += (k4.x > ke || (k4.x == ke && f < e)) + (k4.y > ke || (k4.y == ke && f + 1 < e)) +
                 (k4.z > ke || (k4.z == ke && f + 2 < e)) + (k4.w > ke || (k4.w == ke && f + 3 < e));
        }
        hd.list[r] = e;
    }
    if (warp == 0) {
        int cnt = 0;
        for (int base_e = 0; base_e < a.E; base_e += 32) {
            const int e = base_e + lane;
            cnt += __popc(__ballot_sync(0xffffffffu, e < a.E && hd.key[e] >= 0));
        }
        if (lane == 0) {
            hd.D = cnt;
            hd.abort = 0;
            for (int s = 0; s < kRawStages; ++s) {
                mbar_init(&hd.raw_full[s], 1);
                mbar_init(&hd.raw_empty[s], kConvWarps);
            }
            for (int s = 0; s < kAStages; ++s) {
                mbar_init(&hd.a_full[s], kConvWarps);
                mbar_init(&hd.a_empty[s], 1);
            }
            for (int s = 0; s < kBStages; ++s) {
                mbar_init(&hd.b_full[s], 1);
                mbar_init(&hd.b_empty[s], issuers<P>());
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(&hd.acc_full[s], issuers<P>());
                mbar_init(&hd.acc_empty[s], 4);
            }
            for (int j = 0; j < kTaskQ; ++j) {
                mbar_init(&hd.tq_full[j], 1);
                mbar_init(&hd.tq_empty[j], task_takers<P>());
            }
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
    // activations, prescales and outputs belong to the previous kernel until it completes
    grid_dep_wait();
    const uint32_t tmem = hd.tmem_base;
    const int ntask = hd.D * tiles;

    // stages per column pass: the K chunks, times the matrices of each chunk
    const int nst = nks * mats<P>();
    if (warp == 0) {
        // ---------------- raw weight producer, task fetcher (lane 0) ----------------
        if (lane == 0) {
            int rs = 0;
            unsigned rph = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int j = k % kTaskQ;
                if (!mbar_wait_fast(&hd.tq_empty[j], ((unsigned)(k / kTaskQ) & 1u) ^ 1u, abort, a.status, a.diag, 21,
                                    j, k, 0))
                    break;
                int task = atomicAdd(a.task_ctr + ctr, 1);
                if (task >= ntask) task = -1;
                TcTask t{};
                if (task >= 0) t = tc_task(a, hd, task, tiles);
                *reinterpret_cast<volatile int*>(&hd.tq[j]) = task;
                hd.tqt[j] = t;
                mbar_arrive(&hd.tq_full[j]);
                if (task < 0) break;
                if (!t.valid) continue;
                const CUtensorMap* map = P == 0 ? &a.tmaps[t.phys].w13r : &a.tmaps[t.phys].w2r;
                asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
                const int r0 = t.rb * kBM;
                for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                    for (int st = 0; st < nst; ++st) {
                        if (!mbar_wait_fast(&hd.raw_empty[rs], rph ^ 1u, abort, a.status, a.diag, 12, rs, st, task)) {
                            ok = false;
                            break;
                        }
                        // stage st: chunk st / mats, matrix st % mats (gate/up phase: rows
                        // r0.. of the gate half, then of the up half)
                        const int c = st / mats<P>(), m = st % mats<P>();
                        mbar_arrive_expect_tx(&hd.raw_full[rs], kRawBytes);
                        tma_load_2d(raw + (size_t)rs * kRawBytes, map, c * kRawRow, m * I + r0, &hd.raw_full[rs]);
                        advance(rs, rph, kRawStages);
                    }
                }
            }
            for (int s = 0; s < kRawStages; ++s) mbar_drain(&hd.raw_full[s], (s < rs) ? rph : (rph ^ 1u));
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------- activation producer (lane 0) ----------------
        if (lane == 0) {
            int bs = 0;
            unsigned bph = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                TcTask t;
                const int task = take_task(hd, k, a, abort, 1, t);
                if (task < 0) break;
                if (!t.valid) continue;
                for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                    const int boxes = (ncols16(min(kNMax, t.cnt - tb)) + kActBoxRows - 1) / kActBoxRows;
                    for (int c = 0; c < nks; ++c) {
                        if (!mbar_wait_fast(&hd.b_empty[bs], bph ^ 1u, abort, a.status, a.diag, 13, bs, c, task)) {
                            ok = false;
                            break;
                        }
                        uint8_t* dst = sb + (size_t)bs * kBStageBytes;
                        mbar_arrive_expect_tx(&hd.b_full[bs], (unsigned)(boxes * 2 * kActBoxRows * 128));
                        for (int at = 0; at < 2; ++at)  // the chunk's two 64-element atoms of K
                            for (int bx = 0; bx < boxes; ++bx)
                                tma_load_2d(dst + at * kBAtom + bx * kActBoxRows * 128, &act_map, c * kBK + 64 * at,
                                            t.off + tb + kActBoxRows * bx, &hd.b_full[bs]);
                        advance(bs, bph, kBStages);
                    }
                }
            }
            for (int s = 0; s < kBStages; ++s) mbar_drain(&hd.b_full[s], (s < bs) ? bph : (bph ^ 1u));
        }
        __syncwarp();
    } else if (warp == 1 || (P == 0 && warp == 3)) {
        // ---------------- MMA issuers (lane 0 alone) ----------------
        // one thread per issuer runs this loop and takes no warp-wide votes; in the
        // gate/up phase warp 1 issues the gate stages into the gate accumulator and
        // warp 3 the up stages into the up accumulator
        const int mi = warp == 1 ? 0 : 1;
        if (lane == 0) {
            int bs = 0, buf = 0;
            unsigned bph = 0, accph = 0;  // accph: bit b = phase of accumulator buffer b
            int g0 = 0;                   // stream number of the pass's first stage
            bool ok = true;
            for (int k = 0; ok; ++k) {
                TcTask t;
                const int task = take_task(hd, k, a, abort, 2 + mi, t);
                if (task < 0) break;
                if (!t.valid) continue;
                for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                    const int N = ncols16(min(kNMax, t.cnt - tb));
                    const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
                    if (!mbar_wait_fast(&hd.acc_empty[buf], ((accph >> buf) & 1u) ^ 1u, abort, a.status, a.diag, 14,
                                        buf, 0, task)) {
                        ok = false;
                        break;
                    }
                    accph ^= 1u << buf;
                    tc_fence_after();
                    // gate/up phase: this issuer's matrix's accumulator; down phase: buffer buf
                    const uint32_t d = tmem + (uint32_t)(P == 0 ? mi : buf) * kAccCols;
                    for (int c = 0; c < nks; ++c) {
                        const int g = g0 + c * mats<P>() + (P == 0 ? mi : 0);  // this issuer's stage
                        const int as = g % kAStages;
                        if (!mbar_wait_fast(&hd.a_full[as], (unsigned)(g / kAStages) & 1u, abort, a.status, a.diag, 15,
                                            as, c, task) ||
                            !mbar_wait_fast(&hd.b_full[bs], bph, abort, a.status, a.diag, 16, bs, c, task)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // A: the stage's f16 weights in tensor memory (8 columns per 16-element
                        // k-step); B: descriptor of k-step 0, a 16-element step advances its
                        // start address by 32 bytes
                        const uint32_t at = tmem + kACol0 + (uint32_t)as * kAStageCols;
                        const uint64_t bd = sw128_desc(smem_u32(sb + (size_t)bs * kBStageBytes));
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                            // k-steps 0-3 in the first activation atom, 4-7 in the second
                            const uint64_t b = bd + (uint64_t)((kk >> 2) * (kBAtom >> 4) + 2 * (kk & 3));
                            tc_mma_f16_ta(d, at + 8 * kk, b, idesc, acc);
                        }
                        tc_commit(&hd.a_empty[as]);
                        tc_commit(&hd.b_empty[bs]);
                        advance(bs, bph, kBStages);
                    }
                    if (!ok) break;
                    tc_commit(&hd.acc_full[buf]);
                    g0 += nst;
                    if (P == 1) buf ^= 1;  // the gate/up phase's two accumulators fill [0, 320)
                }
            }
            // no MMA may be in flight when tensor memory is freed: wait (bounded) for the
            // last commit of every weight and activation slot
            for (int s = 0; s < kAStages && s < g0; ++s) {
                const int gl = s + kAStages * ((g0 - 1 - s) / kAStages);  // last stage in slot s
                mbar_drain(&hd.a_empty[s], (unsigned)(gl / kAStages) & 1u);
            }
            for (int s = 0; s < kBStages; ++s) mbar_drain(&hd.b_empty[s], (s < bs) ? bph : (bph ^ 1u));
        }
        __syncwarp();
    } else if (warp >= kFirstConv && warp < kFirstConv + kConvWarps) {
        // ---------------- converters ----------------
        // every stage is one matrix's 128 rows x 128 elements: thread = (half hi of the
        // stage's elements, row); the gate/up phase alternates gate and up stages
        const int cidx = threadIdx.x - kFirstConv * 32;
        const int row = cidx & (kBM - 1);  // = (warp % 4) * 32 + lane: this thread's tensor-memory lane
        const int hi = cidx >> 7;
        const uint32_t lane_base = tmem + ((uint32_t)(warp & 3) * 32u << 16);
        int rs = 0;
        unsigned rph = 0;
        int gs = 0;  // stage number in the CTA's stream
        bool ok = true;
        for (int k = 0; ok; ++k) {
            TcTask t;
            const int task = warp_take_task(hd, k, a, abort, 3, t);
            if (task < 0) break;
            if (!t.valid) continue;
            const uint8_t* blob = t.blob;
            const int r0 = t.rb * kBM;
            const int srl = K / 32;  // scale bytes per row
            // this thread's row of each matrix (gate/up phase: gate, up): its scale row
            // and the exponent its block scales are rebased to
            const uint8_t* sc0 = P == 0 ? blob + a.w13s + (size_t)(r0 + row) * srl : blob + a.w2s + (size_t)(r0 + row) * srl;
            const uint8_t* sc1 = P == 0 ? blob + a.w13s + (size_t)(I + r0 + row) * srl : sc0;
            const int cb0 = row_max_exp(sc0, srl) - 12;
            const int cb1 = P == 0 ? row_max_exp(sc1, srl) - 12 : cb0;
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                // scale word of each stage (the 4 blocks of its chunk), fetched a stage ahead
                uint32_t wcur = ld_u32(sc0);
                for (int st = 0; st < nst && ok; ++st) {
                    const int m = st % mats<P>();  // matrix of this stage (chunk st / mats)
                    const int sn = st + 1, cn = sn / mats<P>(), mn = sn % mats<P>();
                    // unconditional (the last stage rereads its own word): the value is
                    // not needed before the next stage
                    const uint32_t wnext = ld_u32((mn ? sc1 : sc0) + 4 * min(cn, nks - 1));
                    // the weight slot of stage gs was last read by the MMAs of stage gs - kAStages
                    const int as = gs % kAStages;
                    if (!warp_wait(&hd.raw_full[rs], rph, a, abort, 17, rs, st, task) ||
                        !warp_wait(&hd.a_empty[as], ((unsigned)(gs / kAStages) & 1u) ^ 1u, a, abort, 18, as, st,
                                   task)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // this thread's half of the row (64 elements, 8 words of 8) into 32 columns;
                    // the raw stage holds 64-byte rows with the 64-byte swizzle: 16-byte
                    // chunk q of row r sits at chunk q ^ ((r >> 1) & 3), so the 8 rows a
                    // quarter-warp reads fall in distinct banks
                    const uint8_t* rrow = raw + (size_t)rs * kRawBytes + row * kRawRow;
                    const int sw = (row >> 1) & 3;
                    const uint32_t col0 = lane_base + kACol0 + (uint32_t)as * kAStageCols + 32u * (uint32_t)hi;
                    const int cbm = m == 0 ? cb0 : cb1;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {  // 4 words = 32 elements = one scale block
                        const uint4 w = *reinterpret_cast<const uint4*>(rrow + (((2 * hi + g) ^ sw) << 4));
                        const int blk = 2 * hi + g;
                        const uint32_t mf = f16_pow2((int)((wcur >> (8 * blk)) & 0xffu) - cbm);
                        const uint32_t mm = mf | (mf << 16);
                        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                        uint32_t v[16];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 o = convert_chunk(words[q], mm);
                            v[4 * q + 0] = o.x;
                            v[4 * q + 1] = o.y;
                            v[4 * q + 2] = o.z;
                            v[4 * q + 3] = o.w;
                        }
                        tc_st16(col0 + 16u * g, v);
                    }
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&hd.a_full[as]);
                        mbar_arrive(&hd.raw_empty[rs]);
                    }
                    advance(rs, rph, kRawStages);
                    ++gs;
                    wcur = wnext;
                }
            }
        }
    } else if (warp >= kFirstEpi) {
        // ---------------- epilogue ----------------
        const int q4 = warp - kFirstEpi;  // tensor-memory lane quarter (= warp % 4)
        const int t_row = q4 * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        int* cpick = hd.col_pick[q4];
        float* cscale = hd.col_scale[q4];
        // gate/up phase: full 16-token chunks of h leave through two staging buffers
        // of this warp and a bulk tensor store each (lane 0 issues and tracks them)
        float* stage_buf = reinterpret_cast<float*>(base + kEpiOff + (size_t)q4 * 2 * kEpiBufBytes);
        int sbuf = 0;
        int buf = 0;
        unsigned accph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            TcTask t;
            const int task = warp_take_task(hd, k, a, abort, 4, t);
            if (task < 0) break;
            const int r0 = t.rb * kBM;
            if (!t.valid) {
                // zero outputs for an expert whose physical id is out of range
                if (t.rb == 0 && threadIdx.x == kFirstEpi * 32) set_status(a.status, MOE_ERR_BAD_EXPERT);
                for (int c = 0; c < t.cnt; ++c) {
                    if (P == 0) a.h[(size_t)(t.off + c) * I + r0 + t_row] = 0.f;
                    else a.y[(size_t)__ldg(a.entries + t.off + c) * H + r0 + t_row] = 0.f;
                }
                continue;
            }
            const uint8_t* blob = t.blob;
            const int srl = K / 32;
            const int c0 = row_max_exp(blob + (P == 0 ? a.w13s : a.w2s) + (size_t)(r0 + t_row) * srl, srl) - 12;
            const int c1 = P == 0 ? row_max_exp(blob + a.w13s + (size_t)(I + r0 + t_row) * srl, srl) - 12 : c0;
            const float s0 = pow2i(max(-126, min(127, c0 - 127)));
            const float s1 = pow2i(max(-126, min(127, c1 - 127)));
            for (int tb = 0; tb < t.cnt && ok; tb += kNMax) {
                const int nb = min(kNMax, t.cnt - tb);
                // the pass's columns: activation prescale (and for the down phase the
                // pick), fetched before the wait
                for (int n = lane; n < nb; n += 32) {
                    const int pos = t.off + tb + n;
                    cpick[n] = P == 0 ? pos : __ldg(a.entries + pos);
                    cscale[n] = pow2i(__ldg(a.gexp + pos));
                }
                __syncwarp();
                if (!warp_wait(&hd.acc_full[buf], (accph >> buf) & 1u, a, abort, 19, buf, tb, task)) {
                    ok = false;
                    break;
                }
                accph ^= 1u << buf;
                tc_fence_after();
                const uint32_t d = lane_addr + (uint32_t)buf * kAccCols;
                for (int cb = 0; cb < nb; cb += 16) {
                    float v0[16], v1[16];
                    if constexpr (P == 0) tc_ld16x2(d + cb, d + kAccCols + cb, v0, v1);
                    else tc_ld16(d + cb, v0);
                    // the chunk's picks and prescales are read from shared memory before
                    // any store (a store through a generic pointer could alias them and
                    // would order every later read behind it); all 16 columns are
                    // computed (columns past nb hold padding and are not stored)
                    int pk[16];
                    float sxv[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const int4 p4 = *reinterpret_cast<const int4*>(cpick + cb + i);
                        const float4 s4 = *reinterpret_cast<const float4*>(cscale + cb + i);
                        pk[i] = p4.x, pk[i + 1] = p4.y, pk[i + 2] = p4.z, pk[i + 3] = p4.w;
                        sxv[i] = s4.x, sxv[i + 1] = s4.y, sxv[i + 2] = s4.z, sxv[i + 3] = s4.w;
                    }
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float sx = sxv[i];
                        if constexpr (P == 0) {
                            const float gv = v0[i] * s0 * sx;
                            const float uv = v1[i] * s1 * sx;
                            o[i] = silu_tanh(gv) * uv;
                        } else {
                            o[i] = v0[i] * s0 * sx;
                        }
                    }
                    if (P == 0 && cb + kEpiChunk <= nb) {
                        // h rows t.off + tb + cb .. +15 (bucket order), this warp's 32
                        // columns r0 + 32 q4 ..: stage [token][row] and store as one box
                        float* stg = stage_buf + (size_t)sbuf * (kEpiChunk * 32);
                        if (lane == 0) bulk_wait_read_1();  // this buffer's previous store has read it
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 16; ++i) stg[i * 32 + lane] = o[i];
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&h_map, r0 + q4 * 32, t.off + tb + cb, stg);
                            bulk_commit();
                        }
                        sbuf ^= 1;
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (cb + i < nb) {
                                if constexpr (P == 0) a.h[(size_t)pk[i] * I + r0 + t_row] = o[i];  // bucket row
                                else a.y[(size_t)pk[i] * H + r0 + t_row] = o[i];
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hd.acc_empty[buf]);
                if (P == 1) buf ^= 1;
            }
        }
        // the stores must be complete (and done reading shared memory) before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

size_t ffn_tc_smem_bytes() { return kTcSmem; }

cudaError_t launch_ffn_tc(const FfnArgs& a, int phase, int sel, int lo, int sm_count, cudaStream_t st) {
    const int n = a.T * a.k;
    cudaError_t err = cudaSuccess;
    // activation tiles: 64 elements (128 bytes) x 32 bucket rows per box, 128-byte swizzle
    CUtensorMap map, hmap;
    if (!encode_act_map(&map, a, phase, 64, kActBoxRows, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    // h [T·k][I] fp32 in bucket order, boxes of 32 columns x 16 rows (gate/up phase output)
    if (!encode_tmap_2d(&hmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.h, (uint64_t)a.I, (uint64_t)n,
                        (uint64_t)a.I * sizeof(float), 32, kEpiChunk, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const long dmax = (long)(a.E < n / (lo + 1) + 1 ? a.E : n / (lo + 1) + 1);
    const long tasks = dmax * ((phase == 0 ? a.I : a.H) / kBM);
    const int grid = (int)(tasks < sm_count ? tasks : sm_count);
    if (grid <= 0) return cudaSuccess;
    static std::atomic<uint64_t> configured[2];
    err = ensure_smem_limit(phase == 0 ? (const void*)ffn_tc_kernel<0> : (const void*)ffn_tc_kernel<1>, (int)kTcSmem,
                            configured[phase]);
    if (err != cudaSuccess) return err;
    // task counters 12-15 of the call's workspace (zeroed by the gate/up prescale
    // kernel): one per phase and placement class
    const int ctr = 12 + (sel == 2 ? 2 : 0) + phase;
    if (phase == 0)
        return launch_pdl(ffn_tc_kernel<0>, dim3(grid), dim3(kThreadsTC), kTcSmem, st, a, map, hmap, lo, sel, ctr);
    return launch_pdl(ffn_tc_kernel<1>, dim3(grid), dim3(kThreadsTC), kTcSmem, st, a, map, hmap, lo, sel, ctr);
}

}  // namespace moe
