// Grouped SwiGLU expert FFN on block-scaled FP4 tensor cores (the all-FP4 prefill
// mode): tcgen05.mma kind::mxf4 with both operands in MXFP4.
//
// "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1: the layer
// runs all experts in one call; "A 475 GB Model Across Two Workstations, With the
// Table on Disk", Abstract: the routed experts ship in MXFP4 (E2M1 elements, one
// E8M0 scale per 32 elements along the reduction dimension).  The weights feed the
// tensor cores as they are stored; the activations are converted to the same
// format: x once per call (mx_xprep_kernel, bucket order), h by the gate/up
// kernel's epilogue, which owns whole 32-element blocks of h (one 32-row slice of
// the I dimension per warp and token).  The scale factors reach tensor memory
// through tcgen05.st, so the MMA applies them per 32-element block:
//   D[128 weight rows x N tokens] (+)= sum over blocks of (A_blk * 2^sa) (B_blk * 2^sb)^T
// with fp32 accumulation in tensor memory.
//
// Tensor-memory layout of the scale factors (kind::mxf4, M = 128, scale_vec::2X;
// established with in-bounds checks on this GPU against a CPU product): the MMA
// reads the two block scales of weight row m from lane m at column sfa + m / 32,
// bytes sf_id and sf_id + 1; for token column n, a row of D in lane quarter q
// reads them from quarter q, lane n % 32, column sfb + n / 32, so the token scales
// are written to all four quarters.  One 32-bit word holds four blocks (the K
// range of two MMAs, sf_id 0 and 2).
//
// Warp roles of one persistent CTA per SM (25 warps), each task an expert and a
// 128-row tile:
//   warp 0       loads the tile's E2M1 rows by TMA, 256 elements of K per stage
//                (128-byte swizzle; gate and up rows in the gate/up phase, w2 rows
//                in the down phase), with the rows' scale bytes of the stage, into
//                the weight ring;
//   warp 1       loads the tokens' E2M1 activation rows of each stage by TMA (up to
//                192 bucket rows with one term per token, 128 with four; 32 per
//                box), with their scale words, into the shallower activation ring;
//   warp 2       owns tensor memory; one thread issues the MMAs (four of K = 64 per
//                matrix and stage); in the gate/up phase it issues the gate matrix's
//                and a thread of warp 24 the up matrix's, each into its accumulator;
//   warp 3       takes tasks from a launch-wide counter, experts with the most
//                tokens first, and publishes them with their routing values in a
//                shared-memory queue, up to the queue's depth ahead;
//   warps 4-7    scale writers: each thread takes its weight row's scale words and
//                the tokens' activation scale words of a stage from shared memory
//                (loaded by TMA with the stage's operands) and stores them into a
//                ring of scale slots in tensor memory;
//   warps 8-23   epilogue, four warps per lane quarter taking every fourth 16-token
//                chunk: tensor memory -> registers; gate/up phase: h = SiLU(g) u
//                (relative error about 1e-6, so the quantisation of h takes the
//                decisions of an exact evaluation except within that distance of a
//                decision point), converted to MXFP4 across the warp's 32 rows and
//                stored in bucket order; down phase: y rows.
// Every wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT, and the CTA
// drains its copies and MMAs before it frees tensor memory and returns.
#include <cuda.h>

#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kMxBM = 128;                     // weight rows per tile = tensor-memory lanes
constexpr int kMxBK = 256;                     // K elements per stage
constexpr int kMxRowB = kMxBK / 2;             // bytes of a row per stage
constexpr int kMxTile = kMxBM * kMxRowB;       // 16 KB: one matrix's rows of a stage
constexpr int kMxBox = 32;                     // activation rows per TMA box
// activation scale words of a stage, loaded by TMA from a 4-aligned bucket row (the
// box's start must be a whole 16 bytes): 2 rows (the stage's two words) x 200
constexpr int kMxSfbBox = 200;
constexpr int kMxWsc = kMxBM * 16;             // a matrix's scale box: 128 rows x 16 bytes
constexpr int kMxASlot = kMxTile + kMxWsc;     // per matrix: E2M1 rows, then their scales
constexpr int kMxThreads = 800;
constexpr int kMxUpIssuer = 24;  // gate/up phase: the warp that issues the up matrix's MMAs
constexpr int kMxFirstSf = 4;
constexpr int kMxFirstEpi = 8;
constexpr int kMxEpiWarps = 16;  // four per lane quarter, taking every fourth 16-token chunk
constexpr int kMxMaxE = 1024;
constexpr int kMxTaskQ = 4;
constexpr uint32_t kMxTmemCols = 512;
// epilogue staging per warp in the gate/up phase: with four terms, 16 activation rows
// x 16 bytes of h codes; with one term, an 8-column slice of h transposed (32 rows x
// 8 columns of fp32, rows padded to 33 words so that both the row-wise writes and the
// column-wise reads are free of bank conflicts)
template <int P, int TERMS>
__host__ __device__ constexpr int mx_epi_stage() { return P == 1 ? 0 : (TERMS == 1 ? 8 * 33 * 4 : 16 * 16); }

template <int P>
__host__ __device__ constexpr int mx_mats() { return P == 0 ? 2 : 1; }  // weight matrices per stage
// MMA issuing threads: the gate/up phase issues each matrix from its own thread
// (issuing one block-scaled MMA takes a thread about 100 cycles whatever N is).
template <int P, int TERMS>
__host__ __device__ constexpr int mx_issuers() { return P == 0 ? 2 : 1; }
// roles that take each task from the queue: producers, issuers, scale writers, epilogue
template <int P, int TERMS>
__host__ __device__ constexpr int mx_takers() { return 2 + mx_issuers<P, TERMS>() + 4 + kMxEpiWarps; }
// Activation rows (token columns of the MMA) per pass: 192 with one term per token;
// 128 (32 tokens) with four, which leaves shared memory to a deeper weight ring
// (decode-sized calls read far more weight bytes than activation bytes).
template <int TERMS>
__host__ __device__ constexpr int mx_nmax() { return TERMS == 1 ? 192 : 128; }
template <int TERMS>
__host__ __device__ constexpr int mx_bstage() { return mx_nmax<TERMS>() * kMxRowB + 2048; }  // rows, then scale words
// Two rings of stage slots, each the K range of one stage: weight slots (a matrix's
// E2M1 rows and their scale bytes per matrix) and activation slots (rows and scale
// words, with a scale slot in tensor memory); the MMA issuers release both.  The
// weight ring is the deeper: its bytes come from DRAM, the activations mostly from L2.
template <int P, int TERMS>
__host__ __device__ constexpr int mx_astages() { return TERMS == 1 ? (P == 0 ? 3 : 4) : (P == 0 ? 4 : 8); }
template <int P, int TERMS>
__host__ __device__ constexpr int mx_bstages() { return TERMS == 1 ? (P == 0 ? 3 : 4) : 3; }
constexpr int kMxMaxStages = 8;
// Tensor memory: accumulators (gate and up in the gate/up phase, two buffers in the
// down phase) in [0, 2 nmax), then the scale slots.
template <int TERMS>
__host__ __device__ constexpr uint32_t mx_acc_cols() { return (uint32_t)mx_nmax<TERMS>(); }
template <int TERMS>
__host__ __device__ constexpr uint32_t mx_sf0() { return 2u * mx_acc_cols<TERMS>(); }
// scale slot: weight words (8 columns per matrix: two words x four quarter columns),
// then token words (16 columns: word j of the stage at 8j + token group)
template <int P>
__host__ __device__ constexpr uint32_t mx_sfb_col() { return P == 0 ? 16u : 8u; }
template <int P>
__host__ __device__ constexpr uint32_t mx_sf_cols() { return mx_sfb_col<P>() + 16u; }
template <int P, int TERMS>
__host__ __device__ constexpr bool mx_budget_ok() {
    return mx_sf0<TERMS>() + mx_bstages<P, TERMS>() * mx_sf_cols<P>() <= kMxTmemCols &&
           mx_astages<P, TERMS>() <= kMxMaxStages && mx_bstages<P, TERMS>() <= kMxMaxStages &&
           mx_nmax<TERMS>() + 8 <= kMxSfbBox;
}
static_assert(mx_budget_ok<0, 1>() && mx_budget_ok<1, 1>() && mx_budget_ok<0, 4>() && mx_budget_ok<1, 4>(),
              "tensor memory and ring budget");

struct MxTask {
    const uint8_t* blob;
    int e, rb, cnt, off, phys;
    bool valid;
};

struct alignas(16) MxHead {
    uint64_t a_full[kMxMaxStages], a_empty[kMxMaxStages];  // weight ring
    uint64_t b_full[kMxMaxStages], b_empty[kMxMaxStages];  // activation ring (and scale slots)
    uint64_t sf_full[kMxMaxStages];  // scale slot written; empties: one commit per issuer
    uint64_t acc_full[2], acc_empty[2];
    uint64_t tq_full[kMxTaskQ], tq_empty[kMxTaskQ];
    int tq[kMxTaskQ];
    MxTask tqt[kMxTaskQ];
    uint32_t tmem_base;
    int abort;
    int D;
    int list[kMxMaxE];  // active experts, most tokens first
};

template <int P, int TERMS>
struct MxSmem {
    static constexpr size_t kB = (size_t)mx_astages<P, TERMS>() * mx_mats<P>() * kMxASlot;  // after the weight ring
    static constexpr size_t kStg = kB + (size_t)mx_bstages<P, TERMS>() * mx_bstage<TERMS>();
    static constexpr size_t kHead = kStg + (size_t)kMxEpiWarps * mx_epi_stage<P, TERMS>();
    static constexpr size_t kTotal = 1024 + kHead + sizeof(MxHead);
};
static_assert(MxSmem<0, 1>::kTotal <= 232448 && MxSmem<1, 1>::kTotal <= 232448 && MxSmem<0, 4>::kTotal <= 232448 &&
                  MxSmem<1, 4>::kTotal <= 232448,
              "shared memory budget of one CTA");

// kind::mxf4 instruction descriptor: A and B E2M1 (format 1), both K-major, UE8M0
// scales, M = 128, N tokens, scale-factor byte selector sf for both operands.
__device__ __forceinline__ uint32_t mx_idesc(int N, uint32_t sf) {
    return (sf << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kMxBM >> 4) << 24) | (sf << 29);
}

// One block-scaled MMA, issued by one elected lane of a converged warp.  Issued this
// way, from straight-line code, a thread issues one every ~40 cycles and the
// commits cost nothing; a lone lane in a loop with run-time bounds took ~165 cycles
// per MMA (measured on this GPU).
__device__ __forceinline__ void mx_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// The MMAs of one matrix for one stage: NKK steps of K = 64 (4 for a full stage of
// 256, 2 for a tail of 128).  A step of 64 elements advances both start addresses
// by 32 bytes; its two blocks are bytes 2 (kk % 2) .. +1 of the stage's word kk / 2.
template <int NKK>
__device__ __forceinline__ void mx_stage_mmas(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id0, uint32_t id2,
                                              uint32_t sfa, uint32_t sfb, bool first) {
#pragma unroll
    for (int kk = 0; kk < NKK; ++kk)
        mx_mma(d, ad + 2 * kk, bd + 2 * kk, (kk & 1) ? id2 : id0, sfa + 4u * (uint32_t)(kk >> 1),
               sfb + 8u * (uint32_t)(kk >> 1), (first && kk == 0) ? 0u : 1u);
}

__device__ __forceinline__ void mx_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void mx_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ MxTask mx_task(const FfnArgs& a, const MxHead& hd, int task, int tiles) {
    MxTask t;
    t.e = hd.list[task / tiles];
    t.rb = task % tiles;
    t.cnt = __ldg(a.counts + t.e);
    t.off = __ldg(a.offsets + t.e);
    t.phys = __ldg(a.phys_ids + __ldg(a.entries + t.off));
    t.valid = t.phys >= 0 && t.phys < a.n_phys;
    t.blob = t.valid ? a.ptr[t.phys] : nullptr;
    return t;
}

__device__ __forceinline__ int mx_warp_take(MxHead& hd, int k, const FfnArgs& a, volatile int* abort, int who,
                                            MxTask& t) {
    const int j = k % kMxTaskQ;
    if (!warp_wait(&hd.tq_full[j], (unsigned)(k / kMxTaskQ) & 1u, a, abort, 30, j, k, who)) return -1;
    const int task = *reinterpret_cast<volatile int*>(&hd.tq[j]);
    t = hd.tqt[j];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&hd.tq_empty[j]);
    return task;
}

// MMA width of a pass over nb tokens: a multiple of 16 (the M = 128 shape's step).
__device__ __forceinline__ int mx_ncols(int nb) { return (nb + 15) & ~15; }

// TERMS: activation rows per token.  1: x and h converted to MXFP4 by the OCP rule
// (the all-FP4 mode).  4: each activation written as a sum of four MXFP4 terms, the
// first the activation, each further one the residual of those before (exponent
// rule mx_term_exp, so nothing saturates and every residual is exact in fp32), so
// the products reproduce the unquantised layer to about 2e-4; the terms of a token
// are consecutive rows and consecutive accumulator columns, summed in the epilogue.
// The launch takes the experts with lo < tokens <= hi.
template <int P, int TERMS>
__global__ void __launch_bounds__(kMxThreads, 1) ffn_mx_kernel(FfnArgs a, const __grid_constant__ CUtensorMap act_map,
                                                               const __grid_constant__ CUtensorMap sfb_map, int sel,
                                                               int ctr, int lo, int hi) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = base;
    uint8_t* sB = base + MxSmem<P, TERMS>::kB;
    MxHead& hd = *reinterpret_cast<MxHead*>(base + MxSmem<P, TERMS>::kHead);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I;
    const int K = P == 0 ? H : I;
    const int nks = (K + kMxBK - 1) / kMxBK;  // stages per pass; the last may hold 128 elements
    const int tiles = (P == 0 ? I : H) / kMxBM;
    const int R = a.T * a.k * TERMS;  // activation rows: TERMS per bucket row
    const int Rs = (R + 3) & ~3;      // row stride of the activation scale words
    constexpr int TPP = mx_nmax<TERMS>() / TERMS;  // tokens per column pass
    constexpr uint32_t ACC = mx_acc_cols<TERMS>(), SF0 = mx_sf0<TERMS>();
    constexpr int BSTAGE = mx_bstage<TERMS>(), BTILE = mx_nmax<TERMS>() * kMxRowB;
    // the weight scales arrive by TMA with their stage where the plane's rows are whole
    // 16-byte units, else the scale writers read them from global memory
    const bool wsc_tma = mx_scale_maps(K);
    constexpr int NA = mx_astages<P, TERMS>(), NB = mx_bstages<P, TERMS>();
    constexpr int MATS = mx_mats<P>();
    constexpr int ISS = mx_issuers<P, TERMS>();
    volatile int* abort = &hd.abort;
    // tokens of each active expert (-1: inactive), in the weight ring until the
    // producers start
    int* key = reinterpret_cast<int*>(sA);

    // active experts (at least one token, in the selected placement class), most
    // tokens first (ties by id): every thread keys some experts, then ranks its own
    for (int e = threadIdx.x; e < a.E; e += kMxThreads) {
        const int c = __ldg(a.counts + e);
        bool act = c > lo && c <= hi;
        if (act && sel != 0) {
            const bool hot = __ldg(a.loc + e) < a.n_hot;
            act = (sel == 1) ? hot : !hot;
        }
        key[e] = act ? c : -1;
    }
    for (int e = a.E + threadIdx.x; e < ((a.E + 3) & ~3); e += kMxThreads) key[e] = -1;  // pad to 4
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += kMxThreads) {
        const int ke = key[e];
        if (ke < 0) continue;
        int r = 0;
        for (int f = 0; f < a.E; f += 4) {
            const int4 k4 = *reinterpret_cast<const int4*>(&key[f]);
            r += (k4.x > ke || (k4.x == ke && f < e)) + (k4.y > ke || (k4.y == ke && f + 1 < e)) +
                 (k4.z > ke || (k4.z == ke && f + 2 < e)) + (k4.w > ke || (k4.w == ke && f + 3 < e));
        }
        hd.list[r] = e;
    }
    if (warp == 0) {
        int cnt = 0;
        for (int b0 = 0; b0 < a.E; b0 += 32) {
            const int e = b0 + lane;
            cnt += __popc(__ballot_sync(0xffffffffu, e < a.E && key[e] >= 0));
        }
        if (lane == 0) {
            hd.D = cnt;
            hd.abort = 0;
            // every consumed slot is released by each issuer's commit (one per matrix)
            for (int s = 0; s < NA; ++s) {
                mbar_init(&hd.a_full[s], 1);
                mbar_init(&hd.a_empty[s], ISS);
            }
            for (int s = 0; s < NB; ++s) {
                mbar_init(&hd.b_full[s], 1);
                mbar_init(&hd.b_empty[s], ISS);
                mbar_init(&hd.sf_full[s], 4);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(&hd.acc_full[s], ISS);
                mbar_init(&hd.acc_empty[s], kMxEpiWarps);
            }
            for (int j = 0; j < kMxTaskQ; ++j) {
                mbar_init(&hd.tq_full[j], 1);
                mbar_init(&hd.tq_empty[j], mx_takers<P, TERMS>());
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&hd.tmem_base)),
                     "r"(kMxTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the weight ring is rewritten by the async proxy (TMA) from here on
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the quantised activations and the outputs belong to the previous kernel until it completes
    grid_dep_wait();
    const uint32_t tmem = hd.tmem_base;
    const int ntask = hd.D * tiles;

    if (warp == 3) {
        // ---------------- task fetcher (lane 0) ----------------
        // runs up to a queue's depth ahead of the roles, so the chain of loads behind a
        // task (its expert's picks, first entry, physical id and blob) stays off the
        // operand streams
        if (lane == 0) {
            for (int k = 0;; ++k) {
                const int j = k % kMxTaskQ;
                if (!mbar_wait_fast(&hd.tq_empty[j], ((unsigned)(k / kMxTaskQ) & 1u) ^ 1u, abort, a.status, a.diag,
                                    31, j, k, 0))
                    break;
                int task = atomicAdd(a.task_ctr + ctr, 1);
                if (task >= ntask) task = -1;
                MxTask t{};
                if (task >= 0) t = mx_task(a, hd, task, tiles);
                *reinterpret_cast<volatile int*>(&hd.tq[j]) = task;
                hd.tqt[j] = t;
                mbar_arrive(&hd.tq_full[j]);
                if (task < 0) break;
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------- weight producer ----------------
        // the warp runs converged; one elected lane issues the barrier and TMA operations
        const uint64_t pol = l2_policy_evict_first();  // each weight byte is read once
        int as = 0;
        unsigned aph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            MxTask t;
            const int task = mx_warp_take(hd, k, a, abort, 0, t);
            if (task < 0) break;
            if (!t.valid) continue;
            // the decode kernel's views of the two planes: 128-byte boxes of 32 (w13)
            // or 64 (w2) rows with the 128-byte swizzle, stacked to 128 rows
            const CUtensorMap* map = P == 0 ? &a.tmaps[t.phys].w13n : &a.tmaps[t.phys].w2n;
            const CUtensorMap* smap = P == 0 ? &a.tmaps[t.phys].w13s : &a.tmaps[t.phys].w2s;
            constexpr int box_rows = P == 0 ? 32 : 64;
            asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
            if (wsc_tma) asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(smap) : "memory");
            const int r0 = t.rb * kMxBM;
            for (int tb = 0; tb < t.cnt && ok; tb += TPP) {
                for (int s = 0; s < nks; ++s) {
                    if (!warp_wait(&hd.a_empty[as], aph ^ 1u, a, abort, 32, as, s, task)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(&hd.a_full[as], (unsigned)(MATS * (wsc_tma ? kMxASlot : kMxTile)));
#pragma unroll
                    for (int mt = 0; mt < MATS; ++mt) {
                        uint8_t* dst = sA + (size_t)(as * MATS + mt) * kMxASlot;
#pragma unroll
                        for (int i = 0; i < kMxBM / box_rows; ++i)
                            tma_load_2d_hint_elect(dst + i * box_rows * kMxRowB, map, s * kMxRowB,
                                                   (mt ? I : 0) + r0 + i * box_rows, &hd.a_full[as], pol);
                        // the 16 scale bytes of each row that hold this stage's 8 blocks
                        if (wsc_tma)
#pragma unroll
                            for (int i = 0; i < kMxBM / 32; ++i)
                                tma_load_2d_hint_elect(dst + kMxTile + i * 32 * 16, smap, 16 * (s >> 1),
                                                       (mt ? I : 0) + r0 + 32 * i, &hd.a_full[as], pol);
                    }
                    advance(as, aph, NA);
                }
            }
        }
        if (lane == 0)
            for (int s = 0; s < NA; ++s) mbar_drain(&hd.a_full[s], (s < as) ? aph : (aph ^ 1u));
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- activation producer ----------------
        // the warp runs converged; one elected lane issues the barrier and TMA operations
        const uint64_t pol = l2_policy_evict_last();  // read once per row tile of the expert
        constexpr int kMaxBoxes = (mx_nmax<TERMS>() + kMxBox - 1) / kMxBox;
        int bs = 0;
        unsigned bph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            MxTask t;
            const int task = mx_warp_take(hd, k, a, abort, 1, t);
            if (task < 0) break;
            if (!t.valid) continue;
            for (int tb = 0; tb < t.cnt && ok; tb += TPP) {
                const int row0 = TERMS * (t.off + tb);  // first activation row of the pass
                const int boxes = (mx_ncols(TERMS * min(TPP, t.cnt - tb)) + kMxBox - 1) / kMxBox;
                for (int s = 0; s < nks; ++s) {
                    if (!warp_wait(&hd.b_empty[bs], bph ^ 1u, a, abort, 33, bs, s, task)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(&hd.b_full[bs],
                                                (unsigned)(boxes * kMxBox * kMxRowB + 2 * kMxSfbBox * 4));
                    uint8_t* dst = sB + (size_t)bs * BSTAGE;
#pragma unroll
                    for (int bx = 0; bx < kMaxBoxes; ++bx)
                        if (bx < boxes)
                            tma_load_2d_hint_elect(dst + bx * kMxBox * kMxRowB, &act_map, s * kMxRowB,
                                                   row0 + kMxBox * bx, &hd.b_full[bs], pol);
                    // the stage's two scale words of the pass's tokens, from the 4-aligned
                    // bucket row at or below the first (x is a whole 16 bytes)
                    tma_load_2d_hint_elect(dst + BTILE, &sfb_map, row0 & ~3, 2 * s, &hd.b_full[bs], pol);
                    advance(bs, bph, NB);
                }
            }
        }
        if (lane == 0)
            for (int s = 0; s < NB; ++s) mbar_drain(&hd.b_full[s], (s < bs) ? bph : (bph ^ 1u));
        __syncwarp();
    } else if (warp == 2 || (ISS == 2 && warp == kMxUpIssuer)) {
        // ---------------- MMA issuers ----------------
        // the gate/up phase issues from two warps, warp 2 the gate matrix's MMAs into
        // the gate accumulator and warp 24 the up matrix's into the up accumulator; the
        // down phase has one matrix and one issuer.  Each issuing warp runs its loop
        // converged and one elected lane issues.
        const int mt = warp == 2 ? 0 : 1;
        int as = 0, bs = 0, buf = 0;
        unsigned aph = 0, bph = 0, accph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            MxTask t;
            const int task = mx_warp_take(hd, k, a, abort, 2 + mt, t);
            if (task < 0) break;
            if (!t.valid) continue;
            for (int tb = 0; tb < t.cnt && ok; tb += TPP) {
                const int N = mx_ncols(TERMS * min(TPP, t.cnt - tb));
                const uint32_t id0 = mx_idesc(N, 0u), id2 = mx_idesc(N, 2u);
                if (!warp_wait(&hd.acc_empty[buf], ((accph >> buf) & 1u) ^ 1u, a, abort, 34, buf, 0, task)) {
                    ok = false;
                    break;
                }
                accph ^= 1u << buf;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(P == 0 ? mt : buf) * ACC;
                for (int s = 0; s < nks; ++s) {
                    // the scale writers arrive only after both of the stage's loads landed
                    if (!warp_wait(&hd.sf_full[bs], bph, a, abort, 37, bs, s, task)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf = tmem + SF0 + (uint32_t)bs * mx_sf_cols<P>();
                    const uint64_t bd = sw128_desc(smem_u32(sB + (size_t)bs * BSTAGE));  // its rows
                    const uint64_t ad = sw128_desc(smem_u32(sA + (size_t)(as * MATS + mt) * kMxASlot));
                    const uint32_t sfa = sf + 8u * mt, sfb = sf + mx_sfb_col<P>();
                    if (K - s * kMxBK >= kMxBK)
                        mx_stage_mmas<4>(d, ad, bd, id0, id2, sfa, sfb, s == 0);
                    else  // a K tail of 128 elements (K a multiple of 128)
                        mx_stage_mmas<2>(d, ad, bd, id0, id2, sfa, sfb, s == 0);
                    tc_commit_elect(&hd.a_empty[as]);
                    tc_commit_elect(&hd.b_empty[bs]);
                    advance(as, aph, NA);
                    advance(bs, bph, NB);
                }
                if (!ok) break;
                tc_commit_elect(&hd.acc_full[buf]);
                if (P == 1) buf ^= 1;  // the gate/up phase's two accumulators fill [0, 2 ACC)
            }
        }
        // no MMA may be in flight when tensor memory is freed: wait (bounded) for the
        // last commit of every slot
        if (lane == 0) {
            for (int s = 0; s < NA; ++s) mbar_drain(&hd.a_empty[s], (s < as) ? aph : (aph ^ 1u));
            for (int s = 0; s < NB; ++s) mbar_drain(&hd.b_empty[s], (s < bs) ? bph : (bph ^ 1u));
        }
        __syncwarp();
    } else if (warp >= kMxFirstSf && warp < kMxFirstSf + 4) {
        // ---------------- scale writers ----------------
        // thread = weight row 32 q + lane of the tile (q = lane quarter); every quarter
        // also stores the token words, which each quarter's rows read from their own.
        // The words arrive in shared memory with their stage (the writers follow the
        // weight and activation rings as the MMA issuer does).
        const int q = warp & 3;
        const int rr = 32 * q + lane;
        const uint32_t qaddr = tmem + ((uint32_t)(q * 32) << 16);
        int as = 0, bs = 0;
        unsigned aph = 0, bph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            MxTask t;
            const int task = mx_warp_take(hd, k, a, abort, 3, t);
            if (task < 0) break;
            if (!t.valid) continue;
            const int r0 = t.rb * kMxBM;
            const size_t srl = (size_t)K / 32;  // scale bytes per weight row
            const uint8_t* sg0 = t.blob + (P == 0 ? a.w13s : a.w2s) + (size_t)(r0 + rr) * srl;
            const uint8_t* sg1 = P == 0 ? t.blob + a.w13s + (size_t)(I + r0 + rr) * srl : sg0;
            for (int tb = 0; tb < t.cnt && ok; tb += TPP) {
                const int d0 = (TERMS * (t.off + tb)) & 3;  // first row's place in the loaded words
                for (int s = 0; s < nks; ++s) {
                    const int nj = min(2, (K - s * kMxBK) / 128);  // words of this stage
                    uint32_t wa[2][2] = {{0u, 0u}, {0u, 0u}};
                    if (!wsc_tma) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            wa[0][j] = j < nj ? ld_u32(sg0 + 8 * s + 4 * j) : 0u;
                            if (P == 0) wa[1][j] = j < nj ? ld_u32(sg1 + 8 * s + 4 * j) : 0u;
                        }
                    }
                    // both loads of the stage landed: the producers reused the slot only after
                    // its previous MMAs completed, so its scale slot is free as well
                    if (!warp_wait(&hd.a_full[as], aph, a, abort, 40, as, s, task) ||
                        !warp_wait(&hd.b_full[bs], bph, a, abort, 41, bs, s, task)) {
                        ok = false;
                        break;
                    }
                    if (wsc_tma) {
#pragma unroll
                        for (int mt = 0; mt < MATS; ++mt) {
                            const uint8_t* row = sA + (size_t)(as * MATS + mt) * kMxASlot + kMxTile + rr * 16 + 8 * (s & 1);
                            wa[mt][0] = *reinterpret_cast<const uint32_t*>(row);
                            wa[mt][1] = nj > 1 ? *reinterpret_cast<const uint32_t*>(row + 4) : 0u;
                        }
                    }
                    const uint32_t* wsb = reinterpret_cast<const uint32_t*>(sB + (size_t)bs * BSTAGE + BTILE);
                    constexpr int NG = mx_nmax<TERMS>() / 32;  // token groups of a pass
                    uint32_t wb[2][NG];
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int c = 0; c < NG; ++c) wb[j][c] = j < nj ? wsb[j * kMxSfbBox + d0 + 32 * c + lane] : 0u;
                    tc_fence_after();
                    const uint32_t col = qaddr + SF0 + (uint32_t)bs * mx_sf_cols<P>();
                    // weight words: matrix mt, word j at column 8 mt + 4 j + q (this lane = row 32 q + lane)
                    uint32_t va[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int mt = i >> 3, j = (i >> 2) & 1;
                        va[i] = (mt < MATS && (i & 3) == q) ? wa[mt][j] : 0u;
                    }
                    if constexpr (P == 0) {
                        mx_st16(col, va);
                    } else {
                        uint32_t v8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) v8[i] = va[i];
                        mx_st8(col, v8);
                    }
                    // token words: word j of token group c at column 8 j + c
                    uint32_t vb[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) vb[i] = (i & 7) < NG ? wb[i >> 3][(i & 7) % NG] : 0u;
                    mx_st16(col + mx_sfb_col<P>(), vb);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&hd.sf_full[bs]);
                    advance(as, aph, NA);
                    advance(bs, bph, NB);
                }
            }
        }
    } else if (warp >= kMxFirstEpi && warp < kMxFirstEpi + kMxEpiWarps) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // tensor-memory lane quarter: weight rows 32 q ..
        const int half = (warp - kMxFirstEpi) >> 2;  // this warp's 16-token chunks: 4 i + half
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        uint8_t* stg = base + MxSmem<P, TERMS>::kStg + (size_t)(warp - kMxFirstEpi) * mx_epi_stage<P, TERMS>();
        int buf = 0;
        unsigned accph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            MxTask t;
            const int task = mx_warp_take(hd, k, a, abort, 4, t);
            if (task < 0) break;
            const int r0 = t.rb * kMxBM;
            if (!t.valid) {
                // zero outputs for an expert whose physical id is out of range (its h is
                // never read: the down phase sees the same id)
                if (t.rb == 0 && threadIdx.x == kMxFirstEpi * 32) set_status(a.status, MOE_ERR_BAD_EXPERT);
                if (P == 1)
                    for (int c = half; c < t.cnt; c += 4)
                        a.y[(size_t)__ldg(a.entries + t.off + c) * H + r0 + 32 * q + lane] = 0.f;
                continue;
            }
            for (int tb = 0; tb < t.cnt && ok; tb += TPP) {
                const int nb = min(TPP, t.cnt - tb);  // tokens of the pass
                const int ncol = TERMS * nb;          // accumulator columns (activation rows)
                if (!warp_wait(&hd.acc_full[buf], (accph >> buf) & 1u, a, abort, 39, buf, tb, task)) {
                    ok = false;
                    break;
                }
                accph ^= 1u << buf;
                tc_fence_after();
                const uint32_t d = lane_addr + (uint32_t)buf * ACC;
                for (int cb = 16 * half; cb < ncol; cb += 64) {
                    constexpr int TOK = 16 / TERMS;  // tokens of a 16-column chunk
                    if constexpr (P == 0 && TERMS == 1) {
                        // one term: h of the 16 columns (this lane's row), then per 8-column
                        // slice a transpose through shared memory, so that the four lanes
                        // 4c..4c+3 hold column c's 32-element block, 8 elements each: the
                        // block maximum takes two shuffles, the hardware conversion rounds
                        // element pairs, and each lane stores 4 bytes of the column's row
                        float g[16], u[16];
                        tc_ld16x2(d + cb, d + ACC + cb, g, u);
                        float* tile = reinterpret_cast<float*>(stg);
                        const int col = lane >> 2, part = lane & 3;
#pragma unroll
                        for (int h8 = 0; h8 < 2; ++h8) {
                            __syncwarp();
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const float gs = g[8 * h8 + c];
                                // the fast exponential and division: relative error about 1e-6
                                // for |g| up to 10, far below the quantisation step of h
                                tile[c * 33 + lane] = __fdividef(gs, 1.0f + __expf(-gs)) * u[8 * h8 + c];
                            }
                            __syncwarp();
                            float v[8];
                            uint32_t amax = 0;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                v[i] = tile[col * 33 + part * 8 + i];
                                amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
                            }
                            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                            const int e = mx_block_exp(amax);
                            uint32_t word = 0;
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const uint32_t b0 = __float_as_uint(v[2 * m]), b1 = __float_as_uint(v[2 * m + 1]);
                                const float s0 = __uint_as_float(__float_as_uint(mx_scaled(b0 & 0x7fffffffu, e)) |
                                                                 (b0 & 0x80000000u));
                                const float s1 = __uint_as_float(__float_as_uint(mx_scaled(b1 & 0x7fffffffu, e)) |
                                                                 (b1 & 0x80000000u));
                                word |= e2m1_pair(s0, s1) << (8 * m);
                            }
                            const int cc = cb + 8 * h8 + col;  // accumulator column = activation row offset
                            if (cc < ncol) {
                                const int row = (t.off + tb) + cc;
                                *reinterpret_cast<uint32_t*>(a.hq + (size_t)row * (I / 2) + (r0 + 32 * q) / 2 +
                                                             4 * part) = word;
                                // block (r0 + 32 q) / 32 is byte q of word r0 / 128
                                if (part == 0)
                                    reinterpret_cast<uint8_t*>(a.hs)[((size_t)(r0 / 128) * Rs + row) * 4 + q] =
                                        (uint8_t)(e + 127);
                            }
                        }
                        __syncwarp();
                    } else if constexpr (P == 0) {
                        float g[16], u[16];
                        tc_ld16x2(d + cb, d + ACC + cb, g, u);
                        int es[16];
#pragma unroll
                        for (int n = 0; n < TOK; ++n) {
                            float gs = 0.f, us = 0.f;
#pragma unroll
                            for (int tt = 0; tt < TERMS; ++tt) {
                                gs += g[n * TERMS + tt];
                                us += u[n * TERMS + tt];
                            }
                            // the fast exponential and division: relative error about 1e-6 for
                            // |g| up to 10, far below the quantisation step of h
                            float r = __fdividef(gs, 1.0f + __expf(-gs)) * us;
#pragma unroll
                            for (int tt = 0; tt < TERMS; ++tt) {
                                const int i = n * TERMS + tt;
                                const uint32_t bits = __float_as_uint(r);
                                const uint32_t mag = bits & 0x7fffffffu;
                                // one 32-element block of h per token: this warp's 32 rows
                                const uint32_t amax = __reduce_max_sync(0xffffffffu, mag);
                                const int e = TERMS == 1 ? mx_block_exp(amax) : mx_term_exp(amax);
                                const uint32_t code = e2m1_code(mx_scaled(mag, e)) | ((bits >> 31) << 3);
                                const uint32_t odd = __shfl_down_sync(0xffffffffu, code, 1);
                                if ((lane & 1) == 0) stg[i * 16 + (lane >> 1)] = (uint8_t)(code | (odd << 4));
                                es[i] = e;
                                if (TERMS > 1) r -= mx_decode(code, e);  // exact: the next term's input
                            }
                        }
                        __syncwarp();
                        int my_e = es[0];
#pragma unroll
                        for (int i = 1; i < 16; ++i) my_e = lane == i ? es[i] : my_e;
                        if (lane < 16 && cb + lane < ncol) {
                            const int row = TERMS * (t.off + tb) + cb + lane;  // activation row of this column
                            *reinterpret_cast<uint4*>(a.hq + (size_t)row * (I / 2) + (r0 + 32 * q) / 2) =
                                *reinterpret_cast<const uint4*>(stg + lane * 16);
                            // block (r0 + 32 q) / 32 is byte q of word r0 / 128
                            reinterpret_cast<uint8_t*>(a.hs)[((size_t)(r0 / 128) * Rs + row) * 4 + q] =
                                (uint8_t)(my_e + 127);
                        }
                        __syncwarp();
                    } else {
                        float v[16];
                        tc_ld16(d + cb, v);
                        int pk[TOK];
#pragma unroll
                        for (int n = 0; n < TOK; ++n) {
                            const int tok = cb / TERMS + n;
                            pk[n] = tok < nb ? __ldg(a.entries + t.off + tb + tok) : 0;
                        }
#pragma unroll
                        for (int n = 0; n < TOK; ++n) {
                            float sum = 0.f;
#pragma unroll
                            for (int tt = 0; tt < TERMS; ++tt) sum += v[n * TERMS + tt];
                            if (cb / TERMS + n < nb) a.y[(size_t)pk[n] * H + r0 + 32 * q + lane] = sum;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hd.acc_empty[buf]);
                if (P == 1) buf ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kMxTmemCols) : "memory");
    }
}

// One CTA per bucket row i: x of token entries[i] / k converted to TERMS rows of
// MXFP4 (rows TERMS i .. TERMS i + TERMS - 1 of xq; see ffn_mx_kernel), and their block
// scales into the words of xs (word g of row j at g * Rs + j).  Thread b takes block
// b (32 elements, 64 bytes of bf16).
template <int TERMS>
__global__ void __launch_bounds__(128) mx_xprep_kernel(const __nv_bfloat16* __restrict__ x, int H, int k, int Rs,
                                                       const int32_t* __restrict__ entries, uint8_t* __restrict__ xq,
                                                       uint32_t* __restrict__ xs, int32_t* __restrict__ task_ctr) {
    const int i = blockIdx.x;
    if (i == 0 && threadIdx.x < kTaskCounters) task_ctr[threadIdx.x] = 0;
    const int t = __ldg(entries + i) / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int nblk = H / 32;  // a multiple of 4: a word's four blocks sit in four consecutive lanes
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
        const int lane = threadIdx.x & 31;
        const int active = min(32, nblk - (b - lane));
        const unsigned mask = active >= 32 ? 0xffffffffu : ((1u << active) - 1u);
        float r[32];  // the block (bf16 widens exactly), then each term's residual
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = __ldg(src + 4 * b + j);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                r[8 * j + 2 * q] = __uint_as_float(w4[q] << 16);
                r[8 * j + 2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
            }
        }
#pragma unroll
        for (int tt = 0; tt < TERMS; ++tt) {
            uint32_t amax = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = max(amax, __float_as_uint(r[j]) & 0x7fffffffu);
            const int e = TERMS == 1 ? mx_block_exp(amax) : mx_term_exp(amax);
            uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                // elements j, j + 1 -> byte j / 2 (j in the low nibble), rounded in pairs
                // by the hardware conversion (the same codes as e2m1_code, tested)
                const uint32_t b0 = __float_as_uint(r[j]), b1 = __float_as_uint(r[j + 1]);
                const float s0 = __uint_as_float(__float_as_uint(mx_scaled(b0 & 0x7fffffffu, e)) | (b0 & 0x80000000u));
                const float s1 = __uint_as_float(__float_as_uint(mx_scaled(b1 & 0x7fffffffu, e)) | (b1 & 0x80000000u));
                const uint32_t pair = e2m1_pair(s0, s1);
                o[j >> 3] |= pair << (4 * (j & 7));
                if (TERMS > 1) {  // exact: the next term's input
                    r[j] -= mx_decode(pair & 0xFu, e);
                    r[j + 1] -= mx_decode(pair >> 4, e);
                }
            }
            const size_t row = (size_t)TERMS * i + tt;
            *reinterpret_cast<uint4*>(xq + row * (H / 2) + 16 * b) = make_uint4(o[0], o[1], o[2], o[3]);
            uint32_t word = (uint32_t)(e + 127) << (8 * (b & 3));
            word |= __shfl_xor_sync(mask, word, 1);
            word |= __shfl_xor_sync(mask, word, 2);
            if ((b & 3) == 0) xs[(size_t)(b >> 2) * Rs + row] = word;
        }
    }
}

inline size_t mx_align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct MxWs {
    size_t ctr, xq, xs, hq, hs, total;
};

MxWs mx_ws(int T, int k, int H, int I, int terms) {
    MxWs w;
    const size_t R = (size_t)T * k * terms, Rs = (R + 3) & ~(size_t)3;
    size_t o = 0;
    w.ctr = o;
    o = mx_align256(o + kTaskCounters * sizeof(int32_t));
    w.xq = o;
    o = mx_align256(o + R * (size_t)(H / 2));
    w.xs = o;
    o = mx_align256(o + (size_t)(H / 128) * Rs * 4);
    w.hq = o;
    o = mx_align256(o + R * (size_t)(I / 2));
    w.hs = o;
    o = mx_align256(o + (size_t)(I / 128) * Rs * 4);
    w.total = o;
    return w;
}

template <int P, int TERMS>
cudaError_t launch_mx(const FfnArgs& a, const CUtensorMap& map, const CUtensorMap& smap, int sel, int lo, int hi,
                      int grid, cudaStream_t st) {
    static std::atomic<uint64_t> configured{0};
    const size_t smem = MxSmem<P, TERMS>::kTotal;
    cudaError_t err = ensure_smem_limit((const void*)ffn_mx_kernel<P, TERMS>, (int)smem, configured);
    if (err != cudaSuccess) return err;
    // task counters 12-15 of the call's workspace (zeroed by the prep kernel): one per
    // phase and placement class
    const int ctr = 12 + (sel == 2 ? 2 : 0) + P;
    return launch_pdl(ffn_mx_kernel<P, TERMS>, dim3(grid), dim3(kMxThreads), smem, st, a, map, smap, sel, ctr, lo, hi);
}

}  // namespace

size_t ffn_mx_workspace(int T, int k, int H, int I, int terms) { return mx_ws(T, k, H, I, terms).total; }

cudaError_t launch_ffn_mx_prep(FfnArgs& a, void* workspace, int terms, cudaStream_t st) {
    const MxWs w = mx_ws(a.T, a.k, a.H, a.I, terms);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.task_ctr = reinterpret_cast<int32_t*>(ws + w.ctr);
    a.xq = ws + w.xq;
    a.xs = reinterpret_cast<uint32_t*>(ws + w.xs);
    a.hq = ws + w.hq;
    a.hs = reinterpret_cast<uint32_t*>(ws + w.hs);
    if (a.T == 0) return cudaSuccess;
    const int R = a.T * a.k;
    const int Rs = (R * terms + 3) & ~3;
    if (terms == 1)
        mx_xprep_kernel<1><<<R, 128, 0, st>>>(a.x, a.H, a.k, Rs, a.entries, a.xq, a.xs, a.task_ctr);
    else
        mx_xprep_kernel<4><<<R, 128, 0, st>>>(a.x, a.H, a.k, Rs, a.entries, a.xq, a.xs, a.task_ctr);
    return cudaGetLastError();
}

cudaError_t launch_ffn_mx(const FfnArgs& a, int phase, int sel, int lo, int hi, int terms, int sm_count,
                          cudaStream_t st) {
    const int R = a.T * a.k * terms;
    if (R == 0) return cudaSuccess;
    // activations of the phase: [R rows][K/2 bytes] E2M1, boxes of 128 bytes x 32 rows, 128-byte swizzle
    CUtensorMap map;
    const int K = phase == 0 ? a.H : a.I;
    if (!encode_tmap_2d(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, phase == 0 ? a.xq : a.hq, (uint64_t)(K / 2), (uint64_t)R,
                        (uint64_t)(K / 2), kMxRowB, kMxBox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // their scale words [K/128 rows][Rs words], boxes of 200 words x 2 rows
    CUtensorMap smap;
    const int Rs = (R + 3) & ~3;
    if (!encode_tmap_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT32, phase == 0 ? a.xs : a.hs, (uint64_t)Rs,
                        (uint64_t)(K / 128), (uint64_t)Rs * 4, kMxSfbBox, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const long picks = (long)a.T * a.k;
    const long dmax = a.E < picks ? a.E : picks;
    const long tasks = dmax * ((phase == 0 ? a.I : a.H) / kMxBM);
    const int grid = (int)(tasks < sm_count ? tasks : sm_count);
    if (grid <= 0) return cudaSuccess;
    if (terms == 1)
        return phase == 0 ? launch_mx<0, 1>(a, map, smap, sel, lo, hi, grid, st)
                          : launch_mx<1, 1>(a, map, smap, sel, lo, hi, grid, st);
    return phase == 0 ? launch_mx<0, 4>(a, map, smap, sel, lo, hi, grid, st)
                      : launch_mx<1, 4>(a, map, smap, sel, lo, hi, grid, st);
}

}  // namespace moe
