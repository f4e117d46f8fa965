// Internal declarations shared by the library's translation units (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "moehost.h"

namespace moe {

constexpr int kMaxSwaps = 64;

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device (the
// attribute belongs to the device the calling thread has current): `done` holds
// one bit per device ordinal below 64; higher ordinals set it on every call.
// Setting it twice is harmless, so racing first calls need no lock.
inline cudaError_t ensure_smem_limit(const void* kernel, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launches `kernel` so that it may start while the previous kernel on the stream
// finishes (programmatic dependent launch); the kernel waits with grid_dep_wait
// before it touches that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Blob plane offsets for (H, I); see the blob format in moehost.h.
struct BlobLayout {
    size_t w13n, w13s, w2n, w2s, total;
};

inline BlobLayout blob_layout(int H, int I) {
    BlobLayout b;
    size_t a = (size_t)2 * I * (H / 2);
    size_t s = (size_t)2 * I * (H / 32);
    size_t c = (size_t)H * (I / 2);
    size_t d = (size_t)H * (I / 32);
    b.w13n = 0;
    b.w13s = a;
    b.w2n = a + s;
    b.w2s = a + s + c;
    b.total = a + s + c + d;
    return b;
}

__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---- launchers (implemented in the .cu files) -------------------------------

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids, float* w,
                         int32_t* counts, int32_t* offsets, int32_t* entries, int32_t* window, int* status,
                         cudaStream_t st);

// Remap (phys ids, picked cold slots) on the caller's stream.
cudaError_t launch_cold_remap(const int32_t* ids, int n_picks, const int32_t* loc, int E, int n_hot, int n_cold,
                              int32_t* phys, int32_t* cold_list, int32_t* n_picked, int* status, cudaStream_t st);
// Byte copy of the picked cold slots (derives the slot list from the picks itself);
// marks each copied slot's tag with uid.
// Copies bytes [part_lo, part_hi) (multiples of 16) of every picked cold expert's
// host blob into its scratch slot.
cudaError_t launch_cold_copy(const int32_t* ids, int n_picks, const int32_t* loc, int E, int n_hot, int n_cold,
                             const uint8_t* const* cold_src, uint8_t* slot_base, size_t blob_bytes, size_t part_lo,
                             size_t part_hi, int32_t* slot_tag, int uid, int ctas, cudaStream_t st);

cudaError_t launch_link_probe(const uint8_t* src, uint8_t* dst, size_t bytes, int ctas, cudaStream_t st);

// 2D TMA descriptors of the two nibble planes of the blob at one physical id:
// a swizzled view for the decode kernel and a plain one for the prefill kernel.
struct ExpertMaps {
    CUtensorMap w13n;  // [2I rows][H/2 bytes], box 128 B x 32 rows, 128-byte swizzle
    CUtensorMap w2n;   // [H rows][I/2 bytes], box 128 B x 64 rows, 128-byte swizzle
    CUtensorMap w13r;  // [2I rows][H/2 bytes], box 64 B x 128 rows, 64-byte swizzle
    CUtensorMap w2r;   // [H rows][I/2 bytes], same box
    // the two scale planes, box 16 B x 32 rows: encoded only where a row is a multiple
    // of 16 bytes (H, resp. I, a multiple of 512), else zero and unused (see
    // mx_scale_maps); the kernels then read the scales from global memory
    CUtensorMap w13s;  // [2I rows][H/32 bytes]
    CUtensorMap w2s;   // [H rows][I/32 bytes]
};

// Whether the scale plane of a matrix with reduction length K has a tensor map
// (TMA needs row strides that are multiples of 16 bytes).
__host__ __device__ inline bool mx_scale_maps(int K) { return (K / 32) % 16 == 0; }

// Buckets with more than this many tokens run on the tensor-core prefill kernel.
constexpr int kTcMinTokens = 64;
// Task counters in the FFN workspace: one per decode kernel launch of a call
// (2 placement classes x 2 phases x 3 token-count ranges).
constexpr int kTaskCounters = 16;

// Encodes a 2D tiled TMA descriptor (inner dimension contiguous); false on failure.
bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

struct FfnArgs {
    const uint8_t* const* ptr;  // phys id -> blob base (device)
    const ExpertMaps* tmaps;    // phys id -> descriptors (device)
    const int32_t* loc;         // placement map, for the hot/cold split
    int n_hot;
    int n_phys;
    const int32_t* phys_ids;  // [T*k]
    const int32_t* counts;    // [E]
    const int32_t* offsets;   // [E+1]
    const int32_t* entries;   // [T*k]
    int E, k, H, I, T;
    const __nv_bfloat16* x;  // [T][H]
    // workspace, all in bucket order (row i = entries[i]):
    __half* g;               // [T*k][max(H, I)] prescaled f16 activations: x rows for the
                             // gate/up phase, then h rows for the down phase
    int32_t* gexp;           // [T*k] their power-of-two prescale exponents
    float* h;                // [T*k][I] SiLU(gate) * up
    float* y;                // [T*k][H]
    int32_t* task_ctr;       // workspace [kTaskCounters] per-launch task counters (zeroed by xprep)
    int* status;
    int* diag;               // [16] where the first timed-out wait gave up
    size_t w13s, w2n, w2s;   // plane offsets in a blob
    // zero-copy launches: cold slot c's blob read in place from pinned host memory
    // (device-mapped pointers), no scratch copy
    const uint8_t* const* cold_host;
    // block-scaled (all-FP4) prefill, in bucket order (row i = entries[i]): x and h
    // quantised to MXFP4, element k of a row in byte k/2, and their E8M0 block
    // scales as 32-bit words of four blocks, word (g, i) = blocks 4g..4g+3 of row i
    // at index g * Rs + i
    uint8_t* xq;   // [T*k][H/2]
    uint32_t* xs;  // [H/128][Rs], Rs = T*k rounded up to a multiple of 4 (row stride of
                   // whole 16-byte units, so the words can be loaded by TMA)
    uint8_t* hq;   // [T*k][I/2]
    uint32_t* hs;  // [I/128][Rs]
};

size_t ffn_decode_workspace(int T, int k, int H, int I);
// 2D TMA descriptor of the bucket-ordered activations a.g for a phase (0: H
// columns, 1: I columns), rows T*k, with the given box and swizzle.
bool encode_act_map(CUtensorMap* m, const FfnArgs& a, int phase, uint32_t box_inner, uint32_t box_rows,
                    CUtensorMapSwizzle sw);
// Points the workspace fields of `a` at `workspace` and launches the x prescale
// into bucket order.
cudaError_t launch_ffn_prep(FfnArgs& a, void* workspace, cudaStream_t st);
// One phase (0: gate/up -> h, 1: down -> y) over the experts selected by sel
// (0: all, 1: placed in HBM, 2: placed in cold slots).
// zc: the launch reads the weights of cold experts (sel == 2) in place from host
// memory (decode-sized calls only: T <= kTcMinTokens).
cudaError_t launch_ffn_phase(const FfnArgs& a, int phase, int sel, int sm_count, cudaStream_t st, bool zc = false);
// The tensor-core kernel of one phase over the selected experts with more than lo tokens.
cudaError_t launch_ffn_tc(const FfnArgs& a, int phase, int sel, int lo, int sm_count, cudaStream_t st);

// Block-scaled (all-FP4) prefill path: workspace bytes for T tokens; the prep that
// points the workspace fields of `a` at `workspace`, zeroes the task counters and
// quantises x into bucket order; one phase (0: gate/up -> h quantised, 1: down -> y)
// over every selected expert with at least one token.
// terms: activation rows per token (1: the all-FP4 mode; 4: a sum of four MXFP4
// terms that reproduces the activation, the decode path); lo < tokens <= hi selects
// the experts of a launch.
size_t ffn_mx_workspace(int T, int k, int H, int I, int terms);
cudaError_t launch_ffn_mx_prep(FfnArgs& a, void* workspace, int terms, cudaStream_t st);
cudaError_t launch_ffn_mx(const FfnArgs& a, int phase, int sel, int lo, int hi, int terms, int sm_count,
                          cudaStream_t st);

cudaError_t launch_combine(const float* y, const float* w, int T, int k, int H, void* out, int out_fp32,
                           cudaStream_t st);

struct SwapList {
    int n;
    uint8_t* hot[kMaxSwaps];   // device blob of the HBM slot
    uint8_t* host[kMaxSwaps];  // device-mapped pointer of the host blob
};
// Exchanges hot[i] and host[i] in place for every pair, with `ctas` CTAs.
cudaError_t launch_swap(const SwapList& s, size_t blob_bytes, int ctas, cudaStream_t st);
// Copies host[i] -> hot[i] (blob_bytes each) for every pair, with `ctas` CTAs.
cudaError_t launch_copy_list(const SwapList& s, size_t blob_bytes, int ctas, cudaStream_t st);

cudaError_t launch_debug_e2m1(uint32_t* out, cudaStream_t st);

}  // namespace moe
