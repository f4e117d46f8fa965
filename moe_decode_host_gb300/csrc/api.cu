// Host side of the C ABI declared in moehost.h: argument checks, layer state,
// launches, and the residency manager.
//
// Residency ("DeepSeek-V4.1-Flash on One GB300 Without the Second GPU", section 1:
// between steps a manager swaps often-picked experts into the hot set and quiet
// ones out; section 3: a hysteresis threshold of 3.0 is the published default and
// halved the swap count without slowing the step).  The pick counters of the
// window are accumulated on the device by moe_route; on an acting step the host
// reads them, builds the swap list, exchanges the bytes with one kernel and
// rewrites the placement map.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "internal.cuh"

using namespace moe;

struct moe_scratch {
    int n_slots;
    size_t expert_bytes;
    uint8_t* base;
    int32_t* d_tag = nullptr;  // [n_slots] id of the layer that last copied into the slot, or -1
    int32_t* h_tag = nullptr;  // pinned [n_slots] staging for reads of d_tag
};

struct moe_layer {
    moe_params p;
    moe_scratch* scratch;
    BlobLayout lay;
    int sm_count;
    std::vector<uint8_t*> hot;        // device blobs of the HBM slots
    std::vector<uint8_t*> cold_dev;   // device-mapped pointers of the cold slots' host blobs
    std::vector<uint8_t*> mirror_dev;  // host_mirror: device-mapped pointer of every expert's host copy
    int uid = 0;                      // this layer's id in the scratch slot tags
    std::vector<int32_t> loc;         // host mirror of the placement map
    int32_t* d_loc = nullptr;         // [E]
    const uint8_t** d_ptr = nullptr;  // [n_hot + n_cold] phys id -> blob base
    const uint8_t** d_cold_src = nullptr;  // [n_cold] host blobs (device-mapped)
    int32_t* d_window = nullptr;      // [E] picks in the current window
    int32_t* d_window_alt = nullptr;  // [E] the other window buffer (deferred residency snapshots)
    int* d_status = nullptr;
    int* d_diag = nullptr;            // [16] record of the first device-side wait that timed out
    int32_t* h_counts = nullptr;      // pinned [E]
    int32_t* h_loc = nullptr;         // pinned [E]
    const uint8_t** h_cold_src = nullptr;  // pinned [n_cold] staging of d_cold_src updates
    ExpertMaps* d_tmaps = nullptr;      // [E] TMA descriptors per physical id
    cudaStream_t copy_stream = nullptr;  // cold slot copies run here, joined by moe_grouped_ffn
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    cudaEvent_t ev_join_w13 = nullptr;  // the copy's first launch (the gate/up planes) has completed
    bool copy_pending = false;
    bool copy_pending_w13 = false;
    // residency (moe_layer_set_residency_defer): ev_counts follows the D2H copy of a
    // window snapshot; ev_swap follows the last exchange and map upload
    cudaEvent_t ev_counts = nullptr, ev_swap = nullptr;
    int residency_defer = 1;
    bool plan_pending = false;   // a snapshot in h_counts awaits its plan
    std::vector<int32_t> plan_pro, plan_dem;  // the current plan's pairs (deferred: paced)
    int plan_next = 0;  // pairs [0, plan_next) have been applied
    int plan_age = 0;   // calls since the current plan was made
    bool swap_recorded = false;  // ev_swap has been recorded (the staging buffers may be in use)
    bool swap_pending = false;   // the caller's stream has not yet waited for ev_swap
    int copy_ctas = 0;
    std::vector<cudaEvent_t> prof_ev;  // pairs of events around recorded cold copies
    int prof_n = 0;
    std::vector<cudaEvent_t> fprof_ev;  // six per recorded FFN call (see moe_layer_profile_read_ffn)
    int fprof_n = 0;
    long steps = 0;
    int fault = 0;
    int prefill_kind = 0;  // moe_layer_set_prefill_kind
    int decode_kind = 0;   // moe_layer_set_decode_kind
};

namespace {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_device_ptr(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Returns the device pointer of pinned, mapped host memory, or nullptr.
void* mapped_host_ptr(void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost) return nullptr;
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return d;
}

cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

bool moe::encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// 2D u8 view [rows][row_bytes] at base: the decode kernel's box (128 bytes x
// box_rows rows, 128-byte swizzle) and the prefill kernel's (64 bytes x 128 rows,
// 64-byte swizzle).
bool encode_plane(CUtensorMap* m, const uint8_t* base, size_t row_bytes, size_t rows, uint32_t box_rows) {
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, row_bytes, rows, row_bytes, 128, box_rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}
bool encode_plane_raw(CUtensorMap* m, const uint8_t* base, size_t row_bytes, size_t rows) {
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, row_bytes, rows, row_bytes, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_64B);
}

// Scale plane [rows][row_bytes]: 16-byte x 32-row boxes (a decode task's gate or up
// rows; four of them make a prefill tile).
bool encode_scales(CUtensorMap* m, const uint8_t* base, size_t row_bytes, size_t rows) {
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, row_bytes, rows, row_bytes, 16, 32,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Default grid of the cold copy: 3/16 of the SMs (28 on a GB300) keep the host link
// as busy as 38 do with up to ten cold experts a step (measured: 208.6 against
// 208.7 GB/s at 32 tokens) and leave the other SMs to the FFN over HBM-resident
// experts that runs meanwhile; 19 CTAs streamed ten experts 4% slower.
int default_copy_ctas(int sm_count) { return sm_count * 3 / 16 > 0 ? sm_count * 3 / 16 : 1; }

// Makes `st` wait for the layer's cold copy in flight, if any.
cudaError_t join_copy(moe_layer* L, cudaStream_t st) {
    if (!L->copy_pending) return cudaSuccess;
    L->copy_pending = false;
    L->copy_pending_w13 = false;
    return cudaStreamWaitEvent(st, L->ev_join, 0);
}

// Makes `st` wait for the first half of the cold copy in flight (every picked cold
// expert's gate/up planes), if any: the gate/up phase over the cold experts can then
// run while their down planes still stream.
cudaError_t join_copy_w13(moe_layer* L, cudaStream_t st) {
    if (!L->copy_pending_w13) return cudaSuccess;
    L->copy_pending_w13 = false;
    return cudaStreamWaitEvent(st, L->ev_join_w13, 0);
}

// Makes `st` wait for a residency exchange (and its map upload) that ran on the
// layer's copy stream, if the caller's stream has not waited for it yet.
cudaError_t join_swap(moe_layer* L, cudaStream_t st) {
    if (!L->swap_pending) return cudaSuccess;
    L->swap_pending = false;
    return cudaStreamWaitEvent(st, L->ev_swap, 0);
}

// Blocks the host until the copies that read the pinned staging buffers (h_loc,
// h_cold_src) of the last exchange have completed, before they are rewritten.
cudaError_t settle_staging(moe_layer* L) {
    return L->swap_recorded ? cudaEventSynchronize(L->ev_swap) : cudaSuccess;
}

void free_prof(moe_layer* L) {
    for (cudaEvent_t e : L->prof_ev) cudaEventDestroy(e);
    L->prof_ev.clear();
    L->prof_n = 0;
    for (cudaEvent_t e : L->fprof_ev) cudaEventDestroy(e);
    L->fprof_ev.clear();
    L->fprof_n = 0;
}

std::atomic<int> g_next_uid{1};

void free_layer(moe_layer* L) {
    if (!L) return;
    if (L->copy_stream) cudaStreamSynchronize(L->copy_stream);
    free_prof(L);
    if (L->copy_stream) cudaStreamDestroy(L->copy_stream);
    if (L->ev_fork) cudaEventDestroy(L->ev_fork);
    if (L->ev_join) cudaEventDestroy(L->ev_join);
    if (L->ev_join_w13) cudaEventDestroy(L->ev_join_w13);
    if (L->ev_counts) cudaEventDestroy(L->ev_counts);
    if (L->ev_swap) cudaEventDestroy(L->ev_swap);
    cudaFree(L->d_tmaps);
    cudaFree(L->d_loc);
    cudaFree(L->d_ptr);
    cudaFree(L->d_cold_src);
    cudaFree(L->d_window);
    cudaFree(L->d_window_alt);
    cudaFree(L->d_status);
    cudaFree(L->d_diag);
    cudaFreeHost(L->h_counts);
    cudaFreeHost(L->h_loc);
    cudaFreeHost(L->h_cold_src);
    delete L;
}

}  // namespace

extern "C" {

size_t moe_expert_bytes(int H, int I) {
    if (H <= 0 || I <= 0 || H % 128 || I % 128) return 0;
    return blob_layout(H, I).total;
}

int moe_scratch_create(int n_slots, size_t expert_bytes, void* slot_dev, moe_scratch** out) {
    if (!out || n_slots < 0 || expert_bytes == 0 || expert_bytes % 16) return MOE_ERR_INVALID_ARG;
    if (n_slots > 0 && (!slot_dev || !aligned(slot_dev, 256) || !is_device_ptr(slot_dev))) return MOE_ERR_INVALID_ARG;
    moe_scratch* s = new (std::nothrow) moe_scratch;
    if (!s) return MOE_ERR_NOMEM;
    s->n_slots = n_slots;
    s->expert_bytes = expert_bytes;
    s->base = static_cast<uint8_t*>(slot_dev);
    const size_t tb = sizeof(int32_t) * (n_slots > 0 ? n_slots : 1);
    cudaError_t err = cudaMalloc(&s->d_tag, tb);
    err = err ? err : cudaMemset(s->d_tag, 0xff, tb);
    err = err ? err : cudaHostAlloc(&s->h_tag, tb, cudaHostAllocDefault);
    if (err != cudaSuccess) {
        cudaGetLastError();
        cudaFree(s->d_tag);
        cudaFreeHost(s->h_tag);
        delete s;
        return err == cudaErrorMemoryAllocation ? MOE_ERR_NOMEM : MOE_ERR_CUDA;
    }
    *out = s;
    return MOE_OK;
}

int moe_scratch_destroy(moe_scratch* s) {
    if (s) {
        cudaFree(s->d_tag);
        cudaFreeHost(s->h_tag);
    }
    delete s;
    return MOE_OK;
}

int moe_layer_create(const moe_params* pp, moe_scratch* scratch, void* const* hot_blobs_dev,
                     void* const* cold_blobs_host, const int32_t* init_loc, moe_layer** out) {
    if (!pp || !out || !init_loc) return MOE_ERR_INVALID_ARG;
    const moe_params p = *pp;
    if (p.E < 1 || p.E > 1024 || p.k < 1 || p.k > 32 || p.k > p.E) return MOE_ERR_INVALID_ARG;
    if (moe_expert_bytes(p.H, p.I) == 0) return MOE_ERR_INVALID_ARG;
    if (p.n_hot < 0 || p.n_cold < 0 || p.n_hot + p.n_cold != p.E || p.n_cold > 4096) return MOE_ERR_INVALID_ARG;
    if (p.renorm != 0 && p.renorm != 1) return MOE_ERR_INVALID_ARG;
    if (p.swap_every < 0 || p.max_swaps < 0 || p.max_swaps > kMaxSwaps) return MOE_ERR_INVALID_ARG;
    if (!(p.hysteresis >= 0.0f) || p.hysteresis > 1e30f) return MOE_ERR_INVALID_ARG;
    if (p.host_mirror != 0 && p.host_mirror != 1) return MOE_ERR_INVALID_ARG;
    if (p.zero_copy != 0 && p.zero_copy != 1) return MOE_ERR_INVALID_ARG;
    const size_t eb = moe_expert_bytes(p.H, p.I);
    if (p.n_cold > 0 && (!scratch || scratch->expert_bytes != eb || scratch->n_slots < p.n_cold))
        return MOE_ERR_INVALID_ARG;
    if (p.n_hot > 0 && !hot_blobs_dev) return MOE_ERR_INVALID_ARG;
    const int n_host = p.host_mirror ? p.E : p.n_cold;  // host blobs passed
    if (n_host > 0 && !cold_blobs_host) return MOE_ERR_INVALID_ARG;
    // placement map: a bijection onto [0, E)
    std::vector<char> seen(p.E, 0);
    for (int e = 0; e < p.E; ++e) {
        const int v = init_loc[e];
        if (v < 0 || v >= p.E || seen[v]) return MOE_ERR_INVALID_ARG;
        seen[v] = 1;
    }
    moe_layer* L = new (std::nothrow) moe_layer;
    if (!L) return MOE_ERR_NOMEM;
    L->p = p;
    L->scratch = scratch;
    L->lay = blob_layout(p.H, p.I);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&L->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        delete L;
        return MOE_ERR_CUDA;
    }
    L->hot.resize(p.n_hot);
    for (int h = 0; h < p.n_hot; ++h) {
        void* b = hot_blobs_dev[h];
        if (!b || !aligned(b, 16) || !is_device_ptr(b)) {
            delete L;
            return MOE_ERR_INVALID_ARG;
        }
        L->hot[h] = static_cast<uint8_t*>(b);
    }
    std::vector<uint8_t*> host_dev(n_host);
    for (int i = 0; i < n_host; ++i) {
        void* b = cold_blobs_host[i];
        void* d = b ? mapped_host_ptr(b) : nullptr;
        if (!d || !aligned(b, 16) || !aligned(d, 16)) {
            delete L;
            return MOE_ERR_INVALID_ARG;
        }
        host_dev[i] = static_cast<uint8_t*>(d);
    }
    L->cold_dev.resize(p.n_cold);
    if (p.host_mirror) {
        L->mirror_dev = host_dev;
        for (int e = 0; e < p.E; ++e)
            if (init_loc[e] >= p.n_hot) L->cold_dev[init_loc[e] - p.n_hot] = host_dev[e];
    } else {
        for (int c = 0; c < p.n_cold; ++c) L->cold_dev[c] = host_dev[c];
    }
    L->uid = g_next_uid.fetch_add(1);
    L->loc.assign(init_loc, init_loc + p.E);
    std::vector<const uint8_t*> ptr(p.E);
    for (int h = 0; h < p.n_hot; ++h) ptr[h] = L->hot[h];
    for (int c = 0; c < p.n_cold; ++c) ptr[p.n_hot + c] = scratch->base + (size_t)c * eb;
    cudaError_t err = cudaSuccess;
    err = err ? err : cudaMalloc(&L->d_loc, sizeof(int32_t) * p.E);
    err = err ? err : cudaMalloc(&L->d_ptr, sizeof(uint8_t*) * p.E);
    err = err ? err : cudaMalloc(&L->d_cold_src, sizeof(uint8_t*) * (p.n_cold > 0 ? p.n_cold : 1));
    err = err ? err : cudaMalloc(&L->d_window, sizeof(int32_t) * p.E);
    err = err ? err : cudaMalloc(&L->d_window_alt, sizeof(int32_t) * p.E);
    err = err ? err : cudaMalloc(&L->d_status, sizeof(int));
    err = err ? err : cudaMalloc(&L->d_diag, sizeof(int) * 16);
    err = err ? err : cudaMemset(L->d_diag, 0, sizeof(int) * 16);
    err = err ? err : cudaHostAlloc(&L->h_counts, sizeof(int32_t) * p.E, cudaHostAllocDefault);
    err = err ? err : cudaHostAlloc(&L->h_loc, sizeof(int32_t) * p.E, cudaHostAllocDefault);
    err = err ? err
              : cudaHostAlloc(&L->h_cold_src, sizeof(uint8_t*) * (p.n_cold > 0 ? p.n_cold : 1), cudaHostAllocDefault);
    err = err ? err : cudaMemcpy(L->d_loc, init_loc, sizeof(int32_t) * p.E, cudaMemcpyHostToDevice);
    err = err ? err : cudaMemcpy(L->d_ptr, ptr.data(), sizeof(uint8_t*) * p.E, cudaMemcpyHostToDevice);
    if (p.n_cold > 0)
        err = err ? err
                  : cudaMemcpy(L->d_cold_src, L->cold_dev.data(), sizeof(uint8_t*) * p.n_cold, cudaMemcpyHostToDevice);
    err = err ? err : cudaMemset(L->d_window, 0, sizeof(int32_t) * p.E);
    err = err ? err : cudaMemset(L->d_window_alt, 0, sizeof(int32_t) * p.E);
    err = err ? err : cudaMemset(L->d_status, 0, sizeof(int));
    err = err ? err : cudaStreamCreateWithFlags(&L->copy_stream, cudaStreamNonBlocking);
    err = err ? err : cudaEventCreateWithFlags(&L->ev_fork, cudaEventDisableTiming);
    err = err ? err : cudaEventCreateWithFlags(&L->ev_join, cudaEventDisableTiming);
    err = err ? err : cudaEventCreateWithFlags(&L->ev_join_w13, cudaEventDisableTiming);
    err = err ? err : cudaEventCreateWithFlags(&L->ev_counts, cudaEventDisableTiming);
    err = err ? err : cudaEventCreateWithFlags(&L->ev_swap, cudaEventDisableTiming);
    if (err == cudaSuccess) {
        std::vector<ExpertMaps> maps(p.E);
        memset(maps.data(), 0, sizeof(ExpertMaps) * maps.size());
        for (int i = 0; i < p.E; ++i) {
            if ((mx_scale_maps(p.H) && !encode_scales(&maps[i].w13s, ptr[i] + L->lay.w13s, (size_t)p.H / 32,
                                                      (size_t)2 * p.I)) ||
                (mx_scale_maps(p.I) && !encode_scales(&maps[i].w2s, ptr[i] + L->lay.w2s, (size_t)p.I / 32,
                                                      (size_t)p.H))) {
                free_layer(L);
                return MOE_ERR_CUDA;
            }
            if (!encode_plane(&maps[i].w13n, ptr[i] + L->lay.w13n, (size_t)p.H / 2, (size_t)2 * p.I, 32) ||
                !encode_plane(&maps[i].w2n, ptr[i] + L->lay.w2n, (size_t)p.I / 2, (size_t)p.H, 64) ||
                !encode_plane_raw(&maps[i].w13r, ptr[i] + L->lay.w13n, (size_t)p.H / 2, (size_t)2 * p.I) ||
                !encode_plane_raw(&maps[i].w2r, ptr[i] + L->lay.w2n, (size_t)p.I / 2, (size_t)p.H)) {
                free_layer(L);
                return MOE_ERR_CUDA;
            }
        }
        err = cudaMalloc(&L->d_tmaps, sizeof(ExpertMaps) * p.E);
        err = err ? err : cudaMemcpy(L->d_tmaps, maps.data(), sizeof(ExpertMaps) * p.E, cudaMemcpyHostToDevice);
    }
    L->copy_ctas = default_copy_ctas(L->sm_count);
    if (err != cudaSuccess) {
        cudaGetLastError();
        free_layer(L);
        return err == cudaErrorMemoryAllocation ? MOE_ERR_NOMEM : MOE_ERR_CUDA;
    }
    *out = L;
    return MOE_OK;
}

int moe_layer_destroy(moe_layer* L) {
    if (!L) return MOE_ERR_INVALID_ARG;
    free_layer(L);
    return MOE_OK;
}

int moe_route(moe_layer* L, const float* logits, int T, int32_t* topk_ids, float* topk_w, int32_t* counts,
              int32_t* offsets, int32_t* entries, void* stream) {
    if (!L || T < 0 || !counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_ids || !topk_w || !entries)) return MOE_ERR_INVALID_ARG;
    if ((long)T * L->p.k > (1L << 30)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route(logits, T, L->p.E, L->p.k, L->p.renorm, topk_ids, topk_w, counts, offsets,
                                    entries, L->d_window, L->d_status, S(stream)));
}

int cold_gather(moe_layer* L, const int32_t* topk_ids, int T, int32_t* phys_ids, int32_t* cold_list,
                int32_t* n_cold_picked, void* stream) {
    if (!L || T < 0 || !n_cold_picked) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !phys_ids)) return MOE_ERR_INVALID_ARG;
    if (L->p.n_cold > 0 && T > 0 && !cold_list) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = S(stream);
    // the remap reads the placement map, which a deferred residency exchange updates
    cudaError_t err = join_swap(L, st);
    // zero copy (decode-sized calls): the FFN reads the cold experts in place, no copy
    const bool zc = L->p.zero_copy && T <= kTcMinTokens;
    if (L->p.n_cold > 0 && T > 0 && !zc) {
        // the byte copy forks onto the layer's copy stream first, so that it starts
        // while the remap kernel runs and the FFN over HBM-resident experts can run
        // while the link streams the cold ones.  It moves every picked blob's gate/up
        // planes first, then its down planes, with an event between, so that the
        // gate/up phase over the cold experts overlaps the second launch.
        err = cudaEventRecord(L->ev_fork, st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(L->copy_stream, L->ev_fork, 0);
        const bool prof = L->prof_n < (int)L->prof_ev.size() / 2;
        if (err == cudaSuccess && prof) err = cudaEventRecord(L->prof_ev[2 * L->prof_n], L->copy_stream);
        const size_t split = L->lay.w2n;  // the gate/up planes (nibbles, scales) end where w2 begins
        if (err == cudaSuccess)
            err = launch_cold_copy(topk_ids, T * L->p.k, L->d_loc, L->p.E, L->p.n_hot, L->p.n_cold, L->d_cold_src,
                                   L->scratch->base, L->lay.total, 0, split, L->scratch->d_tag, L->uid, L->copy_ctas,
                                   L->copy_stream);
        if (err == cudaSuccess) err = cudaEventRecord(L->ev_join_w13, L->copy_stream);
        if (err == cudaSuccess)
            err = launch_cold_copy(topk_ids, T * L->p.k, L->d_loc, L->p.E, L->p.n_hot, L->p.n_cold, L->d_cold_src,
                                   L->scratch->base, L->lay.total, split, L->lay.total, L->scratch->d_tag, L->uid,
                                   L->copy_ctas, L->copy_stream);
        if (err == cudaSuccess && prof) {
            err = cudaEventRecord(L->prof_ev[2 * L->prof_n + 1], L->copy_stream);
            ++L->prof_n;
        }
        if (err == cudaSuccess) err = cudaEventRecord(L->ev_join, L->copy_stream);
        if (err == cudaSuccess) {
            L->copy_pending = true;
            L->copy_pending_w13 = true;
        }
    }
    if (err == cudaSuccess)
        err = launch_cold_remap(topk_ids, T * L->p.k, L->d_loc, L->p.E, L->p.n_hot, L->p.n_cold, phys_ids, cold_list,
                                n_cold_picked, L->d_status, st);
    return cuda_status(err);
}

int moe_gather_join(moe_layer* L, void* stream) {
    if (!L) return MOE_ERR_INVALID_ARG;
    cudaError_t err = join_copy(L, S(stream));
    if (err == cudaSuccess) err = join_swap(L, S(stream));
    return cuda_status(err);
}

namespace {
// The kernels a call runs.  Prefill-sized calls (more than 64 tokens): the all-FP4
// block-scaled kernels when the layer asks for them (1 activation term), else the
// dequant-GEMV kernel for buckets of at most 64 tokens and the f16 tensor-core kernel
// above.  Decode-sized calls: the block-scaled kernels with activations as sums of
// four MXFP4 terms (kinds 0 and 2; measured faster than the dequant-GEMV kernel from
// one token up), the dequant-GEMV kernel for kind 1 and whenever the layer reads cold
// experts in place (zero copy), which only that kernel does.
int mx_terms(const moe_layer* L, int T) {
    if (T > kTcMinTokens) return L->prefill_kind == 1 ? 1 : 0;
    if (L->decode_kind == 1 || (L->p.zero_copy && L->p.n_cold > 0)) return 0;
    return 4;
}

size_t ffn_workspace(const moe_layer* L, int T) {
    const size_t d = ffn_decode_workspace(T, L->p.k, L->p.H, L->p.I);
    const int terms = mx_terms(L, T);
    if (terms == 0) return d;
    const size_t m = ffn_mx_workspace(T, L->p.k, L->p.H, L->p.I, terms);
    return d > m ? d : m;
}
}  // namespace

int moe_ffn_workspace_bytes(const moe_layer* L, int T, size_t* bytes) {
    if (!L || T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ffn_workspace(L, T);
    return MOE_OK;
}

int moe_layer_set_prefill_kind(moe_layer* L, int kind) {
    if (!L || kind < 0 || kind > 1) return MOE_ERR_INVALID_ARG;
    L->prefill_kind = kind;
    return MOE_OK;
}

int moe_layer_set_decode_kind(moe_layer* L, int kind) {
    if (!L || kind < 0 || kind > 2) return MOE_ERR_INVALID_ARG;
    L->decode_kind = kind;
    return MOE_OK;
}

int moe_grouped_ffn(moe_layer* L, const void* x, int T, const int32_t* phys_ids, const int32_t* counts,
                    const int32_t* offsets, const int32_t* entries, float* y, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (!L || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !phys_ids || !counts || !offsets || !entries || !y || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < ffn_workspace(L, T)) return MOE_ERR_INVALID_ARG;
    if (join_swap(L, S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    FfnArgs a;
    memset(&a, 0, sizeof a);
    a.ptr = L->d_ptr;
    a.tmaps = L->d_tmaps;
    a.loc = L->d_loc;
    a.n_hot = L->p.n_hot;
    a.n_phys = L->p.E;
    a.phys_ids = phys_ids;
    a.counts = counts;
    a.offsets = offsets;
    a.entries = entries;
    a.E = L->p.E;
    a.k = L->p.k;
    a.H = L->p.H;
    a.I = L->p.I;
    a.T = T;
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.y = y;
    a.status = L->d_status;
    a.diag = L->d_diag;
    a.w13s = L->lay.w13s;
    a.w2n = L->lay.w2n;
    a.w2s = L->lay.w2s;
    cudaStream_t st = S(stream);
    // profiled calls record six events: start, end of the work over HBM-resident
    // experts, after the join of the cold gate/up planes, after the cold gate/up
    // phase, after the join of the rest of the copy, end (the events between the
    // joins coincide when no copy is pending)
    cudaEvent_t* pe = L->fprof_n < (int)L->fprof_ev.size() / 6 ? &L->fprof_ev[6 * L->fprof_n++] : nullptr;
    cudaError_t err = cudaSuccess;
    auto mark = [&](int i) {
        if (err == cudaSuccess && pe) err = cudaEventRecord(pe[i], st);
    };
    mark(0);
    // While the cold experts stream over the link (copy, or zero-copy chain) on the
    // layer's copy stream, that stream's CTAs hold copy_ctas SMs: the persistent FFN
    // launches that run meanwhile take the other SMs, so that all their CTAs are
    // resident and they complete as soon as their work does (a launch with CTAs
    // waiting for an SM would end only when the copy frees one, and the next kernel
    // waits for it).
    const int hot_sms = L->sm_count > L->copy_ctas ? L->sm_count - L->copy_ctas : L->sm_count;
    // block-scaled path: x converted to MXFP4 terms once, then per placement class the
    // gate/up kernel (h converted in its epilogue) and the down kernel; otherwise the
    // dequant-GEMV / f16 tensor-core kernels, whose down phase starts with its own h
    // prescale
    const int terms = mx_terms(L, T);
    auto phase = [&](int ph, int sel, int grid, cudaStream_t s, bool zc) -> cudaError_t {
        return terms > 0 ? launch_ffn_mx(a, ph, sel, 0, 1 << 30, terms, grid, s)
                         : launch_ffn_phase(a, ph, sel, grid, s, zc);
    };
    if (err == cudaSuccess) err = terms > 0 ? launch_ffn_mx_prep(a, workspace, terms, st) : launch_ffn_prep(a, workspace, st);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (terms == 0 && L->p.zero_copy && L->p.n_cold > 0 && T <= kTcMinTokens) {
        // zero copy: the cold experts' chain (gate/up, prescale, down) reads their
        // weights in place over the host link on the layer's copy stream, on at least
        // a quarter of the SMs (its kernels stream less per CTA than the copy: 28 CTAs
        // reached 131 GB/s, 38 about 170), while the experts in HBM run on the rest;
        // profiled calls record the cold chain as the layer's copy
        const int zc_ctas = L->copy_ctas > L->sm_count / 4 ? L->copy_ctas : (L->sm_count / 4 > 0 ? L->sm_count / 4 : 1);
        const int zc_hot = L->sm_count > zc_ctas ? L->sm_count - zc_ctas : L->sm_count;
        a.cold_host = L->d_cold_src;
        err = cudaEventRecord(L->ev_fork, st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(L->copy_stream, L->ev_fork, 0);
        const bool prof = L->prof_n < (int)L->prof_ev.size() / 2;
        if (err == cudaSuccess && prof) err = cudaEventRecord(L->prof_ev[2 * L->prof_n], L->copy_stream);
        if (err == cudaSuccess) err = phase(0, 2, zc_ctas, L->copy_stream, true);
        if (err == cudaSuccess) err = phase(1, 2, zc_ctas, L->copy_stream, true);
        if (err == cudaSuccess && prof) {
            err = cudaEventRecord(L->prof_ev[2 * L->prof_n + 1], L->copy_stream);
            ++L->prof_n;
        }
        if (err == cudaSuccess) err = cudaEventRecord(L->ev_join, L->copy_stream);
        if (err == cudaSuccess) err = phase(0, 1, zc_hot, st, false);
        if (err == cudaSuccess) err = phase(1, 1, zc_hot, st, false);
        mark(1);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(st, L->ev_join, 0);
        mark(2);
        mark(3);
        mark(4);
    } else if (L->copy_pending) {
        // experts in HBM first, on the SMs the cold copy leaves free; then the cold
        // experts' gate/up phase once their gate/up planes have landed (beside the copy
        // of their down planes), and their down phase after the whole copy
        err = phase(0, 1, hot_sms, st, false);
        if (err == cudaSuccess) err = phase(1, 1, hot_sms, st, false);
        mark(1);
        if (err == cudaSuccess) err = join_copy_w13(L, st);
        mark(2);
        if (err == cudaSuccess) err = phase(0, 2, hot_sms, st, false);
        mark(3);
        if (err == cudaSuccess) err = join_copy(L, st);
        mark(4);
        if (err == cudaSuccess) err = phase(1, 2, L->sm_count, st, false);
    } else {
        mark(1);
        mark(2);
        mark(3);
        mark(4);
        if (err == cudaSuccess) err = phase(0, 0, L->sm_count, st, false);
        if (err == cudaSuccess) err = phase(1, 0, L->sm_count, st, false);
    }
    mark(5);
    return cuda_status(err);
}

int moe_combine(const float* y, const float* topk_w, int T, int k, int H, void* out, int out_fp32, void* stream) {
    if (T < 0 || k < 1 || k > 32 || H <= 0 || H % 4) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !topk_w || !out || !aligned(y, 16) || !aligned(out, out_fp32 ? 16 : 8)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(y, topk_w, T, k, H, out, out_fp32, S(stream)));
}

// The ranking and pairing of one acting residency update, on the host: cold
// experts picked at least once (count desc, id asc) against hot experts (count
// asc, id asc); pair i swaps while count(cold) > hysteresis * count(hot), at most
// max_swaps pairs, stopping at the first pair that fails. loc_out is the placement
// after the swaps; promoted[i] takes demoted[i]'s HBM slot and demoted[i] takes
// promoted[i]'s cold slot. Returns the number of swaps.
static int plan_residency(const int32_t* cnt, const int32_t* loc, int E, int n_hot, int max_swaps, float hysteresis,
                          int32_t* loc_out, int32_t* promoted, int32_t* demoted) {
    std::vector<int> cold, hot;
    for (int e = 0; e < E; ++e) {
        if (loc[e] >= n_hot) {
            if (cnt[e] >= 1) cold.push_back(e);
        } else {
            hot.push_back(e);
        }
    }
    std::sort(cold.begin(), cold.end(), [&](int a, int b) { return cnt[a] != cnt[b] ? cnt[a] > cnt[b] : a < b; });
    std::sort(hot.begin(), hot.end(), [&](int a, int b) { return cnt[a] != cnt[b] ? cnt[a] < cnt[b] : a < b; });
    const size_t lim = std::min({(size_t)max_swaps, cold.size(), hot.size()});
    std::vector<int32_t> next(loc, loc + E);
    int n = 0;
    for (size_t i = 0; i < lim; ++i) {
        const int a = cold[i], b = hot[i];
        if (!((double)cnt[a] > (double)hysteresis * (double)cnt[b])) break;
        promoted[n] = a;
        demoted[n] = b;
        ++n;
        std::swap(next[a], next[b]);
    }
    std::memcpy(loc_out, next.data(), sizeof(int32_t) * (size_t)E);
    return n;
}

int moe_residency_plan(const int32_t* counts, const int32_t* loc, int E, int n_hot, int max_swaps, float hysteresis,
                       int32_t* loc_out, int32_t* promoted, int32_t* demoted) {
    if (!counts || !loc || !loc_out || E < 1 || E > 1024 || n_hot < 0 || n_hot > E || max_swaps < 0 ||
        max_swaps > kMaxSwaps || !(hysteresis >= 0.0f) || hysteresis > 1e30f)
        return MOE_ERR_INVALID_ARG;
    if (max_swaps > 0 && (!promoted || !demoted)) return MOE_ERR_INVALID_ARG;
    std::vector<char> seen(E, 0);
    for (int e = 0; e < E; ++e) {
        if (counts[e] < 0 || loc[e] < 0 || loc[e] >= E || seen[loc[e]]) return MOE_ERR_INVALID_ARG;
        seen[loc[e]] = 1;
    }
    return plan_residency(counts, loc, E, n_hot, max_swaps, hysteresis, loc_out, promoted, demoted);
}

namespace {
// The plan of the window counts in h_counts from the current placement, kept in
// plan_pro / plan_dem (pair i: promoted, demoted); returns the number of pairs.
int make_plan(moe_layer* L) {
    const moe_params& p = L->p;
    int32_t promoted[kMaxSwaps], demoted[kMaxSwaps];
    std::vector<int32_t> loc(p.E);
    const int n = plan_residency(L->h_counts, L->loc.data(), p.E, p.n_hot, p.max_swaps, p.hysteresis, loc.data(),
                                 promoted, demoted);
    L->plan_pro.assign(promoted, promoted + (n > 0 ? n : 0));
    L->plan_dem.assign(demoted, demoted + (n > 0 ? n : 0));
    L->plan_next = 0;
    L->plan_age = 0;
    return n > 0 ? n : 0;
}

// Applies pairs [i0, i1) of the current plan: the byte moves (in-place exchange, or
// with host copies a copy of the promoted expert into the HBM slot), the cold-source
// table and the placement map.  Every expert is in at most one pair, so the pairs
// commute and any prefix of the plan is a valid placement.  Deferred: on the layer's
// copy stream, forked from `st` (after this layer's FFN, which read the slots) and
// recorded in ev_swap, which the layer's next cold_gather or moe_grouped_ffn waits
// for; the promoted expert is read from its host blob, never from the shared
// scratch (a later layer's copy may overwrite its slot meanwhile).  Otherwise on
// `st`, with h_tag read and the scratch slot used while it holds this layer's copy.
int apply_pairs(moe_layer* L, cudaStream_t st, bool deferred, int i0, int i1) {
    const moe_params& p = L->p;
    if (i1 <= i0) return MOE_OK;
    // the pinned staging buffers are rewritten below
    if (settle_staging(L) != cudaSuccess) return MOE_ERR_CUDA;
    std::vector<int32_t> loc = L->loc;
    SwapList sw;
    sw.n = 0;
    std::vector<int> moved_slots;  // host_mirror: cold slots whose expert changes
    for (int i = i0; i < i1; ++i) {
        const int a = L->plan_pro[i], b = L->plan_dem[i];
        const int slot_h = loc[b];            // HBM slot of the demoted expert
        const int slot_c = loc[a] - p.n_hot;  // cold slot of the promoted expert
        sw.hot[sw.n] = L->hot[slot_h];
        if (p.host_mirror) {
            // promote from the scratch slot if this layer's copy of the expert is still
            // there (synchronous mode only), else from the expert's host copy; the
            // demoted expert's bytes are already in its host copy
            const bool in_scratch = !deferred && L->scratch->h_tag[slot_c] == L->uid;
            sw.host[sw.n] = in_scratch ? L->scratch->base + (size_t)slot_c * L->lay.total : L->mirror_dev[a];
            moved_slots.push_back(slot_c);
        } else {
            sw.host[sw.n] = L->cold_dev[slot_c];
        }
        ++sw.n;
        loc[a] = slot_h;
        loc[b] = p.n_hot + slot_c;
    }
    cudaStream_t xs = deferred ? L->copy_stream : st;
    cudaError_t err = cudaSuccess;
    if (deferred) {
        err = cudaEventRecord(L->ev_fork, st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(xs, L->ev_fork, 0);
    }
    // deferred moves run in the background of later layers' steps, beside their cold
    // copies on the same host link: a sixteenth of the SMs (about a quarter of a cold
    // copy's link rate) still finishes a move long before this layer's next step and
    // leaves the critical-path copies most of the link (measured on 20 layers: 9 CTAs
    // 263 tokens/s, 38 CTAs 217, 4 CTAs 235, 2 CTAs 211)
    const int ctas = deferred ? (L->sm_count / 16 > 0 ? L->sm_count / 16 : 1) : 2 * L->sm_count;
    if (err == cudaSuccess)
        err = p.host_mirror ? launch_copy_list(sw, L->lay.total, ctas, xs) : launch_swap(sw, L->lay.total, ctas, xs);
    if (err == cudaSuccess && p.host_mirror) {
        // each moved cold slot now belongs to the demoted expert: point the copy at its
        // host copy and drop the slot's tag (the scratch holds the promoted one)
        for (int i = i0; i < i1; ++i) {
            const int c = moved_slots[i - i0];
            L->cold_dev[c] = L->mirror_dev[L->plan_dem[i]];
            if (err == cudaSuccess) err = cudaMemsetAsync(L->scratch->d_tag + c, 0xff, sizeof(int32_t), xs);
        }
        std::memcpy(L->h_cold_src, L->cold_dev.data(), sizeof(uint8_t*) * p.n_cold);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(L->d_cold_src, L->h_cold_src, sizeof(uint8_t*) * p.n_cold, cudaMemcpyHostToDevice,
                                  xs);
    }
    std::memcpy(L->h_loc, loc.data(), sizeof(int32_t) * p.E);
    if (err == cudaSuccess) err = cudaMemcpyAsync(L->d_loc, L->h_loc, sizeof(int32_t) * p.E, cudaMemcpyHostToDevice, xs);
    if (err == cudaSuccess) err = cudaEventRecord(L->ev_swap, xs);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    L->swap_recorded = true;
    L->swap_pending = deferred;
    L->loc = loc;
    L->plan_next = i1;
    return MOE_OK;
}
}  // namespace

int residency_update(moe_layer* L, int32_t* n_swaps_out, void* stream) {
    if (!L || !n_swaps_out) return MOE_ERR_INVALID_ARG;
    *n_swaps_out = 0;
    const moe_params& p = L->p;
    cudaStream_t st = S(stream);
    L->steps += 1;
    const bool acting = p.swap_every > 0 && (L->steps % p.swap_every) == 0;
    if (acting && L->fault == 1) {
        L->fault = 0;
        return MOE_ERR_INJECTED;
    }
    int applied = 0;
    if (L->plan_pending) {
        // the previous closing call's snapshot: its copy to h_counts completes behind that
        // call's step, so by now the host rarely waits here, and the GPU never idles.
        // Pairs of the plan before it that are still unapplied land first.
        L->plan_pending = false;
        const int rest = (int)L->plan_pro.size() - L->plan_next;
        int rc = apply_pairs(L, st, true, L->plan_next, (int)L->plan_pro.size());
        if (rc != MOE_OK) return rc;
        applied += rest;
        if (cudaEventSynchronize(L->ev_counts) != cudaSuccess) return MOE_ERR_CUDA;
        make_plan(L);
    }
    const int n_plan = (int)L->plan_pro.size();
    if (L->plan_next < n_plan) {
        // paced: pair i lands at the plan's call floor(i * span / n), span the calls
        // before the next window closes, so that each call moves a few experts while
        // later layers run instead of every layer moving its whole plan at once
        const int span = p.swap_every > 1 ? p.swap_every - 1 : 1;
        const int i0 = L->plan_next;
        int i1 = i0;
        while (i1 < n_plan && (long)i1 * span / n_plan <= L->plan_age) ++i1;
        const int rc = apply_pairs(L, st, true, i0, i1);
        if (rc != MOE_OK) return rc;
        applied += i1 - i0;
    }
    ++L->plan_age;
    if (!acting) {
        *n_swaps_out = applied;
        return MOE_OK;
    }
    cudaError_t err = cudaSuccess;
    if (L->residency_defer) {
        // snapshot the window (its counts go to the host behind this step's work) and
        // count the next window in the other buffer; the plan follows at the next call
        err = cudaMemcpyAsync(L->h_counts, L->d_window, sizeof(int32_t) * p.E, cudaMemcpyDeviceToHost, st);
        if (err == cudaSuccess) err = cudaEventRecord(L->ev_counts, st);
        if (err == cudaSuccess) {
            std::swap(L->d_window, L->d_window_alt);
            err = cudaMemsetAsync(L->d_window, 0, sizeof(int32_t) * p.E, st);
        }
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        L->plan_pending = true;
        *n_swaps_out = applied;
        return MOE_OK;
    }
    // synchronous: read the counters now (this drains the caller's stream), move the
    // bytes on it and clear the window
    err = join_copy(L, st);
    if (err == cudaSuccess) err = join_swap(L, st);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(L->h_counts, L->d_window, sizeof(int32_t) * p.E, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess && p.host_mirror && p.n_cold > 0)
        err = cudaMemcpyAsync(L->scratch->h_tag, L->scratch->d_tag, sizeof(int32_t) * p.n_cold,
                              cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    const int n = make_plan(L);
    const int rc = apply_pairs(L, st, false, 0, n);
    if (rc != MOE_OK) return rc;
    err = cudaMemsetAsync(L->d_window, 0, sizeof(int32_t) * p.E, st);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    *n_swaps_out = applied + n;
    return MOE_OK;
}

int moe_layer_set_residency_defer(moe_layer* L, int defer) {
    if (!L || defer < 0 || defer > 1) return MOE_ERR_INVALID_ARG;
    L->residency_defer = defer;
    return MOE_OK;
}

int moe_layer_get_loc(moe_layer* L, int32_t* loc_host) {
    if (!L || !loc_host) return MOE_ERR_INVALID_ARG;
    // a deferred exchange uploads the map on the layer's copy stream
    if (settle_staging(L) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(cudaMemcpy(loc_host, L->d_loc, sizeof(int32_t) * L->p.E, cudaMemcpyDeviceToHost));
}

int moe_layer_get_counts(moe_layer* L, int32_t* counts_host) {
    if (!L || !counts_host) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemcpy(counts_host, L->d_window, sizeof(int32_t) * L->p.E, cudaMemcpyDeviceToHost));
}

int moe_get_status(moe_layer* L, int* status) {
    if (!L || !status) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemcpy(status, L->d_status, sizeof(int), cudaMemcpyDeviceToHost));
}

int moe_clear_status(moe_layer* L) {
    if (!L) return MOE_ERR_INVALID_ARG;
    cudaError_t e = cudaMemset(L->d_status, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(L->d_diag, 0, sizeof(int) * 16);
    return cuda_status(e);
}

int moe_get_diag(moe_layer* L, int32_t* diag_host) {
    if (!L || !diag_host) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemcpy(diag_host, L->d_diag, sizeof(int32_t) * 16, cudaMemcpyDeviceToHost));
}

const char* moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_NONFINITE: return "non-finite router logit";
        case MOE_ERR_BAD_EXPERT: return "expert id out of range";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_NOMEM: return "out of memory";
        case MOE_ERR_INJECTED: return "injected fault (test hook)";
        case MOE_ERR_SCRATCH_TOO_SMALL: return "batch needs more workspace than the static no-allocation array holds";
        default: return "unknown status";
    }
}

int moe_layer_set_copy_ctas(moe_layer* L, int ctas) {
    if (!L || ctas < 0 || ctas > 64 * 1024) return MOE_ERR_INVALID_ARG;
    L->copy_ctas = ctas > 0 ? ctas : default_copy_ctas(L->sm_count);
    return MOE_OK;
}

int moe_layer_profile(moe_layer* L, int max_records) {
    if (!L || max_records < 0 || max_records > (1 << 20)) return MOE_ERR_INVALID_ARG;
    if (L->copy_stream && cudaStreamSynchronize(L->copy_stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    free_prof(L);
    for (int i = 0; i < 8 * max_records; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) {
            cudaGetLastError();
            free_prof(L);
            return MOE_ERR_CUDA;
        }
        (i < 2 * max_records ? L->prof_ev : L->fprof_ev).push_back(e);
    }
    return MOE_OK;
}

int moe_layer_profile_read(moe_layer* L, float* copy_ms, int max, int* n_out) {
    if (!L || !n_out || max < 0 || (max > 0 && !copy_ms)) return MOE_ERR_INVALID_ARG;
    const int n = L->prof_n < max ? L->prof_n : max;
    for (int i = 0; i < n; ++i) {
        if (cudaEventSynchronize(L->prof_ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&copy_ms[i], L->prof_ev[2 * i], L->prof_ev[2 * i + 1]) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    }
    *n_out = n;
    return MOE_OK;
}

int moe_layer_profile_read_ffn(moe_layer* L, float* ffn_ms, int max, int* n_out) {
    if (!L || !n_out || max < 0 || (max > 0 && !ffn_ms)) return MOE_ERR_INVALID_ARG;
    const int n = L->fprof_n < max ? L->fprof_n : max;
    for (int i = 0; i < n; ++i) {
        const cudaEvent_t* e = &L->fprof_ev[6 * i];
        float part[3] = {0.f, 0.f, 0.f};
        if (cudaEventSynchronize(e[5]) != cudaSuccess || cudaEventElapsedTime(&part[0], e[0], e[1]) != cudaSuccess ||
            cudaEventElapsedTime(&part[1], e[2], e[3]) != cudaSuccess ||
            cudaEventElapsedTime(&part[2], e[4], e[5]) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        ffn_ms[i] = part[0] + part[1] + part[2];
    }
    *n_out = n;
    return MOE_OK;
}

int moe_layer_inject_fault(moe_layer* L, int what) {
    if (!L || what < 0 || what > 1) return MOE_ERR_INVALID_ARG;
    L->fault = what;
    return MOE_OK;
}

int moe_link_probe(const void* src_host, void* dst_dev, size_t bytes, int ctas, void* stream) {
    if (!src_host || !dst_dev || bytes == 0 || bytes % 16 || ctas < 0) return MOE_ERR_INVALID_ARG;
    void* d = mapped_host_ptr(const_cast<void*>(src_host));
    if (!d || !aligned(d, 16) || !aligned(dst_dev, 16) || !is_device_ptr(dst_dev)) return MOE_ERR_INVALID_ARG;
    if (ctas == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        ctas = sms;
    }
    return cuda_status(launch_link_probe(static_cast<const uint8_t*>(d), static_cast<uint8_t*>(dst_dev), bytes, ctas,
                                         S(stream)));
}

int moe_debug_e2m1_pairs(uint32_t* out_dev, void* stream) {
    if (!out_dev) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_debug_e2m1(out_dev, S(stream)));
}

}  // extern "C"
