// Grouped expert FFN for callers that cannot allocate device memory.
//
// Some callers of this layer cannot call cudaMalloc at the point where they run
// it: a serving engine that has handed every free byte of HBM to its own pools
// (KV cache, weights, graph workspaces) and forbids allocations once it serves;
// code that runs while a stream is being captured in global capture mode, where
// allocation calls are not permitted; or embedders whose allocator is not CUDA's.
// moe_grouped_ffn_noalloc gives them the same FFN with its workspace in a
// fixed-size array that lives in the library's own device image, so the call
// allocates nothing.  The method as published has no counterpart of this entry point.
#include <mutex>

#include "internal.cuh"

namespace {

// Workspace of moe_grouped_ffn_noalloc: MOE_NOALLOC_SCRATCH_BYTES, 256-byte aligned,
// one copy per GPU that loads the library, kept until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];  // device address of g_noalloc_scratch per device

}  // namespace

extern "C" int moe_grouped_ffn_noalloc(moe_layer* L, const void* x, int T, const int32_t* phys_ids,
                                       const int32_t* counts, const int32_t* offsets, const int32_t* entries,
                                       float* y, void* stream) {
    if (!L || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    size_t need = 0;
    int rc = moe_ffn_workspace_bytes(L, T, &need);
    if (rc != MOE_OK) return rc;
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_SCRATCH_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_dev[dev]) {
            // host code sees only a stand-in for the array; its device address comes
            // from the runtime, looked up once per device with that device current
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return MOE_ERR_CUDA;
            }
            g_scratch_dev[dev] = p;
        }
        ws = g_scratch_dev[dev];
    }
    return moe_grouped_ffn(L, x, T, phys_ids, counts, offsets, entries, y, ws, (size_t)MOE_NOALLOC_SCRATCH_BYTES,
                           stream);
}
