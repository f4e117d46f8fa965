// MXFP4 quantisation of bf16 activation rows, for the all-FP4 prefill mode: a
// block-scaled FP4 x FP4 tensor-core product takes both operands in MXFP4, so
// x (and h) must be converted.  The rule is the OCP Microscaling conversion for
// an E2M1 element: each 32-element block gets the shared exponent
// floor(log2(max |v|)) - 2 (2 = the exponent of E2M1's largest value,
// 6 = 1.5 * 2^2), clamped to the E8M0 range [-127, 127] (an all-zero block takes
// -127); each element gets |v| / 2^exp rounded to the nearest E2M1 magnitude
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, above 6 saturating to 6,
// with v's sign bit.  The weights' format ("A 475 GB Model Across Two
// Workstations, With the Table on Disk", Abstract: routed experts in MXFP4) is
// the output layout: element k of a row in byte k/2, low nibble when k is even,
// one scale byte per block.
#include "internal.cuh"
#include "mx.cuh"

namespace {

constexpr int kQuantThreads = 256;  // 8 warps, one 32-element block each

// One warp per block of 32 consecutive elements of the flattened [rows][K] input
// (K a multiple of 32, so blocks never straddle rows): lane i takes element i.
__global__ void __launch_bounds__(kQuantThreads) quant_mxfp4_kernel(const uint16_t* __restrict__ x, long n_blocks,
                                                                    uint8_t* __restrict__ nib,
                                                                    uint8_t* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const long blk = (long)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
    if (blk >= n_blocks) return;  // the same for every lane of the warp
    const uint16_t h = x[blk * 32 + lane];
    const uint32_t mag = (uint32_t)(h & 0x7fffu) << 16;  // |v| as fp32 bits (bf16 widens exactly)
    const uint32_t amax = __reduce_max_sync(0xffffffffu, mag);  // bit order = value order for |v|
    const int e = moe::mx_block_exp(amax);
    const uint32_t code = moe::e2m1_code(moe::mx_scaled(mag, e)) | ((uint32_t)(h >> 15) << 3);
    const uint32_t odd = __shfl_down_sync(0xffffffffu, code, 1);
    if ((lane & 1) == 0) nib[blk * 16 + (lane >> 1)] = (uint8_t)(code | (odd << 4));
    if (lane == 0) scale[blk] = (uint8_t)(e + 127);
}

// Both E2M1 roundings of each value: out[2i] from the hardware pair conversion the
// block-scaled kernels use, out[2i + 1] from the comparison rule (sign in bit 3).
__global__ void e2m1_round_kernel(const float* __restrict__ v, int n, uint32_t* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float x = v[i];
    const uint32_t bits = __float_as_uint(x);
    out[2 * i] = moe::e2m1_pair(x, 0.0f) & 0xFu;
    out[2 * i + 1] = moe::e2m1_code(__uint_as_float(bits & 0x7fffffffu)) | ((bits >> 31) << 3);
}

}  // namespace

extern "C" int moe_debug_e2m1_round(const float* v_dev, int n, uint32_t* out_dev, void* stream) {
    if (n < 0 || (n > 0 && (!v_dev || !out_dev))) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    e2m1_round_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(v_dev, n, out_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_quant_mxfp4(const void* x_bf16, int rows, int K, uint8_t* nib, uint8_t* scales, void* stream) {
    if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x_bf16 || !nib || !scales || (reinterpret_cast<uintptr_t>(x_bf16) & 1u)) return MOE_ERR_INVALID_ARG;
    const long n_blocks = (long)rows * (K / 32);
    const long grid = (n_blocks + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
    if (grid > 0x7fffffffL) return MOE_ERR_INVALID_ARG;
    quant_mxfp4_kernel<<<(unsigned)grid, kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x_bf16), n_blocks, nib, scales);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
