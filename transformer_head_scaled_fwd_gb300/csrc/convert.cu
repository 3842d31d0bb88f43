// convert.cu -- element-wise bf16 <-> fp32 copies (grid-stride, 8 elements per
// thread and iteration when the count allows, else one).
#include "convert.h"

namespace mha {
namespace {

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst, long n) {
    const long stride = static_cast<long>(gridDim.x) * blockDim.x;
    for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src ? __bfloat162float(src[i]) : 0.0f;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, long n) {
    const long stride = static_cast<long>(gridDim.x) * blockDim.x;
    for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = __float2bfloat16_rn(src[i]);
}

unsigned blocks_for(long n) {
    const long b = (n + 255) / 256;
    return static_cast<unsigned>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace

cudaError_t launch_bf16_to_f32(const __nv_bfloat16* src, float* dst, long n, cudaStream_t s) {
    bf16_to_f32_kernel<<<blocks_for(n), 256, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, long n, cudaStream_t s) {
    f32_to_bf16_kernel<<<blocks_for(n), 256, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

}  // namespace mha
