// layernorm.cu -- row LayerNorm in front of the attention sublayer.
//
// The residual sublayer of "The Annotated Transformer" (SublayerConnection:
// x + sublayer(norm(x))) normalises its input first. Two forms are on the pages:
//   kind 0  "The Annotated Transformer", LayerNorm:
//           a_2 (x - mean) / (std + eps) + b_2, std unbiased (divide by d - 1)
//   kind 1  nn.LayerNorm ("003-Transformer", SublayerConnection):
//           a (x - mean) / sqrt(var + eps) + b, var biased (divide by d)
// One warp per row; the row stays in registers (d <= 2048), mean and squared
// deviations are two exact passes over the registers with warp-shuffle sums.
// HBM-bound: reads x once, writes y once.
#include "mha_internal.h"

namespace mha {
namespace {

constexpr int kMaxPerLane = 64;   // d <= 2048

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T, int kPer>
__global__ void __launch_bounds__(256) layernorm_kernel(const LayerNormParams p) {
    const long row = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.rows) return;
    const T* x = static_cast<const T*>(p.x) + row * p.d;
    T* y = static_cast<T*>(p.y) + row * p.d;
    const T* a = static_cast<const T*>(p.gain);
    const T* b = static_cast<const T*>(p.bias);
    float v[kPer];
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        v[k] = (i < p.d) ? to_f<T>(x[i]) : 0.0f;
        s += v[k];
    }
    const float mean = warp_sum(s) / p.d;
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        const float c = (i < p.d) ? v[k] - mean : 0.0f;
        ss = fmaf(c, c, ss);
    }
    ss = warp_sum(ss);
    const float denom = p.kind == 0 ? sqrtf(ss / (p.d - 1)) + p.eps : sqrtf(ss / p.d + p.eps);
    const float inv = 1.0f / denom;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        if (i < p.d) {
            const float g = a ? to_f<T>(a[i]) : 1.0f;
            const float o = b ? to_f<T>(b[i]) : 0.0f;
            y[i] = from_f<T>(fmaf(g * (v[k] - mean), inv, o));
        }
    }
}

}  // namespace

int layernorm_max_d() { return 32 * kMaxPerLane; }

template <typename T>
static void launch_t(const LayerNormParams& p, unsigned grid, cudaStream_t s) {
    const int per = (p.d + 31) / 32;
    if (per <= 8)
        layernorm_kernel<T, 8><<<grid, 256, 0, s>>>(p);
    else if (per <= 16)
        layernorm_kernel<T, 16><<<grid, 256, 0, s>>>(p);
    else if (per <= 32)
        layernorm_kernel<T, 32><<<grid, 256, 0, s>>>(p);
    else
        layernorm_kernel<T, 64><<<grid, 256, 0, s>>>(p);
}

cudaError_t launch_layernorm(const LayerNormParams& p, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((p.rows + 7) / 8);
    if (p.bf16)
        launch_t<__nv_bfloat16>(p, grid, s);
    else
        launch_t<float>(p, grid, s);
    return cudaGetLastError();
}

}  // namespace mha
