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
// bf16 rows with d % 256 == 0 move 16 bytes per lane per access.
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

// bf16 rows with d % 256 == 0: 16-byte loads and stores, 8 elements per lane per chunk.
template <int kChunks>
__global__ void __launch_bounds__(256) layernorm_bf16_vec_kernel(const LayerNormParams p) {
    const long row = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.rows) return;
    const uint4* x = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.x) + row * p.d);
    uint4* y = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + row * p.d);
    const uint4* a = reinterpret_cast<const uint4*>(p.gain);
    const uint4* b = reinterpret_cast<const uint4*>(p.bias);
    float v[kChunks][8];
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        const uint4 raw = x[lane + 32 * k];
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            v[k][2 * e] = f.x;
            v[k][2 * e + 1] = f.y;
            s += f.x + f.y;
        }
    }
    const float mean = warp_sum(s) / p.d;
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kChunks; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float c = v[k][e] - mean;
            ss = fmaf(c, c, ss);
        }
    ss = warp_sum(ss);
    const float denom = p.kind == 0 ? sqrtf(ss / (p.d - 1)) + p.eps : sqrtf(ss / p.d + p.eps);
    const float inv = 1.0f / denom;
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        const int c16 = lane + 32 * k;
        uint4 ga = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);   // bf16 1.0 pairs
        uint4 gb = make_uint4(0, 0, 0, 0);
        if (a) ga = a[c16];
        if (b) gb = b[c16];
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&ga);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&gb);
        uint4 o;
        uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(a2[e]);
            const float2 fb = __bfloat1622float2(b2[e]);
            const float y0 = fmaf(fa.x * (v[k][2 * e] - mean), inv, fb.x);
            const float y1 = fmaf(fa.y * (v[k][2 * e + 1] - mean), inv, fb.y);
            __nv_bfloat162 r = __floats2bfloat162_rn(y0, y1);
            o32[e] = *reinterpret_cast<uint32_t*>(&r);
        }
        y[c16] = o;
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
    const bool vec = p.bf16 && p.d % 256 == 0 && p.d <= 2048 &&
                     (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.gain) & 15) == 0 && (reinterpret_cast<uintptr_t>(p.bias) & 15) == 0;
    if (vec) {
        switch (p.d / 256) {
            case 1: layernorm_bf16_vec_kernel<1><<<grid, 256, 0, s>>>(p); break;
            case 2: layernorm_bf16_vec_kernel<2><<<grid, 256, 0, s>>>(p); break;
            case 3: layernorm_bf16_vec_kernel<3><<<grid, 256, 0, s>>>(p); break;
            case 4: layernorm_bf16_vec_kernel<4><<<grid, 256, 0, s>>>(p); break;
            case 5: layernorm_bf16_vec_kernel<5><<<grid, 256, 0, s>>>(p); break;
            case 6: layernorm_bf16_vec_kernel<6><<<grid, 256, 0, s>>>(p); break;
            case 7: layernorm_bf16_vec_kernel<7><<<grid, 256, 0, s>>>(p); break;
            default: layernorm_bf16_vec_kernel<8><<<grid, 256, 0, s>>>(p); break;
        }
    } else if (p.bf16)
        launch_t<__nv_bfloat16>(p, grid, s);
    else
        launch_t<float>(p, grid, s);
    return cudaGetLastError();
}

}  // namespace mha
