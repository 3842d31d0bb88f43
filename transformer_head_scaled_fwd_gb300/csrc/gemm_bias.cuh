// gemm_bias.cuh -- bias vectors for the epilogues of the projection GEMMs (gemm_tc.cu,
// gemm_tc2.cu): y = x W^T + b of the nn.Linear layers ("003-Transformer" tutorial,
// section "Multi-head attention" and the position-wise FFN).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace mha {

// The 64 bias values of the output columns [n, n + 64) as eight 16-byte vectors
// (zero without a bias, and for columns at or past N).
__device__ __forceinline__ void load_bias_slab(const __nv_bfloat16* bias, int n, int N, uint4 (&dst)[8]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        dst[ch] = (bias != nullptr && n + ch * 8 < N) ? *reinterpret_cast<const uint4*>(bias + n + ch * 8)
                                                      : make_uint4(0, 0, 0, 0);
}

// The 64 residual values of one output row at columns [n, n + 64) as eight 16-byte vectors
// (zero when the row has no residual, i.e. row == nullptr, and for columns at or past N).
__device__ __forceinline__ void load_residual_slab(const __nv_bfloat16* row, int n, int N, uint4 (&dst)[8]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        dst[ch] = (row != nullptr && n + ch * 8 < N) ? *reinterpret_cast<const uint4*>(row + n + ch * 8)
                                                     : make_uint4(0, 0, 0, 0);
}

}  // namespace mha
