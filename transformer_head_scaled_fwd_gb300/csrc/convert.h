// convert.h -- element-wise conversions between bf16 and fp32 (convert.cu), used to
// run bf16 problems whose head width the tensor-core kernels do not take on the
// fp32 kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mha {

// dst[i] = float(src[i]) for i < n; src may be nullptr (dst = 0)
cudaError_t launch_bf16_to_f32(const __nv_bfloat16* src, float* dst, long n, cudaStream_t s);
// dst[i] = bf16(src[i]), round to nearest even
cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, long n, cudaStream_t s);

}  // namespace mha
