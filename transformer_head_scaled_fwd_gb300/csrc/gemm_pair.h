// gemm_pair.h -- the projection GEMM on pairs of SMs (gemm_tc2.cu). Same
// parameters as launch_gemm_tc (mha_internal.h) except that the weight maps'
// box is {64, 128}: each CTA of a pair loads its half of a 256-column tile of W.
#pragma once

#include "mha_internal.h"

namespace mha {

size_t gemm_tc2_smem_bytes();
cudaError_t launch_gemm_tc2(const GemmParams& p, cudaStream_t s);

}  // namespace mha
