// gemv.h -- projections of a few rows (gemv.cu): y = x W^T + b for up to three
// weight matrices W_g [N, K] per launch, x [M, K] bf16 with M <= kGemvMaxRows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mha {

constexpr int kGemvMaxRows = 64;

struct GemvParams {
    const __nv_bfloat16* x;          // [M, K]
    const __nv_bfloat16* w[3];       // [N, K] each
    const __nv_bfloat16* bias[3];    // [N] or nullptr
    __nv_bfloat16* out[3];           // head-split [planes, M, dk] or plain [M, N]
    int j0[3];                       // head-split: first plane of this matrix's output
    int M, N, K, ngroups;
    int head_split;
    int dk;                          // head width (64 or 128) of the head-split and cache layouts
    // Key/value caches (decode): when k_cache != nullptr, matrices 1 and 2 write row m
    // (sequence m) into k_cache / v_cache [M, N / dk, L_max, dk] at position
    // cache_len[m] instead of out[1] / out[2]; nothing is written when that position
    // is not below L_max (full cache).
    __nv_bfloat16* k_cache;
    __nv_bfloat16* v_cache;
    const int32_t* cache_len;
    int L_max;
};

bool gemv_supported(int M, int K);   // K in {256, 512, 1024, 2048}, 1 <= M <= kGemvMaxRows
cudaError_t launch_gemv_bf16(const GemvParams& p, cudaStream_t s);

}  // namespace mha
