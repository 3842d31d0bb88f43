// mha_internal.h -- parameter blocks and launchers shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mha {

// Sets the message mha_last_error() returns on this thread.
void set_last_error(const char* msg);

// ------------------------------------------------------------ bf16 tensor-core GEMM
// out[g] = A[g] . W[g]^T + bias[g] for up to three groups (the Q, K and V
// projections share one launch). A[g] is [B, L_g, K]; tiles never straddle two
// batch items, so rows past L_g inside a tile are zero-filled on load and
// clipped on store. Persistent: one CTA per SM walks the tiles.
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;

struct GemmGroup {
    int L;             // rows per batch item
    int tiles_per_b;   // ceil(L / 128)
    int m_tiles;       // B * tiles_per_b
    int out_j0;        // first head plane of this group in a head-split output
    const __nv_bfloat16* bias;       // [N] or nullptr
    const __nv_bfloat16* residual;   // plain output only: [B, L, N] added after the bias, or nullptr
};

struct GemmParams {
    CUtensorMap a[3];     // {K, L, B}, box {64, 128, 1}
    CUtensorMap w[3];     // {K, N},    box {64, 256}
    CUtensorMap out[3];   // head-split {64, d_k/64, L, planes, B} box {64,1,128,1,1}, or plain {N, L, B} box {64,128,1}
    GemmGroup g[3];
    int ngroups;
    int K;
    int N;
    int out_plain;        // 1: plain [B, L, N] output
    int dk_slabs;         // head-split output: d_k / 64 (64-column slabs per head)
    int narrow_shift;     // head-split output of heads narrower than 64: log2(d_k) (3, 4, 5), else 0;
                          // out map {d_k, L, planes, B}, box {d_k, 128, 64/d_k, 1}, unswizzled
    int relu;             // 1: max(0, .) after the bias (first FFN layer)
    int* status;
    int* zero_words;      // or nullptr: 2 ints set to zero (the attention schedule counter of the workspace)
};

// The tile bookkeeping of a GemmParams is consistent: 1 to 3 groups, K a positive
// multiple of 64, N positive, and every group's tiles cover its rows exactly.
__host__ __device__ inline bool gemm_params_ok(const GemmParams& p) {
    if (p.ngroups < 1 || p.ngroups > 3 || p.K <= 0 || p.K % kGemmBK != 0 || p.N <= 0) return false;
    for (int g = 0; g < p.ngroups; ++g) {
        const GemmGroup& G = p.g[g];
        if (G.L <= 0 || G.tiles_per_b != (G.L + kGemmBM - 1) / kGemmBM || G.m_tiles <= 0 ||
            G.m_tiles % G.tiles_per_b != 0)
            return false;
    }
    return p.out_plain != 0 || p.dk_slabs >= 1;
}

size_t gemm_tc_smem_bytes();
cudaError_t launch_gemm_tc(const GemmParams& p, int max_m_tiles, cudaStream_t s);

// ------------------------------------------------------------ bf16 tensor-core attention
constexpr int kAttnBM = 128;       // queries per Q tile
constexpr int kAttnBN = 128;       // keys per K/V tile
constexpr int kAttnD = 64;         // head width d_k
constexpr int kAttnStages = 4;     // K/V ring depth
constexpr int kAttnThreads = 384;  // 2 softmax warpgroups (one per Q tile) + 1 warpgroup: TMA warp, 3 MMA warps

struct AttnParams {
    CUtensorMap q_map;     // Qh as {64, L_q, B*h}
    CUtensorMap kv_map;    // KVh as {64, L_k, B*2h}
    CUtensorMap ctx_map;   // ctx as {d_model, L_q, B} (store)
    int B, h, Lq, Lk;
    int causal;
    const int32_t* valid_lens;
    const uint8_t* dense;
    int dense_mq;
    float* stats;          // [B, h, L_q, 2] (max in log2 units, sum) or nullptr
    float scale_log2;      // log2(e) / sqrt(d_k)
    int q_pairs;           // ceil(L_q / 256)
    int narrow_dk;         // d_k of heads narrower than 64 (8, 16, 32: q_map / kv_map zero-pad
                           // them to 64 columns, ctx_map stores d_k columns unswizzled); 0 otherwise
    float* p_attn;         // p_attn kernel only: fp32 [B, h, L_q, L_k]
    int* status;
    int* sched;            // d_k = 128 kernel: 2 ints in the workspace (next unit, CTAs finished), zero at launch
    // p_attn kernel only: fp32 {L_k, L_q, B*h}, box {32, 128, 1} (when L_k % 4 == 0). Kept last:
    // placed first, it moved the attention kernel's own tensor maps and fields and made that
    // kernel 1.8 % slower on the long workload (0.5205 against 0.5113 ms, same box).
    CUtensorMap p_map;
};

size_t attn_tc_smem_bytes();
cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s);
// d_k = 128: same parameters with q_map / kv_map as {64, 2, L, planes}, q_pairs = ceil(L_q / 128)
// and sched set (persistent: one CTA per SM drawing query tiles from the counter)
cudaError_t launch_attn_tc_d128(const AttnParams& p, cudaStream_t s);

// p_attn for the bf16 path (pattn_tc.cu): the scores recomputed on the tensor cores from
// Qh and KVh (q_map, kv_map as for the attention), normalised with the row statistics
// the attention kernel wrote (stats), written to p_attn. halves: 1 (d_k <= 64), 2 (d_k = 128).
cudaError_t launch_pattn_tc(const AttnParams& p, int halves, cudaStream_t s);

// ------------------------------------------------------------ diagnostics
// One warp waits on an mbarrier nothing arrives on, through the bounded pipeline wait
// with a small budget; on giving up it records `code` in *status (selftest.cu).
cudaError_t launch_wait_timeout_selftest(int* status, int code, cudaStream_t s);

// ------------------------------------------------------------ fp32 SIMT path
struct F32GemmGroup {
    const float* A;      // [B, L, K]
    const float* W;      // [N, K]
    const float* bias;   // [N] or nullptr
    const float* residual;   // plain output only: [B, L, N] added after the bias, or nullptr
    float* out;          // head-split [B, slabs, L, dk] or plain [B, L, N]
    int L;
    int out_j0;
    int slabs;           // head-split output: slabs per batch item of this group's tensor
};
struct F32GemmParams {
    F32GemmGroup g[3];
    int ngroups;
    int B, K, N;
    int dk;
    int out_plain;
    int relu;            // 1: max(0, .) after the bias
};
cudaError_t launch_gemm_f32(const F32GemmParams& p, cudaStream_t s);

struct F32AttnParams {
    const float* q;      // Qh [B, h, Lq, dk]
    const float* kv;     // KVh [B, 2, h, Lk, dk]
    float* ctx;          // [B, Lq, h*dk]
    float* p_attn;       // [B, h, Lq, Lk] or nullptr
    int B, h, Lq, Lk, dk;
    int causal;
    const int32_t* valid_lens;
    const uint8_t* dense;
    int dense_mq;
};
cudaError_t launch_attn_f32(const F32AttnParams& p, cudaStream_t s);

// ------------------------------------------------------------ incremental decoding (d_k = 64 or 128, bf16)
struct DecodeParams {
    const __nv_bfloat16* q_new;    // Qh of the step [1, h, B, dk]
    const __nv_bfloat16* kv_new;   // KVh of the step [1, 2, h, B, dk] (tiled projections only)
    __nv_bfloat16* k_cache;        // [B, h, L_max, dk]
    __nv_bfloat16* v_cache;        // [B, h, L_max, dk]
    int32_t* cache_len;            // [B]; the step's token sits at cache_len[b], counted by the combine kernel
    __nv_bfloat16* ctx;            // [1, B, h * dk]
    float* partial;                // [B * h, n_split, dk + 2]: max (log2 units), sum, o[dk]
    int dk;                        // 64 or 128
    int B, h, L_max, n_split;
    float scale_log2;
    int* status;
    // Keys each attention CTA prefetches into L2 before its wait on the step's projections
    // (0: none). Only set when the kernel before the attention triggers its dependents after
    // its own wait, so that cache_len is final when the attention starts.
    int prefetch_keys;
};
constexpr int kDecodeMaxSplit = 64;
cudaError_t launch_kv_append(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_attention(const DecodeParams& p, cudaStream_t s);

// ------------------------------------------------------------ LayerNorm (rows of length d)
struct LayerNormParams {
    const void* x;       // [rows, d]
    void* y;             // [rows, d]
    const void* gain;    // [d] or nullptr (ones)
    const void* bias;    // [d] or nullptr (zeros)
    long rows;
    int d;
    float eps;
    int kind;            // 0: unbiased std + eps ("The Annotated Transformer"); 1: nn.LayerNorm
    int bf16;            // element type: 1 bf16, 0 fp32
};
int layernorm_max_d();
cudaError_t launch_layernorm(const LayerNormParams& p, cudaStream_t s);

}  // namespace mha
