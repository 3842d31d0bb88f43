// simt_f32.cu -- fp32 path of the multi-head attention forward pass.
//
// fp32 storage and fp32 CUDA-core arithmetic (no TF32 tensor cores), for
// workloads that ask for fp32 results within 1e-4 and for any head width
// d_k <= 256. Same stages and workspace layout as the bf16 path:
//   gemm_f32_kernel  nn.Linear y = x W^T + b ("003-Transformer" tutorial,
//                    MultiHeadedAttention), with the head split
//                    (view(B, L, h, d_k).transpose(1, 2)) done by the store
//                    addressing, or a plain [B, L, N] store for W_o.
//   attn_f32_kernel  attention() of "The Annotated Transformer", section
//                    "Attention": scores / sqrt(d_k), masked_fill(mask == 0,
//                    -1e9), softmax over keys, P.V; one warp per query row,
//                    two passes over the keys (row max and sum, then weights);
//                    writes the head's slab of the concatenated context and,
//                    if asked, p_attn.
#include <math_constants.h>

#include "mha_internal.h"

namespace mha {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;   // block tile; 256 threads x (4 x 4) outputs

__global__ void __launch_bounds__(256) gemm_f32_kernel(const __grid_constant__ F32GemmParams p) {
    const F32GemmGroup& G = p.g[blockIdx.z];
    const long M = static_cast<long>(p.B) * G.L;
    const long m0 = static_cast<long>(blockIdx.y) * kTM;
    const int n0 = blockIdx.x * kTN;
    if (m0 >= M) return;
    __shared__ float As[kTK][kTM + 4];
    __shared__ float Ws[kTK][kTN + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < p.K; k0 += kTK) {
        for (int e = threadIdx.x; e < kTM * kTK; e += 256) {
            const int r = e / kTK, c = e % kTK;
            const long m = m0 + r;
            const int k = k0 + c;
            As[c][r] = (m < M && k < p.K) ? G.A[m * p.K + k] : 0.0f;
            const int n = n0 + r;
            Ws[c][r] = (n < p.N && k < p.K) ? G.W[static_cast<long>(n) * p.K + k] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kTK; ++kk) {
            float a[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long m = m0 + ty * 4 + i;
        if (m >= M) continue;
        const long b = m / G.L;
        const long l = m - b * G.L;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= p.N) continue;
            float y = acc[i][j] + (G.bias ? G.bias[n] : 0.0f);
            if (p.relu) y = fmaxf(y, 0.0f);
            if (G.residual) y += G.residual[m * p.N + n];
            if (p.out_plain) {
                G.out[m * p.N + n] = y;
            } else {
                const int slab = G.out_j0 + n / p.dk;
                const int c = n % p.dk;
                G.out[((b * p.slabs + slab) * G.L + l) * p.dk + c] = y;
            }
        }
    }
}

// Few rows (M = B * L <= kSmallM, e.g. the tiny workload's 20 tokens): the tiled kernel
// above would run a handful of CTAs through a long chain of dependent k-steps. Here one
// warp owns one output feature n of one group and all rows: its lanes stream the weight
// row and the input rows (consecutive k per lane, so every load is coalesced) four rows
// at a time, and a butterfly reduction finishes each dot product.
constexpr int kSmallM = 64;
constexpr int kSmallWarps = 8;

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kSmallRows = 16;   // rows accumulated per pass

__global__ void __launch_bounds__(32 * kSmallWarps) gemm_f32_small_m_kernel(const __grid_constant__ F32GemmParams p) {
    const F32GemmGroup& G = p.g[blockIdx.y];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kSmallWarps + warp;
    if (n >= p.N) return;   // whole warp
    const int K = p.K;
    const long M = static_cast<long>(p.B) * G.L;
    const float* __restrict__ A = G.A;
    const float* __restrict__ w = G.W + static_cast<long>(n) * K;
    const float bias = G.bias ? G.bias[n] : 0.0f;
    for (long m0 = 0; m0 < M; m0 += kSmallRows) {
        float acc[kSmallRows];
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) acc[r] = 0.f;
        // unrolled so that the loads of several k-steps are in flight together
        const int rows = static_cast<int>(min(static_cast<long>(kSmallRows), M - m0));
        const float* __restrict__ a0 = A + m0 * K;
#pragma unroll 4
        for (int k = lane; k < K; k += 32) {
            const float wk = __ldg(w + k);
#pragma unroll
            for (int r = 0; r < kSmallRows; ++r)
                if (r < rows) acc[r] = fmaf(__ldg(a0 + static_cast<long>(r) * K + k), wk, acc[r]);
        }
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) acc[r] = warp_sum_f32(acc[r]);
        float mine = 0.f;   // lane r keeps row m0 + r's sum
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r)
            if (lane == r) mine = acc[r];
        if (lane < kSmallRows && m0 + lane < M) {
            const long m = m0 + lane;
            float y = mine + bias;
            if (p.relu) y = fmaxf(y, 0.0f);
            if (G.residual) y += G.residual[m * p.N + n];
            if (p.out_plain) {
                G.out[m * p.N + n] = y;
            } else {
                const long b = m / G.L, l = m - b * G.L;
                const int slab = G.out_j0 + n / p.dk;
                G.out[((b * p.slabs + slab) * G.L + l) * p.dk + n % p.dk] = y;
            }
        }
    }
}

constexpr int kMaxDk = 256;
constexpr int kRowsPerBlock = 8;   // one warp per query row

__device__ __forceinline__ bool allowed_f32(const F32AttnParams& p, int b, int qi, int kj, int vl) {
    if (p.causal && kj > qi) return false;
    if (kj >= vl) return false;
    if (p.dense != nullptr) {
        const long mrow = (p.dense_mq == 1) ? 0 : qi;
        const long mq = (p.dense_mq == 1) ? 1 : p.Lq;
        if (p.dense[(static_cast<long>(b) * mq + mrow) * p.Lk + kj] == 0) return false;
    }
    return true;
}

__global__ void __launch_bounds__(32 * kRowsPerBlock) attn_f32_kernel(const __grid_constant__ F32AttnParams p) {
    __shared__ float qs[kRowsPerBlock][kMaxDk];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int b = bh / p.h, head = bh % p.h;
    const int qi = blockIdx.x * kRowsPerBlock + warp;
    if (qi >= p.Lq) return;   // no block-wide barrier below
    const int dk = p.dk;
    const float* q = p.q + (static_cast<long>(bh) * p.Lq + qi) * dk;
    const float* K = p.kv + (static_cast<long>(b) * 2 * p.h + head) * p.Lk * dk;
    const float* V = p.kv + (static_cast<long>(b) * 2 * p.h + p.h + head) * p.Lk * dk;
    for (int c = lane; c < dk; c += 32) qs[warp][c] = q[c];
    __syncwarp();
    int vl = p.Lk;
    if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[b], 0), p.Lk);
    const float sqrt_dk = sqrtf(static_cast<float>(dk));

    auto score = [&](int kj) {
        const float* kr = K + static_cast<long>(kj) * dk;
        float dot = 0.0f;
        for (int c = 0; c < dk; ++c) dot = fmaf(qs[warp][c], kr[c], dot);
        const float s = dot / sqrt_dk;
        return allowed_f32(p, b, qi, kj, vl) ? s : -1.0e9f;   // fill after scaling
    };

    // pass 1: row max and sum (per lane, then merged)
    float m = -CUDART_INF_F, z = 0.0f;
    for (int kj = lane; kj < p.Lk; kj += 32) {
        const float s = score(kj);
        const float mn = fmaxf(m, s);
        z = z * expf(m - mn) + expf(s - mn);
        m = mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float zo = __shfl_xor_sync(0xffffffffu, z, off);
        const float mn = fmaxf(m, mo);
        const float a = (m == -CUDART_INF_F) ? 0.0f : z * expf(m - mn);
        const float c = (mo == -CUDART_INF_F) ? 0.0f : zo * expf(mo - mn);
        z = a + c;
        m = mn;
    }
    // pass 2: weights, p_attn, and P.V with lanes owning output features
    float o[kMaxDk / 32];
#pragma unroll
    for (int i = 0; i < kMaxDk / 32; ++i) o[i] = 0.0f;
    for (int k0 = 0; k0 < p.Lk; k0 += 32) {
        const int kj = k0 + lane;
        float w = 0.0f;
        if (kj < p.Lk) {
            w = expf(score(kj) - m) / z;
            if (p.p_attn != nullptr) p.p_attn[(static_cast<long>(bh) * p.Lq + qi) * p.Lk + kj] = w;
        }
        const int cnt = min(32, p.Lk - k0);
        for (int t = 0; t < cnt; ++t) {
            const float wt = __shfl_sync(0xffffffffu, w, t);
            const float* vr = V + static_cast<long>(k0 + t) * dk;
#pragma unroll
            for (int i = 0; i < kMaxDk / 32; ++i) {
                const int c = lane + 32 * i;
                if (c < dk) o[i] = fmaf(wt, vr[c], o[i]);
            }
        }
    }
    float* out = p.ctx + (static_cast<long>(b) * p.Lq + qi) * (static_cast<long>(p.h) * dk) + head * dk;
#pragma unroll
    for (int i = 0; i < kMaxDk / 32; ++i) {
        const int c = lane + 32 * i;
        if (c < dk) out[c] = o[i];
    }
}

}  // namespace

cudaError_t launch_gemm_f32(const F32GemmParams& p, cudaStream_t s) {
    int maxL = 0;
    for (int g = 0; g < p.ngroups; ++g) maxL = max(maxL, p.g[g].L);
    const long M = static_cast<long>(p.B) * maxL;
    if (M <= kSmallM) {
        dim3 grid((p.N + kSmallWarps - 1) / kSmallWarps, p.ngroups);
        gemm_f32_small_m_kernel<<<grid, 32 * kSmallWarps, 0, s>>>(p);
        return cudaGetLastError();
    }
    dim3 grid((p.N + kTN - 1) / kTN, static_cast<unsigned>((M + kTM - 1) / kTM), p.ngroups);
    gemm_f32_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attn_f32(const F32AttnParams& p, cudaStream_t s) {
    dim3 grid((p.Lq + kRowsPerBlock - 1) / kRowsPerBlock, p.B * p.h);
    attn_f32_kernel<<<grid, 32 * kRowsPerBlock, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mha
