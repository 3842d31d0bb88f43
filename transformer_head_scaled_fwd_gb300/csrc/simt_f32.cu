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
//                    if asked, p_attn. attn_f32_short_kernel does the same for
//                    L_k <= 64 from K and V staged in shared memory.
// Every kernel is launched with programmatic dependent launch (launch.h) and waits
// for the previous kernel's results before its first read of them.
#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;   // block tile; 256 threads x (4 x 4) outputs

__global__ void __launch_bounds__(256) gemm_f32_kernel(const __grid_constant__ F32GemmParams p) {
    pdl_trigger();
    pdl_wait();   // the inputs may come from the previous kernel
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
                G.out[((b * G.slabs + slab) * G.L + l) * p.dk + c] = y;
            }
        }
    }
}

// Few rows (M = B * L <= kSmallM, e.g. the tiny workload's 20 tokens): the tiled kernel
// above would run a handful of CTAs through a long chain of dependent k-steps. Here one
// warp owns one output feature n of one group and all rows: the CTA stages up to 16 input
// rows in shared memory with coalesced 16-byte loads, each warp keeps its weight row in
// registers (lane l holds k = l, l + 32, ...) and forms the 16 dot products from shared
// memory, and a butterfly reduction finishes each of them.
constexpr int kSmallM = 64;
constexpr int kSmallWarps = 8;
constexpr int kSmallRows = 16;   // rows per pass
constexpr int kSmallMaxK = 1024; // weight row held in registers: K / 32 <= 32 values per lane

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int KW>   // K / 32: weight values per lane
__global__ void __launch_bounds__(32 * kSmallWarps) gemm_f32_small_m_kernel(const __grid_constant__ F32GemmParams p) {
    extern __shared__ float4 xs4[];   // kSmallRows x K fp32
    float* xs = reinterpret_cast<float*>(xs4);
    pdl_trigger();
    pdl_wait();   // the inputs may come from the previous kernel
    const F32GemmGroup& G = p.g[blockIdx.y];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kSmallWarps + warp;
    constexpr int K = KW * 32;
    const long M = static_cast<long>(p.B) * G.L;
    float w[KW];
#pragma unroll
    for (int i = 0; i < KW; ++i) w[i] = n < p.N ? __ldg(G.W + static_cast<long>(n) * K + i * 32 + lane) : 0.0f;
    const float bias = (G.bias != nullptr && n < p.N) ? G.bias[n] : 0.0f;
    for (long m0 = 0; m0 < M; m0 += kSmallRows) {
        const int rows = static_cast<int>(min(static_cast<long>(kSmallRows), M - m0));
        __syncthreads();   // the previous pass has finished reading xs
        const float4* a4 = reinterpret_cast<const float4*>(G.A + m0 * K);
        for (int e = threadIdx.x; e < rows * K / 4; e += 32 * kSmallWarps) xs4[e] = __ldg(a4 + e);
        __syncthreads();
        if (n >= p.N) continue;   // whole warp; still takes part in the barriers
        float acc[kSmallRows];
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) {
            float a = 0.0f;
            if (r < rows) {
#pragma unroll
                for (int i = 0; i < KW; ++i) a = fmaf(xs[r * K + i * 32 + lane], w[i], a);
            }
            acc[r] = a;
        }
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) acc[r] = warp_sum_f32(acc[r]);
        float mine = 0.f;   // lane r keeps row m0 + r's sum
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r)
            if (lane == r) mine = acc[r];
        if (lane < rows) {
            const long m = m0 + lane;
            float y = mine + bias;
            if (p.relu) y = fmaxf(y, 0.0f);
            if (G.residual) y += G.residual[m * p.N + n];
            if (p.out_plain) {
                G.out[m * p.N + n] = y;
            } else {
                const long b = m / G.L, l = m - b * G.L;
                const int slab = G.out_j0 + n / p.dk;
                G.out[((b * G.slabs + slab) * G.L + l) * p.dk + n % p.dk] = y;
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
    pdl_trigger();
    pdl_wait();   // Qh and KVh come from the projection kernel
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

// Short key ranges (L_k <= 64, K and V of the head fit in shared memory): the CTA stages
// K^T and V of its (batch, head) once; each warp takes one query row with one score per
// lane (keys lane and lane + 32) computed from shared memory, the row's max and sum by
// warp shuffles, and P.V with the lanes owning output features.
constexpr int kShortLk = 64;

__global__ void __launch_bounds__(32 * kRowsPerBlock) attn_f32_short_kernel(const __grid_constant__ F32AttnParams p) {
    extern __shared__ float sh[];   // Kt [dk][kShortLk], V [L_k][dk], q [kRowsPerBlock][dk]
    pdl_trigger();
    pdl_wait();   // Qh and KVh come from the projection kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int b = bh / p.h, head = bh % p.h;
    const int dk = p.dk, Lk = p.Lk;
    float* Kt = sh;
    float* Vs = sh + dk * kShortLk;
    float* qs = Vs + Lk * dk;
    const float* K = p.kv + (static_cast<long>(b) * 2 * p.h + head) * Lk * dk;
    const float* V = p.kv + (static_cast<long>(b) * 2 * p.h + p.h + head) * Lk * dk;
    for (int e = threadIdx.x; e < Lk * dk; e += blockDim.x) {
        const int j = e / dk, c = e - j * dk;
        Kt[c * kShortLk + j] = K[e];
        Vs[e] = V[e];
    }
    const int qi = blockIdx.x * kRowsPerBlock + warp;
    if (qi < p.Lq) {
        const float* q = p.q + (static_cast<long>(bh) * p.Lq + qi) * dk;
        for (int c = lane; c < dk; c += 32) qs[warp * dk + c] = q[c];
    }
    __syncthreads();
    if (qi >= p.Lq) return;   // no barrier below
    int vl = Lk;
    if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[b], 0), Lk);
    const float sqrt_dk = sqrtf(static_cast<float>(dk));
    float s[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int kj = lane + 32 * t;
        s[t] = -CUDART_INF_F;   // not a key
        if (kj < Lk) {
            float dot = 0.0f;
            for (int c = 0; c < dk; ++c) dot = fmaf(qs[warp * dk + c], Kt[c * kShortLk + kj], dot);
            const float sc = dot / sqrt_dk;
            s[t] = allowed_f32(p, b, qi, kj, vl) ? sc : -1.0e9f;   // fill after scaling
        }
    }
    float m = fmaxf(s[0], s[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float e[2], z = 0.0f;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        e[t] = (lane + 32 * t < Lk) ? expf(s[t] - m) : 0.0f;
        z += e[t];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    float w[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        w[t] = e[t] / z;
        const int kj = lane + 32 * t;
        if (p.p_attn != nullptr && kj < Lk) p.p_attn[(static_cast<long>(bh) * p.Lq + qi) * Lk + kj] = w[t];
    }
    float o[kMaxDk / 32];
#pragma unroll
    for (int i = 0; i < kMaxDk / 32; ++i) o[i] = 0.0f;
    for (int kj = 0; kj < Lk; ++kj) {
        const float wt = __shfl_sync(0xffffffffu, kj < 32 ? w[0] : w[1], kj & 31);
#pragma unroll
        for (int i = 0; i < kMaxDk / 32; ++i) {
            const int c = lane + 32 * i;
            if (c < dk) o[i] = fmaf(wt, Vs[kj * dk + c], o[i]);
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

template <int KW>
cudaError_t launch_small(const F32GemmParams& p, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(kSmallRows) * KW * 32 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(gemm_f32_small_m_kernel<KW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kSmallWarps - 1) / kSmallWarps, p.ngroups);
    return launch_pdl(gemm_f32_small_m_kernel<KW>, grid, dim3(32 * kSmallWarps), smem, s, p);
}

cudaError_t launch_gemm_f32(const F32GemmParams& p, cudaStream_t s) {
    int maxL = 0;
    bool aligned = true;   // the small-M kernel reads its input rows as float4
    for (int g = 0; g < p.ngroups; ++g) {
        maxL = max(maxL, p.g[g].L);
        aligned = aligned && (reinterpret_cast<uintptr_t>(p.g[g].A) & 15u) == 0;
    }
    const long M = static_cast<long>(p.B) * maxL;
    if (M <= kSmallM && aligned && p.K % 32 == 0 && p.K <= kSmallMaxK) {
        switch (p.K / 32) {
            case 8: return launch_small<8>(p, s);
            case 16: return launch_small<16>(p, s);
            case 24: return launch_small<24>(p, s);
            case 32: return launch_small<32>(p, s);
            default: break;
        }
    }
    dim3 grid((p.N + kTN - 1) / kTN, static_cast<unsigned>((M + kTM - 1) / kTM), p.ngroups);
    return launch_pdl(gemm_f32_kernel, grid, dim3(256), 0, s, p);
}

cudaError_t launch_attn_f32(const F32AttnParams& p, cudaStream_t s) {
    dim3 grid((p.Lq + kRowsPerBlock - 1) / kRowsPerBlock, p.B * p.h);
    if (p.Lk <= kShortLk && p.dk <= kMaxDk) {
        const size_t smem = sizeof(float) * (static_cast<size_t>(p.dk) * kShortLk + static_cast<size_t>(p.Lk) * p.dk +
                                             static_cast<size_t>(kRowsPerBlock) * p.dk);
        cudaError_t e = cudaFuncSetAttribute(attn_f32_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        return launch_pdl(attn_f32_short_kernel, grid, dim3(32 * kRowsPerBlock), smem, s, p);
    }
    return launch_pdl(attn_f32_kernel, grid, dim3(32 * kRowsPerBlock), 0, s, p);
}

}  // namespace mha
