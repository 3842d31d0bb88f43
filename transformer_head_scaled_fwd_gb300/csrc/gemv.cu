// gemv.cu -- projections of a few rows (incremental decoding: one new token per
// sequence), y = x W^T + b for up to three weight matrices per launch.
//
// With M <= 64 rows the work is reading W once (2 * N * K bytes per matrix), so
// the kernel spreads W over many CTAs instead of tiling M: a CTA computes 8
// output features of one matrix for all rows. Each warp owns 2 features; its
// lanes stream the two W rows with 16-byte loads and multiply them with the x
// rows staged in shared memory as fp32 (16 rows per pass), accumulating 2 x 16
// sums with packed fp32 FMAs. A 5-step butterfly (reduce-scatter over the 32 lanes) leaves lane l with
// the complete sum of (feature l / 16, row l % 16), which it finishes with the
// bias and stores as bf16: head-split [planes, M, 64] (the q of the step),
// straight into the key / value caches at each sequence's current length (k and v
// of the step), or plain [M, N].
#include "gemv.h"
#include "launch.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kGemvWarps = 4;
constexpr int kGemvFeatures = 2 * kGemvWarps;   // per CTA
constexpr int kGemvRows = 16;                   // rows per pass (one butterfly)

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

template <int KC>   // K / 256: 16-byte chunks of W per lane per W row
__global__ void __launch_bounds__(32 * kGemvWarps) gemv_bf16_kernel(const __grid_constant__ GemvParams p) {
    // x rows staged once per pass as fp32, laid out so that lane l's 8 elements of chunk j
    // of row r are two float4 at ((r * KC + j) * 2 + half) * 32 + l: every ld.shared.v4 of
    // a warp reads 512 contiguous bytes
    extern __shared__ float4 xs[];
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = KC * 256;
    const int n0 = blockIdx.x * kGemvFeatures + 2 * warp;   // this warp's features n0, n0 + 1
    const __nv_bfloat16* W = p.w[g];
    pdl_wait();   // x (and the cache lengths) may come from the previous kernel
    // Dependents launch only once every CTA has passed its wait: what the kernels before
    // this one wrote (the cache lengths) is final when they start.
    pdl_trigger();

    // the two W rows as fp32 pairs, all chunks loaded at once (16 bytes per lane per chunk)
    float2 wf[2][KC][4];
#pragma unroll
    for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            const int n = n0 + f;
            const uint4 raw = n < p.N ? *reinterpret_cast<const uint4*>(W + static_cast<long>(n) * K + (j * 32 + lane) * 8)
                                      : make_uint4(0, 0, 0, 0);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) wf[f][j][e] = __bfloat1622float2(h2[e]);
        }

    for (int mb = 0; mb < p.M; mb += kGemvRows) {
        // After the butterfly lane l holds (feature l / 16, row l % 16): its bias and, for
        // the cache writes, its sequence's cache length are requested now so that their
        // latency overlaps the staging and the products.
        const int n_out = n0 + (lane >> 4);
        const int m_out = mb + (lane & 15);
        const float bias_out = (p.bias[g] != nullptr && n_out < p.N) ? __bfloat162float(p.bias[g][n_out]) : 0.0f;
        const int pos_out = (g > 0 && p.k_cache != nullptr && m_out < p.M) ? p.cache_len[m_out] : -1;
        __syncthreads();   // the previous pass has finished reading xs
        {
            // every thread's 16-byte loads of the 16 x rows in flight together
            constexpr int kPer = kGemvRows * KC * 32 / (32 * kGemvWarps);
            uint4 t[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int i = threadIdx.x + u * 32 * kGemvWarps;   // chunk i of the 16 rows: row i / (K/8)
                const int r = i / (K / 8), c = i - r * (K / 8);
                t[u] = (mb + r < p.M) ? *reinterpret_cast<const uint4*>(p.x + static_cast<long>(mb + r) * K + c * 8)
                                      : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int i = threadIdx.x + u * 32 * kGemvWarps;
                const int r = i / (K / 8), c = i - r * (K / 8);   // c = j * 32 + l
                const int j = c >> 5, l = c & 31;
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&t[u]);
                const float2 a = __bfloat1622float2(h2[0]), b = __bfloat1622float2(h2[1]);
                const float2 cc = __bfloat1622float2(h2[2]), d = __bfloat1622float2(h2[3]);
                xs[((r * KC + j) * 2 + 0) * 32 + l] = make_float4(a.x, a.y, b.x, b.y);
                xs[((r * KC + j) * 2 + 1) * 32 + l] = make_float4(cc.x, cc.y, d.x, d.y);
            }
        }
        __syncthreads();
        float2 acc2[2 * kGemvRows];   // index f * 16 + row; the two halves of a packed sum
#pragma unroll
        for (int i = 0; i < 2 * kGemvRows; ++i) acc2[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < KC; ++j) {
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                const float4 xa = xs[((r * KC + j) * 2 + 0) * 32 + lane];
                const float4 xb = xs[((r * KC + j) * 2 + 1) * 32 + lane];
                const float2 x2[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w), make_float2(xb.x, xb.y),
                                      make_float2(xb.z, xb.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc2[r] = ffma2(wf[0][j][e], x2[e], acc2[r]);
                    acc2[kGemvRows + r] = ffma2(wf[1][j][e], x2[e], acc2[kGemvRows + r]);
                }
            }
        }
        float acc[2 * kGemvRows];
#pragma unroll
        for (int i = 0; i < 2 * kGemvRows; ++i) acc[i] = acc2[i].x + acc2[i].y;
        // reduce-scatter: after the step of width s, lane keeps the half of its values
        // selected by (lane & s); at the end acc[0] = total of value index `lane`
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) {
            const bool upper = (lane & s) != 0;
#pragma unroll
            for (int i = 0; i < s; ++i) {
                const float send = upper ? acc[i] : acc[i + s];
                const float keep = upper ? acc[i + s] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
            }
        }
        const int n = n_out;
        const int m = m_out;
        if (n < p.N && m < p.M) {
            const float y = p.bias[g] != nullptr ? acc[0] + bias_out : acc[0];
            if (g > 0 && p.k_cache != nullptr) {   // the step's key / value: straight into the cache
                const int pos = pos_out;
                if (pos >= 0 && pos < p.L_max)
                    (g == 1 ? p.k_cache : p.v_cache)[((static_cast<long>(m) * (p.N / p.dk) + n / p.dk) * p.L_max + pos) *
                                                          p.dk + n % p.dk] = __float2bfloat16_rn(y);
            } else {
                long off;
                if (p.head_split)   // plane j0 + n / dk, row m, column n % dk of [planes, M, dk]
                    off = (static_cast<long>(p.j0[g] + n / p.dk) * p.M + m) * p.dk + n % p.dk;
                else
                    off = static_cast<long>(m) * p.N + n;
                p.out[g][off] = __float2bfloat16_rn(y);
            }
        }
    }
}

}  // namespace

bool gemv_supported(int M, int K) {
    return M >= 1 && M <= kGemvMaxRows && (K == 256 || K == 512 || K == 1024 || K == 2048);
}

template <int KC>
cudaError_t launch_kc(const GemvParams& p, dim3 grid, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(kGemvRows) * KC * 256 * sizeof(float);   // fp32 x rows
    cudaError_t e = cudaFuncSetAttribute(gemv_bf16_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv_bf16_kernel<KC>, grid, dim3(32 * kGemvWarps), smem, s, p);
}

cudaError_t launch_gemv_bf16(const GemvParams& p, cudaStream_t s) {
    dim3 grid((p.N + kGemvFeatures - 1) / kGemvFeatures, p.ngroups);
    switch (p.K / 256) {
        case 1: return launch_kc<1>(p, grid, s);
        case 2: return launch_kc<2>(p, grid, s);
        case 4: return launch_kc<4>(p, grid, s);
        case 8: return launch_kc<8>(p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mha
