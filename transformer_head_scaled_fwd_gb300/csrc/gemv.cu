// gemv.cu -- projections of a few rows (incremental decoding: one new token per
// sequence), y = x W^T + b for up to three weight matrices per launch.
//
// With M <= 64 rows the work is reading W once (2 * N * K bytes per matrix), so
// the kernel spreads W over many CTAs instead of tiling M: a CTA computes 8
// output features of one matrix for all rows. Each warp owns 2 features; its
// lanes stream the two W rows with 16-byte loads and multiply them with the x
// rows staged in shared memory (16 rows per pass), accumulating 2 x 16 sums in
// fp32. A 5-step butterfly (reduce-scatter over the 32 lanes) leaves lane l with
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

template <int KC>   // K / 256: 16-byte chunks per lane per W row
__global__ void __launch_bounds__(32 * kGemvWarps) gemv_bf16_kernel(const __grid_constant__ GemvParams p) {
    extern __shared__ uint4 xs[];   // [kGemvRows][K / 8] 16-byte chunks of the staged x rows
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = KC * 256;
    const int n0 = blockIdx.x * kGemvFeatures + 2 * warp;   // this warp's features n0, n0 + 1
    const __nv_bfloat16* W = p.w[g];
    pdl_trigger();
    pdl_wait();   // x (and the cache lengths) may come from the previous kernel

    // the two W rows, all chunks in flight at once (16 bytes per lane per chunk)
    uint4 wv[2][KC];
#pragma unroll
    for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            const int n = n0 + f;
            wv[f][j] = n < p.N ? *reinterpret_cast<const uint4*>(W + static_cast<long>(n) * K + (j * 32 + lane) * 8)
                               : make_uint4(0, 0, 0, 0);
        }

    for (int mb = 0; mb < p.M; mb += kGemvRows) {
        __syncthreads();   // the previous pass has finished reading xs
        {
            // every thread's 16-byte loads of the 16 x rows in flight together
            constexpr int kPer = kGemvRows * KC * 32 / (32 * kGemvWarps);
            uint4 t[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int i = threadIdx.x + u * 32 * kGemvWarps;
                const int r = i / (K / 8), c = i - r * (K / 8);
                t[u] = (mb + r < p.M) ? *reinterpret_cast<const uint4*>(p.x + static_cast<long>(mb + r) * K + c * 8)
                                      : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) xs[threadIdx.x + u * 32 * kGemvWarps] = t[u];
        }
        __syncthreads();
        float acc[2 * kGemvRows];   // index f * 16 + row
#pragma unroll
        for (int i = 0; i < 2 * kGemvRows; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            float w0[8], w1[8];
            bf16x8_to_f32(wv[0][j], w0);
            bf16x8_to_f32(wv[1][j], w1);
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                float xv[8];
                bf16x8_to_f32(xs[r * (K / 8) + j * 32 + lane], xv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    acc[r] = fmaf(w0[e], xv[e], acc[r]);
                    acc[kGemvRows + r] = fmaf(w1[e], xv[e], acc[kGemvRows + r]);
                }
            }
        }
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
        const int n = n0 + (lane >> 4);
        const int m = mb + (lane & 15);
        if (n < p.N && m < p.M) {
            float y = acc[0];
            if (p.bias[g]) y += __bfloat162float(p.bias[g][n]);
            if (g > 0 && p.k_cache != nullptr) {   // the step's key / value: straight into the cache
                const int pos = p.cache_len[m];
                if (pos >= 0 && pos < p.L_max)
                    (g == 1 ? p.k_cache : p.v_cache)[((static_cast<long>(m) * (p.N / 64) + n / 64) * p.L_max + pos) *
                                                          64 + (n & 63)] = __float2bfloat16_rn(y);
            } else {
                long off;
                if (p.head_split)   // plane j0 + n / 64, row m, column n % 64 of [planes, M, 64]
                    off = (static_cast<long>(p.j0[g] + n / 64) * p.M + m) * 64 + (n & 63);
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

cudaError_t launch_gemv_bf16(const GemvParams& p, cudaStream_t s) {
    const int kc = p.K / 256;
    const size_t smem = static_cast<size_t>(kGemvRows) * p.K * 2;
    dim3 grid((p.N + kGemvFeatures - 1) / kGemvFeatures, p.ngroups);
    switch (kc) {
        case 1: return launch_pdl(gemv_bf16_kernel<1>, grid, dim3(32 * kGemvWarps), smem, s, p);
        case 2: return launch_pdl(gemv_bf16_kernel<2>, grid, dim3(32 * kGemvWarps), smem, s, p);
        case 4: return launch_pdl(gemv_bf16_kernel<4>, grid, dim3(32 * kGemvWarps), smem, s, p);
        case 8: {
            cudaError_t e = cudaFuncSetAttribute(gemv_bf16_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            return launch_pdl(gemv_bf16_kernel<8>, grid, dim3(32 * kGemvWarps), smem, s, p);
        }
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mha
