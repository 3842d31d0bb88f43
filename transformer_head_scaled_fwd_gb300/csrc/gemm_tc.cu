// gemm_tc.cu -- bf16 projection GEMM on the 5th-generation tensor cores.
//
// Computes the nn.Linear layers of MultiHeadedAttention ("003-Transformer"
// tutorial, section "Multi-head attention": four nn.Linear(d_model, d_model)),
// y = x W^T + b with W stored [out, in], for up to three groups per launch
// (the Q, K and V projections). The head split of the same section
// (view(B, L, h, d_k).transpose(1, 2)) is folded into the epilogue: each 64-wide
// column slab of the tile is written by one TMA store straight into its head's
// [L, d_k] plane, so no transpose kernel runs.
//
// CTA = one 128 x 128 output tile of one batch item (tiles never straddle a
// batch boundary). Warp roles:
//   warp 0     TMA producer: A and W k-blocks (64 wide, 128-byte swizzle) into a
//              3-stage shared-memory ring guarded by full/empty mbarriers.
//   warp 1     allocates 128 tensor-memory columns and issues tcgen05.mma
//              (M=128, N=128, K=16) from one thread; tcgen05.commit frees stages.
//   warps 2-5  epilogue: tcgen05.ld the fp32 accumulator, add bias, round to
//              bf16, stage in swizzled shared memory, TMA-store 64-column slabs.
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr uint32_t kTileABytes = kGemmBM * kGemmBK * 2;   // 16 KB
constexpr uint32_t kTileBBytes = kGemmBN * kGemmBK * 2;   // 16 KB
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kTmemCols = 128;

struct GemmSmem {
    // layout after the 1024-aligned stage ring
    uint64_t full[kGemmStages];
    uint64_t empty[kGemmStages];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort_flag;
    float bias[kGemmBN];
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kGemmStages * kStageBytes + sizeof(GemmSmem);

__global__ void __launch_bounds__(kGemmThreads, 2) gemm_bf16_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmSmem* sm = reinterpret_cast<GemmSmem*>(ring + kGemmStages * kStageBytes);

    const int grp = blockIdx.z;
    const GemmGroup& G = p.g[grp];
    const int mt = blockIdx.y;
    if (mt >= G.m_tiles) return;   // whole CTA, before any barrier
    const int b = mt / G.tiles_per_b;
    const int l0 = (mt - b * G.tiles_per_b) * kGemmBM;
    const int n0 = blockIdx.x * kGemmBN;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kblocks = p.K / kGemmBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        mbar_init(&sm->acc_full, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&p.a[grp]);
        tma_prefetch_desc(&p.w[grp]);
        tma_prefetch_desc(&p.out[grp]);
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x >= 64) {
        const int c = threadIdx.x - 64;   // 128 epilogue threads load the bias slice
        const int n = n0 + c;
        sm->bias[c] = (G.bias != nullptr && n < p.N) ? __bfloat162float(G.bias[n]) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int* abort_flag = &sm->abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kGemmStages;
                const uint32_t ph = (kb / kGemmStages) & 1;
                mbar_wait(&sm->empty[s], ph ^ 1, abort_flag, p.status, 0x101);
                uint8_t* a_dst = ring + s * kStageBytes;
                uint8_t* b_dst = a_dst + kTileABytes;
                mbar_arrive_expect_tx(&sm->full[s], kStageBytes);
                tma_load_3d(&p.a[grp], &sm->full[s], a_dst, kb * kGemmBK, l0, b);
                tma_load_2d(&p.w[grp], &sm->full[s], b_dst, kb * kGemmBK, n0);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kGemmBM, kGemmBN, false, false);
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kGemmStages;
                const uint32_t ph = (kb / kGemmStages) & 1;
                mbar_wait(&sm->full[s], ph, abort_flag, p.status, 0x102);
                tc_fence_after();
                const uint32_t a_addr = smem_u32(ring + s * kStageBytes);
                const uint32_t b_addr = a_addr + kTileABytes;
#pragma unroll
                for (int k = 0; k < kGemmBK / 16; ++k) {
                    const uint64_t ad = sdesc_sw128(a_addr + k * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(b_addr + k * 32, 16, 1024);
                    mma_ss(tmem, ad, bd, idesc, (kb | k) != 0);
                }
                tc_commit(&sm->empty[s]);
            }
            tc_commit(&sm->acc_full);
        }
    } else {
        // ---------------- epilogue: warps 2..5, lane quarter = warp % 4
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        mbar_wait(&sm->acc_full, 0, abort_flag, p.status, 0x103);
        __syncwarp();
        tc_fence_after();
        // The ring is idle now (all loads consumed, all MMAs complete): reuse it
        // as the bf16 staging tile, two 64-column slabs of 128 rows x 128 bytes.
        const uint32_t stage_addr = smem_u32(ring);
#pragma unroll
        for (int cb = 0; cb < kGemmBN / 32; ++cb) {
            uint32_t v[32];
            tmem_ld_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cb * 32, v);
            const int slab = cb >> 1;
            const uint32_t slab_addr = stage_addr + slab * (kGemmBM * 128) + row * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = cb * 32 + u * 8 + e * 2;
                    const float x0 = __uint_as_float(v[u * 8 + e * 2]) + sm->bias[c];
                    const float x1 = __uint_as_float(v[u * 8 + e * 2 + 1]) + sm->bias[c + 1];
                    w[e] = pack_bf16x2(x0, x1);
                }
                const int chunk = (cb & 1) * 4 + u;            // 16-byte chunk within the 128-byte row
                const uint32_t addr = slab_addr + ((chunk ^ (row & 7)) << 4);
                st_shared_v4(addr, w[0], w[1], w[2], w[3]);
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (warp == 2 && lane == 0 && !*abort_flag) {
#pragma unroll
            for (int slab = 0; slab < kGemmBN / 64; ++slab) {
                const int n = n0 + slab * 64;
                if (n >= p.N) break;
                const uint8_t* src = ring + slab * (kGemmBM * 128);
                if (p.out_plain)
                    tma_store_3d(&p.out[grp], src, n, l0, b);
                else
                    tma_store_4d(&p.out[grp], src, 0, l0, G.out_j0 + n / 64, b);
            }
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemm_tc(const GemmParams& p, int max_m_tiles, cudaStream_t s) {
    static_assert(kGemmBN == 128 && kGemmBM == 128, "epilogue assumes 128 x 128 tiles");
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kGemmBN - 1) / kGemmBN, max_m_tiles, p.ngroups);
    gemm_bf16_tc_kernel<<<grid, kGemmThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mha
