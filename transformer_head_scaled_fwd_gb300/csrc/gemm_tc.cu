// gemm_tc.cu -- bf16 projection GEMM on the 5th-generation tensor cores.
//
// Computes the nn.Linear layers of MultiHeadedAttention ("003-Transformer"
// tutorial, section "Multi-head attention": four nn.Linear(d_model, d_model)),
// y = x W^T + b with W stored [out, in], for up to three groups per launch
// (the Q, K and V projections), and the two layers of the position-wise FFN
// (same tutorial, feed-forward layer: max(0, x W_1 + b_1) W_2 + b_2). The head split of the same section
// (view(B, L, h, d_k).transpose(1, 2)) is folded into the epilogue: each 64-wide
// column slab of a tile is written by one TMA store straight into its head's
// [L, d_k] plane, so no transpose kernel runs.
//
// Persistent kernel: one CTA per SM walks the output tiles (128 x 256, never
// straddling a batch item) in a static round robin. Warp roles:
//   warp 0     TMA producer: A (128 x 64) and W (256 x 64) k-blocks, 128-byte
//              swizzle, into a 4-stage ring that runs ahead across tiles.
//   warp 1     allocates 512 tensor-memory columns (two 128 x 256 fp32
//              accumulators) and issues tcgen05.mma (M=128, N=256, K=16) from
//              one thread; tcgen05.commit frees ring stages and hands a finished
//              accumulator to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld 64 columns at a time, add the bias (and apply
//              ReLU for the first layer of the position-wise FFN, or the
//              residual of the sublayer connection for W_o), round to
//              bf16, stage in swizzled shared memory (two slab buffers) and
//              TMA-store; the accumulator is released as soon as it is read, so
//              the next tile's MMAs overlap this tile's stores.
#include "gemm_bias.cuh"
#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int BN = kGemmBN;                              // 256
constexpr uint32_t kTileABytes = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr uint32_t kTileBBytes = BN * kGemmBK * 2;       // 32 KB
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kSlabBytes = kGemmBM * 128;           // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;

struct GemmSmem {
    uint64_t full[kGemmStages];
    uint64_t empty[kGemmStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort_flag;
};

// [ring: stages x (A | B)] [2 staging slabs] [GemmSmem]
constexpr uint32_t kOffStage = kGemmStages * kStageBytes;
constexpr uint32_t kOffBar = kOffStage + 2 * kSlabBytes;
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kOffBar + sizeof(GemmSmem);

struct TileCoord {
    int grp, b, l0, n0;
};

__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int tile, int n_tiles) {
    TileCoord c;
    int g = 0;
    while (g + 1 < p.ngroups && tile >= p.g[g].m_tiles * n_tiles) {
        tile -= p.g[g].m_tiles * n_tiles;
        ++g;
    }
    const int mt = tile / n_tiles;
    const int nt = tile - mt * n_tiles;
    c.grp = g;
    c.b = mt / p.g[g].tiles_per_b;
    c.l0 = (mt - c.b * p.g[g].tiles_per_b) * kGemmBM;
    c.n0 = nt * BN;
    return c;
}

// kRes: the instance for launches with a residual (the sublayer's W_o): each slab's residual
// values are requested one slab ahead, like the bias; launches without one keep the lighter epilogue.
// kRelu (the FFN's first layer) and kNarrow (heads narrower than 64 in the head-split store) likewise
// compile their code only into the instances that need it.
template <bool kRes, bool kRelu, bool kNarrow>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmSmem* sm = reinterpret_cast<GemmSmem*>(base + kOffBar);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kblocks = p.K / kGemmBK;
    const int n_tiles = (p.N + BN - 1) / BN;
    int total = 0;
    for (int g = 0; g < p.ngroups; ++g) total += p.g[g].m_tiles * n_tiles;
    MHA_DEVICE_CHECK(gemm_params_ok(p), p.status, 0x1f0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm->acc_full[a], 1);
            mbar_init(&sm->acc_empty[a], 128);
        }
        sm->abort_flag = 0;
        fence_barrier_init();
        for (int g = 0; g < p.ngroups; ++g) {
            tma_prefetch_desc(&p.a[g]);
            tma_prefetch_desc(&p.w[g]);
            tma_prefetch_desc(&p.out[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int* abort_flag = &sm->abort_flag;
    pdl_trigger();
    pdl_wait();   // inputs, bias and residual may come from the previous kernel
    if (p.zero_words != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        // after the wait: every earlier kernel on the stream (an attention launch drawing
        // from this counter included) has completed
        p.zero_words[0] = 0;
        p.zero_words[1] = 0;
    }

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int it = 0;   // ring position across tiles
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                const TileCoord c = tile_coord(p, tile, n_tiles);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % kGemmStages;
                    const uint32_t ph = (it / kGemmStages) & 1;
                    mbar_wait(&sm->empty[s], ph ^ 1, abort_flag, p.status, 0x101);
                    uint8_t* a_dst = base + s * kStageBytes;
                    mbar_arrive_expect_tx(&sm->full[s], kStageBytes);
                    tma_load_3d(&p.a[c.grp], &sm->full[s], a_dst, kb * kGemmBK, c.l0, c.b);
                    tma_load_2d(&p.w[c.grp], &sm->full[s], a_dst + kTileABytes, kb * kGemmBK, c.n0);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kGemmBM, BN, false, false);
            int it = 0, use = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++use) {
                const int acc = use & 1;
                const uint32_t d = tmem + acc * BN;
                mbar_wait(&sm->acc_empty[acc], ((use >> 1) & 1) ^ 1, abort_flag, p.status, 0x104);
                tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % kGemmStages;
                    const uint32_t ph = (it / kGemmStages) & 1;
                    mbar_wait(&sm->full[s], ph, abort_flag, p.status, 0x102);
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(base + s * kStageBytes);
                    const uint32_t b_addr = a_addr + kTileABytes;
#pragma unroll
                    for (int k = 0; k < kGemmBK / 16; ++k)
                        mma_ss(d, sdesc_sw128(a_addr + k * 32, 16, 1024), sdesc_sw128(b_addr + k * 32, 16, 1024),
                               idesc, (kb | k) != 0);
                    tc_commit(&sm->empty[s]);
                }
                tc_commit(&sm->acc_full[acc]);
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5, lane quarter = warp % 4
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const bool issuer = (warp == 2 && lane == 0);
        int use = 0, slabs_issued = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++use) {
            const TileCoord c = tile_coord(p, tile, n_tiles);
            const GemmGroup& G = p.g[c.grp];
            const int acc = use & 1;
            if (G.residual != nullptr && c.l0 + row < G.L) {
                // pull this row's residual (BN bf16 = 4 lines of 128 B) towards L2 while the MMAs run
                const char* rp = reinterpret_cast<const char*>(
                    G.residual + (static_cast<long>(c.b) * G.L + c.l0 + row) * p.N + c.n0);
                const int lines = min(BN, p.N - c.n0) / 64;
                for (int q = 0; q < lines; ++q) asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + q * 128));
            }
            // the first slab's bias is requested before the accumulator is ready, each next
            // slab's while the current one is converted: its load latency stays hidden
            uint4 bias_cur[8];
            load_bias_slab(G.bias, c.n0, p.N, bias_cur);
            // this thread's output row of the residual (nullptr: none, or a row past L)
            const __nv_bfloat16* res_row =
                (kRes && G.residual != nullptr && c.l0 + row < G.L)
                    ? G.residual + (static_cast<long>(c.b) * G.L + c.l0 + row) * p.N
                    : nullptr;
            uint4 res_cur[8];
            if constexpr (kRes) load_residual_slab(res_row, c.n0, p.N, res_cur);
            mbar_wait(&sm->acc_full[acc], (use >> 1) & 1, abort_flag, p.status, 0x103);
            __syncwarp();
            tc_fence_after();
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int slab = 0; slab < BN / 64; ++slab) {
                const int n = c.n0 + slab * 64;
                uint4 bias_next[8];
                load_bias_slab(G.bias, slab + 1 < BN / 64 ? n + 64 : p.N, p.N, bias_next);
                uint4 res_next[8];
                if constexpr (kRes) load_residual_slab(res_row, slab + 1 < BN / 64 ? n + 64 : p.N, p.N, res_next);
                uint32_t v[64];
                tmem_ld_x64(t_row + slab * 64, v);
                if (slab == BN / 64 - 1) {
                    // accumulator fully read: the next tile's MMAs may overwrite it
                    tc_fence_before();
                    mbar_arrive(&sm->acc_empty[acc]);
                }
                if (n >= p.N) {   // uniform across the CTA
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        bias_cur[ch] = bias_next[ch];
                        if constexpr (kRes) res_cur[ch] = res_next[ch];
                    }
                    continue;
                }
                const int sb = slabs_issued & 1;
                // the TMA store that last used this staging buffer must have read it
                if (issuer && slabs_issued >= 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                named_bar_sync(1, 128);
                const uint32_t sbuf = smem_u32(base + kOffStage + sb * kSlabBytes);
                const uint32_t stage = sbuf + row * 128;
                const int nsh = kNarrow ? p.narrow_shift : 0;   // heads narrower than 64: log2(d_k), else 0
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w[4];
                    const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&res_cur[ch]);
                    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bias_cur[ch]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int cc = ch * 8 + 2 * e;
                        const float2 bf = __bfloat1622float2(b2[e]);
                        float y0 = __uint_as_float(v[cc]) + bf.x;
                        float y1 = __uint_as_float(v[cc + 1]) + bf.y;
                        if (kRelu) {
                            y0 = fmaxf(y0, 0.0f);
                            y1 = fmaxf(y1, 0.0f);
                        }
                        if (kRes) {   // residual connection: x + sublayer(...) (zeros past L)
                            const float2 rf = __bfloat1622float2(r2[e]);
                            y0 += rf.x;
                            y1 += rf.y;
                        }
                        w[e] = pack_bf16x2(y0, y1);
                    }
                    // 128-byte swizzled rows, or (narrow heads) dense head-major sub-tiles:
                    // head (8 ch) / d_k at ((head * 128 + row) * d_k + (8 ch) % d_k) * 2
                    const uint32_t dst = nsh ? sbuf + ((((ch * 8) >> nsh) * 128 + row) << (nsh + 1)) +
                                                   (((ch * 8) & ((1 << nsh) - 1)) << 1)
                                             : stage + ((ch ^ (row & 7)) << 4);
                    st_shared_v4(dst, w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (issuer && !*abort_flag) {
                    const uint8_t* src = base + kOffStage + sb * kSlabBytes;
                    if (p.out_plain)
                        tma_store_3d(&p.out[c.grp], src, n, c.l0, c.b);
                    else if (nsh)   // the slab's 64 >> nsh heads, planes from out_j0 + (n/64) * (64 >> nsh)
                        tma_store_4d(&p.out[c.grp], src, 0, c.l0, G.out_j0 + (n / 64) * (64 >> nsh), c.b);
                    else   // slab n/64 of the group: head (n/64) / dk_slabs, half (n/64) % dk_slabs
                        tma_store_5d(&p.out[c.grp], src, 0, (n / 64) % p.dk_slabs, c.l0,
                                     G.out_j0 + (n / 64) / p.dk_slabs, c.b);
                    tma_store_commit();
                }
                ++slabs_issued;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    bias_cur[ch] = bias_next[ch];
                    if constexpr (kRes) res_cur[ch] = res_next[ch];
                }
            }
        }
        if (issuer) tma_store_wait_all();
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

cudaError_t launch_gemm_tc(const GemmParams& p, int /*max_m_tiles*/, cudaStream_t s) {
    static_assert(kGemmBM == 128 && BN == 256, "epilogue assumes 128 x 256 tiles");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    bool res = false;
    for (int g = 0; g < p.ngroups; ++g) res = res || p.g[g].residual != nullptr;
    // the instances the library launches: plain, ReLU (FFN layer 1), narrow heads (Q/K/V), residual (W_o)
    auto* kern = gemm_bf16_tc_kernel<false, false, false>;
    if (p.relu && !res && !p.narrow_shift) kern = gemm_bf16_tc_kernel<false, true, false>;
    else if (p.narrow_shift && !res && !p.relu) kern = gemm_bf16_tc_kernel<false, false, true>;
    else if (res && !p.relu && !p.narrow_shift) kern = gemm_bf16_tc_kernel<true, false, false>;
    else if (res || p.relu || p.narrow_shift) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int n_tiles = (p.N + BN - 1) / BN;
    long total = 0;
    for (int g = 0; g < p.ngroups; ++g) total += static_cast<long>(p.g[g].m_tiles) * n_tiles;
    const int grid = static_cast<int>(total < sms ? total : sms);
    return launch_pdl(kern, dim3(grid), dim3(kGemmThreads), kSmemBytes, s, p);
}

}  // namespace mha
