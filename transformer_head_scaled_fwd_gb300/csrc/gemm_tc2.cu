// gemm_tc2.cu -- the projection GEMM of gemm_tc.cu on pairs of SMs.
//
// Same computation and epilogue as gemm_tc.cu (y = x W^T + b for up to three
// groups, bias / ReLU / residual, head-split or plain TMA-stored output: the
// nn.Linear layers of MultiHeadedAttention and of the position-wise FFN in the
// "003-Transformer" tutorial), but a 2-CTA cluster owns a 256 x 256 output tile
// and one tcgen05.mma of M = 256 (cta_group::2) covers both CTAs: each CTA loads
// its own 128 rows of x and its own 128-row half of W, and the tensor cores of
// the pair read each half of W once for both. Per SM this halves the W traffic
// into shared memory and the operand reads of the MMA for W, which leaves room
// for the epilogue's shared-memory staging and TMA stores.
//
// Warp roles (192 threads per CTA, one CTA per SM, persistent over tile pairs):
//   warp 0     TMA producer (both CTAs): x rows and the W half into a 3-stage ring of
//              two k-blocks per stage; each CTA's loads complete on its own "full" barrier.
//   warp 1     both CTAs allocate 512 tensor-memory columns together. Leader CTA
//              (rank 0): one thread issues the MMAs and multicasts its commits to
//              both CTAs' "empty" and "acc_full" barriers. Peer CTA (rank 1): one
//              thread relays each completed stage of its own ring to the leader's
//              "full" barrier (count 2: the leader's own stage and the peer's).
//   warps 2-5  epilogue (both CTAs): each reads its own 128 accumulator rows and
//              releases the accumulator on the leader's "acc_empty" (one arrival
//              per warp of both CTAs: count 8).
// Every wait is bounded; at the end each producer waits for the last releases of
// its ring and both CTAs meet at a cluster barrier before freeing tensor memory.
#include "gemm_bias.cuh"
#include "gemm_pair.h"
#include "launch.h"
#include "ptx_pair.cuh"

namespace mha {
namespace {

constexpr int BN = kGemmBN;                                     // 256 columns per pair tile
// A ring stage holds two 64-wide k-blocks ([x | W half] twice): one full/empty
// barrier round trip (and one relay arrival) per 128 of K instead of per 64.
constexpr int kKbPerStage = 2;
constexpr int kStages = 3;
constexpr uint32_t kTileABytes = kGemmBM * kGemmBK * 2;         // 16 KB: 128 rows of x
constexpr uint32_t kHalfBBytes = (BN / 2) * kGemmBK * 2;        // 16 KB: 128 rows of W
constexpr uint32_t kKbBytes = kTileABytes + kHalfBBytes;
constexpr uint32_t kStageBytes = kKbPerStage * kKbBytes;
constexpr uint32_t kSlabBytes = kGemmBM * 128;                  // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;

struct Gemm2Smem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort_flag;
};

// [ring: stages x (A | B half)] [2 staging slabs] [Gemm2Smem]
constexpr uint32_t kOffStage = kStages * kStageBytes;
constexpr uint32_t kOffBar = kOffStage + 2 * kSlabBytes;
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kOffBar + sizeof(Gemm2Smem);

struct PairCoord {
    int grp, b, l0, n0;
};

// True when every group has the same rows (batch items and length), as the Q, K
// and V projections of one input do.
__device__ __forceinline__ bool groups_share_rows(const GemmParams& p) {
    for (int g = 1; g < p.ngroups; ++g)
        if (p.g[g].L != p.g[0].L || p.g[g].m_tiles != p.g[0].m_tiles || p.g[g].tiles_per_b != p.g[0].tiles_per_b)
            return false;
    return true;
}

// Unit u -> group, batch item, this CTA's first row and the tile's first column.
// A unit is 256 rows (never straddling a batch item) x 256 columns. When the
// groups share their rows, the units of one row pair are consecutive across all
// groups (row pair, then group, then column tile), so the clusters in flight read
// the same rows of the input and each row block comes from DRAM once; otherwise
// the groups follow one another.
__device__ __forceinline__ PairCoord pair_coord(const GemmParams& p, int u, int n_tiles, int rank,
                                                bool shared_rows) {
    int g = 0;
    int pm, nt;
    if (shared_rows) {
        const int per_pm = p.ngroups * n_tiles;
        pm = u / per_pm;
        const int rem = u - pm * per_pm;
        g = rem / n_tiles;
        nt = rem - g * n_tiles;
    } else {
        for (;;) {
            const int bn = p.g[g].m_tiles / p.g[g].tiles_per_b;
            const int units = bn * ((p.g[g].L + 2 * kGemmBM - 1) / (2 * kGemmBM)) * n_tiles;
            if (u < units || g + 1 >= p.ngroups) break;
            u -= units;
            ++g;
        }
        pm = u / n_tiles;
        nt = u - pm * n_tiles;
    }
    const int ptb = (p.g[g].L + 2 * kGemmBM - 1) / (2 * kGemmBM);
    PairCoord c;
    c.grp = g;
    c.b = pm / ptb;
    c.l0 = (pm - c.b * ptb) * 2 * kGemmBM + rank * kGemmBM;
    c.n0 = nt * BN;
    return c;
}

__device__ __forceinline__ int pair_units(const GemmParams& p, int n_tiles) {
    int total = 0;
    for (int g = 0; g < p.ngroups; ++g) {
        const int bn = p.g[g].m_tiles / p.g[g].tiles_per_b;
        total += bn * ((p.g[g].L + 2 * kGemmBM - 1) / (2 * kGemmBM)) * n_tiles;
    }
    return total;
}

// kRes: the instance for launches with a residual (the sublayer's W_o): each slab's residual
// values are requested one slab ahead, like the bias, so their load latency stays off the
// epilogue's path; launches without one keep the lighter epilogue. kRelu (the FFN's first layer)
// and kNarrow (heads narrower than 64 in the head-split store) likewise compile their code only into
// the instances that need it.
template <bool kRes, bool kRelu, bool kNarrow>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc2_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Gemm2Smem* sm = reinterpret_cast<Gemm2Smem*>(base + kOffBar);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int cid = static_cast<int>(blockIdx.x) >> 1;
    const int ncl = static_cast<int>(gridDim.x) >> 1;
    const int kblocks = p.K / kGemmBK;
    const int n_tiles = (p.N + BN - 1) / BN;
    const int total = pair_units(p, n_tiles);
    const bool shared_rows = groups_share_rows(p);
    MHA_DEVICE_CHECK(gemm_params_ok(p), p.status, 0x1f1);   // uniform: both CTAs of a pair return

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], rank == 0 ? 2 : 1);   // leader: own stage + the peer's relay
            mbar_init(&sm->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm->acc_full[a], 1);
            mbar_init(&sm->acc_empty[a], 2 * 4);          // epilogue warps of both CTAs
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
        tmem_alloc_pair(&sm->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();   // barriers of both CTAs initialised, tensor memory allocated
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
        // ---------------- TMA producer (both CTAs)
        if (lane == 0) {
            int it = 0;   // ring position across tiles
            for (int u = cid; u < total; u += ncl) {
                const PairCoord c = pair_coord(p, u, n_tiles, rank, shared_rows);
                for (int kb = 0; kb < kblocks; kb += kKbPerStage, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    const int nk = min(kKbPerStage, kblocks - kb);   // 1 for the last stage of an odd count
                    mbar_wait(&sm->empty[s], ph ^ 1, abort_flag, p.status, 0x111);
                    uint8_t* a_dst = base + s * kStageBytes;
                    mbar_arrive_expect_tx(&sm->full[s], nk * kKbBytes);
                    for (int q = 0; q < nk; ++q) {
                        tma_load_3d(&p.a[c.grp], &sm->full[s], a_dst + q * kKbBytes, (kb + q) * kGemmBK, c.l0, c.b);
                        tma_load_2d(&p.w[c.grp], &sm->full[s], a_dst + q * kKbBytes + kTileABytes, (kb + q) * kGemmBK,
                                    c.n0 + rank * (BN / 2));
                    }
                }
            }
            // the leader's last commits into this CTA's ring have landed
            for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
                mbar_wait(&sm->empty[j % kStages], (j / kStages) & 1, abort_flag, p.status, 0x115);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (leader CTA)
            constexpr uint32_t idesc = idesc_bf16(2 * kGemmBM, BN, false, false);
            int it = 0, use = 0;
            for (int u = cid; u < total; u += ncl, ++use) {
                const int acc = use & 1;
                const uint32_t d = tmem + acc * BN;
                mbar_wait(&sm->acc_empty[acc], ((use >> 1) & 1) ^ 1, abort_flag, p.status, 0x114);
                tc_fence_after();
                for (int kb = 0; kb < kblocks; kb += kKbPerStage, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    const int nk = min(kKbPerStage, kblocks - kb);
                    mbar_wait(&sm->full[s], ph, abort_flag, p.status, 0x112);
                    tc_fence_after();
                    for (int q = 0; q < nk; ++q) {
                        const uint32_t a_addr = smem_u32(base + s * kStageBytes + q * kKbBytes);
                        const uint32_t b_addr = a_addr + kTileABytes;
#pragma unroll
                        for (int k = 0; k < kGemmBK / 16; ++k)
                            mma_ss_pair(d, sdesc_sw128(a_addr + k * 32, 16, 1024),
                                        sdesc_sw128(b_addr + k * 32, 16, 1024), idesc, ((kb + q) | k) != 0);
                    }
                    tc_commit_pair(&sm->empty[s], 0x3);
                }
                tc_commit_pair(&sm->acc_full[acc], 0x3);
            }
        } else if (lane == 0) {
            // ---------------- relay (peer CTA): own stage filled -> one arrival on the leader's
            uint32_t leader_full[kStages];
            for (int s = 0; s < kStages; ++s) leader_full[s] = mapa_shared(smem_u32(&sm->full[s]), 0);
            int it = 0;
            for (int u = cid; u < total; u += ncl)
                for (int kb = 0; kb < kblocks; kb += kKbPerStage, ++it) {
                    const int s = it % kStages;
                    mbar_wait(&sm->full[s], (it / kStages) & 1, abort_flag, p.status, 0x116);
                    mbar_arrive_remote(leader_full[s]);
                }
        }
    } else {
        // ---------------- epilogue: warps 2..5, lane quarter = warp % 4
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const bool issuer = (warp == 2 && lane == 0);
        const uint32_t leader_acc_empty[2] = {mapa_shared(smem_u32(&sm->acc_empty[0]), 0),
                                              mapa_shared(smem_u32(&sm->acc_empty[1]), 0)};
        int use = 0, slabs_issued = 0;
        for (int u = cid; u < total; u += ncl, ++use) {
            const PairCoord c = pair_coord(p, u, n_tiles, rank, shared_rows);
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
            mbar_wait(&sm->acc_full[acc], (use >> 1) & 1, abort_flag, p.status, 0x113);
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
                    // accumulator fully read: the leader's next MMAs may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank == 0)
                            mbar_arrive(&sm->acc_empty[acc]);
                        else
                            mbar_arrive_remote(leader_acc_empty[acc]);
                    }
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
    __syncwarp();
    cluster_sync_all();   // both CTAs done: no more MMAs, commits or remote arrivals in flight
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_tc2_smem_bytes() { return kSmemBytes; }

// Grid: an even number of CTAs (whole clusters), at most one CTA per SM.
cudaError_t launch_gemm_tc2(const GemmParams& p, cudaStream_t s) {
    static_assert(kGemmBM == 128 && BN == 256, "epilogue assumes 128 x 256 tiles per CTA");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    bool res = false;
    for (int g = 0; g < p.ngroups; ++g) res = res || p.g[g].residual != nullptr;
    // the instances the library launches: plain, ReLU (FFN layer 1), narrow heads (Q/K/V), residual (W_o)
    auto* kern = gemm_bf16_tc2_kernel<false, false, false>;
    if (p.relu && !res && !p.narrow_shift) kern = gemm_bf16_tc2_kernel<false, true, false>;
    else if (p.narrow_shift && !res && !p.relu) kern = gemm_bf16_tc2_kernel<false, false, true>;
    else if (res && !p.relu && !p.narrow_shift) kern = gemm_bf16_tc2_kernel<true, false, false>;
    else if (res || p.relu || p.narrow_shift) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int n_tiles = (p.N + BN - 1) / BN;
    long units = 0;
    for (int g = 0; g < p.ngroups; ++g) {
        const long bn = p.g[g].m_tiles / p.g[g].tiles_per_b;
        units += bn * ((p.g[g].L + 2 * kGemmBM - 1) / (2 * kGemmBM)) * n_tiles;
    }
    const long clusters = units < sms / 2 ? units : sms / 2;
    return launch_pdl(kern, dim3(static_cast<unsigned>(2 * clusters)), dim3(kGemmThreads),
                      kSmemBytes, s, p);
}

}  // namespace mha
