// attn_tc_d128.cu -- fused scaled dot-product attention for head width d_k = 128.
//
// Same computation as attn_tc.cu ("The Annotated Transformer", section
// "Attention", attention(): scores / sqrt(d_k), masked_fill(mask == 0, -1e9),
// softmax over keys, P.V; the head's output written into its slab of the
// concatenated context), for heads of width 128 (e.g. d_model 1024 with
// h = 8). With d_k = 128 each score costs twice the tensor
// work of d_k = 64 for the same exponential, so one 128-row query tile per CTA
// keeps the tensor pipe busy:
//
// Tensor memory (512 columns):
//   S_0 [0,128) S_1 [128,256)   fp32 scores, double-buffered: S(j+1) is
//                               computed while the softmax of S(j) runs
//   P   [256,320)               bf16 weights, two per column
//   O   [320,448)               fp32 output accumulator (128 features)
// Shared memory: Q (two 64-wide 128-byte-swizzled halves), K and V rings of 3
// stages (each tile two halves). S = Q K^T is SS-MMA M=128 N=128 (8 k-steps);
// O += P V takes P from tensor memory and V MN-major with N = 128 (the two
// 64-wide halves are the descriptor's two MN blocks, LBO apart).
// Warps: 0-3 softmax (one thread per query row), 4 TMA, 5 issues the score MMAs
// (and allocates tensor memory), 6 issues the P.V MMAs, 7 idle. With their own
// issuing thread the score MMAs of tile j + 1 start as soon as the softmax has
// released the buffer, instead of queueing behind the P.V MMAs of tile j - 1.
#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr uint32_t kHalf = 128 * 128;        // one 128-row x 64-column bf16 half tile = 16 KB
constexpr uint32_t kTile = 2 * kHalf;        // 128 x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                // + 128 * buffer
constexpr uint32_t kColP = 256;
constexpr uint32_t kColO = 320;
constexpr float kMaskedLog2 = -1.0e9f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kHeadGroup = 8;

struct Smem128 {
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, pv_done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTile;
constexpr uint32_t kOffV = kOffK + kStages * kTile;
constexpr uint32_t kOffBar = kOffV + kStages * kTile;
constexpr size_t kSmemBytes = 1024 + kOffBar + sizeof(Smem128);

__global__ void __launch_bounds__(kThreads, 1) attn_d128_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem128* sm = reinterpret_cast<Smem128*>(base + kOffBar);
    pdl_trigger();
    pdl_wait();   // Qh, KVh and the mask parts come from earlier kernels

    // (batch, head) pairs in groups of kHeadGroup, longest query tiles first
    const int BH = p.B * p.h;
    const int QT = p.q_pairs;   // query tiles of 128 rows
    const int idx = static_cast<int>(blockIdx.x);
    const int grp = idx / (kHeadGroup * QT);
    const int g_heads = min(kHeadGroup, BH - grp * kHeadGroup);
    const int r = idx - grp * kHeadGroup * QT;
    const int qt = QT - 1 - r / g_heads;
    const int bh = grp * kHeadGroup + r % g_heads;
    MHA_DEVICE_CHECK(bh >= 0 && bh < BH && qt >= 0 && qt < QT && p.Lq >= 1 && p.Lk >= 1 && QT * BM >= p.Lq,
                     p.status, 0x2f1);
    const int b = bh / p.h;
    const int head = bh - b * p.h;
    const int q0 = qt * BM;

    int vl = p.Lk;
    if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[b], 0), p.Lk);
    const bool can_skip = (p.dense == nullptr) && (vl >= 1);
    int kend = can_skip ? vl : p.Lk;
    if (can_skip && p.causal) kend = min(kend, q0 + BM);
    const int n = (kend + BN - 1) / BN;   // >= 1

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q_slab = b * p.h + head;
    const int k_slab = b * 2 * p.h + head;
    const int v_slab = k_slab + p.h;

    if (threadIdx.x == 0) {
        mbar_init(&sm->q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->k_full[s], 1);
            mbar_init(&sm->v_full[s], 1);
            mbar_init(&sm->k_empty[s], 1);
            mbar_init(&sm->v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->s_full[i], 1);
            mbar_init(&sm->s_free[i], BM);
        }
        mbar_init(&sm->p_full, BM);
        mbar_init(&sm->pv_done, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&p.q_map);
        tma_prefetch_desc(&p.kv_map);
        tma_prefetch_desc(&p.ctx_map);
    }
    if (warp == 5) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int* abort_flag = &sm->abort_flag;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm->q_full, kTile);
            for (int hf = 0; hf < 2; ++hf)
                tma_load_4d(&p.q_map, &sm->q_full, base + kOffQ + hf * kHalf, 0, hf, q0, q_slab);
            for (int j = 0; j < n; ++j) {
                const int s = j % kStages;
                const uint32_t ph = (j / kStages) & 1;
                mbar_wait(&sm->k_empty[s], ph ^ 1, abort_flag, p.status, 0x401);
                mbar_arrive_expect_tx(&sm->k_full[s], kTile);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_4d(&p.kv_map, &sm->k_full[s], base + kOffK + s * kTile + hf * kHalf, 0, hf, j * BN,
                                k_slab);
                mbar_wait(&sm->v_empty[s], ph ^ 1, abort_flag, p.status, 0x402);
                mbar_arrive_expect_tx(&sm->v_full[s], kTile);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_4d(&p.kv_map, &sm->v_full[s], base + kOffV + s * kTile + hf * kHalf, 0, hf, j * BN,
                                v_slab);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ score MMAs: S(j) = Q K_j^T into buffer j % 2
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(BM, BN, false, false);
            const uint32_t qa = smem_u32(base + kOffQ);
            const uint32_t k_addr = smem_u32(base + kOffK);
            mbar_wait(&sm->q_full, 0, abort_flag, p.status, 0x403);
            for (int j = 0; j < n; ++j) {
                const int s = j % kStages;
                mbar_wait(&sm->k_full[s], (j / kStages) & 1, abort_flag, p.status, 0x404);
                // the buffer is free once the softmax has loaded S(j - 2)
                if (j >= 2) mbar_wait(&sm->s_free[j & 1], ((j - 2) >> 1) & 1, abort_flag, p.status, 0x406);
                tc_fence_after();
                const uint32_t ka = k_addr + s * kTile;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
                    mma_ss(tmem + kColS + (j & 1) * 128, sdesc_sw128(qa + off, 16, 1024),
                           sdesc_sw128(ka + off, 16, 1024), idesc_s, k > 0);
                }
                tc_commit(&sm->s_full[j & 1]);
                tc_commit(&sm->k_empty[s]);
            }
        }
    } else if (warp == 6) {
        // ------------------------------------------------ P.V MMAs: O += P(j) V_j
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16(BM, D, false, true);
            const uint32_t v_addr = smem_u32(base + kOffV);
            for (int j = 0; j < n; ++j) {
                const int s = j % kStages;
                mbar_wait(&sm->v_full[s], (j / kStages) & 1, abort_flag, p.status, 0x407);
                mbar_wait(&sm->p_full, j & 1, abort_flag, p.status, 0x408);
                tc_fence_after();
                const uint32_t va = v_addr + s * kTile;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ts(tmem + kColO, tmem + kColP + k * 8, sdesc_sw128(va + k * 2048, kHalf, 1024), idesc_o,
                           (j > 0 || k > 0) ? 1u : 0u);
                tc_commit(&sm->pv_done);
                tc_commit(&sm->v_empty[s]);
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------ softmax, one thread per query row
        const int row = warp * 32 + lane;
        const int qi = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t p_tmem = tmem + lane_off + kColP;
        const uint32_t o_tmem = tmem + lane_off + kColO;
        float m = -CUDART_INF_F;
        float l = 0.0f;
        // Scores of the current key tile. The load of the next tile's scores is issued
        // as soon as the exponentials of this one have consumed u, so that its latency
        // (and the wait for S(j + 1)) overlaps the P store and the loop turnaround.
        uint32_t u[128];
        mbar_wait(&sm->s_full[0], 0, abort_flag, p.status, 0x409);
        __syncwarp();
        tc_fence_after();
        tmem_ld_x128_nowait(tmem + lane_off + kColS, u);
        for (int j = 0; j < n; ++j) {
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&sm->s_free[j & 1]);
            const int k0 = j * BN;
            const bool edge = (p.dense != nullptr) || (k0 + BN > vl) || (p.causal && k0 + BN - 1 > q0);
            float sc = p.scale_log2;
            if (edge) {
                const int lim = min(vl, p.causal ? qi + 1 : p.Lk) - k0;
                const int oob = p.Lk - k0;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const float x = (c < lim) ? __uint_as_float(u[c]) * sc : kMaskedLog2;
                    u[c] = __float_as_uint((c < oob) ? x : -CUDART_INF_F);
                }
                if (p.dense != nullptr && qi < p.Lq) {
                    const long mrow = (p.dense_mq == 1) ? 0 : qi;
                    const long mq = (p.dense_mq == 1) ? 1 : p.Lq;
                    const uint8_t* mr = p.dense + (static_cast<long>(b) * mq + mrow) * p.Lk + k0;
                    uint32_t keep[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t bits = 0;
#pragma unroll 1
                        for (int c = 0; c < 32; ++c)
                            if (32 * w + c >= oob || mr[32 * w + c] != 0) bits |= 1u << c;
                        keep[w] = bits;
                    }
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (!((keep[c >> 5] >> (c & 31)) & 1u)) u[c] = __float_as_uint(kMaskedLog2);
                }
                sc = 1.0f;
            }
            float a8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float a = fmax3(__uint_as_float(u[16 * k]), __uint_as_float(u[16 * k + 1]),
                                __uint_as_float(u[16 * k + 2]));
#pragma unroll
                for (int e = 3; e < 15; e += 2)
                    a = fmax3(a, __uint_as_float(u[16 * k + e]), __uint_as_float(u[16 * k + e + 1]));
                a8[k] = fmaxf(a, __uint_as_float(u[16 * k + 15]));
            }
            const float mt = fmax3(fmax3(a8[0], a8[1], a8[2]), fmax3(a8[3], a8[4], a8[5]), fmaxf(a8[6], a8[7]));
            const float m_new = fmaxf(m, mt * sc);
            float alpha = 1.0f;
            bool grow = false;
            if (j == 0) {
                m = m_new;
            } else {
                grow = (m_new - m) > kRescaleThreshold;
                if (grow) {
                    alpha = ex2_approx(m - m_new);
                    l *= alpha;
                    m = m_new;
                }
            }
            const float2 sc2 = make_float2(sc, sc);
            const float2 nm2 = make_float2(-m, -m);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float2 x = ffma2(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sc2, nm2);
                x.x = ex2_approx(x.x);
                x.y = ex2_approx(x.y);
                acc[c & 3] = fadd2(acc[c & 3], x);
                pk[c] = pack_bf16x2(x.x, x.y);
            }
            const float2 s4 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
            l += s4.x + s4.y;
            if (j + 1 < n) {
                mbar_wait(&sm->s_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, p.status, 0x409);
                __syncwarp();
                tc_fence_after();
                tmem_ld_x128_nowait(tmem + lane_off + kColS + ((j + 1) & 1) * 128, u);
            }
            if (j > 0) {
                mbar_wait(&sm->pv_done, (j - 1) & 1, abort_flag, p.status, 0x40a);
                __syncwarp();
                tc_fence_after();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        uint32_t o[16];
                        tmem_ld_x16(o_tmem + q8 * 16, o);
#pragma unroll
                        for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st_x16(o_tmem + q8 * 16, o);
                    }
                }
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_st_x16_nowait(p_tmem + q4 * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * q4]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm->p_full);
        }
        // ---------------- epilogue: O / l -> bf16 -> the head's slab (two 64-column halves) of ctx
        mbar_wait(&sm->pv_done, (n - 1) & 1, abort_flag, p.status, 0x40b);
        __syncwarp();
        tc_fence_after();
        const float inv = 1.0f / l;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t o[64];
            tmem_ld_x64(o_tmem + hf * 64, o);
            // the Q tile is free (every S MMA completed before the last softmax): stage there
            const uint32_t stage = smem_u32(base + kOffQ + hf * kHalf) + row * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(o[ch * 8 + 2 * e]) * inv,
                                       __uint_as_float(o[ch * 8 + 2 * e + 1]) * inv);
                st_shared_v4(stage + ((ch ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
            }
        }
        if (p.stats != nullptr && qi < p.Lq) {
            float2* st = reinterpret_cast<float2*>(p.stats) + (static_cast<long>(q_slab) * p.Lq + qi);
            *st = make_float2(m, l);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, BM);
        if (row == 0 && !*abort_flag) {
            for (int hf = 0; hf < 2; ++hf)
                tma_store_3d(&p.ctx_map, base + kOffQ + hf * kHalf, head * D + hf * 64, q0, b);
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_tc_d128(const AttnParams& p, cudaStream_t s) {
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(attn_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.q_pairs) * p.B * p.h;
    cudaError_t e2 = launch_pdl(attn_d128_kernel, dim3(grid), dim3(kThreads), kSmemBytes, s, p);
    if (e2 != cudaSuccess) return e2;
    return cudaGetLastError();
}

}  // namespace mha
