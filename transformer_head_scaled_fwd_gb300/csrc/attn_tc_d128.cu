// attn_tc_d128.cu -- fused scaled dot-product attention for head width d_k = 128.
//
// Same computation as attn_tc.cu ("The Annotated Transformer", section
// "Attention", attention(): scores / sqrt(d_k), masked_fill(mask == 0, -1e9),
// softmax over keys, P.V; the head's output written into its slab of the
// concatenated context), for heads of width 128 (e.g. d_model 1024 with h = 8).
// CTA = one 128-row query tile of one (batch, head); key tiles of 128.
//
// Each query row is shared by two softmax threads: thread (h, row) of warpgroup h
// takes keys 64 h .. 64 h + 63 of every key tile and keeps its own running max m_h,
// sum l_h and output accumulator O_h = sum over its keys of p V. Softmax is exact
// per half (the online rewrite), and the two halves merge once at the end:
//     M = max(m_0, m_1),  f_h = 2^(m_h - M),
//     out = (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1),
// which is the softmax over all keys of the row (a half whose keys are all masked
// carries the -1e9 fill as its max, so its factor underflows to zero whenever the
// other half has an allowed key, and a fully masked row stays uniform over L_k).
// Two threads per row give each sub-partition two softmax warps and halve each
// warp's chain of loads, maxima, exponentials and stores per key tile, so the
// tensor pipe (S = Q K^T and P.V, 8 MMAs of N = 128 each per key tile) no longer
// waits on a single warp's softmax.
//
// Tensor memory (512 columns):
//   S    [0,128)    fp32 scores of the current key tile (released as soon as both
//                   halves have loaded them: S(j+1) is computed during softmax(j))
//   P    [128,192)  bf16 weights, P_0 (keys 0..63) in [128,160), P_1 in [160,192)
//   O_0  [256,384)  fp32 output accumulator of key half 0 (128 features)
//   O_1  [384,512)  fp32 output accumulator of key half 1
// Shared memory: Q (two 64-wide 128-byte-swizzled halves), K and V rings of 3
// stages (each tile two halves). S = Q K^T is SS-MMA M=128 N=128 (8 k-steps);
// O_h += P_h V_h takes P_h from tensor memory and the 64 value rows of half h
// MN-major with N = 128 (the two 64-wide feature halves are the descriptor's two
// MN blocks, LBO apart): 4 k-steps per half.
// Warps: 0-3 / 4-7 softmax of key half 0 / 1 (one thread per query row), 8 TMA,
// 9 score MMAs (and tensor-memory allocation), 10 P.V MMAs, 11 idle. Registers:
// 168 per thread at launch; the third warpgroup drops to 64 and the softmax
// warpgroups rise to 216 (128*64 + 256*216 = 63488 <= 384*168).
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
constexpr int kThreads = 384;
constexpr uint32_t kHalf = 128 * 128;        // one 128-row x 64-column bf16 half tile = 16 KB
constexpr uint32_t kTile = 2 * kHalf;        // 128 x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColP = 128;              // + 32 h
constexpr uint32_t kColO = 256;              // + 128 h
constexpr float kMaskedLog2 = -1.0e9f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kHeadGroup = 8;

struct Smem128 {
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
    uint64_t s_full, s_free;     // S(j) computed (commit) / loaded by both halves (256 arrivals)
    uint64_t p_full, pv_done;    // P(j) written by both halves (256) / P.V(j) done (commit)
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
        mbar_init(&sm->s_full, 1);
        mbar_init(&sm->s_free, 2 * BM);
        mbar_init(&sm->p_full, 2 * BM);
        mbar_init(&sm->pv_done, 1);
        sm->abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&p.q_map);
        tma_prefetch_desc(&p.kv_map);
        tma_prefetch_desc(&p.ctx_map);
    }
    if (warp == 9) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    volatile int* abort_flag = &sm->abort_flag;

    if (warp >= 8) {
      regs_dec<64>();
      if (warp == 8 && lane == 0) {
        // ------------------------------------------------ TMA producer
        mbar_arrive_expect_tx(&sm->q_full, kTile);
        for (int hf = 0; hf < 2; ++hf)
            tma_load_4d(&p.q_map, &sm->q_full, base + kOffQ + hf * kHalf, 0, hf, q0, q_slab);
        for (int j = 0; j < n; ++j) {
            const int s = j % kStages;
            const uint32_t ph = (j / kStages) & 1;
            mbar_wait(&sm->k_empty[s], ph ^ 1, abort_flag, p.status, 0x401);
            mbar_arrive_expect_tx(&sm->k_full[s], kTile);
            for (int hf = 0; hf < 2; ++hf)
                tma_load_4d(&p.kv_map, &sm->k_full[s], base + kOffK + s * kTile + hf * kHalf, 0, hf, j * BN, k_slab);
            mbar_wait(&sm->v_empty[s], ph ^ 1, abort_flag, p.status, 0x402);
            mbar_arrive_expect_tx(&sm->v_full[s], kTile);
            for (int hf = 0; hf < 2; ++hf)
                tma_load_4d(&p.kv_map, &sm->v_full[s], base + kOffV + s * kTile + hf * kHalf, 0, hf, j * BN, v_slab);
        }
      } else if (warp == 9 && lane == 0) {
        // ------------------------------------------------ score MMAs: S(j) = Q K_j^T
        constexpr uint32_t idesc_s = idesc_bf16(BM, BN, false, false);
        const uint32_t qa = smem_u32(base + kOffQ);
        const uint32_t k_addr = smem_u32(base + kOffK);
        mbar_wait(&sm->q_full, 0, abort_flag, p.status, 0x403);
        for (int j = 0; j < n; ++j) {
            const int s = j % kStages;
            mbar_wait(&sm->k_full[s], (j / kStages) & 1, abort_flag, p.status, 0x404);
            // S is free once both halves have loaded S(j - 1)
            if (j > 0) mbar_wait(&sm->s_free, (j - 1) & 1, abort_flag, p.status, 0x406);
            tc_fence_after();
            const uint32_t ka = k_addr + s * kTile;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
                mma_ss(tmem + kColS, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc_s,
                       k > 0);
            }
            tc_commit(&sm->s_full);
            tc_commit(&sm->k_empty[s]);
        }
      } else if (warp == 10 && lane == 0) {
        // ------------------------------------------------ P.V MMAs: O_h += P_h(j) V_j[keys of half h]
        constexpr uint32_t idesc_o = idesc_bf16(BM, D, false, true);
        const uint32_t v_addr = smem_u32(base + kOffV);
        for (int j = 0; j < n; ++j) {
            const int s = j % kStages;
            mbar_wait(&sm->v_full[s], (j / kStages) & 1, abort_flag, p.status, 0x407);
            mbar_wait(&sm->p_full, j & 1, abort_flag, p.status, 0x408);
            tc_fence_after();
            const uint32_t va = v_addr + s * kTile;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ts(tmem + kColO + h * 128, tmem + kColP + h * 32 + k * 8,
                           sdesc_sw128(va + (4 * h + k) * 2048, kHalf, 1024), idesc_o, (j > 0 || k > 0) ? 1u : 0u);
            tc_commit(&sm->pv_done);
            tc_commit(&sm->v_empty[s]);
        }
      }
      tc_fence_before();
      __syncwarp();
      named_bar_sync(3, kThreads);
      if (warp == 9) {
          __syncwarp();
          tc_fence_after();
          tmem_dealloc(tmem, kTmemCols);
      }
    } else {
        regs_inc<216>();
        // ------------------------------------------------ softmax: thread (h, row), keys 64 h .. 64 h + 63
        const int h = warp >> 2;
        const int row = (warp & 3) * 32 + lane;
        const int qi = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + kColS + h * 64;
        const uint32_t p_tmem = tmem + lane_off + kColP + h * 32;
        const uint32_t o_tmem = tmem + lane_off + kColO + h * 128;
        float m = -CUDART_INF_F;
        float l = 0.0f;
        for (int j = 0; j < n; ++j) {
            mbar_wait(&sm->s_full, j & 1, abort_flag, p.status, 0x409);
            __syncwarp();
            tc_fence_after();
            uint32_t u[64];
            tmem_ld_x64(s_tmem, u);
            tc_fence_before();
            mbar_arrive(&sm->s_free);
            const int k0 = j * BN + h * 64;   // first key of this half
            const bool edge = (p.dense != nullptr) || (k0 + 64 > vl) || (p.causal && k0 + 63 > q0);
            float sc = p.scale_log2;
            if (edge) {
                const int lim = min(vl, p.causal ? qi + 1 : p.Lk) - k0;
                const int oob = p.Lk - k0;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float x = (c < lim) ? __uint_as_float(u[c]) * sc : kMaskedLog2;   // -1e9 fill, after scaling
                    u[c] = __float_as_uint((c < oob) ? x : -CUDART_INF_F);                   // not a key at all
                }
                if (p.dense != nullptr && qi < p.Lq) {
                    const long mrow = (p.dense_mq == 1) ? 0 : qi;
                    const long mq = (p.dense_mq == 1) ? 1 : p.Lq;
                    const uint8_t* mr = p.dense + (static_cast<long>(b) * mq + mrow) * p.Lk + k0;
                    uint32_t keep[2];
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        uint32_t bits = 0;
#pragma unroll 1
                        for (int c = 0; c < 32; ++c)
                            if (32 * w + c >= oob || mr[32 * w + c] != 0) bits |= 1u << c;
                        keep[w] = bits;
                    }
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (!((keep[c >> 5] >> (c & 31)) & 1u)) u[c] = __float_as_uint(kMaskedLog2);
                }
                sc = 1.0f;
            }
            float a4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float a = fmax3(__uint_as_float(u[16 * k]), __uint_as_float(u[16 * k + 1]),
                                __uint_as_float(u[16 * k + 2]));
#pragma unroll
                for (int e = 3; e < 15; e += 2)
                    a = fmax3(a, __uint_as_float(u[16 * k + e]), __uint_as_float(u[16 * k + e + 1]));
                a4[k] = fmaxf(a, __uint_as_float(u[16 * k + 15]));
            }
            const float mt = fmaxf(fmax3(a4[0], a4[1], a4[2]), a4[3]);
            const float m_new = fmaxf(m, mt * sc);
            float alpha = 1.0f;
            bool grow = false;
            if (m == -CUDART_INF_F) {
                m = m_new;   // first keys of this half (-inf while every key so far is past L_k)
            } else {
                grow = (m_new - m) > kRescaleThreshold;
                if (grow) {
                    alpha = ex2_approx(m - m_new);
                    l *= alpha;
                    m = m_new;
                }
            }
            // with no key of this half yet (m = -inf) every weight is exp2(-inf) = 0
            const float mref = (m == -CUDART_INF_F) ? 0.0f : m;
            const float2 sc2 = make_float2(sc, sc);
            const float2 nm2 = make_float2(-mref, -mref);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float2 x = ffma2(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sc2, nm2);
                x.x = ex2_approx(x.x);
                x.y = ex2_approx(x.y);
                acc[c & 3] = fadd2(acc[c & 3], x);
                pk[c] = pack_bf16x2(x.x, x.y);
            }
            const float2 s4 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
            l += s4.x + s4.y;
            if (j > 0) {
                // P and O are busy until P.V(j - 1) has completed
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
            for (int q4 = 0; q4 < 2; ++q4)
                tmem_st_x16_nowait(p_tmem + q4 * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * q4]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm->p_full);
        }
        // ---------------- merge the halves; thread (h, row) writes output features 64 h .. 64 h + 63
        // (m_h, l_h) of every half and row go through the K ring, idle since the last score
        // MMA (completed before this thread's last wait on S)
        float2* ml = reinterpret_cast<float2*>(base + kOffK);
        ml[h * BM + row] = make_float2(m, l);
        mbar_wait(&sm->pv_done, (n - 1) & 1, abort_flag, p.status, 0x40b);
        __syncwarp();
        tc_fence_after();
        named_bar_sync(1, 2 * BM);   // both halves' statistics are in shared memory
        const float2 s0 = ml[row], s1 = ml[BM + row];
        const float M = fmaxf(s0.x, s1.x);
        const float f0 = (s0.x == -CUDART_INF_F) ? 0.0f : ex2_approx(s0.x - M);
        const float f1 = (s1.x == -CUDART_INF_F) ? 0.0f : ex2_approx(s1.x - M);
        const float L = s0.y * f0 + s1.y * f1;
        const float inv = 1.0f / L;
        const float g0 = f0 * inv, g1 = f1 * inv;
        uint32_t o0[64], o1[64];
        tmem_ld_x64(tmem + lane_off + kColO + h * 64, o0);          // O_0, features 64 h ..
        tmem_ld_x64(tmem + lane_off + kColO + 128 + h * 64, o1);    // O_1, features 64 h ..
        // the Q tile is free (every S MMA completed before the last softmax): stage half h there
        const uint32_t stage = smem_u32(base + kOffQ + h * kHalf) + row * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = ch * 8 + 2 * e;
                w[e] = pack_bf16x2(__uint_as_float(o0[c]) * g0 + __uint_as_float(o1[c]) * g1,
                                   __uint_as_float(o0[c + 1]) * g0 + __uint_as_float(o1[c + 1]) * g1);
            }
            st_shared_v4(stage + ((ch ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
        if (h == 0 && p.stats != nullptr && qi < p.Lq) {
            // the row's softmax statistics for p_attn: exp2(u - M) / L is the weight of any key
            float2* st = reinterpret_cast<float2*>(p.stats) + (static_cast<long>(q_slab) * p.Lq + qi);
            *st = make_float2(M, L);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 2 * BM);
        if (warp == 0 && lane == 0 && !*abort_flag) {
            for (int hf = 0; hf < 2; ++hf)
                tma_store_3d(&p.ctx_map, base + kOffQ + hf * kHalf, head * D + hf * 64, q0, b);
            tma_store_commit();
            tma_store_wait_all();
        }
        tc_fence_before();
        named_bar_sync(3, kThreads);
    }
}

}  // namespace

cudaError_t launch_attn_tc_d128(const AttnParams& p, cudaStream_t s) {
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(attn_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.q_pairs) * p.B * p.h;
    return launch_pdl(attn_d128_kernel, dim3(grid), dim3(kThreads), kSmemBytes, s, p);
}

}  // namespace mha
