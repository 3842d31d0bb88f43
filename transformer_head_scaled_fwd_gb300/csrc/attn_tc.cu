// attn_tc.cu -- fused scaled dot-product attention on the 5th-generation tensor cores.
//
// Per (batch, head) it computes "The Annotated Transformer", section
// "Attention", attention():
//     scores = Q K^T / sqrt(d_k);  scores.masked_fill(mask == 0, -1e9);
//     p_attn = softmax(scores, dim=-1);  head = p_attn V
// and writes the head's output into its d_k-wide column slab of the
// concatenated context [B, L_q, h*d_k] ("003-Transformer" tutorial,
// MultiHeadedAttention.forward: transpose(1, 2).contiguous().view(B, -1, h*d_k)),
// so the concat is a strided TMA store and no transpose kernel runs.
//
// The softmax is taken online over key tiles (running row max m and row sum l,
// the accumulated output rescaled when m grows), which is an exact rewrite of
// softmax-then-matmul: the L_q x L_k score matrix never leaves the chip.
//
// CTA = two 128-row query tiles (t = 0, 1) of one (batch, head); key tiles of 128
// (when L_q <= 128 the two tiles belong to two consecutive (batch, head) pairs).
// Tensor memory (512 columns, no aliasing):
//   S_0 [0,128)  S_1 [128,256)   fp32 scores
//   P_0 [256,320) P_1 [320,384)  bf16 weights, two per column (A operand of P.V)
//   O_0 [384,448) O_1 [448,512)  fp32 output accumulators
// Because P has its own columns, the next score tile S_t(j+1) is computed while
// the softmax of tile j is still running: the softmax releases S_t as soon as
// it has loaded it, and only waits for P.V(j-1) (to reuse P_t / rescale O_t).
// Warp roles:
//   warps 0-3 / 4-7   softmax for query tile 0 / 1: one thread per query row.
//                     tcgen05.ld the score row, release S, scale to log2 units,
//                     apply the -1e9 fill, update (m, l), rescale O when m grows
//                     by more than 2^8 (lazy: exact, the final O / l uses the
//                     same m), write P with tcgen05.st.
//   warp 8            TMA: K and V tiles through a 4-deep ring (Q and the ring's
//                     first four K/V tiles are issued by thread 0 right after it
//                     has initialised the barriers, before the tensor-memory
//                     allocation and the register split).
//   warp 9            issues S_t = Q_t K^T for both tiles (SS, M=128, N=128)
//                     and allocates the tensor memory.
//   warps 10 / 11     issue O_t += P_t V for tile 0 / 1 (A from tensor memory,
//                     V MN-major, M=128, N=64).
// The score MMAs have their own issuing thread so that S_t(j+1) enters the
// tensor pipe as soon as the softmax has loaded S_t(j), instead of queueing
// behind the P.V MMAs, whose issue the busy pipe holds back.
// Registers: launched at 168 per thread (384 threads); the third warpgroup
// drops to 64 and the two softmax warpgroups rise to 216
// (128*64 + 256*216 = 63488 <= 384*168 = 64512, the launch total).
#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr uint32_t kTileBytes = 128 * 128;          // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // + 128 t
constexpr uint32_t kColP = 256;    // + 64 t
constexpr uint32_t kColO = 384;    // + 64 t
constexpr float kMaskedLog2 = -1.0e9f * 1.4426950408889634f;   // the -1e9 fill, in log2 units
constexpr float kRescaleThreshold = 8.0f;           // lazy rescale: only when m grows by > 2^8
constexpr int kHeadGroup = 8;                       // (batch, head) pairs scheduled together

struct AttnSmem {
    uint64_t q_full;
    uint64_t k_full[kAttnStages];
    uint64_t v_full[kAttnStages];
    uint64_t k_empty[kAttnStages];
    uint64_t v_empty[kAttnStages];
    uint64_t s_full[2];    // S_t(j) computed                      (tcgen05.commit)
    uint64_t s_free[2];    // S_t(j) loaded by the softmax         (128 arrivals)
    uint64_t p_full[2];    // P_t(j) written, O_t rescaled         (128 arrivals)
    uint64_t pv_done[2];   // P_t(j).V done: P_t free, O_t stable  (tcgen05.commit)
    uint32_t tmem_base;
    int abort_flag;
};

// [Q0 | Q1 | K ring | V ring | AttnSmem], tiles 1024-aligned.
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kAttnStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kAttnStages * kTileBytes;
constexpr size_t kSmemBytes = 1024 + kOffBar + sizeof(AttnSmem);

struct TileWork {
    int n;          // key tiles this query tile processes
    bool active;    // query tile has rows < L_q
};

// kShortKeys: the instance for short key ranges (L_k <= kShortKeysMax), where most key
// tiles are cut by the causal or valid-length mask and take the one-select fill
// below; long key ranges use the instance without that branch in the hot loop.
constexpr int kShortKeysMax = 1024;
// kTwo: the instance for query ranges of one tile (L_q <= 128, with short key
// ranges): the CTA's second query tile takes the next (batch, head) pair instead of
// staying idle, each pair with its own K/V ring stages (tile t uses the stages of
// parity t), so the launch has half as many CTAs.

template <bool kShortKeys, bool kTwo>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_bf16_tc_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    AttnSmem* sm = reinterpret_cast<AttnSmem*>(base + kOffBar);
    pdl_trigger();
    pdl_wait();   // Qh, KVh and the mask parts come from earlier kernels

    // Block order: (batch, head) pairs in groups of kHeadGroup, so the CTAs in
    // flight share the K/V of a few heads in L2; inside a group, longest first
    // (with the causal mask the last query tiles carry the most key tiles).
    const int BH = p.B * p.h;
    const int QP = p.q_pairs;
    const int idx = static_cast<int>(blockIdx.x);
    int qp, bh;
    if constexpr (kTwo) {
        qp = 0;
        bh = 2 * idx;
    } else {
        const int grp = idx / (kHeadGroup * QP);
        const int g_heads = min(kHeadGroup, BH - grp * kHeadGroup);
        const int r = idx - grp * kHeadGroup * QP;
        qp = QP - 1 - r / g_heads;
        bh = grp * kHeadGroup + r % g_heads;
    }
    MHA_DEVICE_CHECK(bh >= 0 && bh < BH && qp >= 0 && qp < QP && p.Lq >= 1 && p.Lk >= 1 &&
                         QP * 2 * kAttnBM >= p.Lq,
                     p.status, 0x2f0);
    const int b = bh / p.h;
    const int head = bh - b * p.h;
    const int q0 = qp * 2 * kAttnBM;
    // two-head instance: (batch, head) pair of query tile 1
    const bool two_on = kTwo && bh + 1 < BH;
    const int bh1 = two_on ? bh + 1 : bh;
    const int b1 = bh1 / p.h;
    const int head1 = bh1 - b1 * p.h;

    // Key range. With at least one allowed key per row (valid length >= 1 and
    // no dense mask), key tiles that are fully masked for every row of a query
    // tile add exactly zero and are skipped. Otherwise every key is visited, so
    // that a fully masked row comes out uniform over all L_k keys.
    int vl = p.Lk;
    if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[b], 0), p.Lk);
    const bool can_skip = (p.dense == nullptr) && (vl >= 1);
    int vl1 = vl;
    if (kTwo && p.valid_lens != nullptr) vl1 = min(max(p.valid_lens[b1], 0), p.Lk);
    const bool can_skip1 = (p.dense == nullptr) && (vl1 >= 1);
    TileWork tw[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt0 = kTwo ? 0 : q0 + t * kAttnBM;
        const int vlt = (kTwo && t == 1) ? vl1 : vl;
        const bool skt = (kTwo && t == 1) ? can_skip1 : can_skip;
        tw[t].active = qt0 < p.Lq && (!kTwo || t == 0 || two_on);
        int kend = skt ? vlt : p.Lk;
        if (skt && p.causal) kend = min(kend, qt0 + kAttnBM);
        tw[t].n = tw[t].active ? (kend + kAttnBN - 1) / kAttnBN : 0;
    }
    const int n_all = max(tw[0].n, tw[1].n);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q_slab = b * p.h + head;
    const int k_slab = b * 2 * p.h + head;
    const int v_slab = k_slab + p.h;
    const int q_slab1 = b1 * p.h + head1;
    const int k_slab1 = b1 * 2 * p.h + head1;
    const int v_slab1 = k_slab1 + p.h;
    // two-head instance: stage use g = 2 j + t holds key tile j of query tile t's pair
    auto load_kv2 = [&](int g) {
        const int t = g & 1, j = g >> 1, s = g % kAttnStages;
        mbar_arrive_expect_tx(&sm->k_full[s], kTileBytes);
        tma_load_3d(&p.kv_map, &sm->k_full[s], base + kOffK + s * kTileBytes, 0, j * kAttnBN, t ? k_slab1 : k_slab);
        mbar_arrive_expect_tx(&sm->v_full[s], kTileBytes);
        tma_load_3d(&p.kv_map, &sm->v_full[s], base + kOffV + s * kTileBytes, 0, j * kAttnBN, t ? v_slab1 : v_slab);
    };

    if (threadIdx.x == 0) {
        mbar_init(&sm->q_full, 1);
        for (int s = 0; s < kAttnStages; ++s) {
            mbar_init(&sm->k_full[s], 1);
            mbar_init(&sm->v_full[s], 1);
            mbar_init(&sm->k_empty[s], 1);   // the score issuer
            mbar_init(&sm->v_empty[s], kTwo ? 1 : 2);   // both P.V issuers commit every stage (kTwo: its own)
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sm->s_full[t], 1);
            mbar_init(&sm->s_free[t], kAttnBM);
            mbar_init(&sm->p_full[t], kAttnBM);
            mbar_init(&sm->pv_done[t], 1);
        }
        sm->abort_flag = 0;
        fence_barrier_init();
        // The first loads leave now, before tensor memory is allocated and the warps
        // take their register budgets: Q and the first kAttnStages K/V tiles.
        const uint32_t qbytes = (tw[0].n > 0 ? kTileBytes : 0) + (tw[1].n > 0 ? kTileBytes : 0);
        mbar_arrive_expect_tx(&sm->q_full, qbytes);
        if (tw[0].n > 0) tma_load_3d(&p.q_map, &sm->q_full, base + kOffQ, 0, q0, q_slab);
        if (tw[1].n > 0)
            tma_load_3d(&p.q_map, &sm->q_full, base + kOffQ + kTileBytes, 0, kTwo ? 0 : q0 + kAttnBM,
                        kTwo ? q_slab1 : q_slab);
        if constexpr (kTwo) {
            for (int g = 0; g < kAttnStages && (g >> 1) < n_all; ++g)
                if (tw[g & 1].active) load_kv2(g);
        } else {
            for (int j = 0; j < n_all && j < kAttnStages; ++j) {
                mbar_arrive_expect_tx(&sm->k_full[j], kTileBytes);
                tma_load_3d(&p.kv_map, &sm->k_full[j], base + kOffK + j * kTileBytes, 0, j * kAttnBN, k_slab);
                mbar_arrive_expect_tx(&sm->v_full[j], kTileBytes);
                tma_load_3d(&p.kv_map, &sm->v_full[j], base + kOffV + j * kTileBytes, 0, j * kAttnBN, v_slab);
            }
        }
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

    // The two register-budget regions never rejoin: each ends with its own
    // copy of the teardown barrier (id 3, all 384 threads).
    if (warp >= 8) {
      regs_dec<64>();
      if (warp == 8) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && kTwo) {
            // Q and the first ring's tiles were issued during set-up
            for (int g = kAttnStages; (g >> 1) < n_all; ++g) {
                if (!tw[g & 1].active) continue;
                const int s = g % kAttnStages;
                const uint32_t ph = (g / kAttnStages) & 1;
                mbar_wait(&sm->k_empty[s], ph ^ 1, abort_flag, p.status, 0x201);
                mbar_wait(&sm->v_empty[s], ph ^ 1, abort_flag, p.status, 0x202);
                load_kv2(g);
            }
        } else if (lane == 0) {
            // Q and the first ring's tiles were issued during set-up
            for (int j = kAttnStages; j < n_all; ++j) {
                const int s = j % kAttnStages;
                const uint32_t ph = (j / kAttnStages) & 1;
                mbar_wait(&sm->k_empty[s], ph ^ 1, abort_flag, p.status, 0x201);
                mbar_arrive_expect_tx(&sm->k_full[s], kTileBytes);
                tma_load_3d(&p.kv_map, &sm->k_full[s], base + kOffK + s * kTileBytes, 0, j * kAttnBN, k_slab);
                mbar_wait(&sm->v_empty[s], ph ^ 1, abort_flag, p.status, 0x202);
                mbar_arrive_expect_tx(&sm->v_full[s], kTileBytes);
                tma_load_3d(&p.kv_map, &sm->v_full[s], base + kOffV + s * kTileBytes, 0, j * kAttnBN, v_slab);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------ score MMAs, both query tiles
        if (lane == 0 && n_all > 0 && kTwo) {
            constexpr uint32_t idesc_s = idesc_bf16(kAttnBM, kAttnBN, false, false);
            const uint32_t k_addr = smem_u32(base + kOffK);
            mbar_wait(&sm->q_full, 0, abort_flag, p.status, 0x203);
            for (int j = 0; j < n_all; ++j) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!tw[t].active) continue;
                    const int g = 2 * j + t, s = g % kAttnStages;
                    mbar_wait(&sm->k_full[s], (g / kAttnStages) & 1, abort_flag, p.status, 0x204);
                    if (j < tw[t].n) {
                        if (j > 0) mbar_wait(&sm->s_free[t], (j - 1) & 1, abort_flag, p.status, 0x20a);
                        tc_fence_after();
                        const uint32_t qa = smem_u32(base + kOffQ) + t * kTileBytes;
                        const uint32_t ka = k_addr + s * kTileBytes;
                        const uint32_t d_s = tmem + kColS + t * 128;
#pragma unroll
                        for (int k = 0; k < kAttnD / 16; ++k)
                            mma_ss(d_s, sdesc_sw128(qa + k * 32, 16, 1024), sdesc_sw128(ka + k * 32, 16, 1024),
                                   idesc_s, k > 0);
                        tc_commit(&sm->s_full[t]);
                    }
                    tc_commit(&sm->k_empty[s]);
                }
            }
        } else if (lane == 0 && n_all > 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kAttnBM, kAttnBN, false, false);
            const uint32_t k_addr = smem_u32(base + kOffK);
            mbar_wait(&sm->q_full, 0, abort_flag, p.status, 0x203);
            for (int j = 0; j < n_all; ++j) {
                const int s = j % kAttnStages;
                mbar_wait(&sm->k_full[s], (j / kAttnStages) & 1, abort_flag, p.status, 0x204);
                const uint32_t ka = k_addr + s * kTileBytes;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (j < tw[t].n) {
                        if (j > 0) mbar_wait(&sm->s_free[t], (j - 1) & 1, abort_flag, p.status, 0x20a);
                        tc_fence_after();
                        const uint32_t qa = smem_u32(base + kOffQ) + t * kTileBytes;
                        const uint32_t d_s = tmem + kColS + t * 128;
#pragma unroll
                        for (int k = 0; k < kAttnD / 16; ++k)
                            mma_ss(d_s, sdesc_sw128(qa + k * 32, 16, 1024), sdesc_sw128(ka + k * 32, 16, 1024),
                                   idesc_s, k > 0);
                        tc_commit(&sm->s_full[t]);
                    }
                }
                tc_commit(&sm->k_empty[s]);
            }
        }
    } else if (warp == 10 || warp == 11) {
        // ------------------------------------------------ P.V MMAs of query tile t
        // Both commit every V stage, also for key tiles their own query tile does
        // not use, after waiting for that stage to be filled.
        const int t = warp - 10;
        if (lane == 0 && n_all > 0) {
            constexpr uint32_t idesc_o = idesc_bf16(kAttnBM, kAttnD, false, true);
            const uint32_t v_addr = smem_u32(base + kOffV);
            const uint32_t a_p = tmem + kColP + t * 64;
            const uint32_t d_o = tmem + kColO + t * 64;
            const int n_t = tw[t].n;
            for (int j = 0; j < n_all; ++j) {
                if (kTwo && !tw[t].active) break;   // kTwo: this tile's stages only
                const int g = kTwo ? 2 * j + t : j;
                const int s = g % kAttnStages;
                mbar_wait(&sm->v_full[s], (g / kAttnStages) & 1, abort_flag, p.status, 0x205);
                if (j < n_t) {
                    mbar_wait(&sm->p_full[t], j & 1, abort_flag, p.status, 0x207);
                    tc_fence_after();
                    const uint32_t va = v_addr + s * kTileBytes;
#pragma unroll
                    for (int k = 0; k < kAttnBN / 16; ++k)
                        mma_ts(d_o, a_p + k * 8, sdesc_sw128(va + k * 2048, 8192, 1024), idesc_o,
                               (j > 0 || k > 0) ? 1u : 0u);
                    tc_commit(&sm->pv_done[t]);
                }
                tc_commit(&sm->v_empty[s]);
            }
        }
      }
    tc_fence_before();
    named_bar_sync(3, kAttnThreads);
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    } else {
        regs_inc<216>();
        // ------------------------------------------------ softmax, one thread per query row
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int qt0 = kTwo ? 0 : q0 + t * kAttnBM;
        const int qi = qt0 + row;
        // this query tile's (batch, head) pair (the CTA's, or the second one of kTwo)
        const bool second = kTwo && t == 1;
        const int tb = second ? b1 : b;
        const int thead = second ? head1 : head;
        const int tvl = second ? vl1 : vl;
        const bool tskip = second ? can_skip1 : can_skip;
        const int tq_slab = second ? q_slab1 : q_slab;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + kColS + t * 128;
        const uint32_t p_tmem = tmem + lane_off + kColP + t * 64;
        const uint32_t o_tmem = tmem + lane_off + kColO + t * 64;
        const int n = tw[t].n;
        float m = -CUDART_INF_F;
        float l = 0.0f;
        const uint32_t fill_raw = __float_as_uint(kMaskedLog2 / p.scale_log2);

        for (int j = 0; j < n; ++j) {
            mbar_wait(&sm->s_full[t], j & 1, abort_flag, p.status, 0x208);
            __syncwarp();
            tc_fence_after();
            uint32_t u[128];   // raw fp32 scores of this row
            tmem_ld_x128(s_tmem, u);
            tc_fence_before();
            mbar_arrive(&sm->s_free[t]);   // S_t may now be overwritten by S_t(j+1)
            const int k0 = j * kAttnBN;
            const bool edge = (p.dense != nullptr) || (k0 + kAttnBN > tvl) ||
                              (p.causal && k0 + kAttnBN - 1 > qt0);
            // Full tiles keep raw scores and fold the scale into the exponent
            // (scale > 0, so max commutes with it); edge tiles are rewritten in
            // log2 units with the fill applied, and use scale 1.
            float sc = p.scale_log2;
            if (kShortKeys && edge && tskip && k0 + kAttnBN <= p.Lk) {
                // Only the causal / valid-length parts cut this tile, and every row keeps an
                // allowed key in every visited tile: a masked key gets a raw score that,
                // scaled like a full tile, is the -1e9 fill, and its weight underflows to
                // zero exactly as the fill's does.
                const int lim = min(tvl, p.causal ? qi + 1 : p.Lk) - k0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= lim) u[c] = fill_raw;
            } else if (edge) {
                // keys c < lim pass the causal and valid-length parts; c >= oob are past L_k
                const int lim = min(tvl, p.causal ? qi + 1 : p.Lk) - k0;
                const int oob = p.Lk - k0;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const float x = (c < lim) ? __uint_as_float(u[c]) * sc : kMaskedLog2;   // -1e9 fill, after scaling
                    u[c] = __float_as_uint((c < oob) ? x : -CUDART_INF_F);                   // not a key at all
                }
                if (p.dense != nullptr && qi < p.Lq) {
                    const long mrow = (p.dense_mq == 1) ? 0 : qi;
                    const long mq = (p.dense_mq == 1) ? 1 : p.Lq;
                    const uint8_t* mr = p.dense + (static_cast<long>(tb) * mq + mrow) * p.Lk + k0;
                    uint32_t keep[4];   // bit c: dense mask allows key k0 + c
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
            // row max: 8 independent 3-input max chains of depth 8, then a small tree
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
            // Lazy rescale decision (registers only): the reference max m moves
            // only when the row max grows by more than 2^8.
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
            // p = exp2(u * sc - m): packed FMA for the argument, MUFU ex2, packed sums in
            // four independent accumulators, bf16 pairs kept in registers.
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
            const float2 s01 = fadd2(acc[0], acc[1]);
            const float2 s23 = fadd2(acc[2], acc[3]);
            const float2 s4 = fadd2(s01, s23);
            l += s4.x + s4.y;
            if (j > 0) {
                // P_t and O_t are busy until P.V(j-1) has completed
                mbar_wait(&sm->pv_done[t], (j - 1) & 1, abort_flag, p.status, 0x20b);
                __syncwarp();
                tc_fence_after();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t o[16];
                        tmem_ld_x16(o_tmem + q4 * 16, o);
#pragma unroll
                        for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st_x16(o_tmem + q4 * 16, o);
                    }
                }
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_st_x16_nowait(p_tmem + q4 * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * q4]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm->p_full[t]);
        }

        // ---------------- epilogue: O / l -> bf16 -> the head's slab of ctx
        if (n > 0) {
            mbar_wait(&sm->pv_done[t], (n - 1) & 1, abort_flag, p.status, 0x209);
            __syncwarp();
            tc_fence_after();
            uint32_t o[64];
            tmem_ld_x64(o_tmem, o);
            const float inv = 1.0f / l;
            // Q_t's tile is free (its last S MMA completed before the last softmax): stage there,
            // 128-byte swizzled rows of 64 columns, or for heads narrower than 64 a dense tile of
            // their d_k columns (the rest of O is the zero padding's).
            const int nd = p.narrow_dk;
            const uint32_t stage = smem_u32(base + kOffQ + t * kTileBytes) + row * (nd ? nd * 2 : 128);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                if (nd && ch * 8 >= nd) break;
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(o[ch * 8 + 2 * e]) * inv,
                                       __uint_as_float(o[ch * 8 + 2 * e + 1]) * inv);
                st_shared_v4(stage + ((nd ? ch : (ch ^ (row & 7))) << 4), w[0], w[1], w[2], w[3]);
            }
            if (p.stats != nullptr && qi < p.Lq) {
                float2* st = reinterpret_cast<float2*>(p.stats) + (static_cast<long>(tq_slab) * p.Lq + qi);
                *st = make_float2(m, l);
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + t, kAttnBM);
            if (row == 0 && !*abort_flag) {
                tma_store_3d(&p.ctx_map, base + kOffQ + t * kTileBytes, thead * (nd ? nd : kAttnD), qt0, tb);
                tma_store_commit();
                tma_store_wait_all();
            }
        }
        tc_fence_before();
        named_bar_sync(3, kAttnThreads);
    }
}

}  // namespace

size_t attn_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s) {
    const bool short_keys = p.Lk <= kShortKeysMax;
    const long BH = static_cast<long>(p.B) * p.h;
    const bool two = short_keys && p.Lq <= kAttnBM && BH >= 2;
    auto* kern = two ? attn_bf16_tc_kernel<true, true>
                     : short_keys ? attn_bf16_tc_kernel<true, false> : attn_bf16_tc_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const unsigned grid = two ? static_cast<unsigned>((BH + 1) / 2) : static_cast<unsigned>(p.q_pairs) * p.B * p.h;
    return launch_pdl(kern, dim3(grid), dim3(kAttnThreads), kSmemBytes, s, p);
}

}  // namespace mha
