// attn_tc_d128.cu -- fused scaled dot-product attention for head width d_k = 128.
//
// Same computation as attn_tc.cu ("The Annotated Transformer", section
// "Attention", attention(): scores / sqrt(d_k), masked_fill(mask == 0, -1e9),
// softmax over keys, P.V; the head's output written into its slab of the
// concatenated context), for heads of width 128 (e.g. d_model 1024 with h = 8).
// Unit of work = one 128-row query tile of one (batch, head); key tiles of 128.
//
// Each query row is shared by two softmax threads: thread (h, row) of warpgroup h
// takes keys 64 h .. 64 h + 63 of every key tile. The two halves of a row exchange
// their tile maxima through shared memory (a named barrier per pair of warps), so
// both keep the same reference max m (the lazy online rewrite: m moves only when the
// row max grows by more than 2^8, exact because the final O / l uses the same m),
// each adds its own share l_h of the row sum, writes its 64 weights into one half of
// the tile's P and rescales its 64 features of the one output accumulator O; the row
// ends as O / (l_0 + l_1). Two threads per row give each sub-partition two softmax
// warps and halve each warp's chain of loads, maxima, exponentials and stores.
//
// Persistent: one CTA per SM draws query tiles ("units": (batch, head, 128 query rows))
// from a counter in the workspace, in the order (groups of kHeadGroup (batch, head)
// pairs, longest query tiles first), so the K/V in flight fit L2 and the short tiles
// fill the end. The next unit's Q, K and V tiles are loaded, and its first score tiles
// computed, while the current unit's softmax and output finish: a CTA's set-up is paid
// once, not once per query tile. The last CTA to finish resets the counter; the Q/K/V
// projection kernel also zeroes it before the first use of a workspace.
//
// Tensor memory (512 columns), every tile double-buffered so that neither MMA waits
// on the other's consumer:
//   S_0 S_1  [0,256)    fp32 scores of key tiles j = 0, 2, ... / 1, 3, ...: S(j + 2) is
//                       computed once both halves have loaded S(j)
//   P_0 P_1  [256,384)  bf16 weights of those tiles (keys 0..63 in the first 32 columns,
//                       64..127 in the next 32): the softmax writes P(j) without waiting
//                       for P.V(j - 1), only for P.V(j - 2)
//   O        [384,512)  fp32 output accumulator (128 features)
// Shared memory: two Q buffers (unit u uses buffer u mod 2; after its last score MMA
// the buffer carries the halves' sums and stages the unit's output for the TMA store),
// a K ring of 3 stages and a V ring of 2 (every tile two 64-wide 128-byte-swizzled
// halves), the maxima exchange. S = Q K^T is SS-MMA M=128 N=128 (8 k-steps);
// O += P V takes P from tensor memory and V MN-major with N = 128 (the two 64-wide
// feature halves are the descriptor's two MN blocks, LBO apart): 8 k-steps.
// Warps: 0-3 / 4-7 softmax of key half 0 / 1 (one thread per query row), 8 scheduler
// and Q/K loads, 9 score MMAs (and tensor-memory allocation), 10 P.V MMAs, 11 V loads.
// Registers: 168 per thread at launch; the third warpgroup drops to 64 and the softmax
// warpgroups rise to 216 (128*64 + 256*216 = 63488 <= 384*168).
#include <algorithm>

#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
constexpr int kThreads = 384;
constexpr uint32_t kHalf = 128 * 128;        // one 128-row x 64-column bf16 half tile = 16 KB
constexpr uint32_t kTile = 2 * kHalf;        // 128 x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                // + 128 b: score buffers S_0, S_1
constexpr uint32_t kColP = 256;              // + 64 b + 32 h: weight buffers P_0, P_1 (two halves each)
constexpr uint32_t kColO = 384;              // output accumulator, 128 features
constexpr float kMaskedLog2 = -1.0e9f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kHeadGroup = 8;

// One unit as the scheduler publishes it; n == 0 means no more work.
struct UnitInfo {
    int b, head, q0, n, vl;
};

struct Smem128 {
    uint64_t q_full[2], q_empty[2];                       // Q buffer loaded / output stored from it
    uint64_t k_full[kStagesK], k_empty[kStagesK];
    uint64_t v_full[kStagesV], v_empty[kStagesV];
    uint64_t s_full[2];          // score buffer b holds S(j) (commit)
    uint64_t s_free[2];          // S(j) of buffer b loaded by both halves (256 arrivals)
    uint64_t p_full[2];          // P(j) of weight buffer b written by both halves (256 arrivals)
    uint64_t p_free[2];          // P.V(j) of weight buffer b done (commit): P_b free, O holds tile j
    uint64_t unit_full[2];       // unit slot published by the scheduler
    UnitInfo unit[2];
    uint32_t tmem_base;
    int abort_flag;
    float mx[2][2][BM];          // [tile parity][half][row]: the halves' tile maxima, exchanged
};
constexpr uint32_t kOffQ = 0;                                  // + kTile * buffer
constexpr uint32_t kOffK = 2 * kTile;
constexpr uint32_t kOffV = kOffK + kStagesK * kTile;
constexpr uint32_t kOffBar = kOffV + kStagesV * kTile;
// The dynamic shared memory starts 1024-byte aligned (checked at entry): no alignment slack, which
// leaves room for the maxima exchange beside the rings.
constexpr size_t kSmemBytes = kOffBar + sizeof(Smem128);

// Unit u of the schedule: (batch, head) pairs in groups of kHeadGroup, inside a group the
// query tiles from the last (longest key range under a causal mask) to the first.
__device__ __forceinline__ UnitInfo unit_of(const AttnParams& p, int u) {
    const int BH = p.B * p.h;
    const int QT = p.q_pairs;
    const int grp = u / (kHeadGroup * QT);
    const int g_heads = min(kHeadGroup, BH - grp * kHeadGroup);
    const int r = u - grp * kHeadGroup * QT;
    const int qt = QT - 1 - r / g_heads;
    const int bh = grp * kHeadGroup + r % g_heads;
    UnitInfo x;
    x.b = bh / p.h;
    x.head = bh - x.b * p.h;
    x.q0 = qt * BM;
    int vl = p.Lk;
    if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[x.b], 0), p.Lk);
    const bool can_skip = (p.dense == nullptr) && (vl >= 1);
    int kend = can_skip ? vl : p.Lk;
    if (can_skip && p.causal) kend = min(kend, x.q0 + BM);
    x.n = (kend + BN - 1) / BN;   // >= 1
    x.vl = vl;
    return x;
}

// kDense: the instance for calls with a dense mask; without one the softmax loop carries no
// mask-byte code (1 % faster on the long workload).
template <bool kDense>
__global__ void __launch_bounds__(kThreads, 1) attn_d128_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw;
    Smem128* sm = reinterpret_cast<Smem128*>(base + kOffBar);
    if ((smem_u32(base) & 1023u) != 0) {
        // the 128-byte-swizzled tiles need 1024-byte alignment: refuse rather than compute garbage
        if (threadIdx.x == 0) atomicCAS(p.status, 0, 0x2f2);
        return;
    }
    pdl_trigger();
    pdl_wait();   // Qh, KVh, the mask parts and the schedule counter come from earlier kernels

    const int total = p.B * p.h * p.q_pairs;
    MHA_DEVICE_CHECK(total >= 1 && p.Lq >= 1 && p.Lk >= 1 && p.q_pairs * BM >= p.Lq && p.sched != nullptr,
                     p.status, 0x2f1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->q_full[i], 1);
            mbar_init(&sm->q_empty[i], 1);
            mbar_init(&sm->unit_full[i], 1);
        }
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(&sm->k_full[s], 1);
            mbar_init(&sm->k_empty[s], 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&sm->v_full[s], 1);
            mbar_init(&sm->v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm->s_full[b], 1);
            mbar_init(&sm->s_free[b], 2 * BM);
            mbar_init(&sm->p_full[b], 2 * BM);
            mbar_init(&sm->p_free[b], 1);
        }
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
        // ------------------------------------------------ scheduler, Q and K loads
        int next = atomicAdd(p.sched, 1);
        uint32_t gk = 0;   // K tiles issued so far
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            // unit k - 2 has stored its output from this Q buffer (and every role has read its slot)
            if (k >= 2) mbar_wait(&sm->q_empty[qb], ((k >> 1) - 1) & 1, abort_flag, p.status, 0x400);
            if (next >= total || *abort_flag) {
                sm->unit[qb].n = 0;
                mbar_arrive(&sm->unit_full[qb]);
                break;
            }
            const UnitInfo x = unit_of(p, next);
            sm->unit[qb] = x;
            mbar_arrive(&sm->unit_full[qb]);
            next = atomicAdd(p.sched, 1);   // the unit after this one, fetched while this one loads
            const int q_slab = x.b * p.h + x.head;
            const int k_slab = x.b * 2 * p.h + x.head;
            uint8_t* qbuf = base + kOffQ + qb * kTile;
            mbar_arrive_expect_tx(&sm->q_full[qb], kTile);
            for (int hf = 0; hf < 2; ++hf)
                tma_load_4d(&p.q_map, &sm->q_full[qb], qbuf + hf * kHalf, 0, hf, x.q0, q_slab);
            for (int j = 0; j < x.n; ++j, ++gk) {
                const int s = gk % kStagesK;
                mbar_wait(&sm->k_empty[s], ((gk / kStagesK) & 1) ^ 1, abort_flag, p.status, 0x401);
                mbar_arrive_expect_tx(&sm->k_full[s], kTile);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_4d(&p.kv_map, &sm->k_full[s], base + kOffK + s * kTile + hf * kHalf, 0, hf, j * BN,
                                k_slab);
            }
        }
      } else if (warp == 11 && lane == 0) {
        // ------------------------------------------------ V loads
        uint32_t gv = 0;
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            if (!mbar_wait(&sm->unit_full[qb], (k >> 1) & 1, abort_flag, p.status, 0x40c)) break;
            const UnitInfo x = sm->unit[qb];
            if (x.n == 0) break;
            const int v_slab = x.b * 2 * p.h + p.h + x.head;
            for (int j = 0; j < x.n; ++j, ++gv) {
                const int s = gv % kStagesV;
                mbar_wait(&sm->v_empty[s], ((gv / kStagesV) & 1) ^ 1, abort_flag, p.status, 0x402);
                mbar_arrive_expect_tx(&sm->v_full[s], kTile);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_4d(&p.kv_map, &sm->v_full[s], base + kOffV + s * kTile + hf * kHalf, 0, hf, j * BN,
                                v_slab);
            }
        }
      } else if (warp == 9 && lane == 0) {
        // ------------------------------------------------ score MMAs: S(j) = Q K_j^T
        constexpr uint32_t idesc_s = idesc_bf16(BM, BN, false, false);
        const uint32_t k_addr = smem_u32(base + kOffK);
        uint32_t gk = 0;   // score tiles issued so far
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            if (!mbar_wait(&sm->unit_full[qb], (k >> 1) & 1, abort_flag, p.status, 0x40d)) break;
            const int n = sm->unit[qb].n;
            if (n == 0) break;
            const uint32_t qa = smem_u32(base + kOffQ + qb * kTile);
            mbar_wait(&sm->q_full[qb], (k >> 1) & 1, abort_flag, p.status, 0x403);
            for (int j = 0; j < n; ++j, ++gk) {
                const int s = gk % kStagesK;
                mbar_wait(&sm->k_full[s], (gk / kStagesK) & 1, abort_flag, p.status, 0x404);
                // buffer gk mod 2 is free once both halves have loaded score tile gk - 2
                const int sb = gk & 1;
                if (gk >= 2) mbar_wait(&sm->s_free[sb], ((gk >> 1) - 1) & 1, abort_flag, p.status, 0x406);
                tc_fence_after();
                const uint32_t ka = k_addr + s * kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_ss(tmem + kColS + sb * 128, sdesc_sw128(qa + off, 16, 1024),
                           sdesc_sw128(ka + off, 16, 1024), idesc_s, kk > 0);
                }
                tc_commit(&sm->s_full[sb]);
                tc_commit(&sm->k_empty[s]);
            }
        }
      } else if (warp == 10 && lane == 0) {
        // ------------------------------------------------ P.V MMAs: O += P(j) V_j (128 keys, both halves)
        constexpr uint32_t idesc_o = idesc_bf16(BM, D, false, true);
        const uint32_t v_addr = smem_u32(base + kOffV);
        uint32_t gv = 0;   // P.V steps issued so far
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            if (!mbar_wait(&sm->unit_full[qb], (k >> 1) & 1, abort_flag, p.status, 0x40e)) break;
            const int n = sm->unit[qb].n;
            if (n == 0) break;
            for (int j = 0; j < n; ++j, ++gv) {
                const int s = gv % kStagesV;
                mbar_wait(&sm->v_full[s], (gv / kStagesV) & 1, abort_flag, p.status, 0x407);
                // P(j) written; for j = 0 also: the previous unit's output has been read out of O
                mbar_wait(&sm->p_full[gv & 1], (gv >> 1) & 1, abort_flag, p.status, 0x408);
                tc_fence_after();
                const uint32_t va = v_addr + s * kTile;
                const uint32_t pa = tmem + kColP + (gv & 1) * 64;   // keys 16 kk .. 16 kk + 15: columns 8 kk ..
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColO, pa + kk * 8, sdesc_sw128(va + kk * 2048, kHalf, 1024), idesc_o,
                           (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&sm->p_free[gv & 1]);
                tc_commit(&sm->v_empty[s]);
            }
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
      if (warp == 8 && lane == 0) {
          // the last CTA to finish leaves the schedule counter at zero for the next launch
          __threadfence();
          if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
              atomicExch(p.sched, 0);
              atomicExch(p.sched + 1, 0);
          }
      }
    } else {
        regs_inc<216>();
        // ------------------------------------------------ softmax: thread (h, row), keys 64 h .. 64 h + 63
        const int h = warp >> 2;
        const int q = warp & 3;   // lane quarter; warps q and q + 4 hold the two halves of the same rows
        const int row = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + kColS + h * 64;   // + 128 b
        const uint32_t p_tmem = tmem + lane_off + kColP + h * 32;   // + 64 b
        const uint32_t o_tmem = tmem + lane_off + kColO + h * 64;   // this half's 64 output features
        uint32_t g = 0;   // score tiles consumed so far
        for (int k = 0;; ++k) {
            const int qb = k & 1;
            const bool ok = mbar_wait(&sm->unit_full[qb], (k >> 1) & 1, abort_flag, p.status, 0x40f);
            const UnitInfo x = sm->unit[qb];
            __syncwarp();
            // every softmax thread takes the same decision (a give-up in one thread stops all)
            if (!named_bar_and(1, 2 * BM, ok && x.n > 0)) break;
            const int n = x.n, vl = x.vl, q0 = x.q0, b = x.b;
            const int qi = q0 + row;
            float m = -CUDART_INF_F;   // the row's reference max (log2 units), common to both halves
            float l = 0.0f;            // this half's share of the row sum
            for (int j = 0; j < n; ++j, ++g) {
                const uint32_t sb = g & 1;
                mbar_wait(&sm->s_full[sb], (g >> 1) & 1, abort_flag, p.status, 0x409);
                __syncwarp();
                tc_fence_after();
                uint32_t u[64];
                tmem_ld_x64(s_tmem + sb * 128, u);
                tc_fence_before();
                mbar_arrive(&sm->s_free[sb]);
                const int k0 = j * BN + h * 64;   // first key of this half
                const bool edge = (kDense && p.dense != nullptr) || (k0 + 64 > vl) || (p.causal && k0 + 63 > q0);
                float sc = p.scale_log2;
                if (edge) {
                    const int lim = min(vl, p.causal ? qi + 1 : p.Lk) - k0;
                    const int oob = p.Lk - k0;
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const float xs = (c < lim) ? __uint_as_float(u[c]) * sc : kMaskedLog2;   // -1e9 fill, after scaling
                        u[c] = __float_as_uint((c < oob) ? xs : -CUDART_INF_F);                  // not a key at all
                    }
                    if (kDense && p.dense != nullptr && qi < p.Lq) {
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
                    __syncwarp();   // rows past L_q skip the dense mask: reconverge before warp-wide instructions
                    sc = 1.0f;
                }
                float a4[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    float a = fmax3(__uint_as_float(u[16 * c4]), __uint_as_float(u[16 * c4 + 1]),
                                    __uint_as_float(u[16 * c4 + 2]));
#pragma unroll
                    for (int e = 3; e < 15; e += 2)
                        a = fmax3(a, __uint_as_float(u[16 * c4 + e]), __uint_as_float(u[16 * c4 + e + 1]));
                    a4[c4] = fmaxf(a, __uint_as_float(u[16 * c4 + 15]));
                }
                // this half's tile max (log2 units), exchanged with the other half of the row
                const float mth = fmaxf(fmax3(a4[0], a4[1], a4[2]), a4[3]) * sc;
                sm->mx[sb][h][row] = mth;
                named_bar_sync(4 + q, 64);   // warps q and q + 4
                const float m_new = fmaxf(m, fmaxf(mth, sm->mx[sb][h ^ 1][row]));
                float alpha = 1.0f;
                bool grow = false;
                if (m == -CUDART_INF_F) {
                    m = m_new;   // first keys of the row (-inf while every key so far is past L_k)
                } else {
                    grow = (m_new - m) > kRescaleThreshold;
                    if (grow) {
                        alpha = ex2_approx(m - m_new);
                        l *= alpha;
                        m = m_new;
                    }
                }
                // with no key of the row yet (m = -inf) every weight is exp2(-inf) = 0
                const float mref = (m == -CUDART_INF_F) ? 0.0f : m;
                const float2 sc2 = make_float2(sc, sc);
                const float2 nm2 = make_float2(-mref, -mref);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float2 e2 = ffma2(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sc2, nm2);
                    e2.x = ex2_approx(e2.x);
                    e2.y = ex2_approx(e2.y);
                    acc[c & 3] = fadd2(acc[c & 3], e2);
                    pk[c] = pack_bf16x2(e2.x, e2.y);
                }
                const float2 s4 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                l += s4.x + s4.y;
                // weight buffer sb is free once P.V(g - 2) has read it (P.V(g - 4) was waited for
                // at tile g - 2 and P.V(g) needs this thread's weights: the phase is unambiguous)
                if (g >= 2) {
                    mbar_wait(&sm->p_free[sb], ((g >> 1) - 1) & 1, abort_flag, p.status, 0x40c);
                    __syncwarp();
                    tc_fence_after();
                }
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
                    // O is rescaled (this half's 64 features) once P.V(g - 1) has completed; at j = 0
                    // the first P.V overwrites O, after the previous unit's output has been read
                    mbar_wait(&sm->p_free[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_flag, p.status, 0x40a);
                    __syncwarp();
                    tc_fence_after();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t o[16];
                        tmem_ld_x16(o_tmem + q4 * 16, o);
#pragma unroll
                        for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st_x16(o_tmem + q4 * 16, o);
                    }
                }
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4)
                    tmem_st_x16_nowait(p_tmem + sb * 64 + q4 * 16,
                                       *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * q4]));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&sm->p_full[sb]);
            }
            // ---------------- output: thread (h, row) writes features 64 h .. 64 h + 63 of O / (l_0 + l_1).
            // The unit's Q buffer is idle (its last score MMA completed before this thread's last wait on
            // S): it carries l_h of every half and row, then the bf16 output tile.
            uint8_t* qbuf = base + kOffQ + qb * kTile;
            float* lsum = reinterpret_cast<float*>(qbuf);
            lsum[h * BM + row] = l;
            named_bar_sync(1, 2 * BM);   // both halves' sums are in shared memory
            const float L = lsum[row] + lsum[BM + row];
            const float inv = 1.0f / L;
            const uint32_t gl = g - 1;   // the unit's last tile: its P.V completes O
            mbar_wait(&sm->p_free[gl & 1], (gl >> 1) & 1, abort_flag, p.status, 0x40b);
            __syncwarp();
            tc_fence_after();
            uint32_t o[64];
            tmem_ld_x64(o_tmem, o);
            named_bar_sync(1, 2 * BM);   // every thread has read the sums the staging overwrites
            const uint32_t stage = smem_u32(qbuf + h * kHalf) + row * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = ch * 8 + 2 * e;
                    w[e] = pack_bf16x2(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv);
                }
                st_shared_v4(stage + ((ch ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
            }
            if (h == 0 && p.stats != nullptr && qi < p.Lq) {
                // the row's softmax statistics for p_attn: exp2(u - m) / L is the weight of any key
                float2* st = reinterpret_cast<float2*>(p.stats) +
                             (static_cast<long>(b * p.h + x.head) * p.Lq + qi);
                *st = make_float2(m, L);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 2 * BM);
            if (warp == 0 && lane == 0) {
                if (!*abort_flag) {
                    for (int hf = 0; hf < 2; ++hf)
                        tma_store_3d(&p.ctx_map, qbuf + hf * kHalf, x.head * D + hf * 64, q0, b);
                    tma_store_commit();
                }
                tma_store_wait_read();   // the buffer may take the Q tile of unit k + 2
                mbar_arrive(&sm->q_empty[qb]);
            }
        }
        if (warp == 0 && lane == 0) tma_store_wait_all();
        tc_fence_before();
        named_bar_sync(3, kThreads);
    }
}

}  // namespace

cudaError_t launch_attn_tc_d128(const AttnParams& p, cudaStream_t s) {
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    if (p.sched == nullptr) return cudaErrorInvalidValue;
    auto* kern = p.dense != nullptr ? attn_d128_kernel<true> : attn_d128_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long units = static_cast<long>(p.q_pairs) * p.B * p.h;
    const unsigned grid = static_cast<unsigned>(std::max(1L, std::min<long>(units, sms)));
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, p);
}

}  // namespace mha
