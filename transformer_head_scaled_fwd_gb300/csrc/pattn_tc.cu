// pattn_tc.cu -- the optional attention weights p_attn [B, h, L_q, L_k] (fp32) on the
// tensor cores, for the bf16 path.
//
// attention() of "The Annotated Transformer", section "Attention", returns p_attn
// beside the output, and MultiHeadedAttention keeps it (self.attn = p_attn,
// "003-Transformer" tutorial). The fused attention kernels never materialise the
// scores; when p_attn is asked for they also write each row's softmax statistics
// (reference max m in log2 units, sum l of exp2(u - m)). This kernel then recomputes
// every score tile and writes the normalised weights:
//     p[i, j] = exp2(u_ij - m_i) / l_i,   u_ij = s_ij log2(e) / sqrt(d_k), or the -1e9
//     fill (in log2 units) where the mask is 0,
// which is the softmax row exactly (a fully masked row, whose statistics are the
// fill and L_k, comes out uniform 1/L_k as the pages' -1e9 fill implies).
//
// CTA = one 128-row query tile of one (batch, head); 320 threads:
//   warps 0-7  two threads per query row (warpgroup g takes key columns 64 g .. 64 g + 63
//              of each tile): tcgen05.ld the scores, form the weights and stage them for
//              the store: with L_k a multiple of 4 in a 128-byte-swizzled fp32 tile that
//              one thread TMA-stores as four {32, 128} boxes (full lines), otherwise in a
//              padded tile read back transposed, so each warp store is 32 consecutive
//              floats of one row (rows of L_k % 4 != 0 floats cannot be TMA-addressed).
//   warp 8     TMA: the query tile once, key tiles through a ring (one stage for
//              d_k <= 64, two for d_k = 128).
//   warp 9     allocates 256 tensor-memory columns and issues S(j) = Q K_j^T into
//              buffer j % 2, so the next tile's scores are computed while the rows
//              write the current one.
// With the TMA store a d_k <= 64 CTA takes 97 KB of shared memory and two fit on an SM.
// The weights are HBM-write bound: 4 bytes per (b, h, i, j) written.
#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kRows = 128;
constexpr int kKeys = 128;
constexpr uint32_t kHalf = 128 * 128;            // 128 rows x 64 bf16
constexpr int kStagePitch = kKeys + 1;           // fp32 staging row pitch (conflict-free both ways)
constexpr uint32_t kTmemCols = 256;
constexpr float kMaskedLog2 = -1.0e9f * 1.4426950408889634f;
constexpr int kRowThreads = 256;   // two per query row
constexpr int kThreads = kRowThreads + 64;

constexpr uint32_t kBox = 128 * 128;             // one {32 fp32, 128 rows} store box, 16 KB

struct PSm {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2];
    uint64_t s_full[2], s_free[2];
    uint32_t tmem_base;
    int abort_flag;
};

// kHalves: 64-column halves of the head, 1 (d_k <= 64) or 2 (d_k = 128); kStaged: with
// the fp32 [128][129] transpose tile (rows of L_k % 4 != 0 floats)
template <int kHalves, bool kStaged>
struct PLayout {
    static constexpr int kKStages = kHalves;                              // key ring depth
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kHalves * kHalf;
    static constexpr uint32_t kStage = kK + kKStages * kHalves * kHalf;
    static constexpr uint32_t kBar =
        kStage + (kStaged ? ((kRows * kStagePitch * 4 + 1023) & ~1023u) : 4u * kBox);
    static constexpr size_t kSmem = 1024 + kBar + sizeof(PSm);
};

template <int kHalves>
__device__ __forceinline__ void load_tile(const CUtensorMap* m, uint64_t* bar, uint8_t* dst, int row, int slab) {
    if constexpr (kHalves == 1) {
        tma_load_3d(m, bar, dst, 0, row, slab);
    } else {
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) tma_load_4d(m, bar, dst + hf * kHalf, 0, hf, row, slab);
    }
}

template <int kHalves, bool kStaged>
__global__ void __launch_bounds__(kThreads) pattn_tc_kernel(const __grid_constant__ AttnParams p) {
    using Lay = PLayout<kHalves, kStaged>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PSm* sm = reinterpret_cast<PSm*>(base + Lay::kBar);
    pdl_trigger();
    pdl_wait();   // Qh, KVh and the row statistics come from the earlier kernels

    const int qtiles = (p.Lq + kRows - 1) / kRows;
    const int bh = static_cast<int>(blockIdx.x) / qtiles;
    const int qt = static_cast<int>(blockIdx.x) - bh * qtiles;
    MHA_DEVICE_CHECK(bh < p.B * p.h, p.status, 0x2f2);
    const int b = bh / p.h;
    const int head = bh - b * p.h;
    const int q0 = qt * kRows;
    const int nk = (p.Lk + kKeys - 1) / kKeys;   // every key is written, masked ones included
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&sm->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm->k_full[s], 1);
            mbar_init(&sm->k_empty[s], 1);
            mbar_init(&sm->s_full[s], 1);
            mbar_init(&sm->s_free[s], kRowThreads);
        }
        sm->abort_flag = 0;
        fence_barrier_init();
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

    if (warp == 8) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm->q_full, kHalves * kHalf);
            load_tile<kHalves>(&p.q_map, &sm->q_full, base + Lay::kQ, q0, bh);
            const int k_slab = b * 2 * p.h + head;
            for (int j = 0; j < nk; ++j) {
                const int s = j % Lay::kKStages;
                mbar_wait(&sm->k_empty[s], ((j / Lay::kKStages) & 1) ^ 1, abort_flag, p.status, 0x601);
                mbar_arrive_expect_tx(&sm->k_full[s], kHalves * kHalf);
                load_tile<kHalves>(&p.kv_map, &sm->k_full[s], base + Lay::kK + s * kHalves * kHalf, j * kKeys,
                                   k_slab);
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kRows, kKeys, false, false);
            const uint32_t qa = smem_u32(base + Lay::kQ);
            mbar_wait(&sm->q_full, 0, abort_flag, p.status, 0x602);
            for (int j = 0; j < nk; ++j) {
                const int s = j & 1;                 // score buffer
                const int ks = j % Lay::kKStages;    // key stage
                mbar_wait(&sm->k_full[ks], (j / Lay::kKStages) & 1, abort_flag, p.status, 0x603);
                if (j >= 2) mbar_wait(&sm->s_free[s], ((j - 2) >> 1) & 1, abort_flag, p.status, 0x604);
                tc_fence_after();
                const uint32_t ka = smem_u32(base + Lay::kK + ks * kHalves * kHalf);
#pragma unroll
                for (int k = 0; k < 4 * kHalves; ++k) {
                    const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
                    mma_ss(tmem + s * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc,
                           k > 0);
                }
                tc_commit(&sm->s_full[s]);
                tc_commit(&sm->k_empty[ks]);
            }
        }
    } else {
        // ------------------------------------------------ two threads per query row
        const int half = warp >> 2;             // key columns 64 half .. 64 half + 63 of each tile
        const int row = (warp & 3) * 32 + lane;
        const int qi = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int vl = p.Lk;
        if (p.valid_lens != nullptr) vl = min(max(p.valid_lens[b], 0), p.Lk);
        float m = 0.f, inv_l = 0.f;
        if (qi < p.Lq) {
            const float2 st = reinterpret_cast<const float2*>(p.stats)[static_cast<long>(bh) * p.Lq + qi];
            m = st.x;
            inv_l = 1.0f / st.y;
        }
        const int lim_causal = p.causal ? qi + 1 : p.Lk;   // keys j < lim pass the causal and valid-length parts
        const int lim = min(vl, lim_causal);
        const uint8_t* mrow = nullptr;
        if (p.dense != nullptr && qi < p.Lq)
            mrow = p.dense + (static_cast<long>(b) * (p.dense_mq == 1 ? 1 : p.Lq) + (p.dense_mq == 1 ? 0 : qi)) * p.Lk;
        const int rows_here = min(kRows, p.Lq - q0);
        float* out_base = p.p_attn + (static_cast<long>(bh) * p.Lq + q0) * p.Lk;
        for (int j = 0; j < nk; ++j) {
            const int s = j & 1;
            mbar_wait(&sm->s_full[s], (j >> 1) & 1, abort_flag, p.status, 0x605);
            __syncwarp();
            tc_fence_after();
            uint32_t u[64];
            tmem_ld_x64(tmem + lane_off + s * 128 + half * 64, u);
            tc_fence_before();
            mbar_arrive(&sm->s_free[s]);
            const int k0 = j * kKeys + half * 64;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const int kj = k0 + c;
                bool ok = kj < lim;
                if (mrow != nullptr && ok) ok = mrow[kj] != 0;
                const float x = ok ? __uint_as_float(u[c]) * p.scale_log2 : kMaskedLog2;
                u[c] = __float_as_uint(ex2_approx(x - m) * inv_l);
            }
            if constexpr (!kStaged) {
                // this thread's 64 weights: boxes 2 half and 2 half + 1, 16-byte chunks swizzled
                // like every 128-byte-row tile; the previous tile's store must have read them
                const uint32_t stg = smem_u32(base + Lay::kStage);
                if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                named_bar_sync(1, kRowThreads);
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
                    const uint32_t box = 2 * half + (c4 >> 3), ch = c4 & 7;
                    st_shared_v4(stg + box * kBox + row * 128 + ((ch ^ (row & 7)) << 4), u[4 * c4], u[4 * c4 + 1],
                                 u[4 * c4 + 2], u[4 * c4 + 3]);
                }
                fence_proxy_async_smem();
                named_bar_sync(1, kRowThreads);
                if (threadIdx.x == 0 && !*abort_flag) {
                    for (int bx = 0; bx < 4 && j * kKeys + 32 * bx < p.Lk; ++bx)
                        tma_store_3d(&p.p_map, base + Lay::kStage + bx * kBox, j * kKeys + 32 * bx, q0, bh);
                    tma_store_commit();
                }
            } else {
                float* stage = reinterpret_cast<float*>(base + Lay::kStage);
                float* srow = stage + row * kStagePitch + half * 64;
#pragma unroll
                for (int c = 0; c < 64; ++c) srow[c] = __uint_as_float(u[c]);
                named_bar_sync(1, kRowThreads);
                // transposed store: thread t writes column t % 128 of the tile's rows of parity
                // t / 128 (each warp store: 32 consecutive floats of one row)
                const int t = half * 128 + row;
                const int col = j * kKeys + (t & 127);
                if (col < p.Lk) {
                    for (int r = t >> 7; r < rows_here; r += 2)
                        out_base[static_cast<long>(r) * p.Lk + col] = stage[r * kStagePitch + (t & 127)];
                }
                named_bar_sync(1, kRowThreads);
            }
        }
    }
    if (threadIdx.x == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kHalves, bool kStaged>
cudaError_t launch_one(const AttnParams& p, unsigned grid, cudaStream_t s) {
    auto* k = pattn_tc_kernel<kHalves, kStaged>;
    constexpr size_t smem = PLayout<kHalves, kStaged>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, s, p);
}

}  // namespace

cudaError_t launch_pattn_tc(const AttnParams& p, int halves, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(p.B * p.h * ((p.Lq + kRows - 1) / kRows));
    // TMA stores need the rows of p_attn on 16-byte boundaries (p_map is then encoded)
    const bool staged = (p.Lk % 4) != 0 || (reinterpret_cast<uintptr_t>(p.p_attn) & 15) != 0;
    if (halves == 2) return staged ? launch_one<2, true>(p, grid, s) : launch_one<2, false>(p, grid, s);
    return staged ? launch_one<1, true>(p, grid, s) : launch_one<1, false>(p, grid, s);
}

}  // namespace mha
