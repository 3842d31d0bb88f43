// decode.cu -- incremental decoding: one new query per sequence against a
// key/value cache.
//
// At prediction time the d2l Transformer decoder (d2l Transformer chapter
// summary, DecoderBlock: state[2] keeps the representations decoded so far and
// torch.cat appends the new one, used as keys and values) attends from the
// newest token to every token decoded so far, itself included. Caching the
// projected keys and values instead of the raw representations gives the same
// result: attention() of "The Annotated Transformer" ("Attention") over all
// cached keys, no mask needed (every cached position precedes the query).
//
// Kernels (HBM-bound: the cache is read once per step):
//   kv_append_kernel    (steps with more than 64 new tokens, whose projections
//                       run as tiled GEMMs) copies the new token's projected k, v
//                       into the caches at position cache_len[b]; with fewer, the
//                       projection kernel writes them there itself.
//   decode_attn_kernel  split-K over the cached keys: each CTA takes a chunk of
//                       keys of one (batch, head); a warp takes 32 keys at a
//                       time with coalesced loads (each instruction reads 4
//                       whole key or value rows), scores them with partial dot
//                       products and an 8-lane reduce-scatter, keeps an online
//                       softmax (running max and sum) and accumulates p.V per
//                       lane over its own keys; the CTA's warps merge and write
//                       a partial (max, sum, o[64]). When the projections run on
//                       the small-M kernel, each CTA first issues a bulk L2 prefetch of
//                       the start of its chunk, before waiting for them: the cache
//                       streams in while the projections run.
//   decode_combine_kernel  merges the partials of a (batch, head), writes its
//                       64-wide slab of the concatenated context, and counts the
//                       new token in cache_len[b] (or reports a full cache).
#include <math_constants.h>

#include "launch.h"
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kWarps = 4;

template <int kD>
__global__ void __launch_bounds__(256) kv_append_kernel(const DecodeParams p) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int pos = p.cache_len[b];
    if (pos < 0 || pos >= p.L_max) return;   // full cache: nothing appended (reported by the combine)
    // KVh of the step is [1, 2, h, B, D]: k of (b, head) at ((head) * B + b) * D, v after h planes
    for (int e = threadIdx.x; e < p.h * kD / 8; e += blockDim.x) {
        const int head = e / (kD / 8);
        const int c8 = e % (kD / 8);
        const long src = (static_cast<long>(head) * p.B + b) * kD + c8 * 8;
        const long vsrc = (static_cast<long>(p.h + head) * p.B + b) * kD + c8 * 8;
        const long dst = ((static_cast<long>(b) * p.h + head) * p.L_max + pos) * kD + c8 * 8;
        *reinterpret_cast<uint4*>(p.k_cache + dst) = *reinterpret_cast<const uint4*>(p.kv_new + src);
        *reinterpret_cast<uint4*>(p.v_cache + dst) = *reinterpret_cast<const uint4*>(p.kv_new + vsrc);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Head width kD = 64 or 128. A key (value) row is kD * 2 bytes: kLanesRow = kD / 8 lanes
// read it with one 16-byte load each, so one load instruction of a warp reads kRowsLoad
// whole consecutive rows (512 contiguous bytes); each lane loads 8 rows per group, so a
// group is kGroup = 8 * kRowsLoad keys.
template <int kD>
__global__ void __launch_bounds__(32 * kWarps) decode_attn_kernel(const DecodeParams p) {
    constexpr int kLanesRow = kD / 8;
    constexpr int kRowsLoad = 32 / kLanesRow;
    constexpr int kGroup = 8 * kRowsLoad;
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ float sm_o[kWarps][kD];
    pdl_trigger();
    if (p.prefetch_keys > 0 && threadIdx.x == 0) {
        // The first keys and values of this CTA's chunk stream into L2 while the step's
        // projections still run; the new token's row (written by them) is left out.
        const int pbh = blockIdx.y;
        const int pb = pbh / p.h;
        const int pn = min(max(p.cache_len[pb], 0) + 1, p.L_max);
        const int pchunk = ((pn + p.n_split - 1) / p.n_split + 31) & ~31;
        const int pc0 = blockIdx.x * pchunk;
        const int pc1 = min(pn - 1, pc0 + p.prefetch_keys);
        if (pc1 > pc0) {
            const long off = (static_cast<long>(pbh) * p.L_max + pc0) * kD;
            const uint32_t bytes = static_cast<uint32_t>(pc1 - pc0) * kD * 2;
            prefetch_l2_bulk(p.k_cache + off, bytes);
            prefetch_l2_bulk(p.v_cache + off, bytes);
        }
    }
    pdl_wait();
    const int bh = blockIdx.y;
    const int b = bh / p.h;
    const int head = bh - b * p.h;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the step's key and value sit at position cache_len[b] (unless the cache is full)
    const int n = min(max(p.cache_len[b], 0) + 1, p.L_max);
    const int chunk = ((n + p.n_split - 1) / p.n_split + 31) & ~31;
    const int c0 = blockIdx.x * chunk;
    const int c1 = min(n, c0 + chunk);
    // Lane (grp, sl) = (lane / kLanesRow, lane % kLanesRow) holds dims 8 sl .. 8 sl + 7 of
    // the keys kRowsLoad i + grp (i = 0..7) of each group.
    const int grp = lane / kLanesRow;
    const int sl = lane % kLanesRow;

    // this lane's slice of the query row, pre-scaled so that scores are in log2 units
    float q[8];
    {
        const uint4 raw = *reinterpret_cast<const uint4*>(p.q_new + (static_cast<long>(head) * p.B + b) * kD + 8 * sl);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            q[2 * e] = f.x * p.scale_log2;
            q[2 * e + 1] = f.y * p.scale_log2;
        }
    }
    const __nv_bfloat16* K = p.k_cache + static_cast<long>(bh) * p.L_max * kD + 8 * sl;
    const __nv_bfloat16* V = p.v_cache + static_cast<long>(bh) * p.L_max * kD + 8 * sl;
    float m = -CUDART_INF_F, l = 0.0f;
    float o[8];   // partial p.V over this lane's keys, dims 8 sl ..
#pragma unroll
    for (int f = 0; f < 8; ++f) o[f] = 0.0f;
    for (int g0 = c0 + kGroup * warp; g0 < c1; g0 += kGroup * kWarps) {
        // keys and values of the group, all 16 loads in flight together
        uint4 kr[8], vr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int key = g0 + kRowsLoad * i + grp;
            kr[i] = (key < c1) ? *reinterpret_cast<const uint4*>(K + static_cast<long>(key) * kD) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int key = g0 + kRowsLoad * i + grp;
            vr[i] = (key < c1) ? *reinterpret_cast<const uint4*>(V + static_cast<long>(key) * kD) : make_uint4(0, 0, 0, 0);
        }
        // partial scores of the 8 keys over this lane's 8 dims
        float part[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&kr[i]);
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                a = fmaf(q[2 * e], f.x, a);
                a = fmaf(q[2 * e + 1], f.y, a);
            }
            part[i] = a;
        }
        // reduce-scatter over 8 lanes of the row: lane sl ends with key i = sl % 8's score
        // summed over those lanes (for kD = 128 the two halves of the row are then added)
#pragma unroll
        for (int s = 4; s >= 1; s >>= 1) {
            const bool upper = (sl & s) != 0;
#pragma unroll
            for (int t = 0; t < s; ++t) {
                const float send = upper ? part[t] : part[t + s];
                const float keep = upper ? part[t + s] : part[t];
                part[t] = keep + __shfl_xor_sync(0xffffffffu, send, s);
            }
        }
        if constexpr (kLanesRow == 16) part[0] += __shfl_xor_sync(0xffffffffu, part[0], 8);
        // the lane holds key g0 + kRowsLoad (sl % 8) + grp; with kD = 128 lanes sl and sl + 8
        // hold the same key, and only the first counts in the sums
        const bool owner = sl < 8;
        const float sc = (g0 + kRowsLoad * (sl & 7) + grp < c1) ? part[0] : -CUDART_INF_F;
        const float m_new = fmaxf(m, warp_max(sc));   // finite: key g0 < c1 always exists
        const float alpha = ex2_approx(m - m_new);
        const float pj = ex2_approx(sc - m_new);      // 0 for keys past the chunk
        l = l * alpha + warp_sum(owner ? pj : 0.0f);
#pragma unroll
        for (int f = 0; f < 8; ++f) o[f] *= alpha;
        // this lane's value rows are keys kRowsLoad i + grp, whose weights sit in lanes
        // kLanesRow grp + i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float w = __shfl_sync(0xffffffffu, pj, kLanesRow * grp + i);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&vr[i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 v = __bfloat1622float2(h2[e]);
                o[2 * e] = fmaf(w, v.x, o[2 * e]);
                o[2 * e + 1] = fmaf(w, v.y, o[2 * e + 1]);
            }
        }
        m = m_new;
    }
    // lanes with the same dims (sl) hold partials over disjoint keys: sum the groups
#pragma unroll
    for (int f = 0; f < 8; ++f) {
#pragma unroll
        for (int x = kLanesRow; x < 32; x <<= 1) o[f] += __shfl_xor_sync(0xffffffffu, o[f], x);
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
    if (lane < kLanesRow) {
#pragma unroll
        for (int f = 0; f < 8; ++f) sm_o[warp][8 * lane + f] = o[f];
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int kPer = kD / 32;   // output dims per lane
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
        float L = 0.0f, a[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) a[e] = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = (sm_m[w] == -CUDART_INF_F) ? 0.0f : ex2_approx(sm_m[w] - M);
            L += sm_l[w] * f;
#pragma unroll
            for (int e = 0; e < kPer; ++e) a[e] += sm_o[w][kPer * lane + e] * f;
        }
        float* part = p.partial + (static_cast<long>(bh) * p.n_split + blockIdx.x) * (kD + 2);
        if (lane == 0) {
            part[0] = M;
            part[1] = L;
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) part[2 + kPer * lane + e] = a[e];
    }
}

template <int kD>
__global__ void __launch_bounds__(kD) decode_combine_kernel(const DecodeParams p) {
    pdl_trigger();
    pdl_wait();
    const int bh = blockIdx.x;
    const int b = bh / p.h;
    const int head = bh - b * p.h;
    const int c = threadIdx.x;
    const float* part = p.partial + static_cast<long>(bh) * p.n_split * (kD + 2);
    // all partials of this thread's column in flight together (n_split <= kDecodeMaxSplit)
    float ms[kDecodeMaxSplit], ls[kDecodeMaxSplit], os[kDecodeMaxSplit];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int s = 0; s < kDecodeMaxSplit; ++s) {
        if (s < p.n_split) {
            ms[s] = part[s * (kD + 2)];
            ls[s] = part[s * (kD + 2) + 1];
            os[s] = part[s * (kD + 2) + 2 + c];
            M = fmaxf(M, ms[s]);
        }
    }
    float L = 0.0f, acc = 0.0f;
#pragma unroll
    for (int s = 0; s < kDecodeMaxSplit; ++s) {
        if (s < p.n_split && ms[s] != -CUDART_INF_F) {   // skip empty chunks
            const float f = ex2_approx(ms[s] - M);
            L += ls[s] * f;
            acc += os[s] * f;
        }
    }
    // ctx of the step is [1, B, d_model]: the head's slab of row b
    p.ctx[static_cast<long>(b) * p.h * kD + head * kD + c] = __float2bfloat16_rn(acc / L);
    if (head == 0 && c == 0) {   // every read of the old length is done: count the new token
        const int len = p.cache_len[b];
        if (len >= 0 && len < p.L_max)
            p.cache_len[b] = len + 1;
        else
            atomicCAS(p.status, 0, 0x301);   // cache full: the token was not appended
    }
}

}  // namespace

cudaError_t launch_kv_append(const DecodeParams& p, cudaStream_t s) {
    if (p.dk == 128) return launch_pdl(kv_append_kernel<128>, dim3(p.B), dim3(256), 0, s, p);
    return launch_pdl(kv_append_kernel<64>, dim3(p.B), dim3(256), 0, s, p);
}

template <int kD>
cudaError_t launch_decode_attention_d(const DecodeParams& p, cudaStream_t s) {
    cudaError_t e = launch_pdl(decode_attn_kernel<kD>, dim3(p.n_split, p.B * p.h), dim3(32 * kWarps), 0, s, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_combine_kernel<kD>, dim3(p.B * p.h), dim3(kD), 0, s, p);
}

cudaError_t launch_decode_attention(const DecodeParams& p, cudaStream_t s) {
    return p.dk == 128 ? launch_decode_attention_d<128>(p, s) : launch_decode_attention_d<64>(p, s);
}

}  // namespace mha
