// mha_api.cu -- the C ABI declared in include/mha.h: argument validation,
// workspace layout, TMA tensor-map encoding and the three-stage dispatch of
// MultiHeadedAttention.forward ("003-Transformer" tutorial, section
// "Multi-head attention"): projections + head split, attention per head +
// concat, output projection.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/mha.h"
#include "gemm_pair.h"
#include "gemv.h"
#include "convert.h"
#include "mha_internal.h"

namespace {

thread_local std::string g_last_error;

__device__ int g_device_status;   // bounded-wait give-ups recorded by the kernels

mha_status_t fail(mha_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

mha_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(MHA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- workspace layout
struct Layout {
    size_t q, kv, ctx, stat, sched, total;
};

// Workspace of a bf16 problem run on the fp32 kernels: the fp32 forward's own
// workspace, then fp32 copies of query, key, value, the four weights and biases,
// and the fp32 output.
struct F32Copies {
    size_t ws, q, k, v, w, b, out, total;
};

bool layout_of(mha_dtype_t dt, int B, int Lq, int Lk, int d, int h, Layout* L) {
    if (B <= 0 || Lq <= 0 || Lk <= 0 || d <= 0 || h <= 0 || d % h != 0) return false;
    if (dt != MHA_F32 && dt != MHA_BF16) return false;
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    const size_t dk = static_cast<size_t>(d / h);
    L->q = 0;
    L->kv = align256(L->q + es * B * h * static_cast<size_t>(Lq) * dk);
    L->ctx = align256(L->kv + es * B * 2 * h * static_cast<size_t>(Lk) * dk);
    L->stat = align256(L->ctx + es * B * static_cast<size_t>(Lq) * d);
    L->sched = align256(L->stat + sizeof(float) * 2 * B * h * static_cast<size_t>(Lq));
    L->total = L->sched + 256;   // the persistent attention's schedule counter (2 ints)
    return true;
}

void f32_copies_of(int B, int Lq, int Lk, int d, int h, F32Copies* C) {
    Layout L;
    layout_of(MHA_F32, B, Lq, Lk, d, h, &L);
    const size_t qn = 4ull * B * Lq * d, kn = 4ull * B * Lk * d;
    C->ws = 0;
    C->q = align256(L.total);
    C->k = align256(C->q + qn);
    C->v = align256(C->k + kn);
    C->w = align256(C->v + kn);
    C->b = align256(C->w + 4ull * 4 * d * d);
    C->out = align256(C->b + 4ull * 4 * d);
    C->total = align256(C->out + qn);
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

mha_status_t get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return fail(MHA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return MHA_OK;
}

// bf16 tiled map, 128-byte swizzle (or none), zero fill out of bounds.
mha_status_t encode_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box, const char* what,
                         bool swizzle = true) {
    uint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MHA_ERR_CUDA, "tensor map encode failed for %s (CUresult %d)", what, (int)r);
    return MHA_OK;
}

// [B, L_stride, N] row-major bf16, first L rows of each sequence, as {N, L, B}, box {64, 128, 1}
mha_status_t map_rows(CUtensorMap* m, const void* base, int B, int L, int N, const char* what, int L_stride = 0) {
    if (L_stride <= 0) L_stride = L;
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)L, (uint64_t)B};
    const uint64_t str[2] = {(uint64_t)N * 2, (uint64_t)L_stride * N * 2};
    const uint32_t box[3] = {64, 128, 1};
    return encode_bf16(m, base, 3, dims, str, box, what);
}
// weight [N, K] as {K, N}, box {64, rows}: kGemmBN rows for the one-SM GEMM, half of
// that for the pair GEMM (each CTA of a pair loads its half of the 256 columns)
mha_status_t map_weight(CUtensorMap* m, const void* base, int N, int K, int rows) {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, (uint32_t)rows};
    return encode_bf16(m, base, 2, dims, str, box, "weight");
}

// Launch a projection GEMM whose groups, input and output maps are set: the pair
// kernel (two SMs per 256-row tile, one MMA of M = 256) when every group has at
// least 512 rows per batch item and there is at least a full wave of SM pairs,
// else the one-SM kernel. Builds the weight maps W[g] ([N, K]) for the chosen one.
mha_status_t launch_projection(mha::GemmParams& p, const void* const* W, cudaStream_t s, const char* what) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return fail(MHA_ERR_CUDA, "device query failed");
    const int n_tiles = (p.N + mha::kGemmBN - 1) / mha::kGemmBN;
    bool pair = true;
    long units = 0;
    int max_m = 0;
    for (int g = 0; g < p.ngroups; ++g) {
        if (p.g[g].L < 4 * mha::kGemmBM) pair = false;
        units += static_cast<long>(p.g[g].m_tiles / p.g[g].tiles_per_b) *
                 ((p.g[g].L + 2 * mha::kGemmBM - 1) / (2 * mha::kGemmBM)) * n_tiles;
        max_m = std::max(max_m, p.g[g].m_tiles);
    }
    if (units < sms / 2) pair = false;
    mha_status_t st;
    for (int g = 0; g < p.ngroups; ++g)
        if ((st = map_weight(&p.w[g], W[g], p.N, p.K, pair ? mha::kGemmBN / 2 : mha::kGemmBN)) != MHA_OK) return st;
    cudaError_t e = pair ? mha::launch_gemm_tc2(p, s) : mha::launch_gemm_tc(p, max_m, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return MHA_OK;
}
// head-split [B, planes, L_stride, d_k] (first L rows of each plane used), d_k = 64 * dks, as
// {64, dks, L, planes, B}: a 64-column slab is (0, half, row, plane, b); box {64, 1, 128, 1, 1}
mha_status_t map_heads5(CUtensorMap* m, const void* base, int B, int planes, int L, int dks, int L_stride = 0) {
    if (L_stride <= 0) L_stride = L;
    const uint64_t row = 128ull * dks;
    const uint64_t dims[5] = {64, (uint64_t)dks, (uint64_t)L, (uint64_t)planes, (uint64_t)B};
    const uint64_t str[4] = {128, row, (uint64_t)L_stride * row, (uint64_t)planes * L_stride * row};
    const uint32_t box[5] = {64, 1, 128, 1, 1};
    return encode_bf16(m, base, 5, dims, str, box, "head-split output");
}
// head-split [planes, L, d_k] as {64, dks, L, planes}, box {64, 1, 128, 1} (attention loads)
mha_status_t map_heads4d(CUtensorMap* m, const void* base, int planes, int L, int dks) {
    const uint64_t row = 128ull * dks;
    const uint64_t dims[4] = {64, (uint64_t)dks, (uint64_t)L, (uint64_t)planes};
    const uint64_t str[3] = {128, row, (uint64_t)L * row};
    const uint32_t box[4] = {64, 1, 128, 1};
    return encode_bf16(m, base, 4, dims, str, box, "head-split input");
}
// Heads narrower than 64 (d_k = 8, 16, 32: 64 / d_k heads per 64-column slab of a
// projection tile). Projection store: head-split [B, planes, L_stride, d_k] as
// {d_k, L, planes, B}, unswizzled; a box {d_k, 128, 64/d_k, 1} holds the slab's heads
// one after the other (the GEMM epilogue stages them head-major, each 128 x d_k dense).
mha_status_t map_heads4_narrow(CUtensorMap* m, const void* base, int B, int planes, int L, int dk,
                               int L_stride = 0) {
    if (L_stride <= 0) L_stride = L;
    const uint64_t plane = (uint64_t)L_stride * dk * 2;
    const uint64_t dims[4] = {(uint64_t)dk, (uint64_t)L, (uint64_t)planes, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)dk * 2, plane, (uint64_t)planes * plane};
    const uint32_t box[4] = {(uint32_t)dk, 128, (uint32_t)(64 / dk), 1};
    return encode_bf16(m, base, 4, dims, str, box, "narrow head-split output", false);
}
// Attention loads of narrow heads: [planes, L, d_k] as {d_k, L, planes} with a box of 64
// columns: the columns past d_k are out of bounds and arrive as zeros, so the d_k = 64
// kernel computes exactly the narrow head's scores and a zero-padded P.V.
mha_status_t map_heads3_narrow(CUtensorMap* m, const void* base, int planes, int L, int dk) {
    const uint64_t dims[3] = {(uint64_t)dk, (uint64_t)L, (uint64_t)planes};
    const uint64_t str[2] = {(uint64_t)dk * 2, (uint64_t)L * dk * 2};
    const uint32_t box[3] = {64, 128, 1};
    return encode_bf16(m, base, 3, dims, str, box, "narrow head-split input");
}
// head-split [planes, L, 64] as {64, L, planes}, box {64, 128, 1}
mha_status_t map_heads3(CUtensorMap* m, const void* base, int planes, int L) {
    const uint64_t dims[3] = {64, (uint64_t)L, (uint64_t)planes};
    const uint64_t str[2] = {128, (uint64_t)L * 128};
    const uint32_t box[3] = {64, 128, 1};
    return encode_bf16(m, base, 3, dims, str, box, "head-split input");
}

int* device_status_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

// ---------------------------------------------------------------- validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Heads narrower than 64 that the d_k = 64 kernels take (zero-padded to 64 columns).
bool narrow_dk(int d, int h) {
    const int dk = d / h;
    return (dk == 8 || dk == 16 || dk == 32) && d % 64 == 0;
}
// bf16 head widths the tensor-core kernels take; other widths up to 256 run (in
// mha_forward only) on the fp32 kernels over converted copies.
bool bf16_native(int d, int h) { return d / h == 64 || d / h == 128 || narrow_dk(d, h); }

mha_status_t check_sizes(mha_dtype_t dt, int B, int Lq, int Lk, int d, int h, bool bf16_any_dk = false) {
    if (dt != MHA_F32 && dt != MHA_BF16) return fail(MHA_ERR_INVALID_ARG, "dtype %d is not MHA_F32 or MHA_BF16", dt);
    if (B <= 0 || Lq <= 0 || Lk <= 0 || d <= 0 || h <= 0)
        return fail(MHA_ERR_INVALID_ARG, "sizes must be positive (B=%d L_q=%d L_k=%d d_model=%d h=%d)", B, Lq, Lk, d,
                    h);
    if (d % h != 0) return fail(MHA_ERR_INVALID_ARG, "d_model %% h != 0 (d_model=%d, h=%d)", d, h);
    const int dk = d / h;
    if (dt == MHA_BF16 && !bf16_native(d, h) && !(bf16_any_dk && dk <= 256))
        return fail(MHA_ERR_UNSUPPORTED,
                    "this bf16 entry point implements d_k = 64 and 128, and 8, 16, 32 with d_model %% 64 == 0 "
                    "(d_k = %d, d_model = %d)", dk, d);
    if (dk > 256) return fail(MHA_ERR_UNSUPPORTED, "d_k <= 256 is implemented (d_k = %d)", dk);
    const double big = static_cast<double>(B) * h * Lq * Lk;
    if (static_cast<double>(B) * Lq * d > 4.0e9 || static_cast<double>(B) * Lk * d * 2 > 4.0e9 || big > 1.0e15)
        return fail(MHA_ERR_UNSUPPORTED, "problem too large for 32-bit tile indices");
    return MHA_OK;
}

mha_status_t check_workspace(mha_dtype_t dt, int B, int Lq, int Lk, int d, int h, const void* ws, size_t bytes,
                             Layout* L) {
    layout_of(dt, B, Lq, Lk, d, h, L);
    if (ws == nullptr) return fail(MHA_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(MHA_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (bytes < L->total)
        return fail(MHA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", bytes, L->total);
    return MHA_OK;
}

mha_status_t check_mask(const mha_mask_t* mask, int Lq, int Lk) {
    if (mask == nullptr) return MHA_OK;
    if (mask->causal && Lq != Lk)
        return fail(MHA_ERR_INVALID_ARG, "causal mask needs L_q == L_k (got %d, %d)", Lq, Lk);
    if (mask->dense != nullptr && mask->dense_mq != 1 && mask->dense_mq != Lq)
        return fail(MHA_ERR_INVALID_ARG, "dense_mq must be 1 or L_q (got %d)", mask->dense_mq);
    return MHA_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }


// Stage implementations without argument checks (defined below). A row window
// [r0, r0 + rows) (rows > 0) restricts a projection to those sequence rows of the
// full-length tensors.
mha_status_t qkv_bf16_impl(const void* query, const void* key, const void* value, const void* w_q, const void* b_q,
                           const void* w_k, const void* b_k, const void* w_v, const void* b_v, int B, int L_q,
                           int L_k, int d_model, int h, const Layout& L, uint8_t* ws, cudaStream_t s, int r0,
                           int rows);
mha_status_t attention_impl(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h, const mha_mask_t* mask,
                            float* p_attn, const Layout& L, uint8_t* ws, cudaStream_t s);
mha_status_t output_projection_impl(mha_dtype_t dt, const void* w_o, const void* b_o, const void* residual,
                                    int B, int L_q, int d_model, int h, void* out, const Layout& L, uint8_t* ws,
                                    cudaStream_t s, int r0 = 0, int rows = 0);
mha_status_t forward_bf16_on_f32(const void* query, const void* key, const void* value, const void* w_q,
                                 const void* b_q, const void* w_k, const void* b_k, const void* w_v, const void* b_v,
                                 const void* w_o, const void* b_o, int B, int L_q, int L_k, int d_model, int h,
                                 const mha_mask_t* mask, void* out, float* p_attn, void* workspace,
                                 size_t workspace_bytes, cudaStream_t s);

}  // namespace

void mha::set_last_error(const char* msg) { g_last_error = msg; }

// ==================================================================== C ABI
extern "C" {

const char* mha_version(void) { return "gb300-mha 0.1 (sm_103a)"; }

const char* mha_last_error(void) { return g_last_error.c_str(); }

size_t mha_workspace_size(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h) {
    Layout L;
    if (!layout_of(dt, B, L_q, L_k, d_model, h, &L)) return 0;
    if (dt == MHA_BF16 && !bf16_native(d_model, h) && d_model / h <= 256) {
        F32Copies C;
        f32_copies_of(B, L_q, L_k, d_model, h, &C);
        return C.total;
    }
    return L.total;
}

mha_status_t mha_qkv_projection(mha_dtype_t dt, const void* query, const void* key, const void* value,
                                const void* w_q, const void* b_q, const void* w_k, const void* b_k,
                                const void* w_v, const void* b_v, int B, int L_q, int L_k, int d_model, int h,
                                void* workspace, size_t workspace_bytes, void* stream) {
    mha_status_t st = check_sizes(dt, B, L_q, L_k, d_model, h);
    if (st != MHA_OK) return st;
    if (!query || !key || !value || !w_q || !w_k || !w_v)
        return fail(MHA_ERR_INVALID_ARG, "query, key, value and W_q, W_k, W_v must not be NULL");
    Layout L;
    if ((st = check_workspace(dt, B, L_q, L_k, d_model, h, workspace, workspace_bytes, &L)) != MHA_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int dk = d_model / h;
    const cudaStream_t s = as_stream(stream);

    if (dt == MHA_F32) {
        mha::F32GemmParams p{};
        const void* A[3] = {query, key, value};
        const void* W[3] = {w_q, w_k, w_v};
        const void* bias[3] = {b_q, b_k, b_v};
        // one launch, three groups: Q -> Qh [B, h, L_q, dk]; K, V -> planes 0..h-1 and h..2h-1
        // of KVh [B, 2h, L_k, dk]
        for (int g = 0; g < 3; ++g) {
            p.g[g].A = static_cast<const float*>(A[g]);
            p.g[g].W = static_cast<const float*>(W[g]);
            p.g[g].bias = static_cast<const float*>(bias[g]);
            p.g[g].out = reinterpret_cast<float*>(ws + (g == 0 ? L.q : L.kv));
            p.g[g].L = g == 0 ? L_q : L_k;
            p.g[g].out_j0 = g == 2 ? h : 0;
            p.g[g].slabs = g == 0 ? h : 2 * h;
        }
        p.ngroups = 3;
        p.B = B;
        p.K = d_model;
        p.N = d_model;
        p.dk = dk;
        p.out_plain = 0;
        cudaError_t e = mha::launch_gemm_f32(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "Q/K/V projection launch");
        return MHA_OK;
    }

    // ---- bf16: one tensor-core launch, three groups
    const void* ptrs[9] = {query, key, value, w_q, w_k, w_v, b_q, b_k, b_v};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    return qkv_bf16_impl(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, B, L_q, L_k, d_model, h, L, ws, s, 0, 0);
}

}  // extern "C"

namespace {

// bf16 Q/K/V projections into the workspace's head-split tensors; no argument checks.
// rows > 0 restricts all three to the sequence rows [r0, r0 + rows) (self-attention,
// L_q == L_k): the maps address that window of the full-length tensors.
mha_status_t qkv_bf16_impl(const void* query, const void* key, const void* value, const void* w_q, const void* b_q,
                           const void* w_k, const void* b_k, const void* w_v, const void* b_v, int B, int L_q,
                           int L_k, int d_model, int h, const Layout& L, uint8_t* ws, cudaStream_t s, int r0,
                           int rows) {
    const int dk = d_model / h;
    const bool narrow = narrow_dk(d_model, h);
    mha_status_t st;
    if ((st = get_encoder()) != MHA_OK) return st;
    mha::GemmParams p;
    memset(&p, 0, sizeof(p));
    const void* A[3] = {query, key, value};
    const void* W[3] = {w_q, w_k, w_v};
    const void* bias[3] = {b_q, b_k, b_v};
    const int Lfull[3] = {L_q, L_k, L_k};
    const int Ls[3] = {rows > 0 ? rows : L_q, rows > 0 ? rows : L_k, rows > 0 ? rows : L_k};
    const size_t in_off = static_cast<size_t>(r0) * d_model * 2;    // window start in an input row block
    const size_t out_off = static_cast<size_t>(r0) * dk * 2;        // ... in a head plane
    int max_m = 0;
    for (int g = 0; g < 3; ++g) {
        if ((st = map_rows(&p.a[g], static_cast<const uint8_t*>(A[g]) + in_off, B, Ls[g], d_model,
                           "projection input", Lfull[g])) != MHA_OK)
            return st;
        if (narrow) {
            st = (g == 0) ? map_heads4_narrow(&p.out[g], ws + L.q + out_off, B, h, Ls[g], dk, L_q)
                          : map_heads4_narrow(&p.out[g], ws + L.kv + out_off, B, 2 * h, Ls[g], dk, L_k);
            if (st != MHA_OK) return st;
        } else if (g == 0) {
            if ((st = map_heads5(&p.out[g], ws + L.q + out_off, B, h, Ls[g], dk / 64, L_q)) != MHA_OK) return st;
        } else {
            if ((st = map_heads5(&p.out[g], ws + L.kv + out_off, B, 2 * h, Ls[g], dk / 64, L_k)) != MHA_OK)
                return st;
        }
        p.g[g].L = Ls[g];
        p.g[g].tiles_per_b = (Ls[g] + mha::kGemmBM - 1) / mha::kGemmBM;
        p.g[g].m_tiles = B * p.g[g].tiles_per_b;
        p.g[g].out_j0 = (g == 2) ? h : 0;   // first plane of V in KVh
        p.g[g].bias = static_cast<const __nv_bfloat16*>(bias[g]);
        max_m = std::max(max_m, p.g[g].m_tiles);
    }
    p.ngroups = 3;
    p.K = d_model;
    p.N = d_model;
    p.out_plain = 0;
    p.dk_slabs = narrow ? 1 : dk / 64;
    p.narrow_shift = narrow ? (dk == 8 ? 3 : dk == 16 ? 4 : 5) : 0;
    p.zero_words = reinterpret_cast<int*>(ws + L.sched);
    p.status = device_status_ptr();
    if (!p.status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    (void)max_m;
    return launch_projection(p, W, s, "QKV projection launch");
}

}  // namespace

extern "C" {

mha_status_t mha_attention_core(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h,
                                const mha_mask_t* mask, float* p_attn, void* workspace, size_t workspace_bytes,
                                void* stream) {
    mha_status_t st = check_sizes(dt, B, L_q, L_k, d_model, h);
    if (st != MHA_OK) return st;
    if ((st = check_mask(mask, L_q, L_k)) != MHA_OK) return st;
    Layout L;
    if ((st = check_workspace(dt, B, L_q, L_k, d_model, h, workspace, workspace_bytes, &L)) != MHA_OK) return st;
    return attention_impl(dt, B, L_q, L_k, d_model, h, mask, p_attn, L, static_cast<uint8_t*>(workspace),
                          as_stream(stream));
}

}  // extern "C"

namespace {

mha_status_t attention_impl(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h, const mha_mask_t* mask,
                            float* p_attn, const Layout& L, uint8_t* ws, cudaStream_t s) {
    mha_status_t st;
    const int dk = d_model / h;
    const int causal = mask ? (mask->causal != 0) : 0;
    const int32_t* vl = mask ? mask->key_valid_lens : nullptr;
    const uint8_t* dense = mask ? mask->dense : nullptr;
    const int dmq = (mask && mask->dense) ? mask->dense_mq : 0;

    if (dt == MHA_F32) {
        mha::F32AttnParams p{};
        p.q = reinterpret_cast<const float*>(ws + L.q);
        p.kv = reinterpret_cast<const float*>(ws + L.kv);
        p.ctx = reinterpret_cast<float*>(ws + L.ctx);
        p.p_attn = p_attn;
        p.B = B; p.h = h; p.Lq = L_q; p.Lk = L_k; p.dk = dk;
        p.causal = causal; p.valid_lens = vl; p.dense = dense; p.dense_mq = dmq;
        cudaError_t e = mha::launch_attn_f32(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 attention launch");
        return MHA_OK;
    }

    if ((st = get_encoder()) != MHA_OK) return st;
    mha::AttnParams p;
    memset(&p, 0, sizeof(p));
    const bool narrow = narrow_dk(d_model, h);
    if (dk == 64) {
        if ((st = map_heads3(&p.q_map, ws + L.q, B * h, L_q)) != MHA_OK) return st;
        if ((st = map_heads3(&p.kv_map, ws + L.kv, B * 2 * h, L_k)) != MHA_OK) return st;
    } else if (narrow) {
        if ((st = map_heads3_narrow(&p.q_map, ws + L.q, B * h, L_q, dk)) != MHA_OK) return st;
        if ((st = map_heads3_narrow(&p.kv_map, ws + L.kv, B * 2 * h, L_k, dk)) != MHA_OK) return st;
    } else {
        if ((st = map_heads4d(&p.q_map, ws + L.q, B * h, L_q, dk / 64)) != MHA_OK) return st;
        if ((st = map_heads4d(&p.kv_map, ws + L.kv, B * 2 * h, L_k, dk / 64)) != MHA_OK) return st;
    }
    if (narrow) {
        // the head's d_k columns of ctx, stored from a dense (unswizzled) 128 x d_k staging tile
        const uint64_t dims[3] = {(uint64_t)d_model, (uint64_t)L_q, (uint64_t)B};
        const uint64_t str[2] = {(uint64_t)d_model * 2, (uint64_t)L_q * d_model * 2};
        const uint32_t box[3] = {(uint32_t)dk, 128, 1};
        if ((st = encode_bf16(&p.ctx_map, ws + L.ctx, 3, dims, str, box, "context (narrow heads)", false)) != MHA_OK)
            return st;
        p.narrow_dk = dk;
    } else if ((st = map_rows(&p.ctx_map, ws + L.ctx, B, L_q, d_model, "context")) != MHA_OK) {
        return st;
    }
    p.B = B; p.h = h; p.Lq = L_q; p.Lk = L_k;
    p.causal = causal; p.valid_lens = vl; p.dense = dense; p.dense_mq = dmq;
    p.stats = p_attn ? reinterpret_cast<float*>(ws + L.stat) : nullptr;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(dk)));
    const bool d128 = dk == 128;
    const int q_rows = d128 ? mha::kAttnBM : 2 * mha::kAttnBM;   // query rows per CTA
    p.q_pairs = (L_q + q_rows - 1) / q_rows;
    p.sched = reinterpret_cast<int*>(ws + L.sched);
    p.status = device_status_ptr();
    if (!p.status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    cudaError_t e = d128 ? mha::launch_attn_tc_d128(p, s) : mha::launch_attn_tc(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    if (p_attn) {
        p.p_attn = p_attn;
        if (L_k % 4 == 0 && aligned16(p_attn)) {
            // fp32 [B*h, L_q, L_k] as {L_k, L_q, B*h}, box {32, 128, 1}, 128-byte swizzle
            const uint64_t dims[3] = {(uint64_t)L_k, (uint64_t)L_q, (uint64_t)B * h};
            const uint64_t str[2] = {(uint64_t)L_k * 4, (uint64_t)L_q * L_k * 4};
            const uint32_t box[3] = {32, 128, 1};
            uint32_t estr[3] = {1, 1, 1};
            CUresult r = g_encode(&p.p_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p_attn, dims, str, box, estr,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return fail(MHA_ERR_CUDA, "tensor map encode failed for p_attn (CUresult %d)", (int)r);
        }
        e = mha::launch_pattn_tc(p, d128 ? 2 : 1, s);
        if (e != cudaSuccess) return cuda_fail(e, "p_attn launch");
    }
    return MHA_OK;
}

// out = ctx W_o^T + b_o (+ residual), reading ctx from the workspace; no argument checks.
mha_status_t output_projection_impl(mha_dtype_t dt, const void* w_o, const void* b_o, const void* residual,
                                    int B, int L_q, int d_model, int h, void* out, const Layout& L, uint8_t* ws,
                                    cudaStream_t s, int r0, int rows) {
    if (dt == MHA_F32) {
        mha::F32GemmParams p{};
        p.ngroups = 1;
        p.B = B; p.K = d_model; p.N = d_model; p.dk = d_model / h; p.g[0].slabs = 1; p.out_plain = 1;
        p.g[0].A = reinterpret_cast<const float*>(ws + L.ctx);
        p.g[0].W = static_cast<const float*>(w_o);
        p.g[0].bias = static_cast<const float*>(b_o);
        p.g[0].residual = static_cast<const float*>(residual);
        p.g[0].out = static_cast<float*>(out);
        p.g[0].L = L_q;
        cudaError_t e = mha::launch_gemm_f32(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 output projection launch");
        return MHA_OK;
    }
    mha_status_t st = get_encoder();
    if (st != MHA_OK) return st;
    mha::GemmParams p;
    memset(&p, 0, sizeof(p));
    const int Lw = rows > 0 ? rows : L_q;
    const size_t off = static_cast<size_t>(r0) * d_model * 2;
    if ((st = map_rows(&p.a[0], ws + L.ctx + off, B, Lw, d_model, "context", L_q)) != MHA_OK) return st;
    if ((st = map_rows(&p.out[0], static_cast<uint8_t*>(out) + off, B, Lw, d_model, "output", L_q)) != MHA_OK)
        return st;
    if (residual && rows > 0)   // the epilogue indexes the residual with the window's own row count
        return fail(MHA_ERR_UNSUPPORTED, "row-window output projection takes no residual");
    p.g[0].L = Lw;
    p.g[0].tiles_per_b = (Lw + mha::kGemmBM - 1) / mha::kGemmBM;
    p.g[0].m_tiles = B * p.g[0].tiles_per_b;
    p.g[0].bias = static_cast<const __nv_bfloat16*>(b_o);
    p.g[0].residual = static_cast<const __nv_bfloat16*>(residual);
    p.ngroups = 1;
    p.K = d_model;
    p.N = d_model;
    p.out_plain = 1;
    p.status = device_status_ptr();
    if (!p.status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    const void* W[1] = {w_o};
    return launch_projection(p, W, s, "output projection launch");
}

// A bf16 problem whose head width the tensor-core kernels do not take: convert the
// activations, weights and biases to fp32 copies in the workspace, run the fp32
// forward on them, convert the output back (round to nearest even).
mha_status_t forward_bf16_on_f32(const void* query, const void* key, const void* value, const void* w_q,
                                 const void* b_q, const void* w_k, const void* b_k, const void* w_v, const void* b_v,
                                 const void* w_o, const void* b_o, int B, int L_q, int L_k, int d_model, int h,
                                 const mha_mask_t* mask, void* out, float* p_attn, void* workspace,
                                 size_t workspace_bytes, cudaStream_t s) {
    F32Copies C;
    f32_copies_of(B, L_q, L_k, d_model, h, &C);
    if (workspace == nullptr) return fail(MHA_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MHA_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (workspace_bytes < C.total)
        return fail(MHA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, C.total);
    const void* ptrs[13] = {query, key, value, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, out, p_attn};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    using bf = const __nv_bfloat16*;
    const long qn = static_cast<long>(B) * L_q * d_model, kn = static_cast<long>(B) * L_k * d_model;
    const long dd = static_cast<long>(d_model) * d_model;
    // A shared input is converted once, but only when both views cover the same rows: a
    // key that starts at the query's address but is longer (L_k > L_q) has rows the query's
    // conversion never touches, so it gets its own copy.
    float* q32 = reinterpret_cast<float*>(ws + C.q);
    const bool k_is_q = key == query && L_k == L_q;
    float* k32 = k_is_q ? q32 : reinterpret_cast<float*>(ws + C.k);
    float* v32 = value == key ? k32 : reinterpret_cast<float*>(ws + C.v);
    float* w32 = reinterpret_cast<float*>(ws + C.w);
    float* b32 = reinterpret_cast<float*>(ws + C.b);
    float* o32 = reinterpret_cast<float*>(ws + C.out);
    cudaError_t e = mha::launch_bf16_to_f32(static_cast<bf>(query), q32, qn, s);
    if (e == cudaSuccess && !k_is_q) e = mha::launch_bf16_to_f32(static_cast<bf>(key), k32, kn, s);
    if (e == cudaSuccess && value != key) e = mha::launch_bf16_to_f32(static_cast<bf>(value), v32, kn, s);
    const void* W[4] = {w_q, w_k, w_v, w_o};
    const void* bias[4] = {b_q, b_k, b_v, b_o};
    const float* b_f32[4] = {nullptr, nullptr, nullptr, nullptr};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) {
        e = mha::launch_bf16_to_f32(static_cast<bf>(W[i]), w32 + i * dd, dd, s);
        if (e == cudaSuccess && bias[i]) {
            e = mha::launch_bf16_to_f32(static_cast<bf>(bias[i]), b32 + i * d_model, d_model, s);
            b_f32[i] = b32 + i * d_model;
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "bf16 to fp32 conversion launch");
    mha_status_t st = mha_forward(MHA_F32, q32, k32, v32, w32, b_f32[0], w32 + dd, b_f32[1], w32 + 2 * dd, b_f32[2],
                                  w32 + 3 * dd, b_f32[3], B, L_q, L_k, d_model, h, mask, o32, p_attn, ws, C.q, s);
    if (st != MHA_OK) return st;
    e = mha::launch_f32_to_bf16(o32, static_cast<__nv_bfloat16*>(out), qn, s);
    if (e != cudaSuccess) return cuda_fail(e, "fp32 to bf16 conversion launch");
    return MHA_OK;
}

}  // namespace

extern "C" {

mha_status_t mha_output_projection(mha_dtype_t dt, const void* w_o, const void* b_o, int B, int L_q, int L_k,
                                   int d_model, int h, void* out, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    mha_status_t st = check_sizes(dt, B, L_q, L_k, d_model, h);
    if (st != MHA_OK) return st;
    if (!w_o || !out) return fail(MHA_ERR_INVALID_ARG, "W_o and out must not be NULL");
    Layout L;
    if ((st = check_workspace(dt, B, L_q, L_k, d_model, h, workspace, workspace_bytes, &L)) != MHA_OK) return st;
    if (dt == MHA_BF16 && (!aligned16(w_o) || !aligned16(out) || (b_o && !aligned16(b_o))))
        return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    return output_projection_impl(dt, w_o, b_o, nullptr, B, L_q, d_model, h, out, L,
                                  static_cast<uint8_t*>(workspace), as_stream(stream));
}

mha_status_t mha_forward(mha_dtype_t dt, const void* query, const void* key, const void* value, const void* w_q,
                         const void* b_q, const void* w_k, const void* b_k, const void* w_v, const void* b_v,
                         const void* w_o, const void* b_o, int B, int L_q, int L_k, int d_model, int h,
                         const mha_mask_t* mask, void* out, float* p_attn, void* workspace, size_t workspace_bytes,
                         void* stream) {
    // Validate everything before enqueueing anything.
    mha_status_t st = check_sizes(dt, B, L_q, L_k, d_model, h, true);
    if (st != MHA_OK) return st;
    if ((st = check_mask(mask, L_q, L_k)) != MHA_OK) return st;
    if (!query || !key || !value || !w_q || !w_k || !w_v || !w_o || !out)
        return fail(MHA_ERR_INVALID_ARG, "query, key, value, W_q, W_k, W_v, W_o and out must not be NULL");
    if (dt == MHA_BF16 && !bf16_native(d_model, h))
        return forward_bf16_on_f32(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, B, L_q, L_k, d_model,
                                   h, mask, out, p_attn, workspace, workspace_bytes, as_stream(stream));
    Layout L;
    if ((st = check_workspace(dt, B, L_q, L_k, d_model, h, workspace, workspace_bytes, &L)) != MHA_OK) return st;
    if (dt == MHA_BF16) {
        const void* ptrs[13] = {query, key, value, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, out, p_attn};
        for (const void* ptr : ptrs)
            if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    }
    if ((st = mha_qkv_projection(dt, query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, B, L_q, L_k, d_model, h,
                                 workspace, workspace_bytes, stream)) != MHA_OK)
        return st;
    if ((st = mha_attention_core(dt, B, L_q, L_k, d_model, h, mask, p_attn, workspace, workspace_bytes, stream)) !=
        MHA_OK)
        return st;
    return mha_output_projection(dt, w_o, b_o, B, L_q, L_k, d_model, h, out, workspace, workspace_bytes, stream);
}

size_t mha_sublayer_workspace_size(mha_dtype_t dt, int B, int L, int L_mem, int d_model, int h) {
    const size_t ws = mha_workspace_size(dt, B, L, L_mem > 0 ? L_mem : L, d_model, h);
    if (ws == 0) return 0;
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    return align256(es * B * static_cast<size_t>(L) * d_model) + ws;
}

mha_status_t mha_sublayer_forward(mha_dtype_t dt, const void* x, const void* memory, const void* ln_gain,
                                  const void* ln_bias, float ln_eps, int ln_kind, const void* w_q, const void* b_q,
                                  const void* w_k, const void* b_k, const void* w_v, const void* b_v,
                                  const void* w_o, const void* b_o, int B, int L, int L_mem, int d_model, int h,
                                  const mha_mask_t* mask, void* out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    const int Lk = memory ? L_mem : L;
    mha_status_t st = check_sizes(dt, B, L, Lk, d_model, h);
    if (st != MHA_OK) return st;
    if ((st = check_mask(mask, L, Lk)) != MHA_OK) return st;
    if (!x || !w_q || !w_k || !w_v || !w_o || !out)
        return fail(MHA_ERR_INVALID_ARG, "x, W_q, W_k, W_v, W_o and out must not be NULL");
    if (ln_kind != 0 && ln_kind != 1) return fail(MHA_ERR_INVALID_ARG, "ln_kind must be 0 or 1 (got %d)", ln_kind);
    if (ln_kind == 0 && d_model < 2) return fail(MHA_ERR_INVALID_ARG, "unbiased std needs d_model >= 2");
    if (!(ln_eps >= 0.0f)) return fail(MHA_ERR_INVALID_ARG, "ln_eps must be >= 0");
    if (d_model > mha::layernorm_max_d())
        return fail(MHA_ERR_UNSUPPORTED, "LayerNorm implements d_model <= %d", mha::layernorm_max_d());
    const size_t need = mha_sublayer_workspace_size(dt, B, L, Lk, d_model, h);
    if (!workspace) return fail(MHA_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MHA_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (workspace_bytes < need) return fail(MHA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
    if (dt == MHA_BF16) {
        const void* ptrs[14] = {x, memory, ln_gain, ln_bias, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, out, workspace};
        for (const void* ptr : ptrs)
            if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    }
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    uint8_t* y = static_cast<uint8_t*>(workspace);
    uint8_t* mws = y + align256(es * B * static_cast<size_t>(L) * d_model);
    const size_t mws_bytes = workspace_bytes - (mws - y);
    const cudaStream_t s = as_stream(stream);
    // 1. y = LayerNorm(x)
    mha::LayerNormParams ln{};
    ln.x = x; ln.y = y; ln.gain = ln_gain; ln.bias = ln_bias;
    ln.rows = static_cast<long>(B) * L; ln.d = d_model; ln.eps = ln_eps; ln.kind = ln_kind;
    ln.bf16 = dt == MHA_BF16;
    cudaError_t e = mha::launch_layernorm(ln, s);
    if (e != cudaSuccess) return cuda_fail(e, "LayerNorm launch");
    // 2. attention sublayer on y (self) or on (y, memory, memory) (source attention)
    const void* kv = memory ? memory : y;
    if ((st = mha_qkv_projection(dt, y, kv, kv, w_q, b_q, w_k, b_k, w_v, b_v, B, L, Lk, d_model, h, mws, mws_bytes,
                                 stream)) != MHA_OK)
        return st;
    if ((st = mha_attention_core(dt, B, L, Lk, d_model, h, mask, nullptr, mws, mws_bytes, stream)) != MHA_OK)
        return st;
    // 3. out = x + (ctx W_o^T + b_o): the residual is added in the W_o epilogue
    Layout Lo;
    layout_of(dt, B, L, Lk, d_model, h, &Lo);
    return output_projection_impl(dt, w_o, b_o, x, B, L, d_model, h, out, Lo, mws, s);
}

static int decode_split(int B, int h, int L_max) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int n = (8 * sms + B * h - 1) / (B * h);    // about 8 CTAs of 4 warps per SM
    n = std::min(n, (L_max + 127) / 128);      // at least 128 keys per chunk
    return std::max(1, std::min(n, mha::kDecodeMaxSplit));
}

size_t mha_decode_workspace_size(int B, int d_model, int h, int L_max) {
    if (B <= 0 || d_model <= 0 || h <= 0 || L_max <= 0 || d_model % h != 0) return 0;
    const size_t ws = mha_workspace_size(MHA_BF16, 1, B, B, d_model, h);
    return ws + align256(sizeof(float) * (d_model / h + 2) * B * h * static_cast<size_t>(mha::kDecodeMaxSplit));
}

mha_status_t mha_kv_cache_prefill(mha_dtype_t dt, const void* x, const void* w_k, const void* b_k, const void* w_v,
                                  const void* b_v, int B, int T, int d_model, int h, void* k_cache, void* v_cache,
                                  int L_max, void* stream) {
    if (dt != MHA_BF16) return fail(MHA_ERR_UNSUPPORTED, "the key/value cache is implemented for bf16 only");
    mha_status_t st = check_sizes(dt, B, T, T, d_model, h);
    if (st != MHA_OK) return st;
    const int dk = d_model / h;
    if (dk != 64 && dk != 128)
        return fail(MHA_ERR_UNSUPPORTED, "the key/value cache is implemented for d_k = 64 and 128 (d_k = %d)", dk);
    if (T > L_max) return fail(MHA_ERR_INVALID_ARG, "T (%d) exceeds the cache length L_max (%d)", T, L_max);
    if (!x || !w_k || !w_v || !k_cache || !v_cache)
        return fail(MHA_ERR_INVALID_ARG, "x, W_k, W_v and the caches must not be NULL");
    const void* ptrs[7] = {x, w_k, b_k, w_v, b_v, k_cache, v_cache};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    if ((st = get_encoder()) != MHA_OK) return st;
    mha::GemmParams p;
    memset(&p, 0, sizeof(p));
    const void* W[2] = {w_k, w_v};
    const void* bias[2] = {b_k, b_v};
    void* cache[2] = {k_cache, v_cache};
    for (int g = 0; g < 2; ++g) {
        if ((st = map_rows(&p.a[g], x, B, T, d_model, "prefill input")) != MHA_OK) return st;
        if ((st = map_heads5(&p.out[g], cache[g], B, h, T, dk / 64, L_max)) != MHA_OK) return st;
        p.g[g].L = T;
        p.g[g].tiles_per_b = (T + mha::kGemmBM - 1) / mha::kGemmBM;
        p.g[g].m_tiles = B * p.g[g].tiles_per_b;
        p.g[g].out_j0 = 0;
        p.g[g].bias = static_cast<const __nv_bfloat16*>(bias[g]);
    }
    p.ngroups = 2;
    p.K = d_model;
    p.N = d_model;
    p.dk_slabs = dk / 64;
    p.status = device_status_ptr();
    if (!p.status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    return launch_projection(p, W, as_stream(stream), "cache prefill launch");
}

mha_status_t mha_decode_step(mha_dtype_t dt, const void* x_new, const void* w_q, const void* b_q, const void* w_k,
                             const void* b_k, const void* w_v, const void* b_v, const void* w_o, const void* b_o,
                             int B, int d_model, int h, void* k_cache, void* v_cache, int32_t* cache_len,
                             int L_max, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (dt != MHA_BF16) return fail(MHA_ERR_UNSUPPORTED, "incremental decoding is implemented for bf16 only");
    mha_status_t st = check_sizes(dt, 1, B, B, d_model, h);
    if (st != MHA_OK) return st;
    const int dk = d_model / h;
    if (dk != 64 && dk != 128)
        return fail(MHA_ERR_UNSUPPORTED, "incremental decoding is implemented for d_k = 64 and 128 (d_k = %d)", dk);
    if (L_max <= 0) return fail(MHA_ERR_INVALID_ARG, "L_max must be positive");
    if (!x_new || !w_q || !w_k || !w_v || !w_o || !k_cache || !v_cache || !cache_len || !out)
        return fail(MHA_ERR_INVALID_ARG, "x_new, weights, caches, cache_len and out must not be NULL");
    const size_t need = mha_decode_workspace_size(B, d_model, h, L_max);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MHA_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    if (workspace_bytes < need) return fail(MHA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
    const void* ptrs[11] = {x_new, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, k_cache, v_cache};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    if (!aligned16(out)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    const size_t ws_mha = mha_workspace_size(MHA_BF16, 1, B, B, d_model, h);
    Layout L;
    layout_of(dt, 1, B, B, d_model, h, &L);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool gemv = mha::gemv_supported(B, d_model);   // a few rows: stream W over many CTAs
    // 1. q, k, v of the B new tokens, head-split as for a [1, B, d_model] sequence
    if (gemv) {
        mha::GemvParams g{};
        g.x = static_cast<const __nv_bfloat16*>(x_new);
        const void* W[3] = {w_q, w_k, w_v};
        const void* bias[3] = {b_q, b_k, b_v};
        for (int i = 0; i < 3; ++i) {
            g.w[i] = static_cast<const __nv_bfloat16*>(W[i]);
            g.bias[i] = static_cast<const __nv_bfloat16*>(bias[i]);
        }
        g.out[0] = reinterpret_cast<__nv_bfloat16*>(ws + L.q);
        g.out[1] = g.out[2] = reinterpret_cast<__nv_bfloat16*>(ws + L.kv);
        g.j0[0] = 0; g.j0[1] = 0; g.j0[2] = h;
        g.M = B; g.N = d_model; g.K = d_model; g.ngroups = 3; g.head_split = 1; g.dk = dk;
        g.k_cache = static_cast<__nv_bfloat16*>(k_cache);   // k, v of the step go straight to the caches
        g.v_cache = static_cast<__nv_bfloat16*>(v_cache);
        g.cache_len = cache_len;
        g.L_max = L_max;
        cudaError_t e = mha::launch_gemv_bf16(g, as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(e, "decode Q/K/V projection launch");
    } else if ((st = mha_qkv_projection(dt, x_new, x_new, x_new, w_q, b_q, w_k, b_k, w_v, b_v, 1, B, B, d_model, h,
                                        workspace, ws_mha, stream)) != MHA_OK) {
        return st;
    }
    mha::DecodeParams p{};
    p.q_new = reinterpret_cast<const __nv_bfloat16*>(ws + L.q);
    p.kv_new = reinterpret_cast<const __nv_bfloat16*>(ws + L.kv);
    p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    p.cache_len = cache_len;
    p.ctx = reinterpret_cast<__nv_bfloat16*>(ws + L.ctx);
    p.partial = reinterpret_cast<float*>(ws + ws_mha);
    p.dk = dk;
    p.B = B;
    p.h = h;
    p.L_max = L_max;
    p.n_split = decode_split(B, h, L_max);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(dk)));
    p.status = device_status_ptr();
    if (!p.status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    // keys each attention CTA prefetches into L2 while the small-M projections run: an eighth
    // of its chunk, at most 64 MB over the grid (half of L2)
    if (gemv) {
        const long ctas = static_cast<long>(p.n_split) * B * h;
        const long chunk = (L_max + p.n_split - 1) / p.n_split;
        p.prefetch_keys = static_cast<int>(std::min<long>(chunk / 8, (64l << 20) / (ctas * 2 * dk * 2)));
    }
    const cudaStream_t s = as_stream(stream);
    // 2. (tiled projections only) append k, v at cache_len[b]; 3. attention over the cache,
    // the new token included; 4. merge, and count the new token in cache_len[b]
    cudaError_t e = cudaSuccess;
    if (!gemv && (e = mha::launch_kv_append(p, s)) != cudaSuccess) return cuda_fail(e, "cache append launch");
    e = mha::launch_decode_attention(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    // 5. out = ctx W_o^T + b_o
    if (gemv) {
        mha::GemvParams g{};
        g.x = reinterpret_cast<const __nv_bfloat16*>(ws + L.ctx);
        g.w[0] = static_cast<const __nv_bfloat16*>(w_o);
        g.bias[0] = static_cast<const __nv_bfloat16*>(b_o);
        g.out[0] = static_cast<__nv_bfloat16*>(out);
        g.M = B; g.N = d_model; g.K = d_model; g.ngroups = 1; g.head_split = 0; g.dk = dk;
        e = mha::launch_gemv_bf16(g, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode output projection launch");
        return MHA_OK;
    }
    return output_projection_impl(dt, w_o, b_o, nullptr, 1, B, d_model, h, out, L, ws, s);
}

size_t mha_ffn_workspace_size(mha_dtype_t dt, int B, int L, int d_model, int d_ff) {
    if (B <= 0 || L <= 0 || d_model <= 0 || d_ff <= 0) return 0;
    if (dt != MHA_F32 && dt != MHA_BF16) return 0;
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    return align256(es * B * static_cast<size_t>(L) * d_ff);
}

mha_status_t mha_ffn_forward(mha_dtype_t dt, const void* x, const void* w_1, const void* b_1, const void* w_2,
                             const void* b_2, int B, int L, int d_model, int d_ff, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (dt != MHA_F32 && dt != MHA_BF16) return fail(MHA_ERR_INVALID_ARG, "dtype %d is not MHA_F32 or MHA_BF16", dt);
    if (B <= 0 || L <= 0 || d_model <= 0 || d_ff <= 0)
        return fail(MHA_ERR_INVALID_ARG, "sizes must be positive (B=%d L=%d d_model=%d d_ff=%d)", B, L, d_model, d_ff);
    if (!x || !w_1 || !w_2 || !out) return fail(MHA_ERR_INVALID_ARG, "x, W_1, W_2 and out must not be NULL");
    if (static_cast<double>(B) * L * d_ff > 4.0e9) return fail(MHA_ERR_UNSUPPORTED, "problem too large");
    const size_t need = mha_ffn_workspace_size(dt, B, L, d_model, d_ff);
    if (!workspace) return fail(MHA_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MHA_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (workspace_bytes < need) return fail(MHA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
    const cudaStream_t s = as_stream(stream);
    if (dt == MHA_F32) {
        mha::F32GemmParams p{};
        p.ngroups = 1;
        p.B = B; p.dk = 1; p.out_plain = 1;
        p.g[0].L = L;
        // layer 1: hidden = relu(x W_1^T + b_1)
        p.K = d_model; p.N = d_ff; p.relu = 1;
        p.g[0].A = static_cast<const float*>(x);
        p.g[0].W = static_cast<const float*>(w_1);
        p.g[0].bias = static_cast<const float*>(b_1);
        p.g[0].out = static_cast<float*>(workspace);
        cudaError_t e = mha::launch_gemm_f32(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "FFN layer 1 launch");
        // layer 2: out = hidden W_2^T + b_2
        p.K = d_ff; p.N = d_model; p.relu = 0;
        p.g[0].A = static_cast<const float*>(workspace);
        p.g[0].W = static_cast<const float*>(w_2);
        p.g[0].bias = static_cast<const float*>(b_2);
        p.g[0].out = static_cast<float*>(out);
        e = mha::launch_gemm_f32(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "FFN layer 2 launch");
        return MHA_OK;
    }
    if (d_model % 64 != 0 || d_ff % 64 != 0)
        return fail(MHA_ERR_UNSUPPORTED, "bf16 FFN needs d_model and d_ff multiples of 64 (got %d, %d)", d_model, d_ff);
    const void* ptrs[6] = {x, w_1, b_1, w_2, b_2, out};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
    mha_status_t st = get_encoder();
    if (st != MHA_OK) return st;
    int* status = device_status_ptr();
    if (!status) return fail(MHA_ERR_CUDA, "device status word unavailable");
    const int tiles_per_b = (L + mha::kGemmBM - 1) / mha::kGemmBM;
    for (int layer = 0; layer < 2; ++layer) {
        mha::GemmParams p;
        memset(&p, 0, sizeof(p));
        const int K = layer == 0 ? d_model : d_ff;
        const int N = layer == 0 ? d_ff : d_model;
        const void* A = layer == 0 ? x : workspace;
        void* O = layer == 0 ? workspace : out;
        if ((st = map_rows(&p.a[0], A, B, L, K, "FFN input")) != MHA_OK) return st;
        if ((st = map_rows(&p.out[0], O, B, L, N, "FFN output")) != MHA_OK) return st;
        p.g[0].L = L;
        p.g[0].tiles_per_b = tiles_per_b;
        p.g[0].m_tiles = B * tiles_per_b;
        p.g[0].bias = static_cast<const __nv_bfloat16*>(layer == 0 ? b_1 : b_2);
        p.ngroups = 1;
        p.K = K;
        p.N = N;
        p.out_plain = 1;
        p.relu = layer == 0;
        p.status = status;
        const void* W[1] = {layer == 0 ? w_1 : w_2};
        if ((st = launch_projection(p, W, s, layer == 0 ? "FFN layer 1 launch" : "FFN layer 2 launch")) != MHA_OK)
            return st;
    }
    return MHA_OK;
}

size_t mha_host_staging_size(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int kv_distinct,
                             int q_distinct) {
    if (B <= 0 || L_q <= 0 || L_k <= 0 || d_model <= 0) return 0;
    if (dt != MHA_F32 && dt != MHA_BF16) return 0;
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    const size_t qb = align256(es * B * static_cast<size_t>(L_q) * d_model);
    const size_t kb = align256(es * B * static_cast<size_t>(L_k) * d_model);
    size_t total = qb /* query */ + qb /* out */;
    if (q_distinct) total += kb;          // key not aliasing query
    if (kv_distinct) total += kb;         // value not aliasing key
    return total;
}

}  // extern "C"

namespace {

// Per-device resources of the host-buffer entry point: an upload stream, a
// download stream, a second compute stream and events, created on first use
// and kept for the life of the process.
constexpr int kHostChunks = 4;                       // chunks of a large call
constexpr int kHostChunksSmall = 2;                  // chunks of a call with less host input
constexpr size_t kHostLargeBytes = size_t(32) << 20;  // host input bytes from which a call is large
constexpr int kHostWindows = 2;   // row windows of the first and the last chunk (self-attention)
constexpr int kHostUnits = kHostChunks + 2 * kHostWindows;
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, compute2 = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kHostUnits] = {}, comp[kHostUnits] = {};
};
HostPipe g_pipes[64];

mha_status_t host_pipe(int dev, HostPipe** hp) {
    if (dev < 0 || dev >= 64) return fail(MHA_ERR_CUDA, "device ordinal %d out of range", dev);
    HostPipe& p = g_pipes[dev];
    if (!p.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.compute2, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming);
        for (int c = 0; c < kHostUnits && e == cudaSuccess; ++c) {
            e = cudaEventCreateWithFlags(&p.in[c], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.comp[c], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_fail(e, "copy stream / event creation");
        p.ready = true;
    }
    *hp = &p;
    return MHA_OK;
}

}  // namespace

extern "C" {

mha_status_t mha_forward_host(mha_dtype_t dt, const void* h_query, const void* h_key, const void* h_value,
                              const void* w_q, const void* b_q, const void* w_k, const void* b_k, const void* w_v,
                              const void* b_v, const void* w_o, const void* b_o, int B, int L_q, int L_k,
                              int d_model, int h, const mha_mask_t* mask, void* h_out, void* staging,
                              size_t staging_bytes, void* workspace, size_t workspace_bytes, void* stream) {
    mha_status_t st = check_sizes(dt, B, L_q, L_k, d_model, h);
    if (st != MHA_OK) return st;
    if ((st = check_mask(mask, L_q, L_k)) != MHA_OK) return st;
    if (!h_query || !h_key || !h_value || !h_out || !staging)
        return fail(MHA_ERR_INVALID_ARG, "host query/key/value/out and staging must not be NULL");
    const int q_distinct = h_key != h_query;
    const int kv_distinct = h_value != h_key;
    const size_t need = mha_host_staging_size(dt, B, L_q, L_k, d_model, kv_distinct, q_distinct);
    if (staging_bytes < need) return fail(MHA_ERR_INVALID_ARG, "staging too small: %zu < %zu", staging_bytes, need);
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0)
        return fail(MHA_ERR_INVALID_ARG, "staging not 256-byte aligned");
    Layout L;
    if ((st = check_workspace(dt, B, L_q, L_k, d_model, h, workspace, workspace_bytes, &L)) != MHA_OK) return st;
    const size_t es = dt == MHA_BF16 ? 2 : 4;
    const size_t qrow = es * static_cast<size_t>(L_q) * d_model;   // bytes of one sequence of query / out
    const size_t krow = es * static_cast<size_t>(L_k) * d_model;
    uint8_t* p = static_cast<uint8_t*>(staging);
    uint8_t* d_q = p;
    p += align256(qrow * B);
    uint8_t* d_out = p;
    p += align256(qrow * B);
    uint8_t* d_k = d_q;
    if (q_distinct) {
        d_k = p;
        p += align256(krow * B);
    }
    uint8_t* d_v = d_k;
    if (kv_distinct) {
        d_v = p;
        p += align256(krow * B);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    HostPipe* hp = nullptr;
    std::lock_guard<std::mutex> lock(g_pipes[dev < 0 || dev >= 64 ? 0 : dev].mu);
    if ((st = host_pipe(dev, &hp)) != MHA_OK) return st;
    const cudaStream_t s = as_stream(stream);
    // Pipeline over chunks of sequences: uploads on one library stream, downloads on
    // another, and the chunks' compute alternating between `stream` and a second
    // library stream (each with its own part of the workspace), so that one chunk's
    // kernels fill the SMs the previous chunk's last waves leave idle. For
    // self-attention (one tensor as query, key and value) the two exposed ends are cut
    // into row windows: the first chunk is uploaded window by window and each window's
    // Q/K/V projection starts as soon as its rows have arrived, and the last chunk's
    // output projection and download run window by window after its attention.
    // Small calls take fewer chunks: their kernels are latency-bound, so every extra
    // chunk adds launches that cost more than the copy overlap they buy.
    const size_t in_bytes = qrow * B + (q_distinct ? krow * B : 0) + (kv_distinct ? krow * B : 0);
    const int nch = std::min(B, in_bytes >= kHostLargeBytes ? kHostChunks : kHostChunksSmall);
    const int per = (B + nch - 1) / nch;
    Layout Lc;
    layout_of(dt, per, L_q, L_k, d_model, h, &Lc);
    const bool two = nch >= 2 && 2 * Lc.total <= workspace_bytes;
    uint8_t* ws_of[2] = {static_cast<uint8_t*>(workspace), static_cast<uint8_t*>(workspace) + Lc.total};
    const size_t ws_bytes = two ? Lc.total : workspace_bytes;
    constexpr int kWinRows = mha::kGemmBM;   // window boundaries on whole GEMM row tiles
    const bool split = dt == MHA_BF16 && !q_distinct && !kv_distinct && L_q == L_k &&
                       L_q >= kHostWindows * kWinRows;
    const int nwin = split ? kHostWindows : 1;
    int wr[kHostWindows + 1];
    wr[0] = 0;
    for (int w = 1; w < nwin; ++w) wr[w] = static_cast<int>(static_cast<long>(L_q) * w / nwin / kWinRows) * kWinRows;
    wr[nwin] = L_q;
    if (split) {   // the stages run without mha_forward's own checks
        const void* ptrs[8] = {w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o};
        for (const void* ptr : ptrs)
            if (ptr && !aligned16(ptr)) return fail(MHA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
        if (!w_q || !w_k || !w_v || !w_o) return fail(MHA_ERR_INVALID_ARG, "W_q, W_k, W_v and W_o must not be NULL");
    }
    const size_t rowq = es * static_cast<size_t>(d_model);   // bytes of one token row
    // windows of chunk c on the input side (its upload + projection) and the output side
    auto in_windows = [&](int c) { return (split && c == 0) ? nwin : 1; };
    auto out_windows = [&](int c) { return (split && c == nch - 1) ? nwin : 1; };
    auto win_lo = [&](int n, int w) { return n == 1 ? 0 : wr[w]; };
    auto win_hi = [&](int n, int w) { return n == 1 ? L_q : wr[w + 1]; };
    e = cudaEventRecord(hp->start, s);   // staging / out / workspace may still be in use by earlier work on `stream`
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->h2d, hp->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->start, 0);
    if (e == cudaSuccess && two) e = cudaStreamWaitEvent(hp->compute2, hp->start, 0);
    int n_in = 0;
    for (int c = 0; c < nch && e == cudaSuccess; ++c) {
        const int b0 = c * per, bc = std::min(per, B - b0);
        if (bc <= 0) break;
        const int nw = in_windows(c);
        for (int w = 0; w < nw && e == cudaSuccess; ++w) {
            const int r0 = win_lo(nw, w), r1 = win_hi(nw, w);
            const size_t off = qrow * b0 + rowq * r0;
            e = cudaMemcpy2DAsync(d_q + off, qrow, static_cast<const uint8_t*>(h_query) + off, qrow,
                                  rowq * (r1 - r0), bc, cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess && q_distinct)
                e = cudaMemcpyAsync(d_k + krow * b0, static_cast<const uint8_t*>(h_key) + krow * b0, krow * bc,
                                    cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess && kv_distinct)
                e = cudaMemcpyAsync(d_v + krow * b0, static_cast<const uint8_t*>(h_value) + krow * b0, krow * bc,
                                    cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess) e = cudaEventRecord(hp->in[n_in++], hp->h2d);
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "host to device copy");
    int n_in_used = 0, n_out = 0;
    for (int c = 0; c < nch; ++c) {
        const int b0 = c * per, bc = std::min(per, B - b0);
        if (bc <= 0) break;
        const int lane = two ? (c & 1) : 0;
        const cudaStream_t sc = lane ? hp->compute2 : s;
        mha_mask_t mc;
        const mha_mask_t* mp = nullptr;
        if (mask) {
            mc = *mask;
            if (mc.key_valid_lens) mc.key_valid_lens += b0;
            if (mc.dense) mc.dense += static_cast<size_t>(b0) * mc.dense_mq * L_k;
            mp = &mc;
        }
        Layout Lb;
        layout_of(dt, bc, L_q, L_k, d_model, h, &Lb);
        const int nwi = in_windows(c), nwo = out_windows(c);
        if (split) {
            uint8_t* xq = d_q + qrow * b0;
            for (int w = 0; w < nwi; ++w) {
                if ((e = cudaStreamWaitEvent(sc, hp->in[n_in_used++], 0)) != cudaSuccess)
                    return cuda_fail(e, "stream wait");
                const int r0 = win_lo(nwi, w), r1 = win_hi(nwi, w);
                if ((st = qkv_bf16_impl(xq, xq, xq, w_q, b_q, w_k, b_k, w_v, b_v, bc, L_q, L_k, d_model, h, Lb,
                                        ws_of[lane], sc, r0, nwi == 1 ? 0 : r1 - r0)) != MHA_OK)
                    return st;
            }
            if ((st = attention_impl(dt, bc, L_q, L_k, d_model, h, mp, nullptr, Lb, ws_of[lane], sc)) != MHA_OK)
                return st;
        } else {
            if ((e = cudaStreamWaitEvent(sc, hp->in[n_in_used++], 0)) != cudaSuccess)
                return cuda_fail(e, "stream wait");
        }
        for (int w = 0; w < nwo; ++w) {
            const int r0 = win_lo(nwo, w), r1 = win_hi(nwo, w);
            if (split) {
                if ((st = output_projection_impl(dt, w_o, b_o, nullptr, bc, L_q, d_model, h, d_out + qrow * b0, Lb,
                                                 ws_of[lane], sc, r0, nwo == 1 ? 0 : r1 - r0)) != MHA_OK)
                    return st;
            } else {
                st = mha_forward(dt, d_q + qrow * b0, d_k + krow * b0, d_v + krow * b0, w_q, b_q, w_k, b_k, w_v, b_v,
                                 w_o, b_o, bc, L_q, L_k, d_model, h, mp, d_out + qrow * b0, nullptr, ws_of[lane],
                                 ws_bytes, sc);
                if (st != MHA_OK) return st;
            }
            const int u = n_out++;
            e = cudaEventRecord(hp->comp[u], sc);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->comp[u], 0);
            if (e == cudaSuccess) {
                const size_t off = qrow * b0 + rowq * r0;
                e = cudaMemcpy2DAsync(static_cast<uint8_t*>(h_out) + off, qrow, d_out + off, qrow, rowq * (r1 - r0),
                                      bc, cudaMemcpyDeviceToHost, hp->d2h);
            }
            if (e != cudaSuccess) return cuda_fail(e, "device to host copy");
        }
    }
    // Every chunk's compute precedes its download, so `done` covers all of the call.
    e = cudaEventRecord(hp->done, hp->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "stream wait");
    return MHA_OK;
}

mha_status_t mha_selftest_wait_timeout(void* stream) {
    int* st = device_status_ptr();
    if (!st) return fail(MHA_ERR_CUDA, "device status word unavailable");
    cudaError_t e = mha::launch_wait_timeout_selftest(st, MHA_SELFTEST_WAIT_CODE, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait-timeout self-test launch");
    return MHA_OK;
}

mha_status_t mha_check_device_status(int* status, int reset) {
    if (!status) return fail(MHA_ERR_INVALID_ARG, "status must not be NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    *status = v;
    if (reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "status reset");
    }
    return MHA_OK;
}

}  // extern "C"
