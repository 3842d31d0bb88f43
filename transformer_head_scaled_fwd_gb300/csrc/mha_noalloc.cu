// mha_noalloc.cu -- mha_forward_noalloc: the forward pass without a caller
// workspace, for callers that cannot allocate device memory.
//
// Who needs it: code that is handed only its inputs and outputs and may not
// allocate -- a plugin whose host application owns every byte of device memory
// through its own pool and forbids allocations behind its back, a serving path
// that must never hit cudaMalloc's implicit device-wide synchronisation, or an
// interface with no workspace argument to thread through. Such callers cannot
// size and pass the workspace that mha_forward asks for.
//
// How: the scratch (head-split Q/K/V, context, softmax statistics) lives in one
// file-scope device array of fixed size, MHA_NOALLOC_SCRATCH_BYTES. It is
// reserved on every GPU that loads this part of the library and stays reserved
// until the process exits. Host code cannot use the array's name as a device
// address (on the host it is only a stand-in symbol), so the first call on each
// device looks up the real address with cudaGetSymbolAddress while that device
// is current, and caches it together with the identity of the CUDA context it
// belongs to. That first call per device should therefore be made before any
// stream capture begins. If the context is destroyed and re-created (for
// example by cudaDeviceReset), the array is re-created at a new address; the
// next call notices the new context and looks the address up again, so that
// call, too, should come before any stream capture.
//
// Every call on a device shares the same array: calls whose work overlaps on
// the GPU (different streams, or host threads racing) corrupt each other's
// scratch. Serialise them, e.g. issue them all on one stream. Nothing in the
// scratch has to start at zero: every byte a kernel reads was written earlier
// in the same call, so no clearing is done.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "../../include/mha.h"
#include "mha_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MHA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;

// The scratch address of each device and the context it was looked up in.
struct ScratchAddr {
    unsigned long long ctx_id;   // 0: not looked up yet
    void* addr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Driver entry points that identify the current context (fetched once; absent
// entry points make every call look the address up again).
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the context current on this thread, or 0 if there is none (or it
// cannot be told).
unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

extern "C" mha_status_t mha_forward_noalloc(mha_dtype_t dt, const void* query, const void* key, const void* value,
                                            const void* w_q, const void* b_q, const void* w_k, const void* b_k,
                                            const void* w_v, const void* b_v, const void* w_o, const void* b_o,
                                            int B, int L_q, int L_k, int d_model, int h, const mha_mask_t* mask,
                                            void* out, float* p_attn, void* stream) {
    const size_t need = mha_workspace_size(dt, B, L_q, L_k, d_model, h);
    if (need == 0) {
        // invalid sizes: let mha_forward report the precise reason (it enqueues nothing)
        return mha_forward(dt, query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, B, L_q, L_k, d_model, h,
                           mask, out, p_attn, nullptr, 0, stream);
    }
    if (need > MHA_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "mha_forward_noalloc: this problem needs %zu bytes of scratch, more than the fixed "
                 "%zu bytes (MHA_NOALLOC_SCRATCH_BYTES); use mha_forward with a caller workspace",
                 need, static_cast<size_t>(MHA_NOALLOC_SCRATCH_BYTES));
        mha::set_last_error(msg);
        return MHA_ERR_INVALID_ARG;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        mha::set_last_error("mha_forward_noalloc: no usable current CUDA device");
        return MHA_ERR_CUDA;
    }
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        ScratchAddr& c = g_scratch[dev];
        const unsigned long long id = current_context_id();
        if (c.addr == nullptr || id == 0 || c.ctx_id != id) {
            // first call on this device, or a context other than the one the cached
            // address belongs to: look the array up in the current context
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                char msg[256];
                snprintf(msg, sizeof(msg), "mha_forward_noalloc: scratch address lookup failed on device %d: %s",
                         dev, cudaGetErrorString(e));
                mha::set_last_error(msg);
                c = ScratchAddr{0, nullptr};
                return MHA_ERR_CUDA;
            }
            c = ScratchAddr{current_context_id(), p};   // the lookup made the device's context current
        }
        base = c.addr;
    }
    return mha_forward(dt, query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, B, L_q, L_k, d_model, h, mask,
                       out, p_attn, base, MHA_NOALLOC_SCRATCH_BYTES, stream);
}
