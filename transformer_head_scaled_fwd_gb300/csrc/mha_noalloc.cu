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
// is current, and caches it. That first call per device should therefore be
// made before any stream capture begins.
//
// Every call on a device shares the same array: calls whose work overlaps on
// the GPU (different streams, or host threads racing) corrupt each other's
// scratch. Serialise them, e.g. issue them all on one stream. Nothing in the
// scratch has to start at zero: every byte a kernel reads was written earlier
// in the same call, so no clearing is done.
#include <cstdio>
#include <mutex>

#include "../../include/mha.h"
#include "mha_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MHA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

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
        if (g_scratch_addr[dev] == nullptr) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                char msg[256];
                snprintf(msg, sizeof(msg), "mha_forward_noalloc: scratch address lookup failed on device %d: %s",
                         dev, cudaGetErrorString(e));
                mha::set_last_error(msg);
                return MHA_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        base = g_scratch_addr[dev];
    }
    return mha_forward(dt, query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, B, L_q, L_k, d_model, h, mask,
                       out, p_attn, base, MHA_NOALLOC_SCRATCH_BYTES, stream);
}
