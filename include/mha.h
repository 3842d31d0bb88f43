/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head attention forward library.
 *
 * The operation is the forward pass of the Transformer's multi-head attention
 * sublayer, as the pages define it:
 *
 *   "003-Transformer" tutorial, section "Multi-head attention",
 *   MultiHeadedAttention.forward(query, key, value, mask):
 *     Q = query W_q^T + b_q, K = key W_k^T + b_k, V = value W_v^T + b_v
 *         (nn.Linear(d_model, d_model), weights stored [out, in]);
 *     each viewed as (B, L, h, d_k) and transposed to (B, h, L, d_k), so head i
 *         owns features [i*d_k, (i+1)*d_k), with d_k = d_model / h;
 *     per head: "The Annotated Transformer", section "Attention", attention():
 *         scores = Q K^T / sqrt(d_k); scores.masked_fill(mask == 0, -1e9);
 *         p_attn = softmax(scores, dim=-1); head = p_attn V;
 *     heads transposed back and concatenated to (B, L_q, h*d_k);
 *     out = concat W_o^T + b_o.
 *
 * Mask (1 = may attend): the AND of up to three parts, broadcast over heads
 * (mask.unsqueeze(1) in MultiHeadedAttention.forward):
 *   causal          key j allowed for query i iff j <= i ("The Annotated
 *                   Transformer", subsequent_mask(); diagonal allowed).
 *   key_valid_lens  key j allowed iff j < key_valid_lens[b] (d2l
 *                   MultiHeadAttention valid_lens, d2l Transformer chapter).
 *   dense           byte mask [B, dense_mq, L_k], dense_mq in {1, L_q};
 *                   0 = masked; dense_mq == 1 broadcasts over queries.
 * A masked score is REPLACED by -1e9 after the 1/sqrt(d_k) scaling, so a
 * query row whose keys are all masked gets uniform weights 1/L_k over all L_k
 * keys. Dropout is the identity (forward / evaluation).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers into buffers the caller owns,
 *     row-major and contiguous, unless an entry point says otherwise. The
 *     library never allocates or frees device memory and never synchronises
 *     the stream (except mha_check_device_status, which says so).
 *   - dt selects the storage type of query/key/value/weights/biases/out and of
 *     the workspace tensors: MHA_F32 (fp32 everywhere, fp32 SIMT arithmetic,
 *     any d_k <= 256) or MHA_BF16 (bf16 storage, fp32 accumulation on the
 *     tensor cores, d_k = 64 or 128, or d_k = 8, 16, 32 when d_model is a
 *     multiple of 64 (those heads run on the d_k = 64 kernels, zero-padded to 64
 *     columns on load); mha_forward and mha_forward_noalloc also take any other
 *     d_k <= 256 in bf16, which they run on the fp32 kernels over fp32 copies held
 *     in the workspace, then round the output to bf16).
 *     p_attn is always fp32.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting for it.
 *   - Arguments are validated on the host before anything is enqueued. On a
 *     non-OK status returned by validation, no output buffer is touched.
 *     mha_last_error() then gives a message (thread-local).
 *   - B, L_q, L_k, d_model, h >= 1; d_model % h == 0 (the pages assert
 *     embedding_dim % head == 0). causal requires L_q == L_k (the subsequent
 *     mask is square).
 *   - MHA_BF16 also requires every tensor pointer to be 16-byte aligned.
 */
#ifndef GB300_MHA_H
#define GB300_MHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1,   /* bad size, null required pointer, small workspace */
    MHA_ERR_UNSUPPORTED = 2,   /* valid per the pages but not implemented (e.g. d_k > 256) */
    MHA_ERR_CUDA = 3           /* a CUDA call failed; see mha_last_error() */
} mha_status_t;

typedef enum { MHA_F32 = 0, MHA_BF16 = 1 } mha_dtype_t;

typedef struct {
    int causal;                     /* nonzero: subsequent mask, key j <= query i */
    const int32_t* key_valid_lens;  /* device [B] or NULL: key j allowed iff j < len[b]; len < 0 reads as 0 */
    const uint8_t* dense;           /* device [B, dense_mq, L_k] or NULL: 0 = masked */
    int dense_mq;                   /* 1 (broadcast over queries) or L_q; ignored if dense is NULL */
} mha_mask_t;

/*
 * Workspace the forward pass needs, in bytes (a multiple of 256).
 * Layout (each part starts on a 256-byte boundary, element type = dt):
 *   Qh   [B, h, L_q, d_k]      head-split projected queries
 *   KVh  [B, 2, h, L_k, d_k]   head-split projected keys (slot 0) and values (slot 1)
 *   ctx  [B, L_q, d_model]     concatenated head outputs (input of W_o)
 *   stat [B, h, L_q, 2] fp32   per-row softmax statistics (max, sum) used for p_attn
 *   sched 256 bytes            2 ints: the d_k = 128 attention's work counter (zeroed by the
 *                              Q/K/V projection stage, left at zero by the attention stage)
 * For MHA_BF16 with a d_k the tensor-core kernels do not take (d_k <= 256): the MHA_F32
 * workspace of the same sizes, then fp32 copies of query, key, value [B, L, d_model], of
 * the four weights and biases and of out, each 256-byte aligned.
 * Returns 0 for invalid sizes.
 */
size_t mha_workspace_size(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h);

/*
 * mha_forward -- the whole sublayer: out = MultiHeadedAttention(query, key, value, mask).
 *   query [B, L_q, d_model]; key, value [B, L_k, d_model]   (may alias each other)
 *   w_q, w_k, w_v, w_o [d_model, d_model] stored (out, in); b_* [d_model] or NULL (= zero bias)
 *   mask   NULL = no mask
 *   out    [B, L_q, d_model], type dt; must not alias any input or the workspace
 *   p_attn NULL, or fp32 [B, h, L_q, L_k]: the attention weights of every head
 *          (the pages keep them as self.attn for visualisation)
 *   workspace >= mha_workspace_size(...) bytes of device memory, 256-byte aligned
 * Three stages run in order on `stream`: mha_qkv_projection, mha_attention_core,
 * mha_output_projection.
 */
mha_status_t mha_forward(mha_dtype_t dt,
                         const void* query, const void* key, const void* value,
                         const void* w_q, const void* b_q,
                         const void* w_k, const void* b_k,
                         const void* w_v, const void* b_v,
                         const void* w_o, const void* b_o,
                         int B, int L_q, int L_k, int d_model, int h,
                         const mha_mask_t* mask,
                         void* out, float* p_attn,
                         void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Stage 1 -- the three input projections of MultiHeadedAttention.forward, written
 * head-split into the workspace (Qh and KVh above). One launch covers all three.
 */
mha_status_t mha_qkv_projection(mha_dtype_t dt,
                                const void* query, const void* key, const void* value,
                                const void* w_q, const void* b_q,
                                const void* w_k, const void* b_k,
                                const void* w_v, const void* b_v,
                                int B, int L_q, int L_k, int d_model, int h,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stage 2 -- attention() for every (batch, head): scores, scale, -1e9 fill,
 * softmax, P.V, written concatenated into ctx of the workspace; and, if p_attn
 * is not NULL, the normalised weights fp32 [B, h, L_q, L_k]. Reads Qh and KVh.
 */
mha_status_t mha_attention_core(mha_dtype_t dt, int B, int L_q, int L_k, int d_model, int h,
                                const mha_mask_t* mask, float* p_attn,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stage 3 -- the fourth Linear of MultiHeadedAttention: out = ctx W_o^T + b_o,
 * reading ctx from the workspace. out [B, L_q, d_model], type dt.
 */
mha_status_t mha_output_projection(mha_dtype_t dt, const void* w_o, const void* b_o,
                                   int B, int L_q, int L_k, int d_model, int h,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * mha_forward_host -- the same sublayer with the activations in HOST memory:
 * query/key/value are read from host buffers and out is written to a host
 * buffer; weights, biases, mask parts and the workspace are device pointers as
 * above. The host buffers should be page-locked for the copies to be
 * asynchronous. `staging` is device memory of at least
 * mha_host_staging_size(...) bytes that receives the activations. The call is
 * pipelined over chunks of sequences (up to 4 when query, key and value hold
 * at least 32 MiB of host data together, else up to 2; never more than B) with
 * library-owned streams (one set
 * per device, created on first use): an upload stream, a download stream and a
 * second compute stream. Chunks alternate between `stream` and the second
 * compute stream when the workspace holds two chunk workspaces (each
 * mha_workspace_size(dt, ceil(B / chunks), ...) bytes; true whenever B >= 2 at
 * realistic sizes), otherwise all run on `stream`. When query, key and value
 * are the same host buffer (bf16, L >= 256), the first chunk is uploaded and
 * projected in two row windows and the last chunk's output projection and
 * download run in two row windows. Copies: host->device of query (and of key and value unless they
 * alias query / each other), device->host of out; all ordered by events. When
 * the call returns, all of it is enqueued behind `stream`: synchronise `stream`
 * before reading out. The workspace must not be used by other work on other
 * streams while the call runs.
 */
size_t mha_host_staging_size(mha_dtype_t dt, int B, int L_q, int L_k, int d_model,
                             int kv_distinct, int q_distinct);
mha_status_t mha_forward_host(mha_dtype_t dt,
                              const void* h_query, const void* h_key, const void* h_value,
                              const void* w_q, const void* b_q,
                              const void* w_k, const void* b_k,
                              const void* w_v, const void* b_v,
                              const void* w_o, const void* b_o,
                              int B, int L_q, int L_k, int d_model, int h,
                              const mha_mask_t* mask,
                              void* h_out,
                              void* staging, size_t staging_bytes,
                              void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * mha_forward_noalloc -- mha_forward for callers that cannot allocate device
 * memory. (The pages have no counterpart: this is an interface choice of this
 * library.) Some callers are handed only their inputs and outputs: a plugin
 * whose host application owns all device memory through its own pool, a
 * serving path that must never hit cudaMalloc (which can synchronise the whole
 * device), an interface with no workspace argument. This entry point takes the
 * same arguments as mha_forward minus the workspace, allocates nothing, and
 * uses a fixed scratch area built into the library instead:
 *   - MHA_NOALLOC_SCRATCH_BYTES (48 MiB) of device memory, reserved on every
 *     GPU that loads this part of the library and held until the process exits.
 *   - Problems whose mha_workspace_size(...) exceeds it are rejected with
 *     MHA_ERR_INVALID_ARG and a message naming both sizes (e.g. the encoder,
 *     decoder and cross-attention workloads of this library fit; B=4, L=8192,
 *     d_model=1024 does not).
 *   - The first call on each device looks up the scratch address with that
 *     device current; make that first call before any stream capture begins.
 *     The address belongs to the device's current CUDA context: after the
 *     context is destroyed and re-created (e.g. cudaDeviceReset), the next
 *     call sees the new context and looks the address up again, so that call
 *     too belongs outside stream capture.
 *   - All calls on a device share the one scratch area: calls whose work
 *     overlaps on the GPU (other streams, other host threads) race and corrupt
 *     each other. Serialise them, e.g. on one stream.
 *   - Nothing in the scratch needs to start at zero; it is not cleared.
 */
#define MHA_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)
mha_status_t mha_forward_noalloc(mha_dtype_t dt,
                                 const void* query, const void* key, const void* value,
                                 const void* w_q, const void* b_q,
                                 const void* w_k, const void* b_k,
                                 const void* w_v, const void* b_v,
                                 const void* w_o, const void* b_o,
                                 int B, int L_q, int L_k, int d_model, int h,
                                 const mha_mask_t* mask,
                                 void* out, float* p_attn,
                                 void* stream);

/*
 * The residual sublayer around multi-head attention, pre-norm form
 * ("The Annotated Transformer", SublayerConnection: x + dropout(sublayer(norm(x))),
 * dropout = identity):
 *   y   = LayerNorm(x)
 *   out = x + MultiHeadedAttention(y, y, y, mask)              if memory == NULL (self-attention)
 *   out = x + MultiHeadedAttention(y, memory, memory, mask)    otherwise (source attention,
 *         "The Annotated Transformer", DecoderLayer: src_attn(x, m, m, src_mask))
 * LayerNorm over the last dimension, ln_kind selects the pages' two forms:
 *   0  a (x - mean) / (std + eps) + b, std unbiased ("The Annotated Transformer", LayerNorm, eps 1e-6)
 *   1  a (x - mean) / sqrt(var + eps) + b, var biased (nn.LayerNorm, "003-Transformer")
 *   ln_gain / ln_bias [d_model] or NULL (ones / zeros), type dt.
 * x [B, L, d_model]; memory [B, L_mem, d_model] or NULL; out [B, L, d_model] (may alias x: each
 * element of x is read by the thread that then writes the same element of out).
 * d_model <= 2048. Workspace >= mha_sublayer_workspace_size(...): LayerNorm(x) followed by the
 * workspace of mha_forward. Launches: LayerNorm, the three stages of mha_forward, with the
 * residual added in the W_o epilogue.
 */
size_t mha_sublayer_workspace_size(mha_dtype_t dt, int B, int L, int L_mem, int d_model, int h);
mha_status_t mha_sublayer_forward(mha_dtype_t dt, const void* x, const void* memory,
                                  const void* ln_gain, const void* ln_bias, float ln_eps, int ln_kind,
                                  const void* w_q, const void* b_q,
                                  const void* w_k, const void* b_k,
                                  const void* w_v, const void* b_v,
                                  const void* w_o, const void* b_o,
                                  int B, int L, int L_mem, int d_model, int h,
                                  const mha_mask_t* mask,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * Incremental decoding with a key/value cache (bf16, d_k = 64 or 128).
 * At prediction time the d2l Transformer decoder (d2l Transformer chapter, DecoderBlock:
 * state[2] keeps the representations decoded so far and torch.cat appends the new one as
 * keys and values) attends from the newest token to every token so far, itself included.
 * This library caches the PROJECTED keys and values, which gives the same result.
 *   k_cache, v_cache  device [B, h, L_max, d_k] bf16: position t of sequence b, head i.
 *   mha_kv_cache_prefill: projects x [B, T, d_model] into positions 0..T-1 of both caches
 *     (K = x W_k^T + b_k, V = x W_v^T + b_v); T <= L_max.
 *   mha_decode_step: one new token per sequence, x_new [B, d_model]:
 *     q, k, v = x_new W^T + b; k, v written at position cache_len[b] (device int32 [B]),
 *     which the step then increments on the device; out [B, d_model] = the sublayer's output
 *     for the new token: attention of q over the cache_len[b] + 1 cached positions (no mask
 *     needed), concat, W_o. A sequence whose cache is full (cache_len[b] >= L_max) appends
 *     nothing and the step records code 0x301 in the device status word
 *     (mha_check_device_status). Workspace >= mha_decode_workspace_size(...), 256-byte aligned.
 */
size_t mha_decode_workspace_size(int B, int d_model, int h, int L_max);
mha_status_t mha_kv_cache_prefill(mha_dtype_t dt, const void* x,
                                  const void* w_k, const void* b_k,
                                  const void* w_v, const void* b_v,
                                  int B, int T, int d_model, int h,
                                  void* k_cache, void* v_cache, int L_max, void* stream);
mha_status_t mha_decode_step(mha_dtype_t dt, const void* x_new,
                             const void* w_q, const void* b_q,
                             const void* w_k, const void* b_k,
                             const void* w_v, const void* b_v,
                             const void* w_o, const void* b_o,
                             int B, int d_model, int h,
                             void* k_cache, void* v_cache, int32_t* cache_len, int L_max,
                             void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Position-wise feed-forward network ("003-Transformer" tutorial, feed-forward
 * layer; "From RNN to Attention", part 3, FFN):
 *   out = max(0, x W_1^T + b_1) W_2^T + b_2        (dropout = identity)
 *   x [B, L, d_model]; w_1 [d_ff, d_model], b_1 [d_ff] or NULL;
 *   w_2 [d_model, d_ff], b_2 [d_model] or NULL; out [B, L, d_model], type dt.
 *   MHA_BF16: d_model and d_ff multiples of 64, 16-byte aligned pointers; the
 *   two layers run on the tensor-core GEMM (ReLU fused into the first epilogue).
 *   The hidden activations [B, L, d_ff] live in the caller's workspace of at
 *   least mha_ffn_workspace_size(...) bytes (256-byte aligned).
 */
size_t mha_ffn_workspace_size(mha_dtype_t dt, int B, int L, int d_model, int d_ff);
mha_status_t mha_ffn_forward(mha_dtype_t dt, const void* x,
                             const void* w_1, const void* b_1,
                             const void* w_2, const void* b_2,
                             int B, int L, int d_model, int d_ff,
                             void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* mha_last_error(void);

/*
 * Device-side status of the bounded waits inside the tensor-core kernels.
 * Every pipeline wait gives up after a fixed iteration budget instead of
 * spinning forever; when one gives up, the kernel records a code here and runs
 * to completion (its outputs are then not valid). This call SYNCHRONISES the
 * device, copies the word to *status (0 = no wait gave up), and, if reset is
 * nonzero, clears it.
 */
mha_status_t mha_check_device_status(int* status, int reset);

/*
 * Diagnostic: exercises the failure path of the bounded pipeline waits on the GPU.
 * Enqueues on `stream` one warp that waits on an mbarrier nothing ever arrives on,
 * through the same bounded wait every tensor-core pipeline uses but with a budget of
 * 1024 rounds; the wait gives up, the kernel records MHA_SELFTEST_WAIT_CODE in the
 * device status word (unless a code is already there) and ends. Read the word with
 * mha_check_device_status. Nothing faults, traps or hangs, and no other work of the
 * library is affected.
 */
#define MHA_SELFTEST_WAIT_CODE 0x7f1
mha_status_t mha_selftest_wait_timeout(void* stream);

/* Library version string. */
const char* mha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_MHA_H */
