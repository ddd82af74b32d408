/*
 * dg_attn -- dual-mode (causal / bidirectional) attention forward pass for
 * DiffusionGemma-style block-autoregressive diffusion decoding, on one GB300
 * (sm_103a) GPU.
 *
 * The operation (DiffusionGemma, agentlenshq page, sections "dual-mode
 * operation", "dynamic per-sequence causal attention" and "symmetric
 * sliding-window attention"; molayo1419 developer guide, "block autoregressive
 * denoising"; 24-ai.news page, "why diffusion differs"):
 *
 *   One call handles a packed batch of B sequences.  Sequence s has
 *   ctx_len[s] = c cached tokens (absolute positions 0..c-1) and
 *   n = cu_q[s+1] - cu_q[s] query tokens (positions c..c+n-1).  Its K/V rows
 *   are its c cached rows followed by the n rows of its own query tokens
 *   (L = c + n rows), stored contiguously right after sequence s-1's rows.
 *
 *   mode[s] == DG_MODE_CAUSAL (encoder mode: prefill, incremental prefill,
 *   commit of a finished canvas): the query at position i sees keys j <= i.
 *   mode[s] == DG_MODE_BIDIRECTIONAL (decoder / denoise mode): every query
 *   sees the whole cached context and every query token of its own block.
 *
 *   window < 0: full layer.  window = W >= 0: sliding-window layer; a causal
 *   query sees the W preceding tokens plus itself (W+1 keys), a bidirectional
 *   query sees W tokens on each side (2W+1), both clipped to [0, L-1].
 *
 *   out[r, h, :] = sum_j softmax_j(scale * q[r,h,:] . k[j,g,:]) v[j,g,:]
 *   lse[r, h]    = ln sum_j exp(scale * q[r,h,:] . k[j,g,:])
 *   over the visible keys j, with g = h / (Hq / Hkv) (grouped-query heads).
 *
 * Conventions for every entry point:
 *   - The caller owns all memory.  Device pointers must be device-accessible
 *     on the current CUDA device.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  dg_attn_forward neither synchronises nor allocates.
 *   - Errors the host can see are returned at once and nothing is enqueued.
 *     Errors found on the device (bad metadata contents, an internal wait
 *     that timed out) are recorded in a per-device status word that
 *     dg_attn_status() reads; the kernels then skip the remaining work and
 *     return instead of hanging.
 *   - Calls are reentrant; concurrent calls must use distinct workspaces.
 */
#ifndef DG_ATTN_H_
#define DG_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dg_status {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or metadata   */
  DG_ERR_UNSUPPORTED = 2,     /* head_dim / group size / GPU not supported  */
  DG_ERR_CUDA = 3,            /* a CUDA runtime call failed                 */
  DG_ERR_WORKSPACE = 4,       /* workspace NULL, misaligned or too small    */
  DG_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait expired         */
  DG_ERR_DEVICE_BOUNDS = 6    /* device-side bounds check failed            */
} dg_status_t;

enum { DG_MODE_CAUSAL = 0, DG_MODE_BIDIRECTIONAL = 1 };

/* Bytes of device workspace dg_attn_forward needs for these sizes on the
 * current device (it depends on the device's SM count).  Returns 0 when the
 * sizes are invalid (negative, Hq % Hkv != 0, unsupported head_dim). */
size_t dg_attn_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim);

/* Kernels one forward call with these sizes launches on its stream: 2 (the
 * attention grid, which builds its work list itself, and the split-KV merge)
 * for contiguous K/V batches of at most 256 query tiles (bounded from the
 * sizes) other than e4m3 at head_dim 128, else 3 (a work-list grid first).
 * paged / e4m3: nonzero for dg_attn_forward_paged / dg_attn_forward_fp8.
 * Host only (no device needed); reads the same environment switch as the
 * call.  Returns 0 when the sizes are invalid. */
int32_t dg_attn_launches_per_call(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t paged,
                                  int32_t e4m3);

/* Dual-mode attention forward.
 *
 *   q          bf16 device [total_q, num_q_heads, head_dim], row-major, 16-byte aligned
 *   k, v       bf16 device [total_kv, num_kv_heads, head_dim], row-major, 16-byte aligned
 *   cu_q       int32 device [num_seqs+1]; cu_q[0] = 0, non-decreasing, cu_q[num_seqs] = total_q
 *   ctx_len    int32 device [num_seqs]; cached tokens before each sequence's queries (>= 0)
 *   mode       uint8 device [num_seqs]; DG_MODE_CAUSAL or DG_MODE_BIDIRECTIONAL
 *   total_kv   rows of k/v; must be >= sum(ctx_len) + total_q
 *   head_dim   64, 128 or 256;  num_q_heads % num_kv_heads == 0 and
 *              num_q_heads / num_kv_heads <= 128
 *   window     -1 (full layer) or W >= 0 (sliding window)
 *   scale      softmax scale (finite, > 0), e.g. 1/sqrt(head_dim)
 *   out        bf16 device [total_q, num_q_heads, head_dim], 16-byte aligned (written)
 *   lse        fp32 device [total_q, num_q_heads] natural-log LSE, or NULL (written)
 *   workspace  device scratch of >= dg_attn_workspace_size(...) bytes, 256-byte
 *              aligned; contents need not be initialised and are clobbered
 *   stream     cudaStream_t
 *
 * Returns DG_OK when the work was enqueued. */
dg_status_t dg_attn_forward(const void* q, const void* k, const void* v,
                            const int32_t* cu_q, const int32_t* ctx_len, const uint8_t* mode,
                            int32_t num_seqs, int32_t total_q, int32_t total_kv,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t window, float scale,
                            void* out, float* lse,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/* Same as dg_attn_forward, and additionally records the caller's CUDA events
 * (cudaEvent_t, either may be NULL) on `stream` immediately before and after
 * the launch of the main attention kernel, so a caller can time that kernel
 * alone (the split-KV merge after it, and the work-list grid before it where
 * there is one, fall outside the two events; batches of at most 256 query
 * tiles with contiguous K/V have no work-list grid, the attention kernel's
 * CTAs build the list themselves, inside the events). */
dg_status_t dg_attn_forward_profiled(const void* q, const void* k, const void* v,
                                     const int32_t* cu_q, const int32_t* ctx_len,
                                     const uint8_t* mode, int32_t num_seqs, int32_t total_q,
                                     int32_t total_kv, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t window, float scale,
                                     void* out, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream, void* attn_begin_event, void* attn_end_event);

/* Capacity, in bytes, of the static scratch array used by
 * dg_attn_forward_noalloc (48 MiB). */
#define DG_ATTN_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)

/* The forward pass for callers that cannot allocate device memory: callers
 * embedded in a host framework that owns every device allocation (a
 * pre-planned arena, a plugin interface that hands out no scratch), or loops
 * that cannot afford cudaMalloc's device-wide synchronisation between steps.
 * The pages describe no such entry point; it exists for those callers only.
 *
 * Same arguments and results as dg_attn_forward without the workspace: the
 * scratch is a file-scope __device__ array of DG_ATTN_NOALLOC_SCRATCH_BYTES
 * inside this library, which every GPU that loads the library holds until the
 * process exits.  The caller still owns q, k, v, the metadata, out and lse.
 *
 *   - Returns DG_ERR_WORKSPACE, having enqueued nothing, when these sizes
 *     need more scratch than the array holds (dg_attn_workspace_size() tells
 *     the requirement).
 *   - Calls no cudaMalloc / cudaFree and no allocating library routine.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents; nothing in it needs to start at zero.  Calls whose
 *     work overlaps on the GPU (other streams, other threads) race on it:
 *     serialise them.
 *   - The first call of any dg_attn entry point on a device looks up the
 *     array's device address (a one-time set-up per device); make that
 *     first call before any stream capture. */
dg_status_t dg_attn_forward_noalloc(const void* q, const void* k, const void* v,
                                    const int32_t* cu_q, const int32_t* ctx_len,
                                    const uint8_t* mode, int32_t num_seqs, int32_t total_q,
                                    int32_t total_kv, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t window, float scale,
                                    void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 variant: the same forward pass with Q, K and V given as e4m3 bytes (the
 * OCP E4M3 format), one fp32 scale per tensor, so that the attention is that
 * of q_scale * q, k_scale * k and v_scale * v.  The pages serve the model from
 * FP8 checkpoints (agentlenshq page, "quantised checkpoints"; the throughput
 * results are FP8 runs) but do not state FP8 attention: this is a variant.
 *
 * Both matrix products run on the tensor cores in e4m3 (tcgen05
 * kind::f8f6f4) with fp32 accumulation; the softmax probabilities are scaled
 * by 2^5 and rounded to e4m3 before P.V (relative error <= 2^-4 each), the
 * running maximum being refreshed once it grew by more than 2^3.  out is
 * bf16, lse fp32 (natural log of the scaled scores' exponential sum).
 *
 *   q  e4m3 bytes device [total_q, Hq, D]; k, v [total_kv, Hkv, D]; 16-byte aligned
 *   head_dim 128 or 256 (64 returns DG_ERR_UNSUPPORTED)
 *   q_scale, k_scale, v_scale  finite, > 0
 * Everything else is as for dg_attn_forward (same workspace size).
 */
dg_status_t dg_attn_forward_fp8(const void* q, const void* k, const void* v, const int32_t* cu_q,
                                const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
                                int32_t total_q, int32_t total_kv, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale,
                                float q_scale, float k_scale, float v_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/* dg_attn_forward_fp8 with two CUDA events recorded around the main kernel. */
dg_status_t dg_attn_forward_fp8_profiled(
    const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* ctx_len,
    const uint8_t* mode, int32_t num_seqs, int32_t total_q, int32_t total_kv, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale, float q_scale,
    float k_scale, float v_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
    void* stream, void* attn_begin_event, void* attn_end_event);

/* ---------------------------------------------------------------------------
 * The same forward pass over a paged KV cache, with the append of the query
 * tokens' K/V fused into the call.  DiffusionGemma pages: the encoder (causal)
 * pass writes finished blocks into the KV cache and every committed canvas is
 * appended to it (agentlenshq page, "dual-mode operation"; developer guide,
 * "block autoregressive denoising", the prefill item); vLLM's prefix caching
 * works unchanged, i.e. the cache is block-based (agentlenshq page,
 * "dual-mode operation").  The pages do not describe the cache layout; this
 * one is the common block-table layout:
 *
 *   k_cache, v_cache  bf16 device [num_pages, page_size, num_kv_heads, head_dim],
 *                     16-byte aligned, caller-owned; the call writes the
 *                     appended rows and reads the rest
 *   page_size         rows per page: a power of two in [8, 65536];
 *                     num_pages * page_size <= INT32_MAX
 *   block_table       int32 device [num_seqs, max_pages_per_seq]:
 *                     block_table[s][p] = physical page of positions
 *                     p*page_size .. p*page_size+page_size-1 of sequence s;
 *                     only entries 0 .. ceil((ctx_len[s]+n_s)/page_size)-1 are
 *                     read, each must lie in [0, num_pages) (device-checked:
 *                     DG_ERR_INVALID_ARG in the status word, nothing computed)
 *   k_new, v_new      bf16 device [total_q, num_kv_heads, head_dim], packed like
 *                     q: the K/V rows of the query tokens, written at positions
 *                     ctx_len[s] .. ctx_len[s]+n_s-1 of their sequence before
 *                     the attention reads the cache (this step's canvas
 *                     overwrites the previous step's); both NULL when those
 *                     rows are already in the cache.  The pages written must
 *                     not be shared with another sequence of the batch.
 *
 * Everything else (q, cu_q, ctx_len, mode, shapes, window, scale, out, lse,
 * status and ordering rules) is as for dg_attn_forward, and the workspace is
 * dg_attn_workspace_size() bytes.  Keys of sequence s are positions
 * 0 .. ctx_len[s]+n_s-1 read through its page-table row.
 */
dg_status_t dg_attn_forward_paged(const void* q, const void* k_new, const void* v_new,
                                  void* k_cache, void* v_cache, int32_t num_pages,
                                  int32_t page_size, const int32_t* block_table,
                                  int32_t max_pages_per_seq, const int32_t* cu_q,
                                  const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
                                  int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t window, float scale, void* out,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* dg_attn_forward_paged with two CUDA events (cudaEvent_t, created by the
 * caller) recorded around the main attention kernel, as in
 * dg_attn_forward_profiled. */
dg_status_t dg_attn_forward_paged_profiled(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    int32_t num_pages, int32_t page_size, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* cu_q, const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
    int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t window,
    float scale, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
    void* attn_begin_event, void* attn_end_event);

/* ---------------------------------------------------------------------------
 * Self-conditioning input of the next denoise step (DiffusionGemma, agentlenshq
 * page, "self-conditioning for stability"; 24-ai.news page, the
 * self-conditioning signal between iterations): every canvas position's
 * softmax distribution over the vocabulary becomes the probability-weighted
 * average of the token embeddings,
 *
 *   out[r, :] = sum_v softmax(logits[r, :])_v * embedding[v, :]
 *
 * (softmax at temperature 1; the gated MLP the model applies afterwards is not
 * part of this call).  The probabilities are rounded to bf16 for the tensor
 * cores; sums are fp32.
 *
 *   logits     bf16 device [rows, vocab], row-major, 16-byte aligned;
 *              vocab % 8 == 0; -inf entries are masked tokens, NaN is not
 *              allowed; a row needs at least one finite logit
 *   embedding  bf16 device [vocab, d_model], row-major, 16-byte aligned;
 *              d_model % 8 == 0
 *   out        fp32 device [rows, d_model], 16-byte aligned, caller-owned
 *   workspace  >= dg_selfcond_workspace_size(rows, vocab, d_model) bytes,
 *              256-byte aligned (row statistics and, for large vocabularies,
 *              per-split fp32 partial sums)
 *
 * Asynchronous on `stream`; no allocation; host-checkable errors return
 * immediately (DG_ERR_INVALID_ARG, DG_ERR_WORKSPACE).
 */
size_t dg_selfcond_workspace_size(int32_t rows, int32_t vocab, int32_t d_model);

dg_status_t dg_selfcond_forward(const void* logits, int32_t rows, int32_t vocab,
                                const void* embedding, int32_t d_model, float* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* dg_selfcond_forward with two CUDA events (cudaEvent_t, created by the caller)
 * recorded around its tensor-core kernel. */
dg_status_t dg_selfcond_forward_profiled(const void* logits, int32_t rows, int32_t vocab,
                                         const void* embedding, int32_t d_model, float* out,
                                         void* workspace, size_t workspace_bytes, void* stream,
                                         void* gemm_begin_event, void* gemm_end_event);

/* ---------------------------------------------------------------------------
 * Entropy-bounded acceptance of one denoise step (DiffusionGemma, agentlenshq
 * page, "sampling loop and entropy-bounded denoising"; 24-ai.news page, "the
 * mechanism for deciding finished tokens").  For every canvas position the
 * LM-head logits give a softmax over the vocabulary; the step computes, per
 * row, the entropy H (nats), the confidence c (largest probability) and the
 * argmax (lowest index on ties).  Per canvas, the rows not yet accepted are
 * ranked by confidence (ties to the lower row) and accepted in that order while
 * the running entropy sum, accumulated in fp32 in ranking order, stays within
 * `entropy_budget`; the most confident open row is always accepted.  The canvas
 * has converged when every argmax equals the previous step's for `patience`
 * consecutive steps (stable_out = stable_in + 1, or 0 when any argmax changed)
 * and the mean entropy (fp32 sum in row order, divided by the row count) is
 * below `entropy_threshold`, or when step + 1 >= max_steps.
 *
 *   logits        bf16 device [rows, vocab], row-major, 16-byte aligned; -inf
 *                 entries are masked tokens (probability 0), NaN is not allowed;
 *                 a row needs at least one logit above the lowest finite bf16
 *                 (otherwise it has no distribution and its outputs are unspecified)
 *   cu_rows       int32 device [num_canvases+1]: canvas b owns rows
 *                 cu_rows[b] .. cu_rows[b+1]-1 (at most 1024 rows per canvas;
 *                 a larger canvas records DG_ERR_INVALID_ARG in the status word)
 *   accepted_in   uint8 device [rows], 1 = accepted in an earlier step
 *   argmax_prev   int32 device [rows], the previous step's argmax
 *   stable_in     int32 device [num_canvases]
 *   entropy_out, confidence_out  fp32 device [rows];  argmax_out int32 [rows]
 *   accepted_out  uint8 device [rows] (accepted_in plus this step's acceptances)
 *   stable_out    int32 device [num_canvases];  converged_out uint8 [num_canvases]
 *   workspace     >= dg_accept_workspace_size(rows, vocab) bytes, 256-byte aligned
 */
size_t dg_accept_workspace_size(int32_t rows, int32_t vocab);

dg_status_t dg_accept_step(const void* logits, int32_t rows, int32_t vocab,
                           const int32_t* cu_rows, int32_t num_canvases,
                           const uint8_t* accepted_in, const int32_t* argmax_prev,
                           const int32_t* stable_in,
                           float entropy_budget, float entropy_threshold,
                           int32_t patience, int32_t step, int32_t max_steps,
                           float* entropy_out, float* confidence_out, int32_t* argmax_out,
                           uint8_t* accepted_out, int32_t* stable_out, uint8_t* converged_out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The sampler's per-step work on one set of LM-head logits, in one call: the
 * acceptance step above and the self-conditioning average (dg_selfcond_forward)
 * of the same logits (DiffusionGemma, agentlenshq page, "sampling loop and
 * entropy-bounded denoising" and "self-conditioning for stability": both are
 * taken from the same step's softmax distribution).  Both need every row's softmax statistics; they are
 * computed once (one pass over the logits instead of two).  Arguments as in
 * the two calls; workspace >= dg_sampler_workspace_size(rows, vocab, d_model)
 * bytes, 256-byte aligned.  The outputs equal those of the two separate calls
 * bit for bit.
 */
size_t dg_sampler_workspace_size(int32_t rows, int32_t vocab, int32_t d_model);

dg_status_t dg_sampler_step(const void* logits, int32_t rows, int32_t vocab, const int32_t* cu_rows,
                            int32_t num_canvases, const uint8_t* accepted_in,
                            const int32_t* argmax_prev, const int32_t* stable_in,
                            float entropy_budget, float entropy_threshold, int32_t patience,
                            int32_t step, int32_t max_steps, const void* embedding, int32_t d_model,
                            float* entropy_out, float* confidence_out, int32_t* argmax_out,
                            uint8_t* accepted_out, int32_t* stable_out, uint8_t* converged_out,
                            float* selfcond_out, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Synchronises `stream`, returns the current device's status word (DG_OK if
 * no device-side error was recorded since the last call) and clears it. */
dg_status_t dg_attn_status(void* stream);

/* Static, human-readable text of a status code. */
const char* dg_attn_error_string(int32_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t dg_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_ATTN_H_ */
