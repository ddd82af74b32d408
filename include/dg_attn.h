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
 * alone (the work-list build before it and the split-KV merge after it fall
 * outside the two events). */
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
