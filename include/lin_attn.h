/*
 * lin_attn.h - C ABI of the GB300 (sm_103a) SANA-Video linear-attention layer core.
 *
 * Operation (page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear
 * attention in quality=high", section 关键源码片段, snippets
 * `sana_video_linear_attention_site.py` (try_sana_video_linear_attention) and
 * `sana_video.py` (SanaVideoLinearAttention.forward, FP32 fallback chain)):
 * for every head h of a batch-1 layer,
 *
 *     KV[h]  = K_rot[h]^T . V[h]                 a D x D matrix, reduced over the N tokens
 *     out[h] = (Q_rot[h] . KV[h]) / den[h]       den[h][n] is the layer's normaliser denominator
 *
 * The page keeps the operands as [B, H, D, N] views and forms scores = V . K_rot^T and
 * (scores @ Q_rot) * normalizer; with contiguous [1, H, N, D] storage those are the
 * transposes of the two products above, so the numbers are the same.
 *
 * Quality tiers (same page, 功能与动机 and the site snippet):
 *   LIN_ATTN_MODE_HIGH      first GEMM on BF16 operands, FP32 accumulation and output;
 *                           second GEMM at FP32 accuracy (here: Q . (KV_hi + KV_mid + KV_lo)
 *                           with KV split into three BF16 terms, FP32 accumulation).
 *   LIN_ATTN_MODE_LOSSLESS  the FP32 chain: Q, K, V upcast to FP32 before both GEMMs.  The
 *                           inputs are BF16, so every product is exact in FP32 either way and
 *                           this tier runs the same tensor-core kernels, with the first GEMM's
 *                           tensor-core sums promoted into IEEE FP32 registers every 64 tokens
 *                           (every 256 in 'high').
 * Both tiers have the same exact result; they differ only in rounding.
 *
 * Conventions shared by every entry point:
 *   - All tensors are contiguous row-major, batch 1.  q_rot, k_rot, v: BF16 [1, H, N, D];
 *     normalizer: FP32 [1, H, N, 1] (the denominator, positive); out: FP32 or BF16 [1, H, N, D].
 *   - Device pointers must live on the context's device and be 16-byte aligned.
 *   - The caller owns every tensor; the context owns only its scratch.
 *   - Calls enqueue on `stream` (a cudaStream_t; NULL = legacy default stream) and return
 *     without synchronising, unless stated otherwise.
 *   - The layer calls (lin_attn_forward, _layout, _fused, _fused_layout) enqueue kernel
 *     launches only - no allocation, no synchronisation - so a sequence of them may be
 *     captured into a CUDA graph (stream capture); the replay gives the same bits.
 *   - A context may be used by one stream at a time (its scratch is shared by all calls);
 *     distinct contexts share no device state and may run at once.
 *   - `out` must not overlap any input.
 *   - Return value: LIN_ATTN_OK or one of the LIN_ATTN_ERR_* codes below; on error nothing
 *     was enqueued (except LIN_ATTN_ERR_CUDA after a failed launch) and
 *     lin_attn_last_error() gives a one-line reason for the calling thread.
 *   - Results are deterministic: for the same inputs the output is bitwise the same from
 *     run to run (the cross-CTA reduction has a fixed order that depends only on the
 *     shape and the tier; see lin_attn_kv_plan).
 */
#ifndef LIN_ATTN_H
#define LIN_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st * */
struct CUevent_st;  /* cudaEvent_t  == struct CUevent_st *  */

typedef struct lin_attn_ctx lin_attn_ctx;

enum lin_attn_mode { LIN_ATTN_MODE_HIGH = 0, LIN_ATTN_MODE_LOSSLESS = 1 };
enum lin_attn_out_dtype { LIN_ATTN_OUT_F32 = 0, LIN_ATTN_OUT_BF16 = 1 };
enum lin_attn_layout {
    LIN_ATTN_LAYOUT_HND = 0, /* q_rot, k_rot, v, out: [1, H, N, D] (each head one N x D block)  */
    LIN_ATTN_LAYOUT_NHD = 1  /* q_rot, k_rot, v: [1, N, H, D]; out: [1, N, H*D] (token-major)   */
};

enum lin_attn_status {
    LIN_ATTN_OK = 0,
    LIN_ATTN_ERR_INVALID_ARG = 1, /* null pointer, size out of range, bad enum value        */
    LIN_ATTN_ERR_UNSUPPORTED = 2, /* head_dim not a multiple of 16 in [16, 128], no sm_100+ */
    LIN_ATTN_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned                */
    LIN_ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a kernel launch failed   */
    LIN_ATTN_ERR_OOM = 5,         /* device or pinned-host allocation failed                */
    LIN_ATTN_ERR_TIMEOUT = 6      /* a kernel gave up waiting on one of its own barriers    */
};

/*
 * Create a context for layers of `heads` heads, up to `max_tokens` tokens and head dim
 * `head_dim` on CUDA device `device`.  Allocates all scratch the forward pass needs
 * (per-chunk partial KV sums, the reduced KV, its three-term BF16 image, a status word),
 * so lin_attn_forward never allocates.  head_dim must be a multiple of 16 in [16, 128];
 * smaller head dims are served by zero-padding D (padding leaves out[..., :D] unchanged).
 * 1 <= heads <= 4096, 1 <= max_tokens <= 2^30.  On success *ctx is set; on failure *ctx
 * is NULL.  The calling thread's current device is left as it was.
 */
int lin_attn_create(lin_attn_ctx **ctx, int heads, int64_t max_tokens, int head_dim, int device);

/* Free the context and its scratch (waits for the device to finish with it).  NULL is OK. */
int lin_attn_destroy(lin_attn_ctx *ctx);

/*
 * One layer call on device tensors (see the conventions above):
 *   q_rot, k_rot, v : BF16 [1, heads, n_tokens, head_dim]
 *   normalizer      : FP32 [1, heads, n_tokens, 1], the denominator den[h][n]
 *   out             : out_dtype (LIN_ATTN_OUT_F32 / LIN_ATTN_OUT_BF16) [1, heads, n_tokens, head_dim];
 *                     BF16 output is rounded to nearest-even from the FP32 result
 *   n_tokens        : 1 <= n_tokens <= max_tokens of the context
 *   mode            : LIN_ATTN_MODE_HIGH or LIN_ATTN_MODE_LOSSLESS
 * Enqueues three kernels (per-chunk KV partial sums, fixed-order reduction, apply +
 * normalise) on `stream`.
 */
int lin_attn_forward(lin_attn_ctx *ctx, const void *q_rot, const void *k_rot, const void *v,
                     const float *normalizer, void *out, int out_dtype, int64_t n_tokens,
                     int mode, struct CUstream_st *stream);

/*
 * lin_attn_forward with a choice of activation layout.  LIN_ATTN_LAYOUT_NHD reads Q_rot,
 * K_rot, V as [1, N, H, D] - the per-head views of the model's packed projection output,
 * before the page's permute to [B, H, D, N] (page 1, 关键源码片段, `sana_video.py`:
 * `.view(batch_size, sequence_length, num_heads, head_dim)`) - and writes out as
 * [1, N, H*D], the `flatten(1, 2).transpose(1, 2)` form the output projection consumes.
 * The normaliser stays [1, H, N, 1] (the page's [B, H, 1, N]).  Same numbers as the
 * head-major call (bitwise); LIN_ATTN_LAYOUT_HND is exactly lin_attn_forward.
 */
int lin_attn_forward_layout(lin_attn_ctx *ctx, const void *q_rot, const void *k_rot, const void *v,
                            const float *normalizer, void *out, int out_dtype, int64_t n_tokens,
                            int mode, int layout, struct CUstream_st *stream);

/*
 * The layer call with the producer step fused in (either tier): what the model does right
 * before the two GEMMs (page 1, 关键源码片段, `sana_video.py`: `F.relu` on the normalised
 * query and key, `apply_interleaved_rotary_emb` on the activated copies, and the normaliser
 * from the un-rotated activated copies) runs inside the kernels, on the tiles they load.
 *   q, k     : BF16 [1, H, N, D], the normalised projections BEFORE ReLU and RoPE
 *   v        : BF16 [1, H, N, D]
 *   rope_cos, rope_sin : FP32 [N, D/2]; pair p (elements 2p, 2p+1) of token n turns by
 *              (rope_cos, rope_sin)[n][p]
 *   out      : as lin_attn_forward (head-major)
 * Computes qa = relu(q), ka = relu(k); Q_rot, K_rot = each pair (x0, x1) of qa, ka turned to
 * (x0 c - x1 s, x0 s + x1 c) with binary32 products and sums in exactly that order, rounded
 * once to BF16 (nearest-even); den[h][n] = qa[h][n] . (sum over m of ka[h][m]) + 1e-6; then
 * the two GEMMs and the normalisation of lin_attn_forward.  The column sums of relu(K) are
 * accumulated with compensated binary32 sums per chunk and reduced in FP64 in a fixed
 * order, then rounded once to FP32.  mode: LIN_ATTN_MODE_HIGH or LIN_ATTN_MODE_LOSSLESS, as
 * for lin_attn_forward.
 */
int lin_attn_forward_fused(lin_attn_ctx *ctx, const void *q, const void *k, const void *v,
                           const float *rope_cos, const float *rope_sin, void *out, int out_dtype,
                           int64_t n_tokens, int mode, struct CUstream_st *stream);

/*
 * lin_attn_forward_fused with a choice of activation layout.  LIN_ATTN_LAYOUT_NHD reads q,
 * k, v as [1, N, H, D] (the per-head views of the model's packed projection output, page 1,
 * 关键源码片段, `sana_video.py`: `.view(batch_size, sequence_length, num_heads, head_dim)`)
 * and writes out as [1, N, H*D]; the rotation tables are per token in both layouts.  Same
 * numbers as the head-major call (bitwise).  LIN_ATTN_ERR_INVALID_ARG for an unknown layout.
 */
int lin_attn_forward_fused_layout(lin_attn_ctx *ctx, const void *q, const void *k, const void *v,
                                  const float *rope_cos, const float *rope_sin, void *out, int out_dtype,
                                  int64_t n_tokens, int mode, int layout, struct CUstream_st *stream);

/*
 * SANA-Video 2.0 softmax anchor layer (page "[sglang] SANA-Video 2.0 anchor attention의
 * FP32 upcast 제거로 720p 생성 52% 단축하기", 코드 분석 §2: F.scaled_dot_product_attention(q,
 * k, v, dropout_p=0.0) on BF16 [B, H, N, D], the page's 'high' path): per head,
 *     out = softmax(scale * Q K^T) V         no mask; scale <= 0 means 1 / sqrt(head_dim)
 *   q, k, v : BF16 [1, heads, n_tokens, head_dim] (the context's heads and head_dim)
 *   out     : FP32 or BF16 [1, heads, n_tokens, head_dim]
 * Flash-attention forward on tensor cores: FP32 scores and accumulator, the softmax
 * weights rounded to BF16 for the second product.  Uses no scratch; timeouts are reported
 * through lin_attn_device_status.
 */
int lin_attn_anchor_forward(lin_attn_ctx *ctx, const void *q, const void *k, const void *v, void *out,
                            int out_dtype, int64_t n_tokens, float scale, struct CUstream_st *stream);

/*
 * Same layer call on HOST buffers (same shapes and dtypes, any alignment).  Copies the
 * inputs to device staging owned by the context, runs the layer, copies the result
 * back and synchronises `stream` before returning: when it returns OK, `out` holds the
 * result (bitwise the same as lin_attn_forward gives).  The work is pipelined over chunks
 * of heads: host-to-device copies, kernels (on `stream`) and device-to-host copies of
 * different chunks overlap, on two extra streams owned by the context.  The staging,
 * streams and events are created on the first call (LIN_ATTN_ERR_OOM if the staging
 * cannot be allocated) and kept until lin_attn_destroy.  Page-locked host buffers give
 * full copy bandwidth and overlap; pageable ones work but copy slower.
 */
int lin_attn_forward_host(lin_attn_ctx *ctx, const void *q_rot, const void *k_rot, const void *v,
                          const float *normalizer, void *out, int out_dtype, int64_t n_tokens,
                          int mode, struct CUstream_st *stream);

/*
 * The fused-producer layer call (lin_attn_forward_fused, head-major) on HOST buffers:
 * q, k, v BF16 [1, heads, n_tokens, head_dim], rope_cos / rope_sin FP32
 * [n_tokens, head_dim / 2], out FP32 or BF16 [1, heads, n_tokens, head_dim], any
 * alignment.  The same pipeline as lin_attn_forward_host (and its staging, streams and
 * events), with the two tables copied once ahead of the first chunk (their staging,
 * 2 x max_tokens x head_dim / 2 FP32, is allocated on the first call: LIN_ATTN_ERR_OOM if
 * it cannot be); synchronises `stream` before returning, and the result is bitwise the
 * one lin_attn_forward_fused gives.  NULL tables: LIN_ATTN_ERR_INVALID_ARG.
 */
int lin_attn_forward_fused_host(lin_attn_ctx *ctx, const void *q, const void *k, const void *v,
                                const float *rope_cos, const float *rope_sin, void *out, int out_dtype,
                                int64_t n_tokens, int mode, struct CUstream_st *stream);

/*
 * Test hook: enqueue a copy of the reduced KV of the last forward call, FP32
 * [heads, head_dim, head_dim] row-major (KV[h][i][j] = sum_n K_rot[h][n][i] V[h][n][j]),
 * into the device buffer kv_out.
 */
int lin_attn_debug_kv(lin_attn_ctx *ctx, float *kv_out, struct CUstream_st *stream);

/*
 * Synchronise `stream`, then return and clear the context's device status word:
 * LIN_ATTN_OK, or LIN_ATTN_ERR_TIMEOUT if a kernel of an earlier call gave up waiting
 * on one of its barriers (its output is then incomplete).
 */
int lin_attn_device_status(lin_attn_ctx *ctx, struct CUstream_st *stream);

/*
 * Work split of the KV reduction for this shape and tier.  k = min(152 / heads, tiles per
 * head, 150) (at least 1) chunks per head take each head's leading 64-token tiles, cut at
 * the same tokens for every head.  On long sequences (at least 256 tiles per such chunk)
 * with k * heads < 152, the 152 - k * heads spare chunks share the remaining tiles of all
 * heads (taken head after head) in equal parts; the number of leading tiles is chosen so
 * that the costliest chunk is as cheap as possible (a chunk that runs into another head
 * counts 6 tiles more per head), and the spare chunks are used only where that beats the
 * split without them.  `*chunks` = one CTA each (152 for the 720p layer at 20 or 32
 * heads), and each head's partial D x D sums - one per chunk run that lies in the head: k,
 * plus one or two from the shared tiles; the most any head has is `*max_segments` - are
 * added in a fixed pairwise order.  The split depends on (heads, n_tokens) only - never on
 * the GPU or the activation layout - which is what makes the summation order, and so the
 * result, reproducible (both tiers and both layouts use the same split).  Either
 * out-pointer may be NULL.  Returns LIN_ATTN_ERR_INVALID_ARG on bad arguments.
 */
int lin_attn_kv_plan(int heads, int64_t n_tokens, int mode, int *chunks, int *max_segments);

/*
 * Test hook: how long a kernel of this context's later calls waits on one of its own
 * barriers before it gives up, in nanoseconds (0 restores the default of 2 s; larger values
 * are LIN_ATTN_ERR_INVALID_ARG).  A kernel that gives up winds down cleanly - it lets its
 * copies and tensor-core operations in flight land, frees its tensor memory and exits -
 * and records LIN_ATTN_ERR_TIMEOUT for lin_attn_device_status; that call's output is then
 * incomplete.  With a limit below 1 ms, a wait that outlasts its first (blocking) probe is
 * then checked with non-blocking probes and gives up within about the limit.  Used to show
 * that the bounded waits report instead of hanging; calls made with the default limit are
 * unaffected.
 */
int lin_attn_set_wait_limit(lin_attn_ctx *ctx, uint64_t limit_ns);

/*
 * Timing hook.  Arms `n_events` (must be 4) CUDA events (created with timing enabled)
 * for the NEXT lin_attn_forward call only: events[0] is recorded before the KV partial
 * kernel, events[1] after it, events[2] after the reduction, events[3] after apply.
 * Passing n_events = 0 disarms.
 */
int lin_attn_set_stage_events(lin_attn_ctx *ctx, struct CUevent_st *const *events, int n_events);

/*
 * Allocation-free variant of lin_attn_forward, for callers that cannot allocate device
 * memory: a plugin whose host forbids allocation inside its execute callback, a process
 * whose device memory is reserved up front by a caching allocator or a hard memory cap,
 * or a latency-critical loop that must not pay cudaMalloc's implicit device
 * synchronisation.  The paper has no counterpart to this entry point; it is an addition
 * of this library.
 *
 * Same tensors, layouts, tiers, checks and results as lin_attn_forward, with the shape
 * given directly (heads, n_tokens, head_dim) and no context; it runs on the calling
 * thread's current device.  Its scratch is one fixed 48 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process exits; the
 * call itself makes no cudaMalloc, cudaFree or other allocating call.
 *   - The scratch a shape needs does not depend on the tier.  With k = the partial slots
 *     per head of lin_attn_kv_plan (max_segments) and every term rounded up to 256 bytes:
 *       heads * k * head_dim^2 * 4          (FP32 partial sums)
 *     + heads * head_dim^2 * 4              (reduced KV)
 *     + heads * 3 * ceil(head_dim / 64) * head_dim * 128   (the KV image)
 *     + 256                                 (status word, at the start of the array)
 *     A shape that needs more than 48 MiB is rejected with LIN_ATTN_ERR_INVALID_ARG.  The
 *     720p/193-frame layer (20 x 180320 x 112, 9 slots) needs ~11.2 MiB; at head_dim 128 and
 *     1 slot per head (heads >= 153) the limit is 219 heads.
 *   - The first call on a device resolves the array's device address (cudaGetSymbolAddress,
 *     with that device current) and keeps it; a failed attempt is not kept, so the next
 *     call retries.  Make that first call before any stream capture.
 *   - Every call uses the same array and it keeps the previous call's contents; each call
 *     clears what has to start at zero.  Calls that overlap on the GPU (from several
 *     streams or host threads) race on the array and corrupt each other's results, so
 *     serialise them.
 *   - A kernel that gives up waiting on one of its barriers (its call's output is then
 *     incomplete) is not reported by the call itself, which returns before the kernels
 *     run: it is recorded in the array's status word, which lin_attn_noalloc_status reads.
 */
int lin_attn_forward_noalloc(const void *q_rot, const void *k_rot, const void *v,
                             const float *normalizer, void *out, int out_dtype, int heads,
                             int64_t n_tokens, int head_dim, int mode, struct CUstream_st *stream);

/*
 * Status of the lin_attn_forward_noalloc calls on the calling thread's current device:
 * waits for `stream` (the stream those calls were made on), then returns
 * LIN_ATTN_ERR_TIMEOUT if a kernel of any of them since the previous query gave up
 * waiting on one of its barriers, else LIN_ATTN_OK, and clears the record.  Makes no
 * allocating call.  LIN_ATTN_ERR_CUDA / LIN_ATTN_ERR_UNSUPPORTED if the device cannot be
 * queried.
 */
int lin_attn_noalloc_status(struct CUstream_st *stream);

/* Static description of a status code. */
const char *lin_attn_error_string(int status);

/* One-line reason for the last error returned on the calling thread ("" if none). */
const char *lin_attn_last_error(void);

/* ABI version of this header (major * 100 + minor). */
int lin_attn_version(void);

#define LIN_ATTN_VERSION 100

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* LIN_ATTN_H */
