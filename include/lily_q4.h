/*
 * lily_q4.h -- C ABI of the GB300 (sm_103a) MLX-affine 4-bit mixture-of-experts hot path.
 *
 * The operations follow the Lily pages' statement of the problem:
 *
 *  - Weight format: MLX affine 4-bit weights in groups of 64 (Lily README, first
 *    paragraph and "Requirements"; Lily-vs-MLX report, "Hardware and software").
 *    Reading taken: dequantised weight
 *    w = s*q + b, q a 4-bit code, eight codes per uint32 along K with the lowest
 *    nibble first, one bf16 scale s and one bf16 bias b per 64 consecutive K.
 *  - The MoE feed-forward of a decode step and of a prefill chunk (the MoE
 *    kernels and the tiling of the expert GEMM, fork page, "How the speed was
 *    achieved"; decode is bandwidth-bound, prefill compute-bound, same
 *    section): router logits, top-k with softmax over the k, SwiGLU experts,
 *    down projection with the weighted combine, and a shared expert gated by
 *    sigmoid(x . g_shared) (fork page, "The model": the shared expert).
 *  - Greedy token selection without logprobs (Lily README, first paragraph;
 *    Lily-vs-MLX report, "Measurement contract"): LM-head GEMV fused with argmax,
 *    the token id staying on the device.
 *
 * Conventions for every call below:
 *  - Matrices are [N rows (outputs) x K columns (inputs)], row-major:
 *      w  uint32 [N][K/8]    (code k of row n = (w[n][k/8] >> 4*(k%8)) & 15)
 *      s  bf16   [N][K/64]   (bit patterns, uint16)
 *      b  bf16   [N][K/64]
 *    Expert stacks add a leading [E] axis (expert e at offset e*N*K/8 words).
 *  - Activations are bf16 bit patterns (uint16), row-major [T][K].
 *  - All data pointers are DEVICE pointers, except in lily_q4_pack/unpack.  The
 *    caller owns every buffer, the workspace included; no call allocates or
 *    frees device memory.
 *  - Every compute call is enqueued on `stream` and returns without waiting.
 *    Argument errors are reported before anything is enqueued.  Calls that
 *    share a workspace must be ordered (same stream, or synchronised).
 *  - Workspace: at least the size the matching *_workspace_bytes call returns,
 *    256-byte aligned, zero-filled once before its first use (lily_q4_workspace_init
 *    or a memset).  The calls leave it reusable; they never need it cleared again.
 *  - Results are deterministic: no floating-point atomics touch an output.
 *  - NaN/Inf inputs are outside the contract (results unspecified).
 */
#ifndef LILY_Q4_H
#define LILY_Q4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LILY_Q4_API __attribute__((visibility("default")))
#else
#define LILY_Q4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *lily_q4_stream_t;

/* Status codes.  0 = success, negative = failure. */
#define LILY_Q4_OK 0
#define LILY_Q4_ERR_INVALID_ARG (-1)          /* null / misaligned pointer, bad size */
#define LILY_Q4_ERR_UNSUPPORTED (-2)          /* valid but outside the shapes built */
#define LILY_Q4_ERR_WORKSPACE_TOO_SMALL (-3)
#define LILY_Q4_ERR_CUDA (-4)                 /* a CUDA launch or query failed */
#define LILY_Q4_ERR_TIMEOUT (-5)              /* a bounded device-side wait gave up */

#define LILY_Q4_GROUP 64

/* One Q4 matrix (or a stack over experts).  Device pointers; w 16-byte aligned,
 * s and b 16-byte aligned. */
typedef struct {
  const uint32_t *w;
  const uint16_t *s;
  const uint16_t *b;
} lily_q4_mat;

/* One MoE layer.  Host struct holding device pointers. */
typedef struct {
  int32_t hidden;      /* H: model width (K of gate/up, N of down) */
  int32_t n_experts;   /* E: routed experts, 1..1024 */
  int32_t top_k;       /* k: experts per token, 1..16, <= E */
  int32_t inter;       /* I: expert intermediate width (N of gate/up, K of down) */
  lily_q4_mat gate;    /* [E][I][H/8] codes, [E][I][H/64] s, b */
  lily_q4_mat up;      /* [E][I][H/8] ... */
  lily_q4_mat down;    /* [E][H][I/8] ... */
  int32_t has_shared;  /* 0 or 1 */
  lily_q4_mat sh_gate; /* [I][H/8] ... shared expert, same widths; ignored if !has_shared */
  lily_q4_mat sh_up;   /* [I][H/8] ... */
  lily_q4_mat sh_down; /* [H][I/8] ... */
  const uint16_t *router;      /* bf16 [E][H] (row e = the weights of expert e's logit) */
  const float *router_bias;    /* fp32 [E] added to the logits, or NULL */
  const uint16_t *shared_gate; /* bf16 [H] (g_shared); required iff has_shared */
  /* Affine 8-bit parts (the report's checkpoint keeps its router gates at 8 bits, "Hardware
   * and software"; the fork page's q4-xl conversion keeps the shared expert at 8 bits, "The
   * model").  8-bit codes: four per uint32 along K, lowest byte first, same bf16 s/b per 64.
   * Zero-initialised fields mean the 4-bit / bf16 layout above.  Both lily_q4_moe_decode and
   * lily_q4_moe_prefill take them (prefill prepares them in its workspace: see there). */
  int32_t shared_bits;         /* 0 or 4: sh_* as above; 8: sh_gate/sh_up [I][H/4], sh_down [H][I/4] */
  int32_t router_bits;         /* 0 or 16: bf16 router; 8: router_q8 [E][H/4] codes (router unused) */
  lily_q4_mat router_q8;       /* the 8-bit router when router_bits == 8 */
} lily_q4_moe_layer;

/* Shapes built: H and I in {64,128,256,512,1024,2048}; E <= 1024; k <= 16.
 * Others return LILY_Q4_ERR_UNSUPPORTED. */

/*
 * lily_q4_moe_decode -- MoE feed-forward of T decode tokens (1 <= T <= 16).
 *
 *   logits[t][e] = sum_h x[t][h] * router[e][h] (+ router_bias[e]), fp32, not rounded;
 *   top-k by (logit desc, index asc); p = softmax over the k selected logits;
 *   sigma[t] = sigmoid(sum_h x[t][h] * shared_gate[h])            (if has_shared);
 *   h_e = silu(Wg_e x) * (Wu_e x);  y[t] = sum_i p_i Wd_{e_i} h_{e_i} + sigma Wd_s h_s.
 *
 * x: bf16 [T][H] (16-byte aligned).  y: bf16 [T][H] output (16-byte aligned).
 * topk_idx: int32 [T][k] output (experts in descending logit order) or NULL.
 * topk_w: fp32 [T][k] output (p, same order) or NULL.
 * An expert chosen by several tokens has its rows dequantised once per row block and
 * applied to each of those tokens.
 * Up to 4 tokens (shapes permitting, see lily_q4_moe_launches) run as one launch of one
 * block per SM with two grid-wide barriers; its waits are bounded, and one that gives up is
 * reported by lily_q4_workspace_status.
 * T == 0 returns LILY_Q4_OK and enqueues nothing.
 */
LILY_Q4_API int lily_q4_moe_decode(const lily_q4_moe_layer *layer, const uint16_t *x, int32_t T,
                       uint16_t *y, int32_t *topk_idx, float *topk_w, void *ws,
                       size_t ws_bytes, lily_q4_stream_t stream);

/*
 * lily_q4_moe_prefill -- the same function for a prompt chunk of T tokens
 * (1 <= T <= 8192), computed as a grouped GEMM per expert on the tensor cores
 * (tcgen05, bf16 operands, fp32 accumulation): tokens are bucketed by expert
 * (stable: token order within an expert), the expert's dequantised weight tiles
 * are multiplied with the gathered token rows, the SwiGLU and the weighted
 * combine are fused into the epilogues.  Arguments as lily_q4_moe_decode.
 * Intermediate activations h are rounded to bf16 (tensor-core operand).
 * Affine 8-bit parts: an 8-bit router is turned, in the workspace, into an exact bf16 form
 * (s*q split into two bf16 halves, the bias term against exact bf16 parts of the per-group
 * sums of x), so its logits are as exact as those of a bf16 router; an 8-bit shared expert is
 * rewritten as 4-bit codes of twice the width (q = lo + 16 hi, the halves centred) and runs on
 * the same tensor-core path.  lily_q4_moe_workspace_bytes includes that space.
 * A bounded device-side wait that gives up is reported by lily_q4_workspace_status.
 */
LILY_Q4_API int lily_q4_moe_prefill(const lily_q4_moe_layer *layer, const uint16_t *x, int32_t T,
                        uint16_t *y, int32_t *topk_idx, float *topk_w, void *ws,
                        size_t ws_bytes, lily_q4_stream_t stream);

/*
 * lily_q4_gemv_argmax -- greedy token of a Q4 LM head:
 *   logit[n] = sum_k W[n][k] x[k] (fp32 accumulation), token = argmax_n logit[n]
 *   (ties to the lower n).
 * W: one Q4 matrix [N][K] (N >= 1).  x: bf16 [K] (16-byte aligned).
 * token: int32 [1] device output.  logits: fp32 [N] device output, or NULL.
 */
LILY_Q4_API int lily_q4_gemv_argmax(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                        int32_t *token, float *logits, void *ws, size_t ws_bytes,
                        lily_q4_stream_t stream);

/*
 * lily_q4_gemv_argmax_logprobs -- lily_q4_gemv_argmax plus the full-vocabulary
 * log-sum-exp and, optionally, the log-probability vector, in the same pass over W
 * (in the Lily-vs-MLX report, "Measurement contract", the MLX path computes both over
 * the whole vocabulary for every token).
 *   token = argmax_n logit[n] (as lily_q4_gemv_argmax),
 *   *lse = log sum_n exp(logit[n]) (fp32; running max and sum of exp, merged in a fixed
 *   order, so repeated calls give identical bits),
 *   logprobs[n] = logit[n] - *lse when logprobs is not NULL.
 * lse: fp32 [1] device output (required).  logprobs: fp32 [N] device output, or NULL; it
 * is written in a second, elementwise launch on `stream`.  Non-finite logits: +inf
 * gives lse = +inf, NaN gives NaN.  The workspace is that of lily_q4_gemv_argmax
 * (lily_q4_gemv_argmax_workspace_bytes covers both calls); errors as there.
 */
LILY_Q4_API int lily_q4_gemv_argmax_logprobs(const lily_q4_mat *W, int32_t N, int32_t K,
                                             const uint16_t *x, int32_t *token, float *lse,
                                             float *logprobs, void *ws, size_t ws_bytes,
                                             lily_q4_stream_t stream);

/*
 * lily_q8_gemv_argmax -- lily_q4_gemv_argmax for an LM head kept at 8 bits (the fork page's
 * q4-xl conversion, "The model", keeps the LM head, the shared expert and attention at 8
 * bits; the report's checkpoint, "Hardware and software", keeps its router gates at 8 bits).
 * Format: the same affine w = s*q + b with q in 0..255, four codes per uint32 along K,
 * lowest byte first (code k of row n = (w[n][k/4] >> 8*(k%4)) & 255); s and b bf16
 * [N][K/64] as for 4 bits.  W->w is uint32 [N][K/4].  K must be 512, 1024 or 2048
 * (else LILY_Q4_ERR_UNSUPPORTED).  Arguments, results and errors otherwise as
 * lily_q4_gemv_argmax; the workspace size comes from lily_q8_gemv_argmax_workspace_bytes.
 */
LILY_Q4_API int lily_q8_gemv_argmax(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                                    int32_t *token, float *logits, void *ws, size_t ws_bytes,
                                    lily_q4_stream_t stream);
/* lily_q8_gemv_argmax_logprobs -- lily_q4_gemv_argmax_logprobs for the 8-bit LM head (same
 * outputs and rules; K as lily_q8_gemv_argmax).  lily_q8_gemv_argmax_workspace_bytes covers
 * both 8-bit calls. */
LILY_Q4_API int lily_q8_gemv_argmax_logprobs(const lily_q4_mat *W, int32_t N, int32_t K,
                                             const uint16_t *x, int32_t *token, float *lse,
                                             float *logprobs, void *ws, size_t ws_bytes,
                                             lily_q4_stream_t stream);
LILY_Q4_API size_t lily_q8_gemv_argmax_workspace_bytes(int32_t N, int32_t K);

/*
 * lily_q4_gemv_argmax_noalloc -- lily_q4_gemv_argmax for callers that cannot allocate.
 *
 * The paper has no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc at all (code running on a memory budget fixed at start-up, or a host
 * framework that owns every device allocation and passes this library only its input
 * and output pointers) and so have no workspace to give.  Arguments, results and errors
 * are those of lily_q4_gemv_argmax without ws/ws_bytes.
 *
 * The kernel's scratch (a 256-byte header with the counter, then the per-block (max,
 * argmax) pairs) lives in a 16,640-byte __device__ array inside the library, held by every
 * GPU that loads the library until the process exits.  It covers up to 2048 blocks; on GPUs
 * with more than 1024 SMs the call returns LILY_Q4_ERR_WORKSPACE_TOO_SMALL.  K must be a
 * power of two from 64 to 2048 (else LILY_Q4_ERR_UNSUPPORTED).
 *  - The first call on a device looks up the array's device address on that device
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call on a device shares the one array and it keeps the last call's contents;
 *    each call clears the counters it needs on `stream` before its kernel.  Calls whose
 *    work overlaps on the GPU (different streams without ordering) race on the array:
 *    order them.
 *  - A bounded device-side wait of the kernel that gives up (the case that
 *    lily_q4_workspace_status reports for a workspace) is recorded in the array's error
 *    word.  Later calls leave that word set; lily_q4_gemv_argmax_noalloc_status reads and
 *    clears it.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
LILY_Q4_API int lily_q4_gemv_argmax_noalloc(const lily_q4_mat *W, int32_t N, int32_t K,
                                            const uint16_t *x, int32_t *token, float *logits,
                                            lily_q4_stream_t stream);

/* Synchronises `stream`, then reads and clears the error word of the fixed scratch of
 * lily_q4_gemv_argmax_noalloc on the current device: LILY_Q4_OK, or LILY_Q4_ERR_TIMEOUT if a
 * bounded wait in one of its calls gave up since the last check (LILY_Q4_ERR_CUDA if the
 * array's address cannot be looked up or the copy fails).  Allocates nothing. */
LILY_Q4_API int lily_q4_gemv_argmax_noalloc_status(lily_q4_stream_t stream);

/* Workspace sizes (bytes) for the calls above; 0 when the arguments are invalid. */
LILY_Q4_API size_t lily_q4_moe_workspace_bytes(const lily_q4_moe_layer *layer, int32_t T, int32_t prefill);
LILY_Q4_API size_t lily_q4_gemv_argmax_workspace_bytes(int32_t N, int32_t K);

/* Number of kernel launches one lily_q4_moe_decode (prefill = 0) or lily_q4_moe_prefill
 * (prefill = 1) call enqueues for this layer and T; 0 when the arguments are invalid.
 * Decode uses one launch when its single-launch kernel covers the shapes and batch (one
 * block per SM, enqueued as a programmatic dependent of the previous kernel on the
 * stream), three launches otherwise (four with an 8-bit shared expert).  Prefill uses 7
 * launches, plus 2 that prepare an 8-bit router and 3 that prepare an 8-bit shared expert. */
LILY_Q4_API int lily_q4_moe_launches(const lily_q4_moe_layer *layer, int32_t T, int32_t prefill);

/* Zero-fill a workspace on `stream` (asynchronous). */
LILY_Q4_API int lily_q4_workspace_init(void *ws, size_t ws_bytes, lily_q4_stream_t stream);

/* Synchronises `stream`, then reads and clears the workspace's device-side error
 * word: LILY_Q4_OK, or LILY_Q4_ERR_TIMEOUT if a bounded wait gave up since the
 * last check. */
LILY_Q4_API int lily_q4_workspace_status(void *ws, lily_q4_stream_t stream);

/*
 * lily_q4_selftest_timeout -- diagnostic of the bounded device-side waits.  Enqueues on
 * `stream` one single-block kernel that waits on something nothing provides -- which = 0: a
 * grid barrier on the workspace's arrival counter whose target no arrival reaches; which = 1:
 * an mbarrier phase that nothing completes -- until the wait's bound (about 1 s and 2 s of
 * SM clock), then records the time-out in the workspace header and exits, as a stalled launch
 * of this library would.  lily_q4_workspace_status then returns LILY_Q4_ERR_TIMEOUT.
 * Afterwards the workspace's barrier count is off: re-initialise it (lily_q4_workspace_init)
 * before the next decode.  ws: any workspace of at least 256 bytes; ws = NULL with
 * ws_bytes = 0 targets the fixed scratch of lily_q4_gemv_argmax_noalloc instead (its status
 * is then read by lily_q4_gemv_argmax_noalloc_status; its next call resets the counters).
 */
LILY_Q4_API int lily_q4_selftest_timeout(void *ws, size_t ws_bytes, int32_t which,
                                         lily_q4_stream_t stream);

/* Human-readable name of a status code (static string). */
LILY_Q4_API const char *lily_q4_status_string(int status);

/* Host-only format helpers.  q: uint8 [N][K] codes 0..15 (higher bits ignored);
 * w: uint32 [N][K/8].  K must be a positive multiple of 8. */
LILY_Q4_API int lily_q4_pack(const uint8_t *q, int32_t N, int32_t K, uint32_t *w);
LILY_Q4_API int lily_q4_unpack(const uint32_t *w, int32_t N, int32_t K, uint8_t *q);

/* Library version (major*10000 + minor*100 + patch). */
LILY_Q4_API int lily_q4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LILY_Q4_H */
