// C-ABI entry points of liblily_q4: argument validation, workspace sizing and the
// host-only format helpers.  Compute is enqueued by the launchers in the other
// translation units; nothing here allocates device memory.
#include <cstring>

#include "internal.h"

namespace lq4 {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LILY_Q4_OK : LILY_Q4_ERR_CUDA;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

static bool width_ok(int v) {
  return v == 64 || v == 128 || v == 256 || v == 512 || v == 1024 || v == 2048;
}

static bool mat_ok(const lily_q4_mat &m) {
  return m.w && m.s && m.b && aligned(m.w, 16) && aligned(m.s, 16) && aligned(m.b, 16);
}

// Returns LILY_Q4_OK, INVALID_ARG or UNSUPPORTED.
static int check_layer(const lily_q4_moe_layer *L) {
  if (!L) return LILY_Q4_ERR_INVALID_ARG;
  if (L->hidden <= 0 || L->inter <= 0 || L->n_experts <= 0 || L->top_k <= 0)
    return LILY_Q4_ERR_INVALID_ARG;
  if (L->hidden % LILY_Q4_GROUP || L->inter % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (L->top_k > L->n_experts) return LILY_Q4_ERR_INVALID_ARG;
  if (L->n_experts > 1024 || L->top_k > 16) return LILY_Q4_ERR_INVALID_ARG;
  if (L->has_shared != 0 && L->has_shared != 1) return LILY_Q4_ERR_INVALID_ARG;
  if (!mat_ok(L->gate) || !mat_ok(L->up) || !mat_ok(L->down)) return LILY_Q4_ERR_INVALID_ARG;
  if (L->shared_bits != 0 && L->shared_bits != 4 && L->shared_bits != 8) return LILY_Q4_ERR_INVALID_ARG;
  if (L->router_bits != 0 && L->router_bits != 16 && L->router_bits != 8) return LILY_Q4_ERR_INVALID_ARG;
  if (L->router_bits == 8) {
    if (!mat_ok(L->router_q8)) return LILY_Q4_ERR_INVALID_ARG;
  } else if (!L->router || !aligned(L->router, 16)) {
    return LILY_Q4_ERR_INVALID_ARG;
  }
  if (L->router_bias && !aligned(L->router_bias, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (L->has_shared) {
    if (!mat_ok(L->sh_gate) || !mat_ok(L->sh_up) || !mat_ok(L->sh_down))
      return LILY_Q4_ERR_INVALID_ARG;
    if (!L->shared_gate || !aligned(L->shared_gate, 16)) return LILY_Q4_ERR_INVALID_ARG;
  }
  if (!width_ok(L->hidden) || !width_ok(L->inter)) return LILY_Q4_ERR_UNSUPPORTED;
  return LILY_Q4_OK;
}

static int check_io(const uint16_t *x, uint16_t *y, int32_t *idx, float *w, void *ws) {
  if (!x || !y || !ws) return LILY_Q4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  if ((idx && !aligned(idx, 4)) || (w && !aligned(w, 4))) return LILY_Q4_ERR_INVALID_ARG;
  return LILY_Q4_OK;
}

}  // namespace lq4

using namespace lq4;

extern "C" {

int lily_q4_version(void) { return 100; }

const char *lily_q4_status_string(int status) {
  switch (status) {
    case LILY_Q4_OK: return "ok";
    case LILY_Q4_ERR_INVALID_ARG: return "invalid argument";
    case LILY_Q4_ERR_UNSUPPORTED: return "unsupported shape";
    case LILY_Q4_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case LILY_Q4_ERR_CUDA: return "CUDA error";
    case LILY_Q4_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int lily_q4_pack(const uint8_t *q, int32_t N, int32_t K, uint32_t *w) {
  if (!q || !w || N < 0 || K <= 0 || K % 8) return LILY_Q4_ERR_INVALID_ARG;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t m = 0; m < K / 8; ++m) {
      uint32_t word = 0;
      const uint8_t *src = q + n * K + 8 * m;
      for (int j = 7; j >= 0; --j) word = (word << 4) | (uint32_t)(src[j] & 0xF);
      w[n * (K / 8) + m] = word;
    }
  return LILY_Q4_OK;
}

int lily_q4_unpack(const uint32_t *w, int32_t N, int32_t K, uint8_t *q) {
  if (!q || !w || N < 0 || K <= 0 || K % 8) return LILY_Q4_ERR_INVALID_ARG;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t m = 0; m < K / 8; ++m) {
      uint32_t word = w[n * (K / 8) + m];
      for (int j = 0; j < 8; ++j, word >>= 4) q[n * K + 8 * m + j] = (uint8_t)(word & 0xF);
    }
  return LILY_Q4_OK;
}

size_t lily_q4_gemv_argmax_workspace_bytes(int32_t N, int32_t K) {
  if (N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return 0;
  return lm_ws_layout(N, K).total;
}

size_t lily_q8_gemv_argmax_workspace_bytes(int32_t N, int32_t K) {
  if (N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return 0;
  return lm_ws_layout(N, K, 8).total;
}

size_t lily_q4_moe_workspace_bytes(const lily_q4_moe_layer *layer, int32_t T, int32_t prefill) {
  if (check_layer(layer) != LILY_Q4_OK || T <= 0) return 0;
  if (prefill) {
    if (T > 8192) return 0;
    return prefill_ws_layout(*layer, T).total;
  }
  if (T > 16) return 0;
  return decode_ws_layout(*layer, T).total;
}

int lily_q4_moe_launches(const lily_q4_moe_layer *layer, int32_t T, int32_t prefill) {
  if (check_layer(layer) != LILY_Q4_OK || T <= 0) return 0;
  if (prefill)
    return T <= 8192 && layer->hidden >= 128 && layer->inter >= 128 ? prefill_launch_count(*layer) : 0;
  return T <= 16 ? decode_launch_count(*layer, T) : 0;
}

int lily_q4_workspace_init(void *ws, size_t ws_bytes, lily_q4_stream_t stream) {
  if (!ws || ws_bytes < kAlign || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? LILY_Q4_OK
                                                                              : LILY_Q4_ERR_CUDA;
}

int lily_q4_workspace_status(void *ws, lily_q4_stream_t stream) {
  if (!ws || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LILY_Q4_ERR_CUDA;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return LILY_Q4_ERR_CUDA;
    return LILY_Q4_ERR_TIMEOUT;
  }
  return LILY_Q4_OK;
}

int lily_q4_selftest_timeout(void *ws, size_t ws_bytes, int32_t which, lily_q4_stream_t stream) {
  if (which != 0 && which != 1) return LILY_Q4_ERR_INVALID_ARG;
  if (!ws && ws_bytes == 0) {  // the fixed scratch of lily_q4_gemv_argmax_noalloc
    const int rc = noalloc_scratch(&ws);
    if (rc != LILY_Q4_OK) return rc;
    ws_bytes = kAlign;
  }
  if (!ws || ws_bytes < kAlign || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  return selftest_wait(ws, which, (cudaStream_t)stream);
}

int lily_q4_gemv_argmax(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                        int32_t *token, float *logits, void *ws, size_t ws_bytes,
                        lily_q4_stream_t stream) {
  if (!W || !mat_ok(*W) || N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (!x || !aligned(x, 16) || !token || !aligned(token, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (logits && !aligned(logits, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  if (!width_ok(K)) return LILY_Q4_ERR_UNSUPPORTED;
  if (ws_bytes < lm_ws_layout(N, K).total) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_gemv_argmax(*W, N, K, x, token, logits, ws, (cudaStream_t)stream);
}

int lily_q4_gemv_argmax_logprobs(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                                 int32_t *token, float *lse, float *logprobs, void *ws,
                                 size_t ws_bytes, lily_q4_stream_t stream) {
  if (!W || !mat_ok(*W) || N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (!x || !aligned(x, 16) || !token || !aligned(token, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (!lse || !aligned(lse, 4) || (logprobs && !aligned(logprobs, 4))) return LILY_Q4_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  if (!width_ok(K)) return LILY_Q4_ERR_UNSUPPORTED;
  if (ws_bytes < lm_ws_layout(N, K).total) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_gemv_argmax(*W, N, K, x, token, logprobs, ws, (cudaStream_t)stream, lse);
}

int lily_q8_gemv_argmax(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                        int32_t *token, float *logits, void *ws, size_t ws_bytes,
                        lily_q4_stream_t stream) {
  if (!W || !mat_ok(*W) || N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (!x || !aligned(x, 16) || !token || !aligned(token, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (logits && !aligned(logits, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  if (K != 512 && K != 1024 && K != 2048) return LILY_Q4_ERR_UNSUPPORTED;
  if (ws_bytes < lm_ws_layout(N, K, 8).total_argmax) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_q8_gemv_argmax(*W, N, K, x, token, logits, ws, (cudaStream_t)stream);
}

int lily_q8_gemv_argmax_logprobs(const lily_q4_mat *W, int32_t N, int32_t K, const uint16_t *x,
                                 int32_t *token, float *lse, float *logprobs, void *ws,
                                 size_t ws_bytes, lily_q4_stream_t stream) {
  if (!W || !mat_ok(*W) || N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (!x || !aligned(x, 16) || !token || !aligned(token, 4)) return LILY_Q4_ERR_INVALID_ARG;
  if (!lse || !aligned(lse, 4) || (logprobs && !aligned(logprobs, 4))) return LILY_Q4_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return LILY_Q4_ERR_INVALID_ARG;
  if (K != 512 && K != 1024 && K != 2048) return LILY_Q4_ERR_UNSUPPORTED;
  if (ws_bytes < lm_ws_layout(N, K, 8).total) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_q8_gemv_argmax(*W, N, K, x, token, logprobs, ws, (cudaStream_t)stream, lse);
}

int lily_q4_moe_decode(const lily_q4_moe_layer *layer, const uint16_t *x, int32_t T,
                       uint16_t *y, int32_t *topk_idx, float *topk_w, void *ws,
                       size_t ws_bytes, lily_q4_stream_t stream) {
  int rc = check_layer(layer);
  if (rc != LILY_Q4_OK) return rc;
  if (T < 0 || T > 16) return LILY_Q4_ERR_INVALID_ARG;
  if (T == 0) return LILY_Q4_OK;
  rc = check_io(x, y, topk_idx, topk_w, ws);
  if (rc != LILY_Q4_OK) return rc;
  if (ws_bytes < decode_ws_layout(*layer, T).total) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_moe_decode(*layer, x, T, y, topk_idx, topk_w, ws, (cudaStream_t)stream);
}

int lily_q4_moe_prefill(const lily_q4_moe_layer *layer, const uint16_t *x, int32_t T,
                        uint16_t *y, int32_t *topk_idx, float *topk_w, void *ws,
                        size_t ws_bytes, lily_q4_stream_t stream) {
  int rc = check_layer(layer);
  if (rc != LILY_Q4_OK) return rc;
  if (T < 0 || T > 8192) return LILY_Q4_ERR_INVALID_ARG;
  if (T == 0) return LILY_Q4_OK;
  rc = check_io(x, y, topk_idx, topk_w, ws);
  if (rc != LILY_Q4_OK) return rc;
  if (ws_bytes < prefill_ws_layout(*layer, T).total) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  return launch_moe_prefill(*layer, x, T, y, topk_idx, topk_w, ws, (cudaStream_t)stream);
}

}  // extern "C"
