// Q4 LM-head GEMV fused with greedy argmax.
//
// Greedy token selection without logprobs, with the generated id kept on the
// device (Lily README, first paragraph; Lily-vs-MLX report, "Measurement
// contract").  One pass over the weights: each warp dequantises rows in
// registers (lane = one 64-wide group of the row), reduces the row with
// shuffles, keeps a running (max, argmax); blocks publish their best pair to
// the workspace and the last block to finish reduces those pairs into the token.
// The pass is bound by HBM bandwidth: 0.5625 bytes per weight.
#include <cfloat>
#include <climits>
#include <mutex>

#include "internal.h"
#include "q4_device.cuh"

namespace lq4 {

constexpr int kLmThreads = 256;
constexpr int kLmWarps = kLmThreads / 32;
constexpr int kLmBlocksPerSm = 2;

LmWsLayout lm_ws_layout(int N, int K) {
  (void)K;
  LmWsLayout l{};
  int sms = sm_count();
  if (sms <= 0) sms = 152;
  // at most one block per 32 rows, at most kLmBlocksPerSm per SM
  int want = (N + 31) / 32;
  l.grid = want < sms * kLmBlocksPerSm ? want : sms * kLmBlocksPerSm;
  if (l.grid < 1) l.grid = 1;
  size_t off = kHdrWords * sizeof(int32_t);
  off = align_up(off);
  l.off_partial_v = off;
  off = align_up(off + sizeof(float) * (size_t)sms * kLmBlocksPerSm);
  l.off_partial_i = off;
  off = align_up(off + sizeof(int32_t) * (size_t)sms * kLmBlocksPerSm);
  l.total = off;
  return l;
}

// G = groups per row (K/64), U = row-steps per iteration: a warp issues the loads of U
// row-steps (U*32 bytes of codes per lane) before computing them.
template <int G, int U>
__global__ void __launch_bounds__(kLmThreads, kLmBlocksPerSm)
    gemv_argmax_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                       const uint16_t *__restrict__ b, int N, const uint16_t *__restrict__ x,
                       float *__restrict__ logits, int32_t *__restrict__ token,
                       int32_t *__restrict__ hdr, float *__restrict__ part_v,
                       int32_t *__restrict__ part_i) {
  constexpr int RPS = 32 / G;  // rows per warp-step
  constexpr int K8 = G * 8;    // words per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;

  XGroupB xg;
  {
    uint4 c[8];
    const uint4 *xp = reinterpret_cast<const uint4 *>(x + kGroup * g);
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
    xgroupb_from_bf16(xg, c);
  }

  float best_v = -INFINITY;
  int best_i = INT_MAX;
  const int gwarp = blockIdx.x * kLmWarps + warp;
  const int nwarps = gridDim.x * kLmWarps;
  constexpr int RPI = RPS * U;  // rows per warp-iteration

#pragma unroll 1
  for (int r0 = gwarp * RPI; r0 < N; r0 += nwarps * RPI) {
    uint4 wa[U], wb[U];
    float sv[U], bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = r0 + u * RPS + rsub;
      if (row < N) {
        const uint32_t *wr = w + (size_t)row * K8 + 8 * g;
        wa[u] = ld_stream(wr);
        wb[u] = ld_stream(wr + 4);
        sv[u] = bf16f(ld_u16(s + (size_t)row * G + g));
        bv[u] = bf16f(ld_u16(b + (size_t)row * G + g));
      } else {
        wa[u] = wb[u] = make_uint4(0, 0, 0, 0);
        sv[u] = bv[u] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float d = seg_sum<G>(q4_group_dot_b(wa[u], wb[u], xg, sv[u], bv[u]));
      const float dc = cand(d);
      const int row = r0 + u * RPS + rsub;
      if (g == 0 && row < N) {
        if (logits) logits[row] = d;
        if (better(dc, row, best_v, best_i)) {
          best_v = dc;
          best_i = row;
        }
      }
    }
  }
  // warp argmax
  warp_argmax(best_v, best_i);
  __shared__ float sv_[kLmWarps];
  __shared__ int si_[kLmWarps];
  __shared__ int is_last;
  if (lane == 0) {
    sv_[warp] = best_v;
    si_[warp] = best_i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv_ = sv_[0];
    int bi_ = si_[0];
    for (int i = 1; i < kLmWarps; ++i)
      if (better(sv_[i], si_[i], bv_, bi_)) {
        bv_ = sv_[i];
        bi_ = si_[i];
      }
    part_v[blockIdx.x] = bv_;
    part_i[blockIdx.x] = bi_;
    __threadfence();
    const int ticket = atomicAdd(hdr + kHdrCounterA, 1);
    is_last = (ticket == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // last block: reduce the per-block pairs
  float v = -INFINITY;
  int i = INT_MAX;
  for (int j = threadIdx.x; j < (int)gridDim.x; j += kLmThreads) {
    const float pv = __ldcg(part_v + j);
    const int pi = __ldcg(part_i + j);
    if (better(pv, pi, v, i)) {
      v = pv;
      i = pi;
    }
  }
  warp_argmax(v, i);
  if (lane == 0) {
    sv_[warp] = v;
    si_[warp] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv_ = sv_[0];
    int bi_ = si_[0];
    for (int j = 1; j < kLmWarps; ++j)
      if (better(sv_[j], si_[j], bv_, bi_)) {
        bv_ = sv_[j];
        bi_ = si_[j];
      }
    *token = bi_;
    hdr[kHdrCounterA] = 0;  // leave the counter ready for the next call
  }
}

template <int G>
static void launch_g(const lily_q4_mat &W, int N, const uint16_t *x, int32_t *token,
                     float *logits, void *ws, const LmWsLayout &l, cudaStream_t st) {
  char *base = static_cast<char *>(ws);
  gemv_argmax_kernel<G, (G >= 16 ? 8 : 4)><<<l.grid, kLmThreads, 0, st>>>(
      W.w, W.s, W.b, N, x, logits, token, reinterpret_cast<int32_t *>(base),
      reinterpret_cast<float *>(base + l.off_partial_v),
      reinterpret_cast<int32_t *>(base + l.off_partial_i));
}

int launch_gemv_argmax(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                       float *logits, void *ws, cudaStream_t st) {
  const LmWsLayout l = lm_ws_layout(N, K);
  switch (K / kGroup) {
    case 1: launch_g<1>(W, N, x, token, logits, ws, l, st); break;
    case 2: launch_g<2>(W, N, x, token, logits, ws, l, st); break;
    case 4: launch_g<4>(W, N, x, token, logits, ws, l, st); break;
    case 8: launch_g<8>(W, N, x, token, logits, ws, l, st); break;
    case 16: launch_g<16>(W, N, x, token, logits, ws, l, st); break;
    case 32: launch_g<32>(W, N, x, token, logits, ws, l, st); break;
    default: return LILY_Q4_ERR_UNSUPPORTED;
  }
  return check_launch();
}

// ---------------------------------------------------------------------------------------
// lily_q4_gemv_argmax_noalloc: the same kernel with its scratch in a fixed device array.
//
// Some callers cannot call cudaMalloc at all: code that runs on a memory budget fixed when
// it started, or a host framework that owns every device allocation and hands this
// library only its input and output pointers.  They have no workspace to pass, so this
// entry point keeps the kernel's scratch (the last-block counter and the per-block
// (max, argmax) pairs) in a file-scope __device__ array that every GPU loading the library
// holds until the process exits.
// ---------------------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = 16640;  // 256-byte header + 2048 (float, int) pairs
static __device__ __align__(256) unsigned char g_gemv_argmax_scratch[kNoAllocScratchBytes];

// Device address of g_gemv_argmax_scratch on the current device, looked up once per device.
// (In host code the array's name is only a host-side stand-in, never a device address.)
static int noalloc_scratch(void **out) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LILY_Q4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemv_argmax_scratch) != cudaSuccess || !p)
      return LILY_Q4_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return LILY_Q4_OK;
}

}  // namespace lq4

extern "C" int lily_q4_gemv_argmax_noalloc(const lily_q4_mat *W, int32_t N, int32_t K,
                                           const uint16_t *x, int32_t *token, float *logits,
                                           lily_q4_stream_t stream) {
  using namespace lq4;
  auto al = [](const void *p, size_t a) { return ((uintptr_t)p % a) == 0; };
  if (!W || !W->w || !W->s || !W->b || !al(W->w, 16) || !al(W->s, 16) || !al(W->b, 16))
    return LILY_Q4_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % LILY_Q4_GROUP) return LILY_Q4_ERR_INVALID_ARG;
  if (!x || !al(x, 16) || !token || !al(token, 4) || (logits && !al(logits, 4)))
    return LILY_Q4_ERR_INVALID_ARG;
  if (K > 2048 || (K & (K - 1))) return LILY_Q4_ERR_UNSUPPORTED;
  if (lm_ws_layout(N, K).total > kNoAllocScratchBytes) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != LILY_Q4_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // start from a zero counter even if an earlier call was cut short
  if (cudaMemsetAsync(scratch, 0, kHdrWords * sizeof(int32_t), st) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  return launch_gemv_argmax(*W, N, K, x, token, logits, scratch, st);
}

