// Q4 (and 8-bit) LM-head GEMV fused with greedy argmax, and optionally with the
// full-vocabulary log-sum-exp and log-probabilities.
//
// Greedy token selection with the generated id kept on the device (Lily README, first
// paragraph; Lily-vs-MLX report, "Measurement contract", where the MLX path also computes
// log-probabilities over the whole vocabulary).  One pass over the weights: each warp
// dequantises rows in registers (lane = one 64-wide group of the row), reduces the row with
// shuffles, keeps a running (max, argmax); blocks publish their best pair to the workspace
// and the last block to finish reduces those pairs into the token.  The pass streams
// 0.5625 bytes per 4-bit weight (1.0625 per 8-bit weight).
#include <cfloat>
#include <climits>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "q4_device.cuh"
#include "tc_sm100.cuh"

namespace lq4 {

constexpr int kLmThreads = 256;
constexpr int kLmWarps = kLmThreads / 32;
constexpr int kLmBlocksPerSm = 2;

// streaming kernel (rows of >= 8 groups)
constexpr int kLsWarps = 24;                     // compute warps
constexpr int kLsThreads = (kLsWarps + 1) * 32;  // + the copy warp
constexpr int kLsStages = 4;
constexpr int kLsStageCodes = 49152;             // code bytes per stage
// stage waits suspend the waiting thread (time hint) instead of spinning
constexpr uint32_t kLsSleepNs = 1000;
// code bytes of a 64-group: 32 for 4-bit codes, 64 for 8-bit codes
__host__ __device__ constexpr int ls_rows_per_stage(int G, int bits = 4) {
  return kLsStageCodes / (8 * bits * G);
}

LmWsLayout lm_ws_layout(int N, int K, int bits) {
  LmWsLayout l{};
  int sms = sm_count();
  if (sms <= 0) sms = 152;
  if (K / kGroup >= 8) {
    // streaming kernel: one block per SM, at most one block per stage of rows, each block a
    // contiguous range of rows
    const int sr = ls_rows_per_stage(K / kGroup, bits);
    const int want = (N + sr - 1) / sr;
    l.grid = want < sms ? want : sms;
    if (l.grid < 1) l.grid = 1;
    l.rows_per_block = (N + l.grid - 1) / l.grid;
  } else {
    // at most one block per 32 rows, at most kLmBlocksPerSm per SM
    int want = (N + 31) / 32;
    l.grid = want < sms * kLmBlocksPerSm ? want : sms * kLmBlocksPerSm;
    if (l.grid < 1) l.grid = 1;
    l.rows_per_block = 0;
  }
  size_t off = kHdrWords * sizeof(int32_t);
  off = align_up(off);
  l.off_partial_v = off;
  off = align_up(off + sizeof(float) * (size_t)sms * kLmBlocksPerSm);
  l.off_partial_i = off;
  off = align_up(off + sizeof(int32_t) * (size_t)sms * kLmBlocksPerSm);
  l.total_argmax = off;
  l.off_partial_m = off;
  off = align_up(off + sizeof(float) * (size_t)sms * kLmBlocksPerSm);
  l.off_partial_s = off;
  off = align_up(off + sizeof(float) * (size_t)sms * kLmBlocksPerSm);
  l.off_logits = off;
  off = align_up(off + sizeof(float) * (size_t)N);
  l.total = off;
  return l;
}

// Running log-sum-exp as (m, s) = (max, sum of exp(v - m)): fold in one value, or merge two
// partials.  m = -inf means nothing folded in yet (s = 0); a NaN value makes s NaN.
// (Equal maxima are added without exp, so that +inf values count rather than give NaN.)
__device__ __forceinline__ void lse_add(float &m, float &s, float v) {
  if (v > m) {
    s = s * expf(m - v) + 1.0f;  // exp(-inf) = 0 on the first value
    m = v;
  } else if (v == m) {
    s += 1.0f;
  } else {
    s += expf(v - m);
  }
}
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else if (m2 == m) {
    s += s2;
  } else {
    s += s2 * expf(m2 - m);  // m2 = -inf: an empty partial adds 0 (or its NaN)
  }
}
// Merge the 32 lanes' partials, every lane getting the result: the warp maximum M first
// (one reduction on the order-preserving key), then each lane's sum rescaled to M with one
// exp, then a fixed-order butterfly sum -- no chain of dependent exps.
__device__ __forceinline__ void lse_warp(float &m, float &s) {
  const float M = key2f(__reduce_max_sync(0xffffffffu, f2key(m)));
  float t = (m == M) ? s : s * expf(m - M);  // equal maxima (also +-inf) need no rescale
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  m = M;
  s = t;
}

// Rows' logits reach the log-sum-exp a warp at a time: lane j of the warp buffers the j-th
// row since the last flush, and every 32 rows all lanes fold their row in at once (one exp
// per lane instead of one per row on a single lane).  n is the warp-uniform buffer count.
__device__ __forceinline__ void lse_buffer(float &m, float &s, float &buf, int &n, float v) {
  if ((int)(threadIdx.x & 31) == n) buf = v;
  if (++n == 32) {
    lse_add(m, s, buf);
    n = 0;
  }
}
__device__ __forceinline__ void lse_flush(float &m, float &s, float buf, int n) {
  if ((int)(threadIdx.x & 31) < n) lse_add(m, s, buf);
}

// logprob[n] = logit[n] - lse, in place.
__global__ void sub_lse_kernel(float *__restrict__ v, int N, const float *__restrict__ lse) {
  const float l = *lse;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
    v[i] -= l;
}

// Block-wide then grid-wide argmax of the threads' (value, row) pairs.  Argmax only: every
// block folds its best pair into one 64-bit maximum in the header (the order-preserving key
// of the value above the complement of the row, so a larger value wins and equal values go to
// the lower row), and the last block to finish (ticket on header counter A) reads it into
// *token and re-arms maximum and counter for the next call.  With the log-sum-exp, every
// block publishes its best pair and partials and the last block reduces them.
// With LSE, the threads' (m, s) log-sum-exp partials are reduced alongside, in a fixed order
// (deterministic), into *lse = m + log(s).
struct LseOut {
  float *part_m, *part_s, *lse;
};

template <int NW, bool LSE = false>
__device__ __forceinline__ void block_argmax_finish(float best_v, int best_i, int32_t *token,
                                                    int32_t *hdr, float *part_v, int32_t *part_i,
                                                    float lm = -INFINITY, float ls = 0.f,
                                                    LseOut lo = LseOut{}) {
  static_assert(NW <= 32, "one warp merges the warps' partials");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_argmax(best_v, best_i);
  __shared__ float sv_[NW];
  __shared__ int si_[NW];
  if constexpr (!LSE) {
    if (lane == 0) {
      sv_[warp] = best_v;
      si_[warp] = best_i;
    }
    __syncthreads();
    if (warp == 0) {
      float v = lane < NW ? sv_[lane] : -INFINITY;
      int i = lane < NW ? si_[lane] : INT_MAX;
      warp_argmax(v, i);
      if (lane == 0) {
        // The block's (value, row) folds into the packed maximum with a fire-and-forget
        // reduction; the ticket is an acquire-release add, so the reduction is ordered before
        // it and the last block, acquiring, sees every block's.  No round trip but the ticket.
        unsigned long long *mx = reinterpret_cast<unsigned long long *>(hdr + kHdrArgmax64);
        const unsigned long long key =
            ((unsigned long long)f2key(v) << 32) | (0xFFFFFFFFu - (uint32_t)i);
        asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(mx), "l"(key) : "memory");
        int ticket;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(ticket)
                     : "l"(hdr + kHdrCounterA)
                     : "memory");
        if (ticket == (int)gridDim.x - 1) {
          unsigned long long k;  // read, and re-arm
          asm volatile("atom.acquire.gpu.global.exch.b64 %0, [%1], 0;" : "=l"(k) : "l"(mx) : "memory");
          *token = (int32_t)(0xFFFFFFFFu - (uint32_t)k);
          hdr[kHdrCounterA] = 0;
        }
      }
    }
    return;
  }
  __shared__ float sm_[LSE ? NW : 1], ss_[LSE ? NW : 1];
  __shared__ int is_last;
  if (LSE) lse_warp(lm, ls);
  if (lane == 0) {
    sv_[warp] = best_v;
    si_[warp] = best_i;
    if (LSE) {
      sm_[warp] = lm;
      ss_[warp] = ls;
    }
  }
  __syncthreads();
  if (LSE && warp == 0) {
    float m_ = lane < NW ? sm_[lane] : -INFINITY, s_ = lane < NW ? ss_[lane] : 0.f;
    lse_warp(m_, s_);
    if (lane == 0) {
      lo.part_m[blockIdx.x] = m_;
      lo.part_s[blockIdx.x] = s_;
    }
  }
  if (threadIdx.x == 0) {
    float bv_ = sv_[0];
    int bi_ = si_[0];
    for (int i = 1; i < NW; ++i)
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
  float v = -INFINITY;
  int i = INT_MAX;
  float m = -INFINITY, sm = 0.f;
  for (int j = threadIdx.x; j < (int)gridDim.x; j += NW * 32) {
    const float pv = __ldcg(part_v + j);
    const int pi = __ldcg(part_i + j);
    if (better(pv, pi, v, i)) {
      v = pv;
      i = pi;
    }
    if (LSE) lse_merge(m, sm, __ldcg(lo.part_m + j), __ldcg(lo.part_s + j));
  }
  warp_argmax(v, i);
  if (LSE) lse_warp(m, sm);
  __syncthreads();
  if (lane == 0) {
    sv_[warp] = v;
    si_[warp] = i;
    if (LSE) {
      sm_[warp] = m;
      ss_[warp] = sm;
    }
  }
  __syncthreads();
  if (LSE && warp == 0) {
    float m_ = lane < NW ? sm_[lane] : -INFINITY, s_ = lane < NW ? ss_[lane] : 0.f;
    lse_warp(m_, s_);
    if (lane == 0) *lo.lse = m_ + logf(s_);
  }
  if (threadIdx.x == 0) {
    float bv_ = sv_[0];
    int bi_ = si_[0];
    for (int j = 1; j < NW; ++j)
      if (better(sv_[j], si_[j], bv_, bi_)) {
        bv_ = sv_[j];
        bi_ = si_[j];
      }
    *token = bi_;
    hdr[kHdrCounterA] = 0;  // leave the counter ready for the next call
  }
}

// G = groups per row (K/64), U = row-steps per iteration: a warp issues the loads of U
// row-steps (U*32 bytes of codes per lane) before computing them.
template <int G, int U, bool LSE>
__global__ void __launch_bounds__(kLmThreads, kLmBlocksPerSm)
    gemv_argmax_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                       const uint16_t *__restrict__ b, int N, const uint16_t *__restrict__ x,
                       float *__restrict__ logits, int32_t *__restrict__ token,
                       int32_t *__restrict__ hdr, float *__restrict__ part_v,
                       int32_t *__restrict__ part_i, LseOut lo) {
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
  float lm = -INFINITY, ls = 0.f, lbuf = 0.f;  // log-sum-exp partial of this lane's rows
  int lnb = 0;
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
      if (LSE) {
#pragma unroll
        for (int r = 0; r < RPS; ++r)
          if (r0 + u * RPS + r < N)
            lse_buffer(lm, ls, lbuf, lnb, RPS == 1 ? d : __shfl_sync(0xffffffffu, d, r * G));
      }
    }
  }
  if (LSE) lse_flush(lm, ls, lbuf, lnb);
  block_argmax_finish<kLmWarps, LSE>(best_v, best_i, token, hdr, part_v, part_i, lm, ls, lo);
}

// ---------------------------------------------------------------------------------------
// Timeline of the streaming kernel's last launch, for profiling builds only (-DLILY_Q4_TRACE):
// %globaltimer stamps by thread 0 of each block ([block][point]: 0 block set up, 1 x prepared,
// 2 first stage landed, 3 last stage computed, 4 the block's argmax folded in, 5 block done)
// and by the copy thread (6 last copy issued).
#ifdef LILY_Q4_TRACE
__device__ unsigned long long g_lm_trace[1024][8];
#define LM_TRACE(i, cond)                                                  \
  do {                                                                     \
    if ((cond) && blockIdx.x < 1024) {                                     \
      unsigned long long t_;                                               \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));               \
      g_lm_trace[blockIdx.x][(i)] = t_;                                    \
    }                                                                      \
  } while (0)
extern "C" __attribute__((visibility("default"))) int lily_q4_lm_trace_read(void *host, size_t bytes) {
  if (bytes > sizeof(g_lm_trace)) bytes = sizeof(g_lm_trace);
  return cudaMemcpyFromSymbol(host, g_lm_trace, bytes) == cudaSuccess ? 0 : -1;
}
#else
#define LM_TRACE(i, cond) \
  do {                    \
  } while (0)
#endif

// Streaming variant for rows of at least 8 groups (K >= 512), the LM-head shapes.
//
// Each block owns a contiguous range of rows -- one contiguous range of codes, of scales and
// of biases -- and streams it through a ring of shared-memory stages with untiled bulk
// copies (one copy thread; completion counted in bytes on the stage's mbarrier), so the
// loads of later stages are in flight while 24 warps dequantise and reduce the current one.
// A warp copies its rows of a stage into registers and hands the stage back at once.
// ---------------------------------------------------------------------------------------
template <int G, int BITS = 4>
struct LsCfg {
  static constexpr int CB = 8 * BITS;                     // code bytes of a 64-group
  static constexpr int RPS = 32 / G;                      // rows per warp-step
  static constexpr int SR = kLsStageCodes / (CB * G);     // rows per stage (CB*G code bytes a row)
  static constexpr int WR = SR / (kLsWarps * RPS);        // warp-steps per warp per stage
  static constexpr int SC = SR * 2 * G;                   // bytes of scales (and of biases)
  static constexpr int STAGE = kLsStageCodes + 2 * SC;
  static constexpr int OFF_BAR = kLsStages * STAGE;
  static constexpr int BYTES = OFF_BAR + 2 * kLsStages * 8;
  static_assert(G >= 8 && WR * kLsWarps * RPS == SR && STAGE % 128 == 0, "stage shape");
};

template <int G, bool LSE, int BITS = 4>
__global__ void __launch_bounds__(kLsThreads, 1)
    gemv_argmax_stream_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                              const uint16_t *__restrict__ b, int N, int rows_per_block,
                              const uint16_t *__restrict__ x, float *__restrict__ logits,
                              int32_t *__restrict__ token, int32_t *__restrict__ hdr,
                              float *__restrict__ part_v, int32_t *__restrict__ part_i,
                              LseOut lo) {
  using C = LsCfg<G, BITS>;
  extern __shared__ __align__(128) uint8_t ls_smem[];
  __shared__ volatile int s_abort;
  const uint32_t sbase = tc::smem_u32(ls_smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (kLsStages + i); };
  // Launched as a programmatic dependent of the previous kernel on the stream: let the next
  // kernel be scheduled early too.  The copy thread streams the weights (which no kernel
  // writes) at once; every other thread waits for the previous kernel before it reads x, the
  // workspace or the outputs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t *err = hdr + kHdrError;
  const int r_begin = min(N, (int)blockIdx.x * rows_per_block);
  const int r_end = min(N, r_begin + rows_per_block);
  const int nst = (r_end - r_begin + C::SR - 1) / C::SR;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kLsStages; ++i) {
      tc::mbar_init(full(i), 1);
      tc::mbar_init(empty(i), kLsWarps);
    }
    tc::mbar_init_fence();
  }
  __syncthreads();
  LM_TRACE(0, threadIdx.x == 0);

  float best_v = -INFINITY;
  int best_i = INT_MAX;
  float lm = -INFINITY, ls = 0.f;  // log-sum-exp partial of this thread's share of the rows
  if (warp == kLsWarps) {
    // ---------------------------------------------------------------- copy thread
    if (lane == 0) {
      int st = 0;
      for (; st < nst; ++st) {
        const int slot = st % kLsStages;
        if (!tc::wait_bar(empty(slot), ((st / kLsStages) & 1) ^ 1, &s_abort, err, kLsSleepNs)) break;
        const int r0 = r_begin + st * C::SR;
        const int rows = min(C::SR, r_end - r0);
        const uint32_t cb = (uint32_t)rows * (uint32_t)C::CB * G, sb = (uint32_t)rows * 2u * G;
        const uint32_t dst = sbase + (uint32_t)(slot * C::STAGE);
        tc::mbar_arrive_expect_tx(full(slot), cb + 2u * sb);
        tc::bulk_g2s(dst, w + (size_t)r0 * (C::CB / 4) * G, cb, full(slot));
        tc::bulk_g2s(dst + kLsStageCodes, s + (size_t)r0 * G, sb, full(slot));
        tc::bulk_g2s(dst + kLsStageCodes + C::SC, b + (size_t)r0 * G, sb, full(slot));
      }
      LM_TRACE(6, true);
      if (s_abort) {
        // after a time-out: let the copies still in flight land before the block exits
        for (int j = st > kLsStages ? st - kLsStages : 0; j < st; ++j) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(full(j % kLsStages), (j / kLsStages) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps
    const int g = lane % G, rsub = lane / G;
    // x is the previous kernel's output: wait for it (the copy thread streams weights, which
    // do not depend on it, from the start)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // x pairs in the order the codes unpack in (4-bit: (x_j, x_j+4); 8-bit: (x_j, x_j+2))
    std::conditional_t<BITS == 8, XGroup8, XGroupB> xg;
    {
      uint4 c[8];
      const uint4 *xp = reinterpret_cast<const uint4 *>(x + kGroup * g);
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
      if constexpr (BITS == 8)
        xgroup8_from_bf16(xg, c);
      else
        xgroupb_from_bf16(xg, c);
    }
    LM_TRACE(1, threadIdx.x == 0);
    constexpr int NV = C::CB / 16;          // 16-byte code vectors of a lane's group
    constexpr int ROW_B = C::CB * G;        // code bytes of a row
    // The warp's rows of a stage are lr = row0 + u * RPS (u < WR); the lane's code and scale
    // offsets inside a stage are fixed, so the per-row addressing is a constant per u.
    const int row0 = warp * C::WR * C::RPS + rsub;
    const int code_off = row0 * ROW_B + C::CB * g;
    const int sc_off = row0 * G + g;
    // Two rows of 32 groups per warp-step pair (the LM-head shape): their sums are reduced
    // together -- lanes 0-15 finish the first row, 16-31 the second -- and lanes 0 and 16
    // each keep their row's argmax candidate.
    constexpr bool PAIR = (G == 32 && C::WR == 2);
#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
      const int slot = st % kLsStages;
      if (!__all_sync(0xffffffffu,
                      tc::wait_bar(full(slot), (st / kLsStages) & 1, &s_abort, err, kLsSleepNs)))
        break;
      LM_TRACE(2, threadIdx.x == 0 && st == 0);
      const int r0 = r_begin + st * C::SR;
      const int rows = min(C::SR, r_end - r0);
      const bool full_stage = rows == C::SR;
      const uint8_t *cs = ls_smem + slot * C::STAGE;
      const uint16_t *ss = reinterpret_cast<const uint16_t *>(cs + kLsStageCodes);
      const uint16_t *bs = reinterpret_cast<const uint16_t *>(cs + kLsStageCodes + C::SC);
      uint4 wc[C::WR][NV];
      float sv[C::WR], bv[C::WR];
#pragma unroll
      for (int u = 0; u < C::WR; ++u) {
        if (full_stage || row0 + u * C::RPS < rows) {
          const uint4 *p = reinterpret_cast<const uint4 *>(cs + code_off + u * C::RPS * ROW_B);
#pragma unroll
          for (int v = 0; v < NV; ++v) wc[u][v] = p[v];
          sv[u] = bf16f(ss[sc_off + u * C::RPS * G]);
          bv[u] = bf16f(bs[sc_off + u * C::RPS * G]);
        } else {
#pragma unroll
          for (int v = 0; v < NV; ++v) wc[u][v] = make_uint4(0, 0, 0, 0);
          sv[u] = bv[u] = 0.f;
        }
      }
      // the warp's rows are in registers: hand the stage back before computing
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(slot));
      float part[C::WR];
#pragma unroll
      for (int u = 0; u < C::WR; ++u) {
        if constexpr (BITS == 8)
          part[u] = q8_group_dot_b(wc[u], xg, sv[u], bv[u]);
        else
          part[u] = q4_group_dot_b(wc[u][0], wc[u][1], xg, sv[u], bv[u]);
      }
      if constexpr (PAIR) {
        const bool hi = lane >= 16;
        float keep = hi ? part[1] : part[0];
        keep += __shfl_xor_sync(0xffffffffu, hi ? part[0] : part[1], 16);
        keep = seg_sum<16>(keep);
        const int lr = row0 + (hi ? 1 : 0);
        const bool owner = (lane & 15) == 0 && (full_stage || lr < rows);
        const int row = r0 + lr;
        if (owner && logits) logits[row] = keep;
        const float dc = cand(keep);
        const bool take = owner && better(dc, row, best_v, best_i);
        best_v = take ? dc : best_v;
        best_i = take ? row : best_i;
      } else {
#pragma unroll
        for (int u = 0; u < C::WR; ++u) {
          const float d = seg_sum<G>(part[u]);
          const int lr = row0 + u * C::RPS;
          const bool owner = g == 0 && (full_stage || lr < rows);
          const int row = r0 + lr;
          if (owner && logits) logits[row] = d;
          const float dc = cand(d);
          const bool take = owner && better(dc, row, best_v, best_i);
          best_v = take ? dc : best_v;
          best_i = take ? row : best_i;
        }
      }
    }
    LM_TRACE(3, threadIdx.x == 0);
  }
  if (warp == kLsWarps) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (LSE) {
    // the block's rows have their logits in `logits` (global, just written): every thread
    // folds a strided share of them into its partial, off the streaming loop
    __syncthreads();
    if (!s_abort)
      for (int r = r_begin + (int)threadIdx.x; r < r_end; r += kLsThreads) lse_add(lm, ls, __ldcg(logits + r));
  }
  LM_TRACE(4, threadIdx.x == 0);
  block_argmax_finish<kLsWarps + 1, LSE>(best_v, best_i, token, hdr, part_v, part_i, lm, ls, lo);
  LM_TRACE(5, threadIdx.x == 0);
}

// The streaming kernel is launched as a programmatic dependent of the previous kernel on the
// stream (its weight copies start while that kernel drains; see the kernel).
template <int G, bool LSE, int BITS>
static void launch_stream(const LmWsLayout &l, cudaStream_t st, const uint32_t *w,
                          const uint16_t *s, const uint16_t *b, int N, const uint16_t *x,
                          float *logits, int32_t *token, int32_t *hdr, float *pv, int32_t *pi,
                          LseOut lo) {
  using C = LsCfg<G, BITS>;
  auto fn = gemv_argmax_stream_kernel<G, LSE, BITS>;
  // set on every call: cheap, and correct for whichever device is current
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.grid);
  cfg.blockDim = dim3(kLsThreads);
  cfg.dynamicSmemBytes = C::BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, fn, w, s, b, N, l.rows_per_block, x, logits, token, hdr, pv, pi, lo);
}

template <int G, bool LSE>
static void launch_g(const lily_q4_mat &W, int N, const uint16_t *x, int32_t *token,
                     float *logits, void *ws, const LmWsLayout &l, cudaStream_t st, float *lse) {
  char *base = static_cast<char *>(ws);
  int32_t *hdr = reinterpret_cast<int32_t *>(base);
  float *pv = reinterpret_cast<float *>(base + l.off_partial_v);
  int32_t *pi = reinterpret_cast<int32_t *>(base + l.off_partial_i);
  const LseOut lo = LSE ? LseOut{reinterpret_cast<float *>(base + l.off_partial_m),
                                 reinterpret_cast<float *>(base + l.off_partial_s), lse}
                        : LseOut{};
  if constexpr (G >= 8) {
    // the log-sum-exp pass reads the logits back: into the workspace when not requested
    if (LSE && !logits) logits = reinterpret_cast<float *>(base + l.off_logits);
    launch_stream<G, LSE, 4>(l, st, W.w, W.s, W.b, N, x, logits, token, hdr, pv, pi, lo);
  } else {
    gemv_argmax_kernel<G, (G >= 16 ? 8 : 4), LSE><<<l.grid, kLmThreads, 0, st>>>(
        W.w, W.s, W.b, N, x, logits, token, hdr, pv, pi, lo);
  }
}

template <bool LSE>
static int launch_k(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                    float *logits, void *ws, const LmWsLayout &l, cudaStream_t st, float *lse) {
  switch (K / kGroup) {
    case 1: launch_g<1, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 2: launch_g<2, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 4: launch_g<4, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 8: launch_g<8, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 16: launch_g<16, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 32: launch_g<32, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    default: return LILY_Q4_ERR_UNSUPPORTED;
  }
  return LILY_Q4_OK;
}

template <int G, bool LSE>
static void launch_q8_g(const lily_q4_mat &W, int N, const uint16_t *x, int32_t *token,
                        float *logits, void *ws, const LmWsLayout &l, cudaStream_t st, float *lse) {
  char *base = static_cast<char *>(ws);
  const LseOut lo = LSE ? LseOut{reinterpret_cast<float *>(base + l.off_partial_m),
                                 reinterpret_cast<float *>(base + l.off_partial_s), lse}
                        : LseOut{};
  if (LSE && !logits) logits = reinterpret_cast<float *>(base + l.off_logits);
  launch_stream<G, LSE, 8>(l, st, W.w, W.s, W.b, N, x, logits, token,
                           reinterpret_cast<int32_t *>(base),
                           reinterpret_cast<float *>(base + l.off_partial_v),
                           reinterpret_cast<int32_t *>(base + l.off_partial_i), lo);
}

template <bool LSE>
static int launch_q8_k(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                       float *logits, void *ws, const LmWsLayout &l, cudaStream_t st, float *lse) {
  switch (K / kGroup) {
    case 8: launch_q8_g<8, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 16: launch_q8_g<16, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    case 32: launch_q8_g<32, LSE>(W, N, x, token, logits, ws, l, st, lse); break;
    default: return LILY_Q4_ERR_UNSUPPORTED;
  }
  return LILY_Q4_OK;
}

int launch_q8_gemv_argmax(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                          float *logits, void *ws, cudaStream_t st, float *lse) {
  const LmWsLayout l = lm_ws_layout(N, K, 8);
  const int rc = lse ? launch_q8_k<true>(W, N, K, x, token, logits, ws, l, st, lse)
                     : launch_q8_k<false>(W, N, K, x, token, logits, ws, l, st, lse);
  if (rc != LILY_Q4_OK) return rc;
  if (lse && logits) {
    int sms = sm_count();
    if (sms <= 0) sms = 152;
    const int want = (N + 1023) / 1024;
    sub_lse_kernel<<<want < 4 * sms ? want : 4 * sms, 256, 0, st>>>(logits, N, lse);
  }
  return check_launch();
}

int launch_gemv_argmax(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                       float *logits, void *ws, cudaStream_t st, float *lse) {
  const LmWsLayout l = lm_ws_layout(N, K);
  const int rc = lse ? launch_k<true>(W, N, K, x, token, logits, ws, l, st, lse)
                     : launch_k<false>(W, N, K, x, token, logits, ws, l, st, lse);
  if (rc != LILY_Q4_OK) return rc;
  if (lse && logits) {
    int sms = sm_count();
    if (sms <= 0) sms = 152;
    const int want = (N + 1023) / 1024;
    sub_lse_kernel<<<want < 4 * sms ? want : 4 * sms, 256, 0, st>>>(logits, N, lse);
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
int noalloc_scratch(void **out) {
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
  if (lm_ws_layout(N, K).total_argmax > kNoAllocScratchBytes) return LILY_Q4_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != LILY_Q4_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // Start from zero counters even if an earlier call was cut short.  The error word (the
  // header's first) is left as it is: a bounded wait that gave up in an earlier call stays
  // recorded until lily_q4_gemv_argmax_noalloc_status reads it.
  if (cudaMemsetAsync(static_cast<int32_t *>(scratch) + kHdrCounterA, 0,
                      (kHdrWords - kHdrCounterA) * sizeof(int32_t), st) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  return launch_gemv_argmax(*W, N, K, x, token, logits, scratch, st);
}


extern "C" int lily_q4_gemv_argmax_noalloc_status(lily_q4_stream_t stream) {
  using namespace lq4;
  void *scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != LILY_Q4_OK) return rc;
  return lily_q4_workspace_status(scratch, stream);
}
