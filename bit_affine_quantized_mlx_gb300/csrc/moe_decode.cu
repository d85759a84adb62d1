// Decode-step MoE feed-forward (1..16 tokens).
//
// The MoE kernels of a decode step, which is bound by its reads (fork page, "How the
// speed was achieved": the decode step was tuned toward the bandwidth its chain of
// dependent reads can reach).  Up to four tokens, the layer is one launch
// (moe_decode_fused_kernel, below), which also takes layers with an 8-bit router and/or
// 8-bit shared expert.  The general path is three launches on the caller's stream:
//
//  1. router_topk_kernel: fp32 router logits (one warp per expert row, bf16 weights)
//     and the shared-expert gate sigmoid(x . g_shared); the last block to finish takes
//     the top-k per token (logit desc, index asc), the softmax over the k, and builds
//     the list of unique experts with their (token, weight) pairs so that an expert
//     chosen by several tokens is streamed once.
//  2. gateup_kernel: for each unique expert and a block of intermediate rows, the Q4
//     gate and up rows are dequantised in registers once and applied to every token of
//     the expert; h = silu(g) * u is written per pair (fp32).
//  3. down_kernel: each block owns a few output rows, runs the Q4 down rows of every
//     pair against its h, and sums the weighted results per token in a fixed order
//     (deterministic), writing y in bf16.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "q4_device.cuh"
#include "tc_sm100.cuh"

namespace lq4 {

constexpr int kMaxT = 16;
constexpr int kMaxK = 16;
constexpr int kMaxPairs = kMaxT * (kMaxK + 1);
constexpr int kRouterThreads = 128;
constexpr int kGateUpThreads = 256;
constexpr int kGateUpSteps = 2;      // row-steps per warp held in registers
constexpr int kDownThreads = 256;
constexpr int kDownRows = 8;         // output rows per down block

DecodeWsLayout decode_ws_layout(const lily_q4_moe_layer &L, int T) {
  DecodeWsLayout l{};
  l.T = T;
  l.E = L.n_experts;
  l.k = L.top_k;
  l.I = L.inter;
  l.H = L.hidden;
  l.P = T * L.top_k + (L.has_shared ? T : 0);
  l.Umax = T * L.top_k + (L.has_shared ? 1 : 0);
  size_t off = align_up(kHdrWords * sizeof(int32_t));
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  l.off_logits = take(sizeof(float) * (size_t)T * l.E);
  l.off_idx = take(sizeof(int32_t) * (size_t)T * l.k);
  l.off_p = take(sizeof(float) * (size_t)T * l.k);
  l.off_sigma = take(sizeof(float) * (size_t)T);
  l.off_meta = take(sizeof(int32_t) * (size_t)(1 + l.Umax + l.Umax + 1 + l.P));
  l.off_pair_tok = take(sizeof(int32_t) * (size_t)l.P);
  l.off_pair_w = take(sizeof(float) * (size_t)l.P);
  l.off_h = take(sizeof(float) * (size_t)l.P * l.I);
  l.total = off;
  return l;
}

struct DecodePtrs {
  int32_t *hdr;
  float *logits;
  int32_t *idx;
  float *p;
  float *sigma;
  int32_t *meta;      // [0] = U, then uexp[Umax], ubase[Umax+1], pair_e[P]
  int32_t *pair_tok;
  float *pair_w;
  float *h;
  int Umax;
  int P;  // pairs the workspace holds
  __host__ __device__ int32_t *uexp() const { return meta + 1; }
  __host__ __device__ int32_t *ubase() const { return meta + 1 + Umax; }
  __host__ __device__ int32_t *pair_e() const { return meta + 1 + Umax + Umax + 1; }
};

static DecodePtrs decode_ptrs(void *ws, const DecodeWsLayout &l) {
  char *b = static_cast<char *>(ws);
  DecodePtrs p;
  p.hdr = reinterpret_cast<int32_t *>(b);
  p.logits = reinterpret_cast<float *>(b + l.off_logits);
  p.idx = reinterpret_cast<int32_t *>(b + l.off_idx);
  p.p = reinterpret_cast<float *>(b + l.off_p);
  p.sigma = reinterpret_cast<float *>(b + l.off_sigma);
  p.meta = reinterpret_cast<int32_t *>(b + l.off_meta);
  p.pair_tok = reinterpret_cast<int32_t *>(b + l.off_pair_tok);
  p.pair_w = reinterpret_cast<float *>(b + l.off_pair_w);
  p.h = reinterpret_cast<float *>(b + l.off_h);
  p.Umax = l.Umax;
  p.P = l.P;
  return p;
}

struct RouterArgs {
  const uint16_t *router;
  const float *bias;
  const uint16_t *shared_gate;
  const uint16_t *x;
  int T, E, H, k, has_shared;
  int32_t *out_idx;
  float *out_w;
  lily_q4_mat router8;  // the 8-bit router when router_bits == 8
  int router_bits;
};

// Routing bookkeeping of T tokens by one block of NT threads: top-k per token (a warp per
// token, logit desc / index asc), softmax over the k, the unique experts (ascending id, the
// shared expert last, id E) and their (token, combine weight) pairs.  `logits` and `sigma`
// were written by other blocks (read through L2).  Outputs go through generic pointers.
struct RouteDst {
  int32_t *idx;
  float *p;
  int32_t *U;
  int32_t *uexp;
  int32_t *ubase;
  int32_t *pair_tok;
  float *pair_w;
  int32_t *pair_e;
  int32_t *out_idx;
  float *out_w;
};

template <int NT, int EC>
__device__ void route_block(const float *logits, const float *sigma, int T, int E, int k,
                            int has_shared, const RouteDst &d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ int s_idx[kMaxT * kMaxK];
  __shared__ float s_p[kMaxT * kMaxK];
  __shared__ int s_cnt[1024];
  __shared__ int s_base[1024];

  // top-k per token: warp per token; each lane holds its EC logits in registers, then k
  // rounds of a warp argmax over the unselected ones
  for (int t = warp; t < T; t += NT / 32) {
    const float *lg = logits + (size_t)t * E;
    float lv[EC];
#pragma unroll
    for (int j = 0; j < EC; ++j) lv[j] = (lane + 32 * j < E) ? cand(__ldcg(lg + lane + 32 * j)) : -INFINITY;
    uint32_t taken = 0;  // bit j: expert lane + 32 j already selected
    float sel_v[kMaxK];
    int sel_e[kMaxK];
    for (int i = 0; i < k; ++i) {
      float bv = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int j = 0; j < EC; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !(taken & (1u << j)) && better(lv[j], e, bv, be)) {
          bv = lv[j];
          be = e;
        }
      }
      warp_argmax(bv, be);
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_v[i] = bv;
      sel_e[i] = be;
    }
    if (lane == 0) {
      const float v0 = sel_v[0];
      float denom = 0.f;
      for (int i = 0; i < k; ++i) denom += expf(sel_v[i] - v0);
      for (int i = 0; i < k; ++i) {
        const float pi = expf(sel_v[i] - v0) / denom;
        s_idx[t * k + i] = sel_e[i];
        s_p[t * k + i] = pi;
        if (d.idx) d.idx[t * k + i] = sel_e[i];
        if (d.p) d.p[t * k + i] = pi;
        if (d.out_idx) d.out_idx[t * k + i] = sel_e[i];
        if (d.out_w) d.out_w[t * k + i] = pi;
      }
    }
  }
  for (int e = threadIdx.x; e < E; e += NT) s_cnt[e] = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < T * k; j += NT) atomicAdd(&s_cnt[s_idx[j]], 1);
  __syncthreads();
  if (warp == 0) {
    // rank (exclusive count of present experts) and base (exclusive sum of counts)
    const int per = (E + 31) / 32;
    const int lo = lane * per, hi = min(E, lo + per);
    int np = 0, nc = 0;
    for (int e = lo; e < hi; ++e) {
      np += s_cnt[e] > 0;
      nc += s_cnt[e];
    }
    int totp, totc;
    int rp = warp_excl_scan(np, &totp);
    int rc = warp_excl_scan(nc, &totc);
    for (int e = lo; e < hi; ++e) {
      s_base[e] = rc;
      if (s_cnt[e] > 0) {
        d.uexp[rp] = e;
        d.ubase[rp] = rc;
        ++rp;
      }
      rc += s_cnt[e];
    }
    if (lane == 0) {
      int U = totp;
      if (has_shared) {
        d.uexp[U] = E;  // the shared expert
        d.ubase[U] = totc;
        ++U;
      }
      d.ubase[U] = totc + (has_shared ? T : 0);
      *d.U = U;
    }
  }
  __syncthreads();
  // pairs: (token t, slot i) -> position base[e] + (number of earlier tokens that chose e)
  for (int j = threadIdx.x; j < T * k; j += NT) {
    const int t = j / k, e = s_idx[j];
    int pos = 0;
    for (int jj = 0; jj < t * k; ++jj) pos += (s_idx[jj] == e);
    const int pr = s_base[e] + pos;
    d.pair_tok[pr] = t;
    d.pair_w[pr] = s_p[j];
    d.pair_e[pr] = e;
  }
  if (has_shared) {
    for (int t = threadIdx.x; t < T; t += NT) {
      const int pr = T * k + t;
      d.pair_tok[pr] = t;
      d.pair_w[pr] = __ldcg(sigma + t);
      d.pair_e[pr] = E;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------------------
// 1. router logits + shared gate; last block: top-k, gates, unique-expert pairs
// ---------------------------------------------------------------------------------------
template <int EC>
__global__ void __launch_bounds__(kRouterThreads)
    router_topk_kernel(RouterArgs a, DecodePtrs w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nrows = a.E + a.has_shared;
  const int row = blockIdx.x * (kRouterThreads / 32) + warp;
  const int nchunk = a.H / 8;  // 16-byte chunks per row
  if (row < a.E && a.router_bits == 8) {
    // an 8-bit router row: lane g < H/64 holds group g (64 code bytes, its s and b)
    const int G = a.H / kGroup;
    uint4 w4[4] = {};
    float rs = 0.f, rb = 0.f;
    if (lane < G) {
      const size_t wo = (size_t)row * (G * 16) + 16 * lane, so = (size_t)row * G + lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) w4[j] = ld_stream(a.router8.w + wo + 4 * j);
      rs = bf16f(ld_u16(a.router8.s + so));
      rb = bf16f(ld_u16(a.router8.b + so));
    }
    for (int t = 0; t < a.T; ++t) {
      float d = 0.f;
      if (lane < G) {
        uint4 c[8];
        const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kGroup * lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
        XGroup8 x8;
        xgroup8_from_bf16(x8, c);
        d = q8_group_dot_b(w4, x8, rs, rb);
      }
      d = seg_sum<32>(d);
      if (lane == 0) w.logits[(size_t)t * a.E + row] = d + (a.bias ? a.bias[row] : 0.f);
    }
  } else if (row < nrows) {
    const uint16_t *wr = row < a.E ? a.router + (size_t)row * a.H : a.shared_gate;
    uint4 wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = lane + 32 * j;
      wv[j] = c < nchunk ? ld_stream(wr + 8 * c) : make_uint4(0, 0, 0, 0);
    }
    for (int t = 0; t < a.T; ++t) {
      const uint16_t *xt = a.x + (size_t)t * a.H;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = lane + 32 * j;
        if (c < nchunk) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(xt + 8 * c));
          const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
          const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc = fmaf(__uint_as_float(ww[i] << 16), __uint_as_float(xx[i] << 16), acc);
            acc = fmaf(__uint_as_float(ww[i] & 0xFFFF0000u), __uint_as_float(xx[i] & 0xFFFF0000u),
                       acc);
          }
        }
      }
      acc = seg_sum<32>(acc);
      if (lane == 0) {
        if (row < a.E) {
          w.logits[(size_t)t * a.E + row] = acc + (a.bias ? a.bias[row] : 0.f);
        } else {
          w.sigma[t] = 1.0f / (1.0f + expf(-acc));
        }
      }
    }
  }
  // ---- last block to finish does the routing bookkeeping
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(w.hdr + kHdrCounterB, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  RouteDst d{w.idx, w.p, w.meta, w.uexp(), w.ubase(), w.pair_tok, w.pair_w, w.pair_e(),
             a.out_idx, a.out_w};
  route_block<kRouterThreads, EC>(w.logits, w.sigma, a.T, a.E, a.k, a.has_shared, d);
  if (threadIdx.x == 0) w.hdr[kHdrCounterB] = 0;
}

// ---------------------------------------------------------------------------------------
// 2. gate/up dequant-GEMV + SwiGLU, per unique expert and row block
// ---------------------------------------------------------------------------------------
struct GateUpArgs {
  lily_q4_mat gate, up, sh_gate, sh_up;
  const uint16_t *x;
  int E, H, I;
  int shared_bits;  // 8: the shared unit is left to gateup_shared8_kernel
};

template <int G>  // groups per row = H / 64
__global__ void __launch_bounds__(kGateUpThreads)
    gateup_kernel(GateUpArgs a, DecodePtrs w) {
  constexpr int RPS = 32 / G;
  constexpr int K8 = G * 8;
  constexpr int ROWS = (kGateUpThreads / 32) * kGateUpSteps * RPS;
  const int u = blockIdx.y;
  const int U = w.meta[0];
  if (u >= U || U > w.Umax) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;
  const int e = w.uexp()[u];
  const int pb = max(w.ubase()[u], 0), pe = min(w.ubase()[u + 1], w.P);
  if (e < 0 || e > a.E) return;
  const bool shared = (e == a.E);
  if (shared && a.shared_bits == 8) return;
  const size_t eoff_w = shared ? 0 : (size_t)e * a.I * K8;
  const size_t eoff_s = shared ? 0 : (size_t)e * a.I * G;
  const uint32_t *gw = (shared ? a.sh_gate.w : a.gate.w) + eoff_w;
  const uint16_t *gs = (shared ? a.sh_gate.s : a.gate.s) + eoff_s;
  const uint16_t *gb = (shared ? a.sh_gate.b : a.gate.b) + eoff_s;
  const uint32_t *uw = (shared ? a.sh_up.w : a.up.w) + eoff_w;
  const uint16_t *us = (shared ? a.sh_up.s : a.up.s) + eoff_s;
  const uint16_t *ub = (shared ? a.sh_up.b : a.up.b) + eoff_s;

  const int row0 = blockIdx.x * ROWS + warp * kGateUpSteps * RPS;
  uint4 ga[kGateUpSteps], gb2[kGateUpSteps], ua[kGateUpSteps], ub2[kGateUpSteps];
  float gsv[kGateUpSteps], gbv[kGateUpSteps], usv[kGateUpSteps], ubv[kGateUpSteps];
#pragma unroll
  for (int st = 0; st < kGateUpSteps; ++st) {
    const int row = row0 + st * RPS + rsub;
    if (row < a.I) {
      const size_t wo = (size_t)row * K8 + 8 * g;
      const size_t so = (size_t)row * G + g;
      ga[st] = ld_stream(gw + wo);
      gb2[st] = ld_stream(gw + wo + 4);
      ua[st] = ld_stream(uw + wo);
      ub2[st] = ld_stream(uw + wo + 4);
      gsv[st] = bf16f(ld_u16(gs + so));
      gbv[st] = bf16f(ld_u16(gb + so));
      usv[st] = bf16f(ld_u16(us + so));
      ubv[st] = bf16f(ld_u16(ub + so));
    } else {
      ga[st] = gb2[st] = ua[st] = ub2[st] = make_uint4(0, 0, 0, 0);
      gsv[st] = gbv[st] = usv[st] = ubv[st] = 0.f;
    }
  }
  for (int pr = pb; pr < pe; ++pr) {
    const int t = w.pair_tok[pr];
    XGroupB xg;
    {
      uint4 c[8];
      const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kGroup * g);
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
      xgroupb_from_bf16(xg, c);
    }
#pragma unroll
    for (int st = 0; st < kGateUpSteps; ++st) {
      const float gd = seg_sum<G>(q4_group_dot_b(ga[st], gb2[st], xg, gsv[st], gbv[st]));
      const float ud = seg_sum<G>(q4_group_dot_b(ua[st], ub2[st], xg, usv[st], ubv[st]));
      const int row = row0 + st * RPS + rsub;
      if (g == 0 && row < a.I) w.h[(size_t)pr * a.I + row] = silu_mul(gd, ud);
    }
  }
}

// The 8-bit shared expert's gate/up rows (q4-xl): one row-step per warp, applied to every
// token (the shared expert is the last unique unit); h in fp32 as above.
template <int G>  // groups per row = H / 64
__global__ void __launch_bounds__(kGateUpThreads)
    gateup_shared8_kernel(GateUpArgs a, DecodePtrs w) {
  constexpr int RPS = 32 / G;
  const int U = w.meta[0];
  if (U < 1 || U > w.Umax) return;
  const int u = U - 1;
  if (w.uexp()[u] != a.E) return;
  const int pb = max(w.ubase()[u], 0), pe = min(w.ubase()[u + 1], w.P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;
  const int row = (blockIdx.x * (kGateUpThreads / 32) + warp) * RPS + rsub;
  const bool valid = row < a.I;
  uint4 gq[4] = {}, uq[4] = {};
  float gs = 0.f, gb = 0.f, us = 0.f, ub = 0.f;
  if (valid) {
    const size_t wo = (size_t)row * (G * 16) + 16 * g, so = (size_t)row * G + g;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gq[j] = ld_stream(a.sh_gate.w + wo + 4 * j);
      uq[j] = ld_stream(a.sh_up.w + wo + 4 * j);
    }
    gs = bf16f(ld_u16(a.sh_gate.s + so));
    gb = bf16f(ld_u16(a.sh_gate.b + so));
    us = bf16f(ld_u16(a.sh_up.s + so));
    ub = bf16f(ld_u16(a.sh_up.b + so));
  }
  for (int pr = pb; pr < pe; ++pr) {
    const int t = w.pair_tok[pr];
    XGroup8 x8;
    {
      uint4 c[8];
      const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kGroup * g);
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
      xgroup8_from_bf16(x8, c);
    }
    const float gd = seg_sum<G>(q8_group_dot_b(gq, x8, gs, gb));
    const float ud = seg_sum<G>(q8_group_dot_b(uq, x8, us, ub));
    if (g == 0 && valid) w.h[(size_t)pr * a.I + row] = silu_mul(gd, ud);
  }
}

// ---------------------------------------------------------------------------------------
// 3. down GEMV + weighted combine (fixed-order sum per token)
// ---------------------------------------------------------------------------------------
struct DownArgs {
  lily_q4_mat down, sh_down;
  uint16_t *y;
  int T, E, H, I;
  int shared_bits;
};

template <int G, bool Q8P>  // groups per row = I / 64; Q8P: the shared expert's codes are 8-bit
__global__ void __launch_bounds__(kDownThreads)
    down_kernel(DownArgs a, DecodePtrs w) {
  constexpr int RPS = 32 / G;
  constexpr int K8 = G * 8;
  constexpr int STEPS = (kDownRows + RPS - 1) / RPS;
  __shared__ float part[kMaxPairs][kDownRows];
  __shared__ int s_tok[kMaxPairs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;
  const int U = min(max(w.meta[0], 0), w.Umax);
  const int P = min(max(w.ubase()[U], 0), w.P);
  const int r0 = blockIdx.x * kDownRows;

  for (int pr = warp; pr < P; pr += kDownThreads / 32) {
    const int e = min(max(w.pair_e()[pr], 0), a.E);
    const bool shared = (e == a.E);
    if (Q8P && shared) {
      // 8-bit shared down rows: 64 code bytes of the lane's group per row-step, fp32 h
      float v[64];
      const float4 *hp = reinterpret_cast<const float4 *>(w.h + (size_t)pr * a.I + kGroup * g);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 f = __ldcg(hp + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      const float pw = w.pair_w[pr];
#pragma unroll
      for (int st = 0; st < STEPS; ++st) {
        const int rr = st * RPS + rsub;
        const int row = r0 + rr;
        uint4 w4[4] = {};
        float sv = 0.f, bv = 0.f;
        if (rr < kDownRows && row < a.H) {
          const size_t wo = (size_t)row * (G * 16) + 16 * g, so = (size_t)row * G + g;
#pragma unroll
          for (int j = 0; j < 4; ++j) w4[j] = ld_stream(a.sh_down.w + wo + 4 * j);
          sv = bf16f(ld_u16(a.sh_down.s + so));
          bv = bf16f(ld_u16(a.sh_down.b + so));
        }
        const float d = seg_sum<G>(q8_group_dot_f32(w4, v, sv, bv));
        if (g == 0 && rr < kDownRows) part[pr][rr] = pw * d;
      }
      if (lane == 0) s_tok[pr] = w.pair_tok[pr];
      continue;
    }
    const uint32_t *dw = shared ? a.sh_down.w : a.down.w + (size_t)e * a.H * K8;
    const uint16_t *ds = shared ? a.sh_down.s : a.down.s + (size_t)e * a.H * G;
    const uint16_t *db = shared ? a.sh_down.b : a.down.b + (size_t)e * a.H * G;
    uint4 wa[STEPS], wb[STEPS];
    float sv[STEPS], bv[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int rr = st * RPS + rsub;
      const int row = r0 + rr;
      if (rr < kDownRows && row < a.H) {
        const size_t wo = (size_t)row * K8 + 8 * g;
        wa[st] = ld_stream(dw + wo);
        wb[st] = ld_stream(dw + wo + 4);
        sv[st] = bf16f(ld_u16(ds + (size_t)row * G + g));
        bv[st] = bf16f(ld_u16(db + (size_t)row * G + g));
      } else {
        wa[st] = wb[st] = make_uint4(0, 0, 0, 0);
        sv[st] = bv[st] = 0.f;
      }
    }
    XGroup xg;
    {
      float v[64];
      const float4 *hp = reinterpret_cast<const float4 *>(w.h + (size_t)pr * a.I + kGroup * g);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 f = __ldcg(hp + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      xgroup_from(xg, v);
    }
    const float pw = w.pair_w[pr];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const float d = seg_sum<G>(q4_group_dot(wa[st], wb[st], xg, sv[st], bv[st]));
      const int rr = st * RPS + rsub;
      if (g == 0 && rr < kDownRows) part[pr][rr] = pw * d;
    }
    if (lane == 0) s_tok[pr] = w.pair_tok[pr];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < a.T * kDownRows; j += kDownThreads) {
    const int t = j / kDownRows, rr = j % kDownRows;
    const int row = r0 + rr;
    if (row >= a.H) continue;
    float acc = 0.f;
    for (int pr = 0; pr < P; ++pr)
      if (s_tok[pr] == t) acc += part[pr][rr];
    a.y[(size_t)t * a.H + row] = f2bf16_rne(acc);
  }
}

// ---------------------------------------------------------------------------------------
// Single-launch decode layer (one block per SM, two grid barriers)
//
//   phase A: router rows (+ the shared gate row) and the shared expert's gate/up rows,
//            none of which depends on the routing; x is prepared once per block in shared
//            memory for the Q4 dot products while the first weight loads are in flight
//   barrier
//   phase B: every block takes the routing of all tokens from the logits (identical
//            result in every block); routed gate/up rows, each warp issuing the loads of
//            a batch of rows before computing; each warp copies the codes and scales of its
//            first down tasks into shared memory (cp.async) so they load across the barrier
//   barrier
//   phase C: h of every pair prepared in shared memory; block b owns down row-steps
//            b, b + grid, ...; the (pair, row-step) tasks are spread over all warps;
//            partials meet in shared memory and are summed per token in a fixed order
//            (deterministic)
// ---------------------------------------------------------------------------------------
constexpr int kFusedThreads = 448;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr size_t kFusedSmemMax = 160 * 1024;
constexpr int kFusedMaxT = 4;
constexpr int kFusedMaxQ = 4;   // down row-steps per block
constexpr int kFusedBatch = 2;  // gate/up rows whose loads a warp issues together
constexpr long long kBarrierCycles = 2000000000LL;  // ~1 s
// Down tasks (pair, row-step) of a block: warp w takes tasks w, w + kFusedWarps, ...; its
// first kFusedStaged tasks have their codes and scales copied into shared memory before the
// second grid barrier.
constexpr int kFusedStaged = 4;
constexpr int kFusedSlots = kFusedWarps * kFusedStaged;
constexpr int kFusedMaxLoads = 7;  // 16-byte loads per thread when preparing x or h

// Dynamic shared memory of the single-launch kernel (byte offsets, 16-byte aligned): x as
// given, x prepared for the Q4 dot products (pair words + per-group sums), the staged down
// codes ([slot][lane][32 bytes]) and scales ([slot][s 32 | b 32] bf16), then h prepared like
// x.  h is sized for P pairs; the rest does not depend on the routing.
struct FusedLayout {
  size_t xr, xp, xX, dsc, dn, hp, hX, total;
};
__host__ __device__ constexpr size_t al16(size_t v) { return (v + 15) / 16 * 16; }
__host__ __device__ inline FusedLayout fused_layout(int P, int T, int H, int I) {
  FusedLayout l{};
  size_t o = 0;
  l.xr = o;  // x as given (bf16), for the router rows
  o = al16(o + (size_t)T * H * 2);
  l.xp = o;
  o = al16(o + (size_t)T * H * 2);
  l.xX = o;
  o = al16(o + (size_t)T * (H / kGroup) * 4);
  l.dsc = o;
  o = al16(o + (size_t)kFusedSlots * 128);
  l.dn = o;
  o = al16(o + (size_t)kFusedSlots * 32 * 32);
  l.hp = o;
  o = al16(o + (size_t)P * I * 2);
  l.hX = o;
  o = al16(o + (size_t)P * (I / kGroup) * 4);
  l.total = o;
  return l;
}

struct FusedArgs {
  lily_q4_mat gate, up, down, sh_gate, sh_up, sh_down;
  const uint16_t *router;
  const float *bias;
  const uint16_t *shared_gate;
  const uint16_t *x;
  uint16_t *y;
  int T, E, H, I, k, has_shared;
  int32_t *out_idx;
  float *out_w;
  lily_q4_mat router8;  // the 8-bit router when router_bits == 8
  int router_bits, shared_bits;
};

// Word offset of chunk c (8 values) of 64-value group g in a prepared vector: each group's
// eight 4-word chunks are rotated by g so that lanes reading different groups at once hit
// different shared-memory banks.
__device__ __forceinline__ int xg_word(int g, int c) { return g * 32 + (((c + g) & 7) << 2); }

// Prepare n8 chunks of 8 bf16 values (src 16-byte aligned, read through L2) for
// q4_group_dot_b: each chunk becomes the four words (v[j] | v[j+4] << 16), j < 4 -- the order
// in which the dequantised codes pair up -- and each 64-value group's sum goes to X (and the
// chunk as given to raw[c], with RAW).  The whole
// block takes part (the group sums are warp reductions over 8 consecutive chunks); every load
// is issued before any is used.  n8 <= kFusedMaxLoads * kFusedThreads, a multiple of 8.
template <bool RAW>
__device__ __forceinline__ void xg_stage(uint32_t *dst, float *X, const uint16_t *src, int n8,
                                         uint4 *raw) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  uint4 v[kFusedMaxLoads];
#pragma unroll
  for (int i = 0; i < kFusedMaxLoads; ++i) {
    const int c = threadIdx.x + i * kFusedThreads;
    if (c < n8) v[i] = __ldcg(s4 + c);
  }
#pragma unroll
  for (int i = 0; i < kFusedMaxLoads; ++i) {
    if (i * kFusedThreads >= n8) break;  // same for every thread of the block
    const int c = threadIdx.x + i * kFusedThreads;
    float sum = 0.f;
    if (c < n8) {
      if (RAW) raw[c] = v[i];
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};  // w[q] = v[2q] | v[2q+1] << 16
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu);
        const uint32_t hi = (j & 1) ? (w[2 + (j >> 1)] >> 16) : (w[2 + (j >> 1)] & 0xFFFFu);
        o[j] = lo | (hi << 16);
        sum += __uint_as_float(lo << 16) + __uint_as_float(hi << 16);
      }
      *reinterpret_cast<uint4 *>(dst + xg_word(c >> 3, c & 7)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    sum = seg_sum<8>(sum);
    if (c < n8 && (c & 7) == 0) X[c >> 3] = sum;
  }
}

// Group g of a vector prepared by xg_stage, into the registers q4_group_dot_b takes.
__device__ __forceinline__ void xg_load(XGroupB &g, const uint32_t *xp, const float *X, int grp) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = *reinterpret_cast<const uint4 *>(xp + xg_word(grp, c));
    g.xp[4 * c + 0] = v.x;
    g.xp[4 * c + 1] = v.y;
    g.xp[4 * c + 2] = v.z;
    g.xp[4 * c + 3] = v.w;
  }
  g.X = X[grp];
  g.X128 = 128.0f * g.X;
}

// The GI bf16 scales (or biases) of one down row, global -> shared (GI = 8: 16 bytes,
// GI = 2: 4 bytes; both addresses aligned to the size).
template <int GI>
__device__ __forceinline__ void cp_async_row_scales(uint32_t dst, const uint16_t *src) {
  static_assert(GI == 8 || GI == 2, "row scales of 16 or 4 bytes");
  if constexpr (GI == 8)
    cp_async16_stream(dst, src);
  else
    cp_async4_stream(dst, src);
}

// Grid barrier on a 64-bit arrival counter that only grows: each block adds 1 per barrier
// (a fire-and-forget release reduction) and polls until the count reaches its target.  The
// count after a completed launch is a multiple of the grid size, so a block derives this
// launch's base from the value it reads before its first arrival (no block can pass the
// first barrier before every block has arrived).  After a timed-out wait the count is off
// and the workspace must be re-initialised.
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long barrier_base(int32_t *hdr) {
  const unsigned long long c =
      ld_acquire_u64(reinterpret_cast<unsigned long long *>(hdr + kHdrBarrier64));
  return c - c % gridDim.x;
}

__device__ bool grid_barrier(int32_t *hdr, unsigned long long target, volatile int *s_abort) {
  __syncthreads();
  if (threadIdx.x == 0 && !*s_abort) {
    unsigned long long *cnt = reinterpret_cast<unsigned long long *>(hdr + kHdrBarrier64);
    // the release reduction itself orders the block's earlier writes (seen by thread 0
    // through the block barrier) before the arrival
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
    const long long t0 = clock64();
    while (ld_acquire_u64(cnt) < target) {
      if (clock64() - t0 > kBarrierCycles) {
        atomicExch(hdr + kHdrError, 2);
        *s_abort = 1;
        break;
      }
    }
  }
  __syncthreads();
  return !*s_abort;
}

// Diagnostic for the bounded waits: one block waits on something nothing provides -- a grid
// barrier whose target no arrival reaches (which = 0) or an mbarrier phase nothing completes
// (which = 1) -- until the wait's bound, then records the time-out in the workspace header as a
// stalled launch of the library would.
__global__ void selftest_wait_kernel(int32_t *hdr, int which) {
  __shared__ volatile int s_abort;
  __shared__ __align__(8) unsigned long long s_bar;
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  if (which == 0) {
    const unsigned long long base = barrier_base(hdr);
    grid_barrier(hdr, base + 1000ull * gridDim.x, &s_abort);
  } else {
    const uint32_t b = tc::smem_u32(&s_bar);
    if (threadIdx.x == 0) {
      tc::mbar_init(b, 1);
      tc::mbar_init_fence();
    }
    __syncthreads();
    tc::wait_bar(b, 0, &s_abort, hdr + kHdrError);
  }
}

int selftest_wait(void *ws, int which, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(static_cast<int32_t *>(ws), which);
  return check_launch();
}

// Routing of up to 4 tokens by one block, for the single-launch path: warps 0..T-1 take
// the top-k of one token each; warp 0 then builds the unique-expert table with a bitmap
// of selected experts (ascending id) and places the (token, weight) pairs.
template <int EC>
__device__ void route_small(const float *logits, const float *sigma, int T, int E, int k,
                            int has_shared, const RouteDst &d) {
  __shared__ int s_idx[4 * kMaxK];
  __shared__ float s_p[4 * kMaxK];
  __shared__ int s_cnt[4 * kMaxK + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the shared expert's gate of token `lane`, loaded together with the logits
  const float sig = (has_shared && warp == 0 && lane < T) ? __ldcg(sigma + lane) : 0.f;
  if (warp < T) {
    const int t = warp;
    float myv;
    int mye;
    warp_topk<EC>(logits + (size_t)t * E, E, k, mye, myv);  // lane i: selection i
    // softmax over the k selected logits (selection 0 holds the largest)
    const float v0 = __shfl_sync(0xffffffffu, myv, 0);
    const float ex = lane < k ? expf(myv - v0) : 0.f;
    const float pi = ex / seg_sum<32>(ex);
    if (lane < k) {
      s_idx[t * k + lane] = mye;
      s_p[t * k + lane] = pi;
      if (d.out_idx) d.out_idx[t * k + lane] = mye;
      if (d.out_w) d.out_w[t * k + lane] = pi;
    }
    if (T == 1) {
      // one token: the k selected experts are the unique experts, each with one pair;
      // lane i places selection i at the rank of its expert id among the k
      int rank = 0;
      for (int j = 0; j < k; ++j) rank += __shfl_sync(0xffffffffu, mye, j) < mye;
      if (lane < k) {
        d.uexp[rank] = mye;
        d.ubase[rank] = rank;
        d.pair_tok[rank] = 0;
        d.pair_w[rank] = pi;
        d.pair_e[rank] = mye;
      }
      if (lane == 0) {
        int U = k;
        if (has_shared) {
          d.uexp[U] = E;
          d.ubase[U] = k;
          d.pair_tok[k] = 0;
          d.pair_w[k] = sig;
          d.pair_e[k] = E;
          ++U;
        }
        d.ubase[U] = k + (has_shared ? 1 : 0);
        *d.U = U;
      }
    }
  }
  __syncthreads();
  if (T == 1) return;
  if (warp == 0) {
    const int n = T * k;  // <= 64
    uint32_t word = 0;    // lane's 32 experts: bit set if selected
    for (int j = 0; j < n; ++j) {
      const int e = s_idx[j];
      if ((e >> 5) == lane) word |= 1u << (e & 31);
    }
    int total;
    const int prefix = warp_excl_scan(__popc(word), &total);
    // unique experts in ascending id
    {
      uint32_t wb = word;
      int r = prefix;
      while (wb) {
        const int b = __ffs(wb) - 1;
        wb &= wb - 1;
        d.uexp[r++] = lane * 32 + b;
      }
    }
    for (int r = lane; r <= 4 * kMaxK; r += 32) s_cnt[r] = 0;
    __syncwarp();
    int rk[2], ek[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      const int e = j < n ? s_idx[j] : 0;
      const uint32_t wsrc = __shfl_sync(0xffffffffu, word, (e >> 5) & 31);
      const int psrc = __shfl_sync(0xffffffffu, prefix, (e >> 5) & 31);
      rk[h] = psrc + __popc(wsrc & ((1u << (e & 31)) - 1u));
      ek[h] = e;
      if (j < n) atomicAdd(&s_cnt[rk[h]], 1);
    }
    __syncwarp();
    // exclusive scan of the counts of the (<= 64) unique experts: two per lane
    const int c0 = lane * 2 < total ? s_cnt[lane * 2] : 0;
    const int c1 = lane * 2 + 1 < total ? s_cnt[lane * 2 + 1] : 0;
    int dummy;
    const int b0 = warp_excl_scan(c0 + c1, &dummy);
    if (lane * 2 < total) d.ubase[lane * 2] = b0;
    if (lane * 2 + 1 < total) d.ubase[lane * 2 + 1] = b0 + c0;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      if (j < n) {
        const int t = j / k, e = ek[h];
        int before = 0;  // earlier tokens that chose e
        for (int jj = 0; jj < t * k; ++jj) before += (s_idx[jj] == e);
        const int pos = d.ubase[rk[h]] + before;
        d.pair_tok[pos] = t;
        d.pair_w[pos] = s_p[j];
        d.pair_e[pos] = e;
      }
    }
    if (lane == 0) {
      int U = total;
      if (has_shared) {
        d.uexp[U] = E;
        d.ubase[U] = n;
        ++U;
      }
      d.ubase[U] = n + (has_shared ? T : 0);
      *d.U = U;
    }
    if (has_shared && lane < T) {
      d.pair_tok[n + lane] = lane;
      d.pair_w[n + lane] = sig;
      d.pair_e[n + lane] = E;
    }
  }
  __syncthreads();
}

// One row of a routed expert's gate and up matrices (lane's group) and one down row.
struct RowPair {
  uint4 a0, a1, b0, b1;
  float as, ab, bs, bb;
};
struct DownRow {
  uint4 w0, w1;
  float s, b;
};

template <int GH>
__device__ __forceinline__ void load_gateup(const FusedArgs &a, const int32_t *uexp, int task,
                                            int steps_h, int I, int gh, int rh, RowPair &r) {
  constexpr int RPS_H = 32 / GH;
  const int u = task / steps_h;
  const int row = (task % steps_h) * RPS_H + rh;
  const size_t e = (size_t)uexp[u];
  const size_t wo = (e * I + row) * (GH * 8) + 8 * gh, so = (e * I + row) * GH + gh;
  r.a0 = ld_stream(a.gate.w + wo);
  r.a1 = ld_stream(a.gate.w + wo + 4);
  r.b0 = ld_stream(a.up.w + wo);
  r.b1 = ld_stream(a.up.w + wo + 4);
  r.as = bf16f(ld_u16(a.gate.s + so));
  r.ab = bf16f(ld_u16(a.gate.b + so));
  r.bs = bf16f(ld_u16(a.up.s + so));
  r.bb = bf16f(ld_u16(a.up.b + so));
}

template <int GI>
__device__ __forceinline__ void load_down_mat(const lily_q4_mat &m, int e, int row, int H, int gi,
                                              DownRow &r) {
  const size_t wo = ((size_t)e * H + row) * (GI * 8) + 8 * gi;
  const size_t so = ((size_t)e * H + row) * GI + gi;
  r.w0 = ld_stream(m.w + wo);
  r.w1 = ld_stream(m.w + wo + 4);
  r.s = bf16f(ld_u16(m.s + so));
  r.b = bf16f(ld_u16(m.b + so));
}

// Weights of one phase-A task into registers: a router row (bf16; the lane's chunks
// lane + 32 j) or one row-step of the shared expert's gate and up rows (codes in wv[0..3],
// raw bf16 scales and biases in sc, converted where they are used).
template <int GH, bool Q8P>
__device__ __forceinline__ void load_phase_a(const FusedArgs &a, int task, int nrouter, int lane,
                                             uint4 (&wv)[8], uint32_t (&sc)[4]) {
  constexpr int RPS_H = 32 / GH;
  if (task < nrouter) {
    if (Q8P && task < a.E && a.router_bits == 8) {
      // an 8-bit router row: lane g < GH holds group g (64 code bytes, its s and b)
      if (lane < GH) {
        const size_t wo = (size_t)task * (GH * 16) + 16 * lane, so = (size_t)task * GH + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = ld_stream(a.router8.w + wo + 4 * j);
        sc[0] = ld_u16(a.router8.s + so);
        sc[1] = ld_u16(a.router8.b + so);
      }
      return;
    }
    const uint16_t *wr = task < a.E ? a.router + (size_t)task * a.H : a.shared_gate;
    const int nchunk = a.H / 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = lane + 32 * j;
      wv[j] = c < nchunk ? ld_stream(wr + 8 * c) : make_uint4(0, 0, 0, 0);
    }
  } else {
    const int gh = lane % GH, rh = lane / GH;
    const int row = (task - nrouter) * RPS_H + rh;
    const size_t so = (size_t)row * GH + gh;
    if (Q8P && a.shared_bits == 8) {
      // 8-bit shared rows: 64 code bytes of the lane's group in each matrix
      const size_t wo = (size_t)row * (GH * 16) + 16 * gh;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wv[j] = ld_stream(a.sh_gate.w + wo + 4 * j);
        wv[4 + j] = ld_stream(a.sh_up.w + wo + 4 * j);
      }
    } else {
      const size_t wo = (size_t)row * (GH * 8) + 8 * gh;
      wv[0] = ld_stream(a.sh_gate.w + wo);
      wv[1] = ld_stream(a.sh_gate.w + wo + 4);
      wv[2] = ld_stream(a.sh_up.w + wo);
      wv[3] = ld_stream(a.sh_up.w + wo + 4);
    }
    sc[0] = ld_u16(a.sh_gate.s + so);
    sc[1] = ld_u16(a.sh_gate.b + so);
    sc[2] = ld_u16(a.sh_up.s + so);
    sc[3] = ld_u16(a.sh_up.b + so);
  }
}

// Phase timeline of the kernel, for profiling builds only (-DLILY_Q4_TRACE): thread 0 of each
// block stamps %globaltimer at fixed points into a device array, [launch parity][block][point]
// (the parity of the launch's index on the workspace, from its grid-barrier count):
// 7 the previous kernel complete (griddepcontrol.wait returned), 0 x prepared, 1 phase A (router
// rows, shared gate/up) done, 2 first grid barrier passed, 3 routed, 4 gate/up done, 5 second
// grid barrier passed, 6 h prepared and down rows landed, 8 down done, 9 y written.
#ifdef LILY_Q4_TRACE
constexpr int kTracePoints = 16;
__device__ unsigned long long g_lq4_trace[2][1024][kTracePoints];
__device__ __forceinline__ unsigned long long lq4_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define LQ4_TRACE_AT(i, par, t)                                 \
  do {                                                          \
    if (threadIdx.x == 0 && blockIdx.x < 1024)                  \
      g_lq4_trace[(par) & 1ull][blockIdx.x][(i)] = (t);         \
  } while (0)
#define LQ4_TRACE(i, par) LQ4_TRACE_AT(i, par, lq4_now())
#define LQ4_TRACE_CLOCK(var) const unsigned long long var = lq4_now()
#else
#define LQ4_TRACE_AT(i, par, t) \
  do {                          \
  } while (0)
#define LQ4_TRACE(i, par) \
  do {                    \
  } while (0)
#define LQ4_TRACE_CLOCK(var) \
  do {                       \
  } while (0)
#endif

// Q8P: the layer has 8-bit parts (router and/or shared expert); the instantiation without
// them carries none of their branches.
template <int GH, int GI, int EC, bool Q8P>
__global__ void __launch_bounds__(kFusedThreads, 1)
    moe_decode_fused_kernel(FusedArgs a, DecodePtrs w) {
  static_assert(kFusedThreads % 8 == 0, "xg_stage groups 8 consecutive threads");
  extern __shared__ __align__(16) uint8_t fsm[];
  __shared__ int32_t s_U;
  __shared__ int32_t s_uexp[kMaxT * kMaxK + 1];
  __shared__ int32_t s_ubase[kMaxT * kMaxK + 2];
  __shared__ int32_t s_pair_tok[kMaxPairs];
  __shared__ int32_t s_pair_e[kMaxPairs];
  __shared__ float s_pair_w[kMaxPairs];
  __shared__ volatile int s_abort;
  __shared__ unsigned long long s_bbase;
  constexpr int RPS_H = 32 / GH;  // rows per warp-step, K = H (gate/up)
  constexpr int RPS_I = 32 / GI;  // rows per warp-step, K = I (down)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = gridDim.x * kFusedWarps;
  const int gw = warp * gridDim.x + blockIdx.x;  // interleaved: consecutive tasks on different SMs
  const int T = a.T, E = a.E, H = a.H, I = a.I, k = a.k;
  const int nrouter = E + a.has_shared;
  const int gh = lane % GH, rh = lane / GH;
  const int gi = lane % GI, ri = lane / GI;
  const int nquads = H / RPS_I;  // down row-steps
  const int GXH = H / kGroup, GXI = I / kGroup;  // groups of an x row, of an h row
  // Launched as a programmatic dependent of the previous kernel on the stream: the block may
  // start while that kernel drains, so it lets its own dependents be scheduled, then waits
  // for the previous kernel to complete before touching anything it may have written (x,
  // the workspace).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Weights do not depend on the previous kernel: each warp issues the loads of its first
  // phase-A row (router row, or shared-expert gate/up row-step) before it waits for that
  // kernel, so they are in flight while it drains.
  const int nshared_tasks = a.has_shared ? I / RPS_H : 0;
  const int ntasks_a = nrouter + nshared_tasks;
  uint4 wv[8];
  uint32_t sc[4];
  if (gw < ntasks_a) load_phase_a<GH, Q8P>(a, gw, nrouter, lane, wv, sc);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  LQ4_TRACE_CLOCK(t_wait);
  // The barrier base is read by the last warp, which has no phase-A rows: the acquire load
  // holds up only that warp while the others issue their weight loads.
  if (threadIdx.x == kFusedThreads - 32) {
    s_abort = 0;
    s_bbase = barrier_base(w.hdr);
  }
  const FusedLayout L0 = fused_layout(0, T, H, I);  // the offsets that do not depend on P
  const uint4 *s_xr = reinterpret_cast<const uint4 *>(fsm + L0.xr);
  uint32_t *s_xp = reinterpret_cast<uint32_t *>(fsm + L0.xp);
  float *s_xX = reinterpret_cast<float *>(fsm + L0.xX);
  uint16_t *s_dsc = reinterpret_cast<uint16_t *>(fsm + L0.dsc);
  uint8_t *s_dn = fsm + L0.dn;
  uint16_t *h16 = reinterpret_cast<uint16_t *>(w.h);  // this path keeps h as bf16 [pair][I]

  // ------------------------------------------------------------------ phase A
  // The first task's weight loads are in flight (above); the block prepares x in shared memory.
  xg_stage<true>(s_xp, s_xX, a.x, T * H / 8, reinterpret_cast<uint4 *>(fsm + L0.xr));
  __syncthreads();
  const unsigned long long bbase = s_bbase;
  [[maybe_unused]] const unsigned long long par = bbase / (2ull * gridDim.x);  // launch index
  LQ4_TRACE_AT(7, par, t_wait);
  LQ4_TRACE(0, par);
  for (int task = gw; task < ntasks_a; task += nw) {
    if (task != gw) load_phase_a<GH, Q8P>(a, task, nrouter, lane, wv, sc);
    if (Q8P && task < E && a.router_bits == 8) {
      // 8-bit router row: lane g < GH dots its group with x re-paired for 8-bit codes
      const int row = task;
      const uint4 w4[4] = {wv[0], wv[1], wv[2], wv[3]};
      const float rs = bf16f(sc[0]), rb = bf16f(sc[1]);
      for (int t = 0; t < T; ++t) {
        float d = 0.f;
        if (lane < GH) {
          XGroupB xg;
          xg_load(xg, s_xp, s_xX, t * GXH + lane);
          XGroup8 x8;
          xgroup8_from_b(x8, xg);
          d = q8_group_dot_b(w4, x8, rs, rb);
        }
        d = seg_sum<32>(d);
        if (lane == 0) __stcg(w.logits + (size_t)t * E + row, d + (a.bias ? a.bias[row] : 0.f));
      }
    } else if (task < nrouter) {
      const int row = task;
      const int nchunk = H / 8;
      for (int t = 0; t < T; ++t) {
        const uint4 *xt = s_xr + (size_t)t * nchunk;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = lane + 32 * j;
          if (c < nchunk) {
            const uint4 xv = xt[c];
            const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
            const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc = fmaf(__uint_as_float(ww[i] << 16), __uint_as_float(xx[i] << 16), acc);
              acc = fmaf(__uint_as_float(ww[i] & 0xFFFF0000u), __uint_as_float(xx[i] & 0xFFFF0000u),
                         acc);
            }
          }
        }
        acc = seg_sum<32>(acc);
        if (lane == 0) {
          if (row < E)
            __stcg(w.logits + (size_t)t * E + row, acc + (a.bias ? a.bias[row] : 0.f));
          else
            __stcg(w.sigma + t, 1.0f / (1.0f + expf(-acc)));
        }
      }
    } else {
      // shared expert gate/up rows (one warp-step of RPS_H rows)
      const int row = (task - nrouter) * RPS_H + rh;
      const float gs = bf16f(sc[0]), gb = bf16f(sc[1]), us = bf16f(sc[2]), ub = bf16f(sc[3]);
      for (int t = 0; t < T; ++t) {
        XGroupB xg;
        xg_load(xg, s_xp, s_xX, t * GXH + gh);
        float gd, ud;
        if (Q8P && a.shared_bits == 8) {
          XGroup8 x8;
          xgroup8_from_b(x8, xg);
          const uint4 g4[4] = {wv[0], wv[1], wv[2], wv[3]}, u4[4] = {wv[4], wv[5], wv[6], wv[7]};
          gd = seg_sum<GH>(q8_group_dot_b(g4, x8, gs, gb));
          ud = seg_sum<GH>(q8_group_dot_b(u4, x8, us, ub));
        } else {
          gd = seg_sum<GH>(q4_group_dot_b(wv[0], wv[1], xg, gs, gb));
          ud = seg_sum<GH>(q4_group_dot_b(wv[2], wv[3], xg, us, ub));
        }
        // shared pairs sit after the T*k routed pairs
        if (gh == 0) h16[(size_t)(T * k + t) * I + row] = f2bf16_rne(silu_mul(gd, ud));
      }
    }
  }
  LQ4_TRACE(1, par);
  if (!grid_barrier(w.hdr, bbase + gridDim.x, &s_abort)) return;
  LQ4_TRACE(2, par);

  // ------------------------------------------------------------------ phase B
  {
    RouteDst d{nullptr, nullptr, &s_U, s_uexp, s_ubase, s_pair_tok, s_pair_w, s_pair_e,
               blockIdx.x == 0 ? a.out_idx : nullptr, blockIdx.x == 0 ? a.out_w : nullptr};
    route_small<EC>(w.logits, w.sigma, T, E, k, a.has_shared, d);
  }
  LQ4_TRACE(3, par);
  const int U = s_U;
  const int Ur = a.has_shared ? U - 1 : U;  // routed unique experts
  // Down tasks (pair pr, row-step qi) -> j = pr * nq_cta + qi.  The first kFusedSlots are
  // split into contiguous runs, one per warp (neighbouring tasks share the pair, so a warp
  // prepares few h vectors); their codes and scales depend on the routing only, so each warp
  // copies its staged tasks into shared memory (cp.async, nothing held in registers) right
  // after issuing the loads of its first gate/up rows: all of the layer's routed weights are
  // then in flight at once, and the copies have landed before the second grid barrier.  Warp
  // w takes the rest, j = nstaged + w + kFusedWarps i, in phase C.
  const int P = s_ubase[U];  // routed pairs, then the shared expert's T pairs
  const int nq_cta = (nquads - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int ntask_c = P * nq_cta;
  // 8-bit shared-expert rows (q4-xl) have twice the code bytes: their tasks (the last T pairs)
  // are run from global memory after the others
  const int ntask_q4 = (Q8P && a.has_shared && a.shared_bits == 8) ? T * k * nq_cta : ntask_c;
  const int nstaged = min(ntask_q4, kFusedSlots);
  const int jlo = warp * nstaged / kFusedWarps, jhi = (warp + 1) * nstaged / kFusedWarps;
  auto stage_down = [&]() {
#pragma unroll
    for (int i = 0; i < kFusedStaged; ++i) {
      const int j = jlo + i;
      if (j < jhi) {
        const int pr = j / nq_cta, qi = j - pr * nq_cta;
        const int e = s_pair_e[pr];
        const bool sh = (e == E);
        const lily_q4_mat &m = sh ? a.sh_down : a.down;
        const size_t ee = sh ? 0 : (size_t)e;
        const int row = (blockIdx.x + qi * gridDim.x) * RPS_I + ri;
        const size_t wo = (ee * H + row) * (GI * 8) + 8 * gi;
        const uint32_t dst = tc::smem_u32(s_dn + ((size_t)j * 32 + lane) * 32);
        cp_async16_stream(dst, m.w + wo);
        cp_async16_stream(dst + 16, m.w + wo + 4);
        if (gi < 2)
          cp_async_row_scales<GI>(tc::smem_u32(s_dsc + j * 64 + gi * 32 + ri * GI),
                                  (gi ? m.b : m.s) + (ee * H + row) * GI);
      }
    }
    tc::cp_async_commit();
  };
  // routed gate/up: tasks (unique expert, row-step), a batch of kFusedBatch per warp with
  // all of the batch's loads issued before any is computed
  const int steps_h = I / RPS_H;
  const int ntasks_b = Ur * steps_h;
  bool staged = false;
  for (int base = gw; base < ntasks_b; base += nw * kFusedBatch) {
    RowPair rp[kFusedBatch];
#pragma unroll
    for (int i = 0; i < kFusedBatch; ++i)
      if (base + i * nw < ntasks_b) load_gateup<GH>(a, s_uexp, base + i * nw, steps_h, I, gh, rh, rp[i]);
    if (!staged) {
      stage_down();
      staged = true;
    }
    int xg_tok = -1;
    XGroupB xg;
#pragma unroll
    for (int i = 0; i < kFusedBatch; ++i) {
      const int task = base + i * nw;
      if (task < ntasks_b) {
        const int u = task / steps_h;
        const int row = (task % steps_h) * RPS_H + rh;
#pragma unroll 1
        for (int pr = s_ubase[u]; pr < s_ubase[u + 1]; ++pr) {
          const int t = s_pair_tok[pr];
          if (t != xg_tok) {
            xg_load(xg, s_xp, s_xX, t * GXH + gh);
            xg_tok = t;
          }
          const float gd = seg_sum<GH>(q4_group_dot_b(rp[i].a0, rp[i].a1, xg, rp[i].as, rp[i].ab));
          const float ud = seg_sum<GH>(q4_group_dot_b(rp[i].b0, rp[i].b1, xg, rp[i].bs, rp[i].bb));
          if (gh == 0) h16[(size_t)pr * I + row] = f2bf16_rne(silu_mul(gd, ud));
        }
      }
    }
  }
  if (!staged) stage_down();
  LQ4_TRACE(4, par);
  if (!grid_barrier(w.hdr, bbase + 2ull * gridDim.x, &s_abort)) {
    tc::cp_async_wait_all();  // no copy may land after the block has left
    return;
  }

  // ------------------------------------------------------------------ phase C
  // h of every pair, prepared in shared memory; block b owns down row-steps b, b + grid, ...;
  // partials meet in shared memory and are summed per token in a fixed order (deterministic)
  const FusedLayout LP = fused_layout(P, T, H, I);
  uint32_t *s_hp = reinterpret_cast<uint32_t *>(fsm + LP.hp);
  float *s_hX = reinterpret_cast<float *>(fsm + LP.hX);
  LQ4_TRACE(5, par);
  xg_stage<false>(s_hp, s_hX, h16, P * I / 8, nullptr);
  tc::cp_async_wait_all();
  __syncthreads();
  LQ4_TRACE(6, par);
  constexpr int ROWS = kFusedMaxQ * RPS_I;  // rows of this block, at most
  __shared__ float s_part[kFusedMaxT * (kMaxK + 1)][ROWS];
  {
    int cur = -1;  // pair whose h is in xg
    XGroupB xg;
    float pw = 0.f;
#pragma unroll 1
    for (int j = jlo; j < jhi; ++j) {
      const int pr = j / nq_cta, qi = j - pr * nq_cta;
      if (pr != cur) {
        xg_load(xg, s_hp, s_hX, pr * GXI + gi);
        pw = s_pair_w[pr];
        cur = pr;
      }
      const uint4 *c = reinterpret_cast<const uint4 *>(s_dn + ((size_t)j * 32 + lane) * 32);
      const float sv = bf16f(s_dsc[j * 64 + lane]), bv = bf16f(s_dsc[j * 64 + 32 + lane]);
      const float dd = seg_sum<GI>(q4_group_dot_b(c[0], c[1], xg, sv, bv));
      if (gi == 0) s_part[pr][qi * RPS_I + ri] = pw * dd;
    }
    // tasks beyond the staged ones (batch above one token): from global memory, kFusedMaxQ
    // at a time with all of their loads issued first
    for (int j0 = nstaged + warp; j0 < ntask_q4; j0 += kFusedMaxQ * kFusedWarps) {
      DownRow dr[kFusedMaxQ];
#pragma unroll
      for (int q = 0; q < kFusedMaxQ; ++q) {
        const int j = j0 + q * kFusedWarps;
        if (j < ntask_q4) {
          const int pr = j / nq_cta, qi = j - pr * nq_cta;
          const int e = s_pair_e[pr];
          const int row = (blockIdx.x + qi * gridDim.x) * RPS_I + ri;
          if (e == E)
            load_down_mat<GI>(a.sh_down, 0, row, H, gi, dr[q]);
          else
            load_down_mat<GI>(a.down, e, row, H, gi, dr[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < kFusedMaxQ; ++q) {
        const int j = j0 + q * kFusedWarps;
        if (j < ntask_q4) {
          const int pr = j / nq_cta, qi = j - pr * nq_cta;
          if (pr != cur) {
            xg_load(xg, s_hp, s_hX, pr * GXI + gi);
            pw = s_pair_w[pr];
            cur = pr;
          }
          const float dd = seg_sum<GI>(q4_group_dot_b(dr[q].w0, dr[q].w1, xg, dr[q].s, dr[q].b));
          if (gi == 0) s_part[pr][qi * RPS_I + ri] = pw * dd;
        }
      }
    }
    // 8-bit shared-expert down rows: one task at a time, h re-paired for 8-bit codes
    for (int j = ntask_q4 + warp; Q8P && j < ntask_c; j += kFusedWarps) {
      const int pr = j / nq_cta, qi = j - pr * nq_cta;
      const int row = (blockIdx.x + qi * gridDim.x) * RPS_I + ri;
      const size_t wo = (size_t)row * (GI * 16) + 16 * gi, so = (size_t)row * GI + gi;
      uint4 w4[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) w4[v] = ld_stream(a.sh_down.w + wo + 4 * v);
      const float sv = bf16f(ld_u16(a.sh_down.s + so)), bv = bf16f(ld_u16(a.sh_down.b + so));
      XGroup8 x8;
      {
        XGroupB hb;
        xg_load(hb, s_hp, s_hX, pr * GXI + gi);
        xgroup8_from_b(x8, hb);
      }
      const float dd = seg_sum<GI>(q8_group_dot_b(w4, x8, sv, bv));
      if (gi == 0) s_part[pr][qi * RPS_I + ri] = s_pair_w[pr] * dd;
    }
  }
  __syncthreads();
  LQ4_TRACE(8, par);
  const int nrows_cta = nq_cta * RPS_I;
  for (int j = threadIdx.x; j < T * nrows_cta; j += kFusedThreads) {
    const int t = j / nrows_cta, rr = j % nrows_cta;
    const int row = (blockIdx.x + (rr / RPS_I) * gridDim.x) * RPS_I + rr % RPS_I;
    float acc = 0.f;
    for (int pr = 0; pr < P; ++pr)
      if (s_pair_tok[pr] == t) acc += s_part[pr][rr];
    a.y[(size_t)t * H + row] = f2bf16_rne(acc);
  }
  LQ4_TRACE(9, par);
}

#ifdef LILY_Q4_TRACE
extern "C" __attribute__((visibility("default"))) int lily_q4_trace_read(void *host, size_t bytes) {
  if (bytes > sizeof(g_lq4_trace)) bytes = sizeof(g_lq4_trace);
  return cudaMemcpyFromSymbol(host, g_lq4_trace, bytes) == cudaSuccess ? 0 : -1;
}
#endif

static bool fused_ok(const lily_q4_moe_layer &L, int T) {
  if (T > kFusedMaxT) return false;
  const int P = T * L.top_k + (L.has_shared ? T : 0);
  if (fused_layout(P, T, L.hidden, L.inter).total > kFusedSmemMax) return false;
  // x and h are prepared with at most kFusedMaxLoads 16-byte loads per thread
  const size_t nload = (size_t)kFusedMaxLoads * kFusedThreads;
  if ((size_t)T * L.hidden / 8 > nload || (size_t)P * L.inter / 8 > nload) return false;
  const int GH = L.hidden / kGroup, GI = L.inter / kGroup;
  // each block owns at most kFusedMaxQ down row-steps
  if (L.hidden / (32 / GI) > sm_count() * kFusedMaxQ) return false;
  return (GH == 32 && GI == 8) || (GH == 4 && GI == 2 && L.n_experts <= 256);
}

template <int GH, int GI, int EC, bool Q8P>
static int launch_fused_q(const FusedArgs &fa, const DecodePtrs &p, size_t smem, cudaStream_t st) {
  static int attr_done[64] = {0};  // per instantiation and device
  int dev = 0;
  cudaGetDevice(&dev);
  auto fn = moe_decode_fused_kernel<GH, GI, EC, Q8P>;
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmemMax) !=
        cudaSuccess)
      return LILY_Q4_ERR_CUDA;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kFusedThreads, kFusedSmemMax) !=
            cudaSuccess ||
        nb < 1)
      return LILY_Q4_ERR_CUDA;
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // One block per SM (the occupancy check above), so on a GPU that runs this stream alone
  // every block is resident at once, which the grid barriers need.  The launch is a
  // programmatic dependent of the previous kernel on the stream: blocks take SMs as that
  // kernel's blocks leave and wait for it (griddepcontrol.wait) before reading anything,
  // which hides the launch gap between consecutive layers.  (A cooperative launch would
  // guarantee co-residency even with other work on the GPU, but the runtime does not accept
  // it together with programmatic serialization.)  Should other work hold SMs so that some
  // blocks start late, the bounded barrier waits give up and the call reports
  // LILY_Q4_ERR_TIMEOUT through lily_q4_workspace_status instead of hanging.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, fa, p) != cudaSuccess) return LILY_Q4_ERR_CUDA;
  return check_launch();
}

template <int GH, int GI, int EC>
static int launch_fused(const FusedArgs &fa, const DecodePtrs &p, size_t smem, cudaStream_t st) {
  const bool q8 = fa.router_bits == 8 || (fa.has_shared && fa.shared_bits == 8);
  return q8 ? launch_fused_q<GH, GI, EC, true>(fa, p, smem, st)
            : launch_fused_q<GH, GI, EC, false>(fa, p, smem, st);
}

template <int G>
static void launch_gateup(const GateUpArgs &a, const DecodePtrs &p, int Umax, cudaStream_t st) {
  constexpr int RPS = 32 / G;
  constexpr int ROWS = (kGateUpThreads / 32) * kGateUpSteps * RPS;
  dim3 grid((a.I + ROWS - 1) / ROWS, Umax);
  gateup_kernel<G><<<grid, kGateUpThreads, 0, st>>>(a, p);
  if (a.shared_bits == 8) {
    constexpr int ROWS8 = (kGateUpThreads / 32) * RPS;
    gateup_shared8_kernel<G><<<(a.I + ROWS8 - 1) / ROWS8, kGateUpThreads, 0, st>>>(a, p);
  }
}

template <int G>
static void launch_down(const DownArgs &a, const DecodePtrs &p, cudaStream_t st) {
  dim3 grid((a.H + kDownRows - 1) / kDownRows);
  if (a.shared_bits == 8)
    down_kernel<G, true><<<grid, kDownThreads, 0, st>>>(a, p);
  else
    down_kernel<G, false><<<grid, kDownThreads, 0, st>>>(a, p);
}

#define LQ4_DISPATCH_G(gval, FN, ...)      \
  switch (gval) {                          \
    case 1: FN<1>(__VA_ARGS__); break;     \
    case 2: FN<2>(__VA_ARGS__); break;     \
    case 4: FN<4>(__VA_ARGS__); break;     \
    case 8: FN<8>(__VA_ARGS__); break;     \
    case 16: FN<16>(__VA_ARGS__); break;   \
    case 32: FN<32>(__VA_ARGS__); break;   \
    default: return LILY_Q4_ERR_UNSUPPORTED; \
  }

int decode_launch_count(const lily_q4_moe_layer &L, int T) {
  if (fused_ok(L, T) && sm_count() > 0) return 1;
  return (L.has_shared && L.shared_bits == 8) ? 4 : 3;
}

int launch_moe_decode(const lily_q4_moe_layer &L, const uint16_t *x, int T, uint16_t *y,
                      int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t st) {
  const DecodeWsLayout l = decode_ws_layout(L, T);
  const DecodePtrs p = decode_ptrs(ws, l);
  if (fused_ok(L, T) && sm_count() > 0) {
    FusedArgs fa{L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down, L.router, L.router_bias,
                 L.shared_gate, x, y, T, L.n_experts, L.hidden, L.inter, L.top_k, L.has_shared,
                 topk_idx, topk_w, L.router_q8, L.router_bits == 8 ? 8 : 16,
                 (L.has_shared && L.shared_bits == 8) ? 8 : 4};
    const size_t smem = fused_layout(l.P, T, L.hidden, L.inter).total;
    if (L.hidden / kGroup == 32) {
      if (L.n_experts <= 256) return launch_fused<32, 8, 8>(fa, p, smem, st);
      if (L.n_experts <= 512) return launch_fused<32, 8, 16>(fa, p, smem, st);
      return launch_fused<32, 8, 32>(fa, p, smem, st);
    }
    return launch_fused<4, 2, 8>(fa, p, smem, st);
  }
  RouterArgs ra{L.router, L.router_bias, L.shared_gate, x, T, L.n_experts, L.hidden, L.top_k,
                L.has_shared, topk_idx, topk_w, L.router_q8, L.router_bits == 8 ? 8 : 16};
  const int shared_bits = (L.has_shared && L.shared_bits == 8) ? 8 : 4;
  const int nrows = L.n_experts + L.has_shared;
  const int rgrid = (nrows + kRouterThreads / 32 - 1) / (kRouterThreads / 32);
  if (L.n_experts <= 256)
    router_topk_kernel<8><<<rgrid, kRouterThreads, 0, st>>>(ra, p);
  else if (L.n_experts <= 512)
    router_topk_kernel<16><<<rgrid, kRouterThreads, 0, st>>>(ra, p);
  else
    router_topk_kernel<32><<<rgrid, kRouterThreads, 0, st>>>(ra, p);

  GateUpArgs ga{L.gate, L.up, L.sh_gate, L.sh_up, x, L.n_experts, L.hidden, L.inter, shared_bits};
  LQ4_DISPATCH_G(L.hidden / kGroup, launch_gateup, ga, p, l.Umax, st);

  DownArgs da{L.down, L.sh_down, y, T, L.n_experts, L.hidden, L.inter, shared_bits};
  LQ4_DISPATCH_G(L.inter / kGroup, launch_down, da, p, st);
  return check_launch();
}

}  // namespace lq4
