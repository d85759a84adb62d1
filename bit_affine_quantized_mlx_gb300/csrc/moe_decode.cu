// Decode-step MoE feed-forward (1..16 tokens).
//
// "The MoE" kernels of a decode step, which is bandwidth-bound (fork page, "How the
// speed was achieved": a decode step's reads, tuned toward "what its chain of reads
// can stream").  Three launches on the caller's stream:
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
};

// ---------------------------------------------------------------------------------------
// 1. router logits + shared gate; last block: top-k, gates, unique-expert pairs
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouterThreads)
    router_topk_kernel(RouterArgs a, DecodePtrs w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nrows = a.E + a.has_shared;
  const int row = blockIdx.x * (kRouterThreads / 32) + warp;
  const int nchunk = a.H / 8;  // 16-byte chunks per row
  if (row < nrows) {
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

  __shared__ int s_idx[kMaxT * kMaxK];
  __shared__ float s_p[kMaxT * kMaxK];
  __shared__ int s_cnt[1024];
  __shared__ int s_base[1024];
  __shared__ int s_rank[1024];
  const int E = a.E, k = a.k, T = a.T;

  // top-k per token: warp per token, k rounds of a warp argmax over unselected experts
  for (int t = warp; t < T; t += kRouterThreads / 32) {
    const float *lg = w.logits + (size_t)t * E;
    uint32_t taken = 0;  // bit j: expert lane + 32 j already selected
    float v0 = 0.f, denom = 0.f;
    float sel_v[kMaxK];
    int sel_e[kMaxK];
    for (int i = 0; i < k; ++i) {
      float bv = -FLT_MAX;
      int be = INT_MAX;
      for (int j = 0; lane + 32 * j < E; ++j) {
        const int e = lane + 32 * j;
        if (taken & (1u << j)) continue;
        const float v = __ldcg(lg + e);
        if (better(v, e, bv, be)) {
          bv = v;
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_v[i] = bv;
      sel_e[i] = be;
    }
    v0 = sel_v[0];
    for (int i = 0; i < k; ++i) denom += expf(sel_v[i] - v0);
    if (lane == 0) {
      for (int i = 0; i < k; ++i) {
        const float pi = expf(sel_v[i] - v0) / denom;
        s_idx[t * k + i] = sel_e[i];
        s_p[t * k + i] = pi;
        w.idx[t * k + i] = sel_e[i];
        w.p[t * k + i] = pi;
        if (a.out_idx) a.out_idx[t * k + i] = sel_e[i];
        if (a.out_w) a.out_w[t * k + i] = pi;
      }
    }
  }
  for (int e = threadIdx.x; e < E; e += kRouterThreads) s_cnt[e] = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < T * k; j += kRouterThreads) atomicAdd(&s_cnt[s_idx[j]], 1);
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
      s_rank[e] = rp;
      s_base[e] = rc;
      if (s_cnt[e] > 0) {
        w.uexp()[rp] = e;
        w.ubase()[rp] = rc;
        ++rp;
      }
      rc += s_cnt[e];
    }
    if (lane == 0) {
      int U = totp;
      if (a.has_shared) {
        w.uexp()[U] = E;  // the shared expert
        w.ubase()[U] = totc;
        ++U;
      }
      w.ubase()[U] = totc + (a.has_shared ? T : 0);
      w.meta[0] = U;
    }
  }
  __syncthreads();
  // pairs: (token t, slot i) -> position base[e] + (number of earlier tokens that chose e)
  for (int j = threadIdx.x; j < T * k; j += kRouterThreads) {
    const int t = j / k, e = s_idx[j];
    int pos = 0;
    for (int jj = 0; jj < t * k; ++jj) pos += (s_idx[jj] == e);
    const int pr = s_base[e] + pos;
    w.pair_tok[pr] = t;
    w.pair_w[pr] = s_p[j];
    w.pair_e()[pr] = e;
  }
  if (a.has_shared) {
    for (int t = threadIdx.x; t < T; t += kRouterThreads) {
      const int pr = T * k + t;
      w.pair_tok[pr] = t;
      w.pair_w[pr] = __ldcg(w.sigma + t);
      w.pair_e()[pr] = E;
    }
  }
  if (threadIdx.x == 0) w.hdr[kHdrCounterB] = 0;
}

// ---------------------------------------------------------------------------------------
// 2. gate/up dequant-GEMV + SwiGLU, per unique expert and row block
// ---------------------------------------------------------------------------------------
struct GateUpArgs {
  lily_q4_mat gate, up, sh_gate, sh_up;
  const uint16_t *x;
  int E, H, I;
};

template <int G>  // groups per row = H / 64
__global__ void __launch_bounds__(kGateUpThreads)
    gateup_kernel(GateUpArgs a, DecodePtrs w) {
  constexpr int RPS = 32 / G;
  constexpr int K8 = G * 8;
  constexpr int ROWS = (kGateUpThreads / 32) * kGateUpSteps * RPS;
  const int u = blockIdx.y;
  const int U = w.meta[0];
  if (u >= U) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;
  const int e = w.uexp()[u];
  const int pb = w.ubase()[u], pe = w.ubase()[u + 1];
  const bool shared = (e == a.E);
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
    XGroup xg;
    {
      uint4 c[8];
      const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kGroup * g);
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = __ldg(xp + i);
      xgroup_from_bf16(xg, c);
    }
#pragma unroll
    for (int st = 0; st < kGateUpSteps; ++st) {
      const float gd = seg_sum<G>(q4_group_dot(ga[st], gb2[st], xg, gsv[st], gbv[st]));
      const float ud = seg_sum<G>(q4_group_dot(ua[st], ub2[st], xg, usv[st], ubv[st]));
      const int row = row0 + st * RPS + rsub;
      if (g == 0 && row < a.I) w.h[(size_t)pr * a.I + row] = silu_mul(gd, ud);
    }
  }
}

// ---------------------------------------------------------------------------------------
// 3. down GEMV + weighted combine (fixed-order sum per token)
// ---------------------------------------------------------------------------------------
struct DownArgs {
  lily_q4_mat down, sh_down;
  uint16_t *y;
  int T, E, H, I;
};

template <int G>  // groups per row = I / 64
__global__ void __launch_bounds__(kDownThreads)
    down_kernel(DownArgs a, DecodePtrs w) {
  constexpr int RPS = 32 / G;
  constexpr int K8 = G * 8;
  constexpr int STEPS = (kDownRows + RPS - 1) / RPS;
  __shared__ float part[kMaxPairs][kDownRows];
  __shared__ int s_tok[kMaxPairs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G, rsub = lane / G;
  const int U = w.meta[0];
  const int P = w.ubase()[U];
  const int r0 = blockIdx.x * kDownRows;

  for (int pr = warp; pr < P; pr += kDownThreads / 32) {
    const int e = w.pair_e()[pr];
    const bool shared = (e == a.E);
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

template <int G>
static void launch_gateup(const GateUpArgs &a, const DecodePtrs &p, int Umax, cudaStream_t st) {
  constexpr int RPS = 32 / G;
  constexpr int ROWS = (kGateUpThreads / 32) * kGateUpSteps * RPS;
  dim3 grid((a.I + ROWS - 1) / ROWS, Umax);
  gateup_kernel<G><<<grid, kGateUpThreads, 0, st>>>(a, p);
}

template <int G>
static void launch_down(const DownArgs &a, const DecodePtrs &p, cudaStream_t st) {
  dim3 grid((a.H + kDownRows - 1) / kDownRows);
  down_kernel<G><<<grid, kDownThreads, 0, st>>>(a, p);
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

int launch_moe_decode(const lily_q4_moe_layer &L, const uint16_t *x, int T, uint16_t *y,
                      int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t st) {
  const DecodeWsLayout l = decode_ws_layout(L, T);
  const DecodePtrs p = decode_ptrs(ws, l);
  RouterArgs ra{L.router, L.router_bias, L.shared_gate, x, T, L.n_experts, L.hidden, L.top_k,
                L.has_shared, topk_idx, topk_w};
  const int nrows = L.n_experts + L.has_shared;
  const int rgrid = (nrows + kRouterThreads / 32 - 1) / (kRouterThreads / 32);
  router_topk_kernel<<<rgrid, kRouterThreads, 0, st>>>(ra, p);

  GateUpArgs ga{L.gate, L.up, L.sh_gate, L.sh_up, x, L.n_experts, L.hidden, L.inter};
  LQ4_DISPATCH_G(L.hidden / kGroup, launch_gateup, ga, p, l.Umax, st);

  DownArgs da{L.down, L.sh_down, y, T, L.n_experts, L.hidden, L.inter};
  LQ4_DISPATCH_G(L.inter / kGroup, launch_down, da, p, st);
  return check_launch();
}

}  // namespace lq4
