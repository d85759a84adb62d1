// Prefill-chunk MoE feed-forward on the tensor cores.
//
// Prefill is compute-bound and runs the expert GEMM on the matrix units ("Prefill on
// the tensor ops ... better tiling for the expert GEMM", fork page, "How the speed was
// achieved"; prompt chunks of 2,048 tokens, Lily-vs-MLX report, "Measurement
// contract").  Launch sequence on the caller's stream:
//
//   router GEMM : logits[T][E] = x Wr^T (+ offsets), bf16 x bf16 -> fp32 on tcgen05
//   topk        : top-k per token, softmax over the k; the same warp writes the token's row
//                 with K permuted inside every 8-element chunk to the order the Q4 unpack
//                 produces (0,4,1,5,2,6,3,7), so dequantised weight words are stored without
//                 a shuffle (a dot product is unchanged when both operands are permuted
//                 alike), and the shared gate sigmoid(x . g)
//   scan        : per-expert offsets of the expert-sorted pairs, GEMM work lists
//   place       : stable bucketing (token order inside an expert) from the top-k blocks'
//                 per-expert counts and their prefixes over the blocks
//   gate/up GEMM: per (expert, 128 intermediate rows, <=128 tokens): dequantised Q4
//                 gate and up tiles x gathered token rows, SwiGLU in the epilogue -> h (bf16)
//   down GEMM   : per (expert, 128 output rows, <=128 tokens): Q4 down tile x h rows,
//                 scaled by the pair's gate weight -> o (bf16)
//   combine     : y[t] = sum over t's k slots (+ shared) of o, in slot order (deterministic)
//
// Layers with affine 8-bit parts (the report's checkpoint keeps its router gates at 8 bits,
// "Hardware and software"; the fork page's q4-xl conversion keeps the shared expert at 8 bits,
// "The model") take two preparation launches in front:
//   8-bit router        : w = s*q + b with s*q exact in 16 bits, split exactly into bf16 hi +
//                         lo; the bias term uses the per-group sums of x split exactly into
//                         three bf16 parts.  The router GEMM then runs on
//                         A = [hi | lo | b | b | b], B = [x | x | X_hi | X_mid | X_lo]: every
//                         product exact, fp32 accumulation, logits not rounded.
//   8-bit shared expert : q = lo + 16 hi, so s*q + b = (s*lo + b + 128 s) + (16 s*hi - 128 s)
//                         -- each row becomes a 4-bit row of twice the width (low nibbles with
//                         (s, b + 128 s), high nibbles with (16 s, -128 s)); the expert GEMMs run
//                         the shared expert's tiles with K doubled, reading its token (or h)
//                         rows twice.
//
// The GEMM kernel is persistent (one CTA per SM) and warp-specialised:
//   warps 0-3  epilogue: tcgen05.ld of the fp32 accumulator (TMEM lanes 0..127)
//   warp  4    TMEM allocation and the single-thread tcgen05.mma issue loop
//   warps 5-7  token-row gather: cp.async into a 128-byte-swizzled K-major tile
//   warps 8-   weight producers: Q4 codes prefetched into registers a group of k-blocks
//              ahead, dequantised (bf16x2 FMA: s*q + b, one rounding) and written with
//              tcgen05.st straight into tensor memory as the MMA's A operand (row i of the
//              tile in lane i); the router GEMM's bf16 A tile is cp.async'd to shared memory.
//              A row's k-block (32 bytes of codes) is taken by one thread with one 256-bit
//              load when the weights are 32-byte aligned (every code sector is requested
//              once), else by two threads with 128-bit loads
// Stages are handed over with mbarriers; the down and router accumulators are
// double-buffered in TMEM so the epilogue of one tile overlaps the main loop of the next
// (gate/up keeps one accumulator pair: its A stages take the other half of TMEM).  Every
// wait is bounded: on time-out the kernel records an error word in the workspace, drains
// and returns.
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "internal.h"
#include "q4_device.cuh"
#include "tc_sm100.cuh"

namespace lq4 {

constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kBN = 128;  // tokens per tile (MMA N, padded to a multiple of 16)
constexpr int kMmaWarp = 4;
constexpr int kBWarp0 = 5, kBThreads = 96;
constexpr int kAWarp0 = 8;  // weight producers: warps 8.. (128 * RT threads per A matrix)
constexpr int kHdrItemsGU = 8, kHdrItemsDN = 9;
// Waiting threads are suspended by the hardware (mbarrier.try_wait with a time hint) instead of
// spinning, so the warps that wait leave the issue slots to the weight producers, which pace
// the pipeline; the bounded-wait checks run between suspensions.
constexpr uint32_t kSleepNs = 1000;

// The router GEMM splits K so that more SMs share its few tiles; the partial logits are
// summed in a fixed order by the top-k kernel.
__host__ __device__ constexpr int kRouterSplit(int H) { return H >= 1024 ? 4 : 1; }
static_assert(kRouterSplit(1 << 30) <= 4 && kRouterSplit(128) <= 4,
              "the top-k kernel sums at most four partial logits per token");

enum { kRouter = 0, kGateUp = 1, kDown = 2 };

// Tile memory.  The router's A operand (bf16 weights) is copied into shared memory; the
// dequantised Q4 tiles of the expert GEMMs are written by the producer threads straight into
// tensor memory (row i in lane i), so shared-memory bandwidth is left to the token tiles.
// TMEM columns: accumulators first (NACC buffers of ACC_COLS), then SA A stages of 32*NA*KS.
// RT = producer threads per weight row (1: the row's whole k-block, 8 code words; 2: 4 each).
// KS = k-blocks (64 of K) per pipeline stage: the expert GEMMs hand over two k-blocks at a
// time, so the MMA thread's per-stage waits, fences and commits are paid once per 16 (gate/up)
// or 8 (down) MMAs; that loop, not the tensor pipe, bounds the small token tiles.  A stage's A
// columns are [matrix][k-block][32]; its B tile is KS 128-byte-swizzled [kBN][64] sub-tiles.
template <int MODE, int RT = 2>
struct Cfg {
  static constexpr bool TMEM_A = MODE != kRouter;
  static constexpr int NA = MODE == kGateUp ? 2 : 1;  // A tiles per k-block
  static constexpr int KS = MODE == kRouter ? 1 : 2;  // k-blocks per stage
  static constexpr int SA = MODE == kGateUp ? 2 : 4;  // A stages
  static constexpr int SB = MODE == kGateUp ? 4 : (MODE == kDown ? 4 : 6);  // B (token) stages
  static constexpr int AT = NA * kBM * RT;            // weight-producer threads
  static constexpr int XB = 0;                        // gather warps after the producers
  static constexpr int BT = kBThreads + 32 * XB;      // token-row gather threads
  static constexpr int THREADS = kAWarp0 * 32 + AT + 32 * XB;
  static constexpr int A_BYTES = kBM * 128;
  static constexpr int B_SUB = kBN * 128;              // one k-block of a B stage
  static constexpr int B_BYTES = KS * B_SUB;
  static constexpr int A_STAGE = NA * A_BYTES;        // shared-memory A stage (router)
  static constexpr int ACC_COLS = NA * kBN;
  static constexpr int NACC = MODE == kGateUp ? 1 : 2;  // accumulator buffers
  static constexpr int A_COL0 = NACC * ACC_COLS;        // first TMEM column of the A stages
  static constexpr int A_COLS = 32 * NA * KS;           // TMEM columns of one A stage
  static constexpr int TMEM_COLS = TMEM_A ? A_COL0 + SA * A_COLS : NACC * ACC_COLS;
  static constexpr int OFF_B = TMEM_A ? 0 : SA * A_STAGE;
  // epilogue staging of one bf16 output tile [kBN tokens][kBM rows] (expert GEMMs)
  static constexpr int STG_BYTES = TMEM_A ? kBN * kBM * 2 : 0;
  static constexpr int OFF_STG = OFF_B + SB * B_BYTES;
  static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
  static constexpr int NBARS = 2 * SA + 2 * SB + 5;
  static constexpr int BYTES = OFF_BAR + NBARS * 8 + 1024;
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation is a power of two");
};

struct GemmArgs {
  lily_q4_mat a0, a1, sh0, sh1;  // routed stacks and shared matrices (a1/sh1: up)
  const uint16_t *a_bf16;        // router weights [E][H]
  int a_rows;                    // rows of one expert matrix (or E for the router)
  int K;                         // reduction length
  int E;
  const uint16_t *b_src;         // permuted token rows / h / x
  const int32_t *perm;
  const int4 *items;
  const int32_t *n_items_ptr;
  int n_items_static, mt_static, T;
  int ksplit;                    // router: K is split in ksplit parts (partial logits)
  int ksh;                       // the shared expert's K is ksh * K (2: an 8-bit shared expert)
  int P;                         // pair rows (h is [I/64][P][64], k-block-major)
  uint16_t *h_out;
  uint16_t *o_out;
  int o_ld;                      // H
  const float *pw;
  float *logits;
  const float *bias;
  int32_t *hdr;
};

// Barrier among the four epilogue warps only (named barrier 1).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The same barrier, returning whether any of the 128 epilogue threads passed `p` true.
__device__ __forceinline__ bool epilogue_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbar.red.or.pred po, 1, 128, pi;\n"
      "selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

constexpr int kSmemItems = 256;  // work items of one block staged in shared memory

// Work item it of this block (it = blockIdx.x + i * gridDim.x).
template <int MODE>
__device__ __forceinline__ int4 get_item(const GemmArgs &a, int it, const int4 *s_items) {
  if (MODE == kRouter) {  // (k split, first token, tokens, m-tile)
    const int mt = it % a.mt_static, rest = it / a.mt_static;
    const int split = rest % a.ksplit, t0 = (rest / a.ksplit) * kBN;
    return make_int4(split, t0, min(kBN, a.T - t0), mt);
  }
  const int i = (it - (int)blockIdx.x) / (int)gridDim.x;
  return i < kSmemItems ? s_items[i] : a.items[it];
}

// k-blocks of work item `item` (the shared expert, id E, may have a K of ksh times K).
template <int MODE>
__device__ __forceinline__ int item_nkb(const GemmArgs &a, const int4 &item, int nkb) {
  return (MODE != kRouter && item.x == a.E) ? nkb * a.ksh : nkb;
}

// Position of element r inside its 8-chunk in the permuted K order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ int kpos(int r) {
  return (r & ~7) | ((r & 3) * 2 + ((r >> 2) & 1));
}

// Dequantise one code word (8 codes) of one row into one 16-byte chunk of bf16 holding the
// pairs (q_j, q_j+4) -- the permuted K order.  s*q + b is formed with two bf16x2 FMAs:
// (128 + q) - 128 is exact, then s*q + b rounds once.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t s2, uint32_t b2) {
  uint32_t ws[4], out[4];
  ws[0] = w;
  asm("shr.b32 %0, %1, 4;" : "=r"(ws[1]) : "r"(w));
  asm("shr.b32 %0, %1, 8;" : "=r"(ws[2]) : "r"(w));
  asm("shr.b32 %0, %1, 12;" : "=r"(ws[3]) : "r"(w));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t v, q;  // q = v * 1 - 128
    asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(v) : "r"(ws[j]));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(v), "r"(0x3F803F80u), "r"(0xC300C300u));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out[j]) : "r"(q), "r"(s2), "r"(b2));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// KG k-blocks of per-group scales (or biases) of one row: 2*KG bytes.
template <int KG>
struct ScaleVec {
  uint32_t v[KG / 2];
  __device__ __forceinline__ void load(const uint16_t *p) {
    if constexpr (KG == 8) {
      const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
      v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else if constexpr (KG == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
      v[0] = u.x; v[1] = u.y;
    } else {
      v[0] = __ldg(reinterpret_cast<const uint32_t *>(p));
    }
  }
  // bf16 i broadcast to both halves
  __device__ __forceinline__ uint32_t pair(int i) const {
    const uint32_t h = (i & 1) ? (v[i >> 1] >> 16) : (v[i >> 1] & 0xFFFFu);
    return h | (h << 16);
  }
};

// The code words of one row's k-block that a producer thread takes: NV 16-byte vectors
// (NV = 2: the whole 32-byte k-block in one 256-bit load; the address is 32-byte aligned).
template <int NV>
__device__ __forceinline__ void ld_codes(const uint32_t *p, uint4 (&r)[NV]) {
  if constexpr (NV == 2)
    ld_stream32(p, r[0], r[1]);
  else
    r[0] = ld_stream(p);
}

template <int MODE, int KG, int RT>
__global__ void __launch_bounds__(Cfg<MODE, RT>::THREADS, 1) grouped_gemm_kernel(const GemmArgs a) {
  using C = Cfg<MODE, RT>;
  static_assert(MODE != kRouter || RT == 2, "the router's A copy takes two threads a row");
  extern __shared__ uint8_t smem_dyn[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_dyn + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto afull = [&](int s) { return bar0 + 8u * s; };
  auto aempty = [&](int s) { return bar0 + 8u * (C::SA + s); };
  auto bfull = [&](int s) { return bar0 + 8u * (2 * C::SA + s); };
  auto bempty = [&](int s) { return bar0 + 8u * (2 * C::SA + C::SB + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::SA + 2 * C::SB + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::SA + 2 * C::SB + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * C::SA + 2 * C::SB + 4);

  __shared__ uint32_t s_taddr;
  __shared__ volatile int s_abort;
  __shared__ int4 s_items[MODE == kRouter ? 1 : kSmemItems];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_allow_next();
  const int G = a.K / 64;  // groups per row
  const int nkb = MODE == kRouter ? G / a.ksplit : G;  // k-blocks per item

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < C::SA; ++s) {
      tc::mbar_init(afull(s), MODE == kRouter ? C::AT : C::AT / 32);
      tc::mbar_init(aempty(s), 1);
    }
    for (int s = 0; s < C::SB; ++s) {
      tc::mbar_init(bfull(s), MODE == kDown ? 1 : C::BT);
      tc::mbar_init(bempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(accf_bar(b), 1);
      tc::mbar_init(acce_bar(b), 128);
    }
    tc::mbar_init(done_bar, 1);
    tc::mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tc::smem_u32(&s_taddr), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  // Set-up above overlaps the previous kernel's tail; the work list (and every operand) is
  // read only after that kernel has completed.
  pdl_wait_prev();
  const int n_items = MODE == kRouter ? a.n_items_static : *(volatile const int32_t *)a.n_items_ptr;
  if (MODE != kRouter) {
    for (int i = threadIdx.x; i < kSmemItems; i += C::THREADS) {
      const int it = (int)blockIdx.x + i * (int)gridDim.x;
      if (it < n_items) s_items[i] = a.items[it];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = s_taddr;
  int32_t *err = a.hdr + kHdrError;

  if (warp < 4) {
    // ------------------------------------------------------------------ epilogue
    const int r = warp * 32 + lane;
    int j = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
      const int4 item = get_item<MODE>(a, it, s_items);
      const int b = j % C::NACC;
      // gate/up: the pairs' gate weights of this tile (token n in lane n % 32 of pwv[n / 32]),
      // fetched before the accumulator is ready
      float pwv[kBN / 32] = {};
      if (MODE == kGateUp) {
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q)
          if (lane + 32 * q < item.z) pwv[q] = __ldg(a.pw + item.y + lane + 32 * q);
      }
      // all four warps take the same decision, so the epilogue's own barriers never wait for
      // a warp that left
      if (epilogue_any(!tc::wait_bar(accf_bar(b), (j / C::NACC) & 1, &s_abort, err, kSleepNs))) break;
      tc::tc_fence_after();
      const int ntok = item.z, npad = (ntok + 15) & ~15;
      const int m = item.w * kBM + r;
      const bool row_ok = m < a.a_rows;
      const uint32_t tcol = taddr + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      if constexpr (MODE != kRouter) {
        // The tile goes to shared memory as bf16 (row r of the tile at its output position),
        // the accumulator is handed back, and then the staged token rows are written out with
        // 16-byte stores.
        uint16_t *stg = reinterpret_cast<uint16_t *>(smem + C::OFF_STG);  // [kBN][kBM]
        const int pos = MODE == kGateUp ? kpos(r) : r;
        for (int c0 = 0; c0 < npad; c0 += 16) {
          float d[16];
          if (MODE == kGateUp) {
            float u[16];
            tc::tmem_ld16x2(tcol + c0, d, tcol + kBN + c0, u);
            const float pwc = c0 < 32 ? pwv[0] : c0 < 64 ? pwv[1] : c0 < 96 ? pwv[2] : pwv[3];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float w = __shfl_sync(0xffffffffu, pwc, (c0 & 31) + i);
              stg[(c0 + i) * kBM + pos] = f2bf16_rne(w * silu_mul(d[i], u[i]));
            }
          } else {
            tc::tmem_ld16(tcol + c0, d);
#pragma unroll
            for (int i = 0; i < 16; ++i) stg[(c0 + i) * kBM + pos] = f2bf16_rne(d[i]);
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(acce_bar(b));
        epilogue_sync();  // the whole tile is staged
        for (int q = r; q < ntok * (kBM / 8); q += 128) {
          const int n = q / (kBM / 8), c = q % (kBM / 8);
          uint16_t *dst;
          if (MODE == kGateUp) {
            // h in k-block-major order, [I/64][P][64], each 128-byte row slice with its 16-byte
            // chunks in the 128-byte-swizzle order of the row's place n in its tile (the down
            // GEMM's tiles cover the same pair rows), so a down B stage is one bulk copy
            const int kbg = item.w * (kBM / 64) + (c >> 3);
            dst = a.h_out + ((size_t)kbg * a.P + item.y + n) * 64 + 8 * ((c & 7) ^ (n & 7));
          } else {
            dst = a.o_out + (size_t)(item.y + n) * a.o_ld + item.w * kBM + 8 * c;
          }
          *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(stg + n * kBM + 8 * c);
        }
        epilogue_sync();  // the staging buffer is free for the next tile
      } else {
        for (int c0 = 0; c0 < npad; c0 += 16) {
          float d[16];
          tc::tmem_ld16(tcol + c0, d);
          float *part = a.logits + (size_t)item.x * a.T * a.E;  // partial of k split item.x
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c0 + i;
            if (row_ok && n < ntok) part[(size_t)(item.y + n) * a.E + m] = d[i];
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(acce_bar(b));
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    // The whole warp runs the loop (descriptors stay warp-uniform); one elected lane issues
    // the MMAs and commits.  Every wait outcome is made warp-uniform.
    int sa = 0, sb = 0, j = 0;
    uint32_t pa = 0, pb = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++j) {
      const int4 item = get_item<MODE>(a, it, s_items);
      const int b = j % C::NACC;
      if (!__all_sync(0xffffffffu,
                      tc::wait_bar(acce_bar(b), ((j / C::NACC) & 1) ^ 1, &s_abort, err, kSleepNs)))
        break;
      tc::tc_fence_after();
      const int npad = (item.z + 15) & ~15;
      const uint32_t idesc = tc::idesc_bf16_f32(kBM, npad);
      const uint32_t d0 = taddr + (uint32_t)(b * C::ACC_COLS);
      const int nk = item_nkb<MODE>(a, item, nkb);  // a multiple of KS
      for (int kb = 0; kb < nk; kb += C::KS) {
        if (!__all_sync(0xffffffffu, tc::wait_bar(afull(sa), pa, &s_abort, err, kSleepNs) &&
                                         tc::wait_bar(bfull(sb), pb, &s_abort, err, kSleepNs))) {
          ok = false;
          break;
        }
        tc::fence_proxy_async();
        tc::tc_fence_after();
        const uint32_t sB = sbase + C::OFF_B + sb * C::B_BYTES;
        if constexpr (C::TMEM_A) {
          // A stage in TMEM: 8 columns (16 bf16 of K) per MMA
#pragma unroll
          for (int ks = 0; ks < C::KS; ++ks) {
            const uint32_t tA = taddr + (uint32_t)(C::A_COL0 + sa * C::A_COLS + 32 * ks);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = tc::desc_k128_sw128(sB + ks * C::B_SUB + 32 * kk);
              const uint32_t acc = (kb | ks | kk) ? 1u : 0u;
              tc::mma_bf16_ts_warp(d0, tA + 8 * kk, bd, idesc, acc);
              if (MODE == kGateUp)
                tc::mma_bf16_ts_warp(d0 + kBN, tA + 32 * C::KS + 8 * kk, bd, idesc, acc);
            }
          }
        } else {
          const uint32_t sA = sbase + sa * C::A_STAGE;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = tc::desc_k128_sw128(sB + 32 * kk);
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            tc::mma_bf16_warp(d0, tc::desc_k128_sw128(sA + 32 * kk), bd, idesc, acc);
          }
        }
        tc::mma_commit_warp(aempty(sa));
        tc::mma_commit_warp(bempty(sb));
        if (++sa == C::SA) { sa = 0; pa ^= 1; }
        if (++sb == C::SB) { sb = 0; pb ^= 1; }
      }
      if (!ok) break;
      tc::mma_commit_warp(accf_bar(b));
    }
    // drain: all issued MMAs complete before TMEM is released
    tc::mma_commit_warp(done_bar);
    tc::wait_bar(done_bar, 0, &s_abort, err, kSleepNs);
    __syncwarp();
  } else if (MODE == kDown && warp >= kBWarp0 && warp < kAWarp0) {
    // ------------------------------------------------------------------ h rows (down)
    // An item's h rows are consecutive pair rows, stored k-block-major and pre-swizzled by the
    // gate/up epilogue: each k-block of a B stage is one bulk copy of the item's ntok rows
    // (rows past ntok keep stale data; they only feed accumulator columns that are not stored).
    if (warp == kBWarp0 && lane == 0) {
      int sb = 0;
      uint32_t pb = 0;
      bool ok = true;
      long long issued = 0;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int4 item = get_item<MODE>(a, it, s_items);
        const uint32_t bytes = (uint32_t)item.z * 128u;
        const int nk = item_nkb<MODE>(a, item, nkb);
        for (int kb = 0; kb < nk; kb += C::KS) {
          if (!tc::wait_bar(bempty(sb), pb ^ 1, &s_abort, err, kSleepNs)) {
            ok = false;
            break;
          }
          const uint32_t sB = sbase + C::OFF_B + sb * C::B_BYTES;
          tc::mbar_arrive_expect_tx(bfull(sb), bytes * C::KS);
#pragma unroll
          for (int ks = 0; ks < C::KS; ++ks) {
            const int kbs = kb + ks < nkb ? kb + ks : kb + ks - nkb;  // a doubled K reads the rows twice
            tc::bulk_g2s(sB + ks * C::B_SUB, a.b_src + ((size_t)kbs * a.P + item.y) * 64, bytes, bfull(sb));
          }
          ++issued;
          if (++sb == C::SB) { sb = 0; pb ^= 1; }
        }
      }
      // No copy may still be landing when the block exits (after an abort the MMA thread
      // stops consuming): wait, bounded, for the last stages issued.
      volatile int no_abort = 0;
      for (long long q = issued - 1; q >= 0 && q >= issued - C::SB; --q)
        tc::wait_bar(bfull((int)(q % C::SB)), (uint32_t)((q / C::SB) & 1), &no_abort, err, kSleepNs);
    }
  } else if ((warp >= kBWarp0 && warp < kAWarp0) || warp >= kAWarp0 + C::AT / 32) {
    // ------------------------------------------------------------------ token-row gather
    constexpr int QB = (kBN * 8 + C::BT - 1) / C::BT;  // 16-byte chunks per thread
    const int tb = warp < kAWarp0 ? (int)threadIdx.x - kBWarp0 * 32
                                  : kBThreads + (int)threadIdx.x - (kAWarp0 * 32 + C::AT);
    int sb = 0;
    uint32_t pb = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 item = get_item<MODE>(a, it, s_items);
      const int ntok = item.z, nchunk = ((ntok + 15) & ~15) * 8;
      const int kb0 = MODE == kRouter ? item.x * nkb : 0;
      const uint16_t *srcp[QB];
      uint32_t dsto[QB], nbytes[QB];
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const int q = tb + i * C::BT;
        const int n = q >> 3, c = q & 7;
        srcp[i] = a.b_src;
        nbytes[i] = 0;
        if (n < ntok) {
          const size_t r = MODE == kGateUp ? (size_t)__ldg(a.perm + item.y + n) : (size_t)(item.y + n);
          srcp[i] = a.b_src + r * a.K + (size_t)kb0 * 64 + 8 * c;
          nbytes[i] = 16;
        }
        dsto[i] = tc::sw128((uint32_t)n, (uint32_t)c);
      }
      const int nk = item_nkb<MODE>(a, item, nkb);
      for (int kb = 0; kb < nk; kb += C::KS) {
        if (!tc::wait_bar(bempty(sb), pb ^ 1, &s_abort, err, kSleepNs)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          const uint32_t sB = sbase + C::OFF_B + sb * C::B_BYTES + ks * C::B_SUB;
          const int kbs = kb + ks < nkb ? kb + ks : kb + ks - nkb;  // a doubled K reads the rows twice
#pragma unroll
          for (int i = 0; i < QB; ++i)
            if (tb + i * C::BT < nchunk)
              tc::cp_async16(sB + dsto[i], srcp[i] + (nbytes[i] ? kbs * 64 : 0), nbytes[i]);
        }
        tc::cp_async_arrive_noinc(bfull(sb));
        if (++sb == C::SB) { sb = 0; pb ^= 1; }
      }
    }
    tc::cp_async_wait_all();
  } else {
    // ------------------------------------------------------------------ weight producers
    const int ta = threadIdx.x - kAWarp0 * 32;  // 0 .. C::AT-1
    const int row = ta & (kBM - 1);
    const int sub = ta >> 7;
    const int mat = C::NA == 2 ? (RT == 2 ? sub >> 1 : sub) : 0;  // GateUp: gate or up
    const int half = RT == 2 ? (sub & 1) : 0;  // which half of the row's k-block (RT = 2)
    int sa = 0;
    uint32_t pa = 0;
    bool ok = true;
    if (MODE == kRouter) {
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int4 item = get_item<MODE>(a, it, s_items);
        const int m = item.w * kBM + row;
        const bool valid = m < a.a_rows;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::wait_bar(aempty(sa), pa ^ 1, &s_abort, err, kSleepNs)) {
            ok = false;
            break;
          }
          const uint32_t sA = sbase + sa * C::A_STAGE;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * half + i;
            const uint16_t *src =
                valid ? a.a_bf16 + (size_t)m * a.K + (item.x * nkb + kb) * 64 + 8 * c : a.a_bf16;
            tc::cp_async16(sA + tc::sw128(row, c), src, valid ? 16u : 0u);
          }
          tc::cp_async_arrive_noinc(afull(sa));
          if (++sa == C::SA) { sa = 0; pa ^= 1; }
        }
      }
      tc::cp_async_wait_all();
    } else {
      // Codes of the next group of KG k-blocks are loaded into registers while the current
      // group is dequantised (prefetch distance KG k-blocks); per-item addressing is done
      // once per item.
      constexpr int NV = 2 / RT;  // 16-byte code vectors (4 words) per thread per k-block
      const int woff = 4 * half;
      // this thread's 16 TMEM columns of an A stage: lane = row (warp w writes lanes
      // 32*(w%4) .. +31, which is where its rows fall), columns mat*32 + half*16 ..
      const uint32_t t_off =
          ((uint32_t)(warp & 3) << 21) + (uint32_t)(C::A_COL0 + mat * 32 * C::KS + half * 16);
      static_assert(KG % C::KS == 0, "register groups hold whole stages");
      struct Src {
        const uint32_t *w;
        const uint16_t *s, *b;
        bool valid;
        int ngrp;  // register groups of the item (the rows of a doubled K are twice as long)
      };
      auto item_src = [&](int it) {
        const int4 item = get_item<MODE>(a, it, s_items);
        const int nk = item_nkb<MODE>(a, item, nkb);
        Src r{nullptr, nullptr, nullptr, false, nk / KG};
        const int e = item.x, m = item.w * kBM + row;
        if (m < a.a_rows) {
          const bool sh = (e == a.E);
          const lily_q4_mat &W = sh ? (mat ? a.sh1 : a.sh0) : (mat ? a.a1 : a.a0);
          const size_t rr = (sh ? 0 : (size_t)e * a.a_rows) + (size_t)m;
          r.w = W.w + rr * (size_t)(nk * 8) + woff;  // nk * 64 / 8 words a row
          r.s = W.s + rr * (size_t)nk;
          r.b = W.b + rr * (size_t)nk;
          r.valid = true;
        }
        return r;
      };
      uint4 raw[KG][NV];
      ScaleVec<KG> sc, bc, scn, bcn;
      int c_it = blockIdx.x, c_grp = 0;
      Src cur{nullptr, nullptr, nullptr, false, 0};
      if (c_it < n_items) {
        cur = item_src(c_it);
        if (cur.valid) {
#pragma unroll
          for (int i = 0; i < KG; ++i) ld_codes<NV>(cur.w + i * 8, raw[i]);
          sc.load(cur.s);
          bc.load(cur.b);
        }
      }
      while (c_it < n_items && ok) {
        // next group
        int n_it = c_it, n_grp = c_grp + 1;
        Src nxt = cur;
        if (n_grp == cur.ngrp) {
          n_grp = 0;
          n_it += gridDim.x;
          if (n_it < n_items) nxt = item_src(n_it);
        }
        const bool have_next = n_it < n_items && nxt.valid;
        if (have_next) {
          scn.load(nxt.s + n_grp * KG);
          bcn.load(nxt.b + n_grp * KG);
        }
#pragma unroll
        for (int i = 0; i < KG; ++i) {
          uint4 outv[NV * 4];
          if (cur.valid) {
            const uint32_t s2 = sc.pair(i), b2 = bc.pair(i);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
              outv[4 * v + 0] = dequant_word(raw[i][v].x, s2, b2);
              outv[4 * v + 1] = dequant_word(raw[i][v].y, s2, b2);
              outv[4 * v + 2] = dequant_word(raw[i][v].z, s2, b2);
              outv[4 * v + 3] = dequant_word(raw[i][v].w, s2, b2);
            }
          } else {
#pragma unroll
            for (int q = 0; q < NV * 4; ++q) outv[q] = make_uint4(0, 0, 0, 0);
          }
          if (have_next) ld_codes<NV>(nxt.w + (n_grp * KG + i) * 8, raw[i]);
          // The decision to go on is warp-uniform, so the warp-wide hand-over below never
          // waits for a lane that left.  A stage is claimed at its first k-block.
          const int ks = i % C::KS;
          if (ks == 0) {
            if (!__all_sync(0xffffffffu, tc::wait_bar(aempty(sa), pa ^ 1, &s_abort, err, kSleepNs))) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
          }
          {
            uint32_t r[16 * NV];
#pragma unroll
            for (int q = 0; q < 4 * NV; ++q) {
              r[4 * q + 0] = outv[q].x;
              r[4 * q + 1] = outv[q].y;
              r[4 * q + 2] = outv[q].z;
              r[4 * q + 3] = outv[q].w;
            }
            tc::tmem_st(taddr + t_off + (uint32_t)(sa * C::A_COLS + 32 * ks), r);
          }
          // The stores are complete (tcgen05.wait::st); one arrival per warp (the barrier
          // expects one per producer warp) after the warp has converged, once the stage's
          // last k-block is in.
          if (ks == C::KS - 1) {
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(afull(sa));
            if (++sa == C::SA) { sa = 0; pa ^= 1; }
          }
        }
        c_it = n_it;
        c_grp = n_grp;
        cur = nxt;
        sc = scn;
        bc = bcn;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, C::TMEM_COLS);
  }
}

// -------------------------------------------------------------------------------------
// small kernels around the GEMMs
// -------------------------------------------------------------------------------------

// xp[t][8c + pos(i)] = x[t][8c + i] for one token row, by one warp; with a shared expert the
// same warp forms its gate sigmoid(x . g) from the chunks it reads (sigma[t]).  Lane l takes
// chunks l, l + 32, ... (8 bf16 each) and accumulates them in that order; the lanes' sums
// meet in a fixed-order warp sum.
__device__ __forceinline__ void permute_token_row(const uint16_t *__restrict__ x, uint16_t *__restrict__ xp,
                                                  int t, int H, const uint16_t *__restrict__ g,
                                                  float *__restrict__ sigma) {
  const int lane = threadIdx.x & 31;
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
  const uint4 *gr = reinterpret_cast<const uint4 *>(g);
  uint4 *pr = reinterpret_cast<uint4 *>(xp + (size_t)t * H);
  const int cpr = H / 8;  // <= 256
  uint4 xv[8], gv[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int ch = lane + 32 * c;
    xv[c] = ch < cpr ? __ldg(xr + ch) : make_uint4(0, 0, 0, 0);
    gv[c] = (g && ch < cpr) ? __ldg(gr + ch) : make_uint4(0, 0, 0, 0);
  }
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int ch = lane + 32 * c;
    if (ch >= cpr) break;
    const uint4 v = xv[c];
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    pr[ch] = o;
    const uint32_t xx[4] = {v.x, v.y, v.z, v.w}, gg[4] = {gv[c].x, gv[c].y, gv[c].z, gv[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(xx[i] << 16), __uint_as_float(gg[i] << 16), acc);
      acc = fmaf(__uint_as_float(xx[i] & 0xFFFF0000u), __uint_as_float(gg[i] & 0xFFFF0000u), acc);
    }
  }
  if (g) {
    acc = seg_sum<32>(acc);
    if (lane == 0) sigma[t] = 1.0f / (1.0f + expf(-acc));
  }
}

struct TopkArgs {
  const float *logits;  // [nsplit][T][E] partials
  const float *bias;    // [E] or NULL
  int nsplit;
  int T, E, k;
  int32_t *idx;
  float *p;
  int32_t *ctab;  // [gridDim.x][E]: the block's selection count per expert
  int32_t *out_idx;
  float *out_w;
  // the token rows in the permuted K order, and the shared gate (g NULL: no shared expert)
  const uint16_t *x;
  uint16_t *xp;
  const uint16_t *g;
  float *sigma;
  int H;
};

// One warp per token: logits = fixed-order sum of the router GEMM's K-split partials plus
// the per-expert offsets, held in registers (EC per lane); the k largest (logit desc, index
// asc); softmax over the k.  The block's selections are counted per expert in shared memory
// and written to the count table (every expert, zeros included): the scan and the placement
// turn the counts into block prefixes, so the bucketing is stable without a global atomic per
// selection (a skewed router sends most tokens to the same experts).  The warp also writes
// its token's row in the permuted K order for the gate/up GEMM and the shared gate.
constexpr int kTopkTokens = 16;  // tokens (warps) per block
constexpr int kMaxTopK = 16;     // the API's top-k limit
template <int EC>
__global__ void __launch_bounds__(32 * kTopkTokens) topk_prefill_kernel(TopkArgs a) {
  pdl_enter();
  __shared__ int s_cnt[32 * EC];
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkTokens + (threadIdx.x >> 5);
  if (t < a.T) permute_token_row(a.x, a.xp, t, a.H, a.g, a.sigma);
  if (t < a.T) {
  // every partial logit of the lane is loaded before any is summed (the split count is at most
  // kRouterSplit(H) = 4), then the partials are summed in split order
  float lv[EC];
#pragma unroll
  for (int j = 0; j < EC; ++j) {
    const int e = lane + 32 * j;
    float pv[4];
#pragma unroll
    for (int sp = 0; sp < 4; ++sp)
      pv[sp] = (sp < a.nsplit && e < a.E) ? __ldcg(a.logits + ((size_t)sp * a.T + t) * a.E + e) : 0.f;
    float v = -INFINITY;
    if (e < a.E) {
      v = 0.f;
#pragma unroll
      for (int sp = 0; sp < 4; ++sp)
        if (sp < a.nsplit) v += pv[sp];
      if (a.bias) v += a.bias[e];
      v = cand(v);
    }
    lv[j] = v;
  }
  uint32_t key[EC];
#pragma unroll
  for (int j = 0; j < EC; ++j) key[j] = lane + 32 * j < a.E ? f2key(lv[j]) : 0u;
  float myv;  // lane i < k keeps selection i
  int mye;
  warp_topk_keys<EC>(key, a.k, mye, myv);
  // softmax over the k selected logits, one selection per lane
  const float v0 = __shfl_sync(0xffffffffu, myv, 0);
  const float ex = lane < a.k ? expf(myv - v0) : 0.f;
  const float denom = seg_sum<32>(ex);
  if (lane < a.k) {
    const float pi = ex / denom;
    a.idx[t * a.k + lane] = mye;
    a.p[t * a.k + lane] = pi;
    if (a.out_idx) a.out_idx[t * a.k + lane] = mye;
    if (a.out_w) a.out_w[t * a.k + lane] = pi;
    atomicAdd(s_cnt + mye, 1);
  }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x)
    a.ctab[(size_t)blockIdx.x * a.E + e] = s_cnt[e];
}

// Rows of the block-prefix table the scan writes: every kPrefixStride-th top-k block; the
// placement adds the counts of the (< kPrefixStride) blocks between.
constexpr int kPrefixStride = 8;
// Tiles whose expert the scan looks up in a shared-memory table (more: binary search).
constexpr int kTileTable = 4096;

struct ScanArgs {
  const int32_t *ctab;  // [nb][E] block counts
  int32_t *cpre;        // [ceil(nb / kPrefixStride)][E] exclusive prefix over the blocks before
                        // every kPrefixStride-th block
  int nb;               // top-k blocks
  int32_t *offsets;  // [E+2]
  int4 *items_gu, *items_dn;
  int32_t *hdr;
  int T, E, k, has_shared, mt_gu, mt_dn;
};

// Single block: the expert totals and, at every kPrefixStride-th top-k block, each expert's
// exclusive prefix over the blocks before it (the placement finishes the prefix of the blocks
// between); the totals give the per-expert offsets, then the GEMM work lists (each tile's
// expert from a table in shared memory).
__global__ void __launch_bounds__(1024) scan_items_kernel(ScanArgs a) {
  pdl_enter();
  __shared__ int s_cnt[1025];
  __shared__ int s_off[1026];
  __shared__ int s_nt[1025];
  __shared__ int s_ibase[1026];
  const int nexp = a.E + a.has_shared;
  // G = blockDim / E thread groups; group g takes the blocks [g*seg, g*seg + seg) of every
  // expert (thread e of the group: expert e, so a warp reads consecutive experts of a block
  // row): the group's sums meet in shared memory, then each group writes the prefixes of its
  // segment's every kPrefixStride-th block.  E > blockDim takes several passes with one group.
  __shared__ int s_gsum[1024];
  const int G = max(1, (int)blockDim.x / a.E);
  const int seg = ((a.nb + G - 1) / G + kPrefixStride - 1) / kPrefixStride * kPrefixStride;
  for (int e0 = 0; e0 < a.E; e0 += (int)blockDim.x / G) {
    const int g = (int)threadIdx.x / (a.E < (int)blockDim.x ? a.E : (int)blockDim.x);
    const int e = e0 + (int)threadIdx.x % (a.E < (int)blockDim.x ? a.E : (int)blockDim.x);
    const bool live = g < G && e < a.E;
    const int b0 = min(a.nb, g * seg), b1 = min(a.nb, b0 + seg);
    // A segment (a multiple of kPrefixStride blocks, so its prefix rows sit at fixed offsets)
    // is read once: its sum, and the partial sums before its prefix rows -- in registers for a
    // segment of at most kSegV blocks, else written to the prefix table and completed after
    // the groups' sums are known.
    constexpr int kSegV = 32;
    int ploc[kSegV / kPrefixStride];
    int sum = 0;
    if (live) {
      if (seg <= kSegV) {
        int v[kSegV];
#pragma unroll
        for (int q = 0; q < kSegV; ++q) v[q] = b0 + q < b1 ? a.ctab[(size_t)(b0 + q) * a.E + e] : 0;
#pragma unroll
        for (int q = 0; q < kSegV; ++q) {
          if (q % kPrefixStride == 0) ploc[q / kPrefixStride] = sum;
          sum += v[q];
        }
      } else {
        for (int c = b0; c < b1; c += kPrefixStride) {
          int u[kPrefixStride];
#pragma unroll
          for (int q = 0; q < kPrefixStride; ++q) u[q] = c + q < b1 ? a.ctab[(size_t)(c + q) * a.E + e] : 0;
          a.cpre[(size_t)(c / kPrefixStride) * a.E + e] = sum;
#pragma unroll
          for (int q = 0; q < kPrefixStride; ++q) sum += u[q];
        }
      }
      s_gsum[g * (a.E < (int)blockDim.x ? a.E : (int)blockDim.x) + (e - e0)] = sum;
    }
    __syncthreads();
    if (live) {
      const int w = a.E < (int)blockDim.x ? a.E : (int)blockDim.x;
      int run = 0, tot = 0;
      for (int h = 0; h < G; ++h) {
        const int gs = s_gsum[h * w + (e - e0)];
        if (h < g) run += gs;
        tot += gs;
      }
      if (seg <= kSegV) {
#pragma unroll
        for (int m = 0; m < kSegV / kPrefixStride; ++m)
          if (b0 + m * kPrefixStride < b1)
            a.cpre[(size_t)(b0 / kPrefixStride + m) * a.E + e] = run + ploc[m];
      } else {
        for (int c = b0; c < b1; c += kPrefixStride) a.cpre[(size_t)(c / kPrefixStride) * a.E + e] += run;
      }
      if (g == 0) s_cnt[e] = min(tot, a.T);
    }
    __syncthreads();
  }
  if (a.has_shared && threadIdx.x == 0) s_cnt[a.E] = a.T;
  __syncthreads();
  for (int e = threadIdx.x; e < nexp; e += blockDim.x) s_nt[e] = (s_cnt[e] + kBN - 1) / kBN;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (nexp + 31) / 32;
    const int lo = lane * per, hi = min(nexp, lo + per);
    int sc = 0, sn = 0;
    for (int e = lo; e < hi; ++e) {
      sc += s_cnt[e];
      sn += s_nt[e];
    }
    int tc_, tn_;
    int rc = warp_excl_scan(sc, &tc_);
    int rn = warp_excl_scan(sn, &tn_);
    for (int e = lo; e < hi; ++e) {
      s_off[e] = rc;
      s_ibase[e] = rn;
      rc += s_cnt[e];
      rn += s_nt[e];
    }
    if (lane == 31) {
      s_off[nexp] = rc;
      s_ibase[nexp] = rn;
    }
  }
  __syncthreads();
  const int ntiles = s_ibase[nexp];
  for (int e = threadIdx.x; e < nexp; e += blockDim.x) a.offsets[e] = s_off[e];
  // one thread per work item: its tile's expert from the table (each expert writes its tiles'
  // entries), or by binary search of the tile bases when the tiles outnumber the table
  __shared__ int16_t s_t2e[kTileTable];
  const bool table = ntiles <= kTileTable && blockDim.x * 4 >= kTileTable;
  if (table) {
    for (int e = threadIdx.x; e < nexp; e += blockDim.x)
      for (int t = s_ibase[e]; t < s_ibase[e + 1]; ++t) s_t2e[t] = (int16_t)e;
  }
  __syncthreads();
  // Work order: the tiles of more than 16 tokens first, then those of at most 16 (tile order
  // within each part), so that the last, partial round of the round-robin hand-out of items
  // (item i to block i mod grid) holds small tiles.  Thread j takes tiles 4j .. 4j+3; a block
  // scan of the large-tile counts gives every tile its place.
  __shared__ int16_t s_ord[kTileTable];
  __shared__ int s_wbig[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  bool big[4] = {false, false, false, false};
  int nbig = 0, pre = 0;
  if (table) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * (int)threadIdx.x + i;
      if (t < ntiles) {
        const int e = s_t2e[t], nt = t - s_ibase[e];
        big[i] = s_cnt[e] - nt * kBN > 16;
      }
      nbig += big[i];
    }
    int wt;
    pre = warp_excl_scan(nbig, &wt);
    if (lane == 0) s_wbig[warp] = wt;
  }
  __syncthreads();
  if (table && warp == 0) {
    int tot;
    const int v = lane < (int)blockDim.x / 32 ? s_wbig[lane] : 0;
    const int ex = warp_excl_scan(v, &tot);
    s_wbig[lane] = ex;
    if (lane == 0) s_wbig[32] = tot;
  }
  __syncthreads();
  if (table) {
    int pb = s_wbig[warp] + pre;  // large tiles before this thread's first tile
    const int nbig_all = s_wbig[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * (int)threadIdx.x + i;
      if (t < ntiles) s_ord[big[i] ? pb : nbig_all + t - pb] = (int16_t)t;
      pb += big[i];
    }
  }
  __syncthreads();
  const int ngu = ntiles * a.mt_gu, nitems = ngu + ntiles * a.mt_dn;
  for (int q = threadIdx.x; q < nitems; q += blockDim.x) {
    const bool gu = q < ngu;
    const int mts = gu ? a.mt_gu : a.mt_dn, qi = gu ? q : q - ngu;
    const int tile = table ? s_ord[qi / mts] : qi / mts, mt = qi % mts;
    int lo = 0;  // last e with s_ibase[e] <= tile
    if (table) {
      lo = s_t2e[tile];
    } else {
      int hi = nexp - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_ibase[mid] <= tile) lo = mid; else hi = mid - 1;
      }
    }
    const int e = lo, nt = tile - s_ibase[e];
    const int4 item = make_int4(e, s_off[e] + nt * kBN, min(kBN, s_cnt[e] - nt * kBN), mt);
    if (gu) a.items_gu[qi] = item; else a.items_dn[qi] = item;
  }
  if (threadIdx.x == 0) {
    a.offsets[nexp] = s_off[nexp];
    a.hdr[kHdrItemsGU] = ntiles * a.mt_gu;
    a.hdr[kHdrItemsDN] = ntiles * a.mt_dn;
  }
}

struct PermArgs {
  const int32_t *idx;
  const float *p;
  const float *sigma;
  const int32_t *offsets;
  const int32_t *ctab;  // [nb][E] block counts
  const int32_t *cpre;  // [ceil(nb / kPrefixStride)][E] prefixes at every kPrefixStride-th block
  int nb;
  int32_t *perm;
  float *pw;
  int32_t *inv;
  int T, E, k, has_shared;
};

// Stable bucketing (token order within an expert): block b places the selections of the
// tokens of top-k block b; a selection's row is its expert's offset, plus the selections of
// that expert in earlier blocks (the scan's prefix at the last kPrefixStride-th block, plus the
// counts of the blocks from there to b), plus its rank among the block's earlier selections
// of the expert.  The blocks past them write the shared expert's rows,
// every token in order.
constexpr int kPlaceThreads = kTopkTokens * kMaxTopK;
__global__ void __launch_bounds__(kPlaceThreads) place_kernel(PermArgs a) {
  pdl_enter();
  __shared__ int s_e[kPlaceThreads];
  const int kk = a.k + 1;
  if ((int)blockIdx.x >= a.nb) {  // shared expert
    const int t = ((int)blockIdx.x - a.nb) * kPlaceThreads + (int)threadIdx.x;
    if (t < a.T) {
      const int pos = a.offsets[a.E] + t;
      a.perm[pos] = t;
      a.pw[pos] = a.sigma[t];
      a.inv[t * kk + a.k] = pos;
    }
    return;
  }
  const int n = a.T * a.k, j0 = blockIdx.x * kTopkTokens * a.k;
  const int nb_sel = min(n - j0, kTopkTokens * a.k);
  const int q = threadIdx.x;
  const int e = q < nb_sel ? a.idx[j0 + q] : -1;
  s_e[q] = e;
  __syncthreads();
  if (q < nb_sel) {
    int rank = 0;
    for (int r = 0; r < q; ++r) rank += s_e[r] == e;
    const int j = j0 + q, t = j / a.k, i = j - t * a.k;
    const int b = blockIdx.x, bc = b - b % kPrefixStride;
    int before = a.cpre[(size_t)(b / kPrefixStride) * a.E + e];
#pragma unroll
    for (int i = 0; i < kPrefixStride - 1; ++i)  // all loads in flight together
      if (bc + i < b) before += a.ctab[(size_t)(bc + i) * a.E + e];
    const int pos = a.offsets[e] + before + rank;
    a.perm[pos] = t;
    a.pw[pos] = a.p[j];
    a.inv[t * kk + i] = pos;
  }
}

// Drop a 128-byte line from L2 without writing it back (its contents become undefined).
__device__ __forceinline__ void l2_discard(const void *p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// y[t][8c..8c+7] = sum over t's slots of o[inv[t][slot]] (fixed slot order).  All of a
// chunk's slot rows are requested before any is summed (NS >= the slot count).
// The chunk's two large intermediates die here and are dropped from L2 without write-back:
// the o lines a warp has read, and (grid-stride) h, whose last reader was the down GEMM.
// Left dirty, ~0.1 GB of dead data would be written back to HBM inside whatever kernels
// run next (measured: the LM head after a step's decode layers, 43 -> 39 us).
template <int NS>
__global__ void combine_kernel(const uint16_t *__restrict__ o, const int32_t *__restrict__ inv,
                               uint16_t *__restrict__ y, int T, int H, int nslots, int kk,
                               const char *dead_h, size_t dead_h_bytes) {
  pdl_enter();
  const int cpr = H / 8;
  {
    const size_t nthr = (size_t)gridDim.x * blockDim.x, tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (size_t off = tid * 128; off < dead_h_bytes; off += nthr * 128) l2_discard(dead_h + off);
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * cpr; i += gridDim.x * blockDim.x) {
    const int t = i / cpr, c = i % cpr;
    int pos[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) pos[s] = s < nslots ? __ldg(inv + t * kk + s) : 0;
    uint4 v[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s)
      v[s] = s < nslots ? __ldcg(reinterpret_cast<const uint4 *>(o + (size_t)pos[s] * H) + c)
                        : make_uint4(0, 0, 0, 0);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      if (s >= nslots) break;
      const uint32_t w[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(w[q] << 16);
        acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    uint4 r;
    r.x = (uint32_t)f2bf16_rne(acc[0]) | ((uint32_t)f2bf16_rne(acc[1]) << 16);
    r.y = (uint32_t)f2bf16_rne(acc[2]) | ((uint32_t)f2bf16_rne(acc[3]) << 16);
    r.z = (uint32_t)f2bf16_rne(acc[4]) | ((uint32_t)f2bf16_rne(acc[5]) << 16);
    r.w = (uint32_t)f2bf16_rne(acc[6]) | ((uint32_t)f2bf16_rne(acc[7]) << 16);
    reinterpret_cast<uint4 *>(y + (size_t)t * H)[c] = r;
    // every lane of the line's 8 chunks has its values (used above): drop the slot lines
    __syncwarp(__activemask());
    if ((c & 7) == 0) {
#pragma unroll
      for (int s = 0; s < NS; ++s)
        if (s < nslots) l2_discard(o + (size_t)pos[s] * H + 8 * c);
    }
  }
}

// -------------------------------------------------------------------------------------
// affine 8-bit parts
// -------------------------------------------------------------------------------------

// Row e of the 8-bit router in its exact bf16 form, A[e] = [hi | lo | b | b | b | 0...]:
// s*q (bf16 s times a byte code) has at most 16 significant bits, so hi = bf16(s*q) and
// lo = s*q - hi are both exact in bf16.
__global__ void router8_prep_a_kernel(lily_q4_mat r8, int E, int H, int Kr, uint16_t *__restrict__ A) {
  pdl_enter();
  const int e = blockIdx.x;
  if (e >= E) return;
  const int G = H / 64;
  const uint8_t *codes = reinterpret_cast<const uint8_t *>(r8.w) + (size_t)e * H;  // byte k = code k
  uint16_t *row = A + (size_t)e * Kr;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    const float w = bf16f(r8.s[(size_t)e * G + k / 64]) * (float)codes[k];  // exact
    const uint16_t hi = f2bf16_rne(w);
    row[k] = hi;
    row[H + k] = f2bf16_rne(w - bf16f(hi));  // exact
  }
  for (int j = threadIdx.x; j < Kr - 2 * H; j += blockDim.x)
    row[2 * H + j] = j < 3 * G ? r8.b[(size_t)e * G + j % G] : (uint16_t)0;
}

// Row t of the router GEMM's token operand to match, B[t] = [x | x | X_hi | X_mid | X_lo | 0...]:
// X_g = the sum of group g of x (fp32, a fixed order), split exactly into three bf16 parts,
// so A . B = sum_k (s*q)_k x_k + sum_g b_g X_g with every product exact.
__global__ void router8_prep_b_kernel(const uint16_t *__restrict__ x, int H, int Kr, uint16_t *__restrict__ B) {
  pdl_enter();
  const int t = blockIdx.x;
  const int G = H / 64;
  const uint16_t *xr = x + (size_t)t * H;
  uint16_t *row = B + (size_t)t * Kr;
  for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr) + c);
    reinterpret_cast<uint4 *>(row)[c] = v;
    reinterpret_cast<uint4 *>(row + H)[c] = v;
  }
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    float X = 0.f;
    for (int k = 0; k < 64; ++k) X += bf16f(xr[64 * g + k]);
    const uint16_t h1 = f2bf16_rne(X);
    const float r1 = X - bf16f(h1);
    const uint16_t h2 = f2bf16_rne(r1);
    row[2 * H + g] = h1;
    row[2 * H + G + g] = h2;
    row[2 * H + 2 * G + g] = f2bf16_rne(r1 - bf16f(h2));
  }
  for (int j = 2 * H + 3 * G + threadIdx.x; j < Kr; j += blockDim.x) row[j] = 0;
}

// An affine 8-bit matrix [N][K] (four byte codes per uint32, lowest byte first) as an affine
// 4-bit matrix [N][2K]: q = lo + 16 hi gives
//     s*q + b = (s*lo + (b + 128 s)) + (16 s * hi - 128 s),
// so row n becomes the low nibbles with scales s and biases b + 128 s, then the high nibbles
// with scales 16 s and biases -128 s (both exact in bf16).  The split is centred so that both
// halves stay about as small as the weight itself (b is near -128 s): the tensor-core path
// rounds each dequantised half to bf16, and uncentred halves of several times the weight's
// size would multiply that rounding.  b + 128 s is rounded once to bf16 (it is small).
struct Q8ToQ4x2 {
  lily_q4_mat src;
  int N, K;
  uint32_t *w;  // [N][2K/8]
  uint16_t *s;  // [N][2K/64]
  uint16_t *b;
};
__global__ void q8_to_q4x2_kernel(Q8ToQ4x2 a) {
  pdl_enter();
  const int words = a.K / 8, G = a.K / 64;
  const size_t nw = (size_t)a.N * words, ng = (size_t)a.N * G;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw + ng;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < nw) {
      const size_t n = i / words;
      const int m = (int)(i % words);
      const uint2 c = __ldg(reinterpret_cast<const uint2 *>(a.src.w + n * (a.K / 4)) + m);  // codes 8m..8m+7
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= ((c.x >> (8 * j)) & 0xFu) << (4 * j);
        hi |= ((c.x >> (8 * j + 4)) & 0xFu) << (4 * j);
        lo |= ((c.y >> (8 * j)) & 0xFu) << (4 * j + 16);
        hi |= ((c.y >> (8 * j + 4)) & 0xFu) << (4 * j + 16);
      }
      a.w[n * 2 * words + m] = lo;
      a.w[n * 2 * words + words + m] = hi;
    } else {
      const size_t j = i - nw, n = j / G;
      const int g = (int)(j % G);
      const uint16_t sv = a.src.s[n * G + g];
      const float sf = bf16f(sv);
      a.s[n * 2 * G + g] = sv;
      a.b[n * 2 * G + g] = f2bf16_rne(bf16f(a.src.b[n * G + g]) + 128.0f * sf);
      a.s[n * 2 * G + G + g] = f2bf16_rne(16.0f * sf);
      a.b[n * 2 * G + G + g] = f2bf16_rne(-128.0f * sf);
    }
  }
}

// The 4-bit form of an 8-bit shared expert in the workspace: gate, up [I][2H], down [H][2I],
// each as codes, scales, biases.
struct Sh8Ptrs {
  lily_q4_mat gate, up, down;
};
static Sh8Ptrs sh8_ptrs(char *base, int H, int I) {
  Sh8Ptrs p;
  char *c = base;
  auto mat = [&](int N, int K) {
    lily_q4_mat m;
    m.w = reinterpret_cast<const uint32_t *>(c);
    c += align_up((size_t)N * (2 * K / 8) * 4);
    m.s = reinterpret_cast<const uint16_t *>(c);
    c += align_up((size_t)N * (2 * K / 64) * 2);
    m.b = reinterpret_cast<const uint16_t *>(c);
    c += align_up((size_t)N * (2 * K / 64) * 2);
    return m;
  };
  p.gate = mat(I, H);
  p.up = mat(I, H);
  p.down = mat(H, I);
  return p;
}
static size_t sh8_bytes(int H, int I) {
  auto one = [](int N, int K) {
    return align_up((size_t)N * (2 * K / 8) * 4) + 2 * align_up((size_t)N * (2 * K / 64) * 2);
  };
  return 2 * one(I, H) + one(H, I);
}

static int q8_to_q4x2(const lily_q4_mat &src, int N, int K, const lily_q4_mat &dst, cudaStream_t st) {
  Q8ToQ4x2 a{src, N, K, const_cast<uint32_t *>(dst.w), const_cast<uint16_t *>(dst.s),
             const_cast<uint16_t *>(dst.b)};
  const size_t n = (size_t)N * (K / 8) + (size_t)N * (K / 64);
  const int sms = sm_count() > 0 ? sm_count() : 1;
  const size_t want = (n + 255) / 256;
  if (launch_pdl(q8_to_q4x2_kernel, dim3((unsigned)(want < (size_t)4 * sms ? want : (size_t)4 * sms)),
                 dim3(256), 0, st, a) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  return check_launch();
}

static bool router8(const lily_q4_moe_layer &L) { return L.router_bits == 8; }
static bool shared8(const lily_q4_moe_layer &L) { return L.has_shared && L.shared_bits == 8; }

int prefill_launch_count(const lily_q4_moe_layer &L) {
  return 7 + (router8(L) ? 2 : 0) + (shared8(L) ? 3 : 0);
}

// -------------------------------------------------------------------------------------
// host side
// -------------------------------------------------------------------------------------

PrefillWsLayout prefill_ws_layout(const lily_q4_moe_layer &L, int T) {
  PrefillWsLayout l{};
  l.T = T;
  l.E = L.n_experts;
  l.k = L.top_k;
  l.I = L.inter;
  l.H = L.hidden;
  l.P = T * L.top_k + (L.has_shared ? T : 0);
  const int nexp = l.E + (L.has_shared ? 1 : 0);
  const int tiles = nexp + (l.P + kBN - 1) / kBN;
  const int mt_gu = (l.I + kBM - 1) / kBM, mt_dn = (l.H + kBM - 1) / kBM;
  l.max_items = tiles * (mt_gu + mt_dn);
  size_t off = align_up(kHdrWords * sizeof(int32_t));
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  l.off_logits = take(sizeof(float) * (size_t)kRouterSplit(l.H) * T * l.E);
  l.off_idx = take(sizeof(int32_t) * (size_t)T * l.k);
  l.off_p = take(sizeof(float) * (size_t)T * l.k);
  l.off_sigma = take(sizeof(float) * (size_t)T);
  const size_t nbk = (size_t)((T + kTopkTokens - 1) / kTopkTokens);
  l.off_ctab = take(sizeof(int32_t) * (size_t)l.E * nbk);
  l.off_cpre = take(sizeof(int32_t) * (size_t)l.E * ((nbk + kPrefixStride - 1) / kPrefixStride));
  l.off_offsets = take(sizeof(int32_t) * (size_t)(l.E + 2));
  l.off_perm = take(sizeof(int32_t) * (size_t)l.P);
  l.off_pw = take(sizeof(float) * (size_t)l.P);
  l.off_inv = take(sizeof(int32_t) * (size_t)T * (l.k + 1));
  l.off_items = take(sizeof(int4) * (size_t)l.max_items);
  l.off_xperm = take(sizeof(uint16_t) * (size_t)T * l.H);
  l.off_h = take(sizeof(uint16_t) * (size_t)l.P * l.I);
  l.off_o = take(sizeof(uint16_t) * (size_t)l.P * l.H);
  // the router GEMM's K is split into kRouterSplit(H) parts of whole 64-wide blocks
  const int kq = 64 * kRouterSplit(l.H);
  l.Kr = router8(L) ? (2 * l.H + 3 * (l.H / 64) + kq - 1) / kq * kq : l.H;
  l.off_r8a = router8(L) ? take(sizeof(uint16_t) * (size_t)l.E * l.Kr) : 0;
  l.off_r8b = router8(L) ? take(sizeof(uint16_t) * (size_t)T * l.Kr) : 0;
  l.off_sh8 = shared8(L) ? take(sh8_bytes(l.H, l.I)) : 0;
  l.total = off;
  return l;
}

template <int MODE, int KG, int RT = 2>
static int launch_gemm_kg(const GemmArgs &a, int grid, cudaStream_t st) {
  const int bytes = Cfg<MODE, RT>::BYTES;
  // set on every call: cheap, and correct for whichever device is current
  if (cudaFuncSetAttribute(grouped_gemm_kernel<MODE, KG, RT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  if (launch_pdl(grouped_gemm_kernel<MODE, KG, RT>, dim3(grid), dim3(Cfg<MODE, RT>::THREADS),
                 (size_t)bytes, st, a) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  return check_launch();
}

static bool aligned32(const void *p) { return ((uintptr_t)p & 31) == 0; }

// KG = k-blocks per register group of the weight producers (K/64 is a power of two >= 2):
// 8 for down; 4 for gate/up, whose producers hold both matrices' rows (a group of 8 k-blocks
// there does not fit the register budget).  Gate/up takes one producer thread per row when
// all four of its code arrays are 32-byte aligned (row and expert strides are multiples of
// 32 bytes, so every row's k-block is then too).
template <int MODE>
static int launch_gemm(const GemmArgs &a, int grid, cudaStream_t st) {
  const int G = a.K / 64;
  if constexpr (MODE == kRouter) {
    return launch_gemm_kg<MODE, 8>(a, grid, st);
  } else if constexpr (MODE == kGateUp) {
    if (G >= 4) {
      const bool al = aligned32(a.a0.w) && aligned32(a.a1.w) &&
                      (!a.sh0.w || (aligned32(a.sh0.w) && aligned32(a.sh1.w)));
      return al ? launch_gemm_kg<MODE, 4, 1>(a, grid, st) : launch_gemm_kg<MODE, 4, 2>(a, grid, st);
    }
    return launch_gemm_kg<MODE, 2>(a, grid, st);
  } else {
    if (G >= 8) return launch_gemm_kg<MODE, 8>(a, grid, st);
    if (G == 4) return launch_gemm_kg<MODE, 4>(a, grid, st);
    return launch_gemm_kg<MODE, 2>(a, grid, st);
  }
}

int launch_moe_prefill(const lily_q4_moe_layer &L, const uint16_t *x, int T, uint16_t *y,
                       int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t st) {
  if (L.hidden < 128 || L.inter < 128) return LILY_Q4_ERR_UNSUPPORTED;
  const PrefillWsLayout l = prefill_ws_layout(L, T);
  char *b = static_cast<char *>(ws);
  int32_t *hdr = reinterpret_cast<int32_t *>(b);
  float *logits = reinterpret_cast<float *>(b + l.off_logits);
  int32_t *idx = reinterpret_cast<int32_t *>(b + l.off_idx);
  float *p = reinterpret_cast<float *>(b + l.off_p);
  float *sigma = reinterpret_cast<float *>(b + l.off_sigma);
  int32_t *ctab = reinterpret_cast<int32_t *>(b + l.off_ctab);
  int32_t *cpre = reinterpret_cast<int32_t *>(b + l.off_cpre);
  const int nbk = (T + kTopkTokens - 1) / kTopkTokens;  // top-k blocks
  int32_t *offsets = reinterpret_cast<int32_t *>(b + l.off_offsets);
  int32_t *perm = reinterpret_cast<int32_t *>(b + l.off_perm);
  float *pw = reinterpret_cast<float *>(b + l.off_pw);
  int32_t *inv = reinterpret_cast<int32_t *>(b + l.off_inv);
  int4 *items = reinterpret_cast<int4 *>(b + l.off_items);
  uint16_t *xperm = reinterpret_cast<uint16_t *>(b + l.off_xperm);
  uint16_t *h = reinterpret_cast<uint16_t *>(b + l.off_h);
  uint16_t *o = reinterpret_cast<uint16_t *>(b + l.off_o);
  const int sms = sm_count() > 0 ? sm_count() : 1;
  const int H = L.hidden, I = L.inter, E = L.n_experts, k = L.top_k;
  const int nexp = E + L.has_shared;
  const int mt_gu = (I + kBM - 1) / kBM, mt_dn = (H + kBM - 1) / kBM;
  const int tiles = nexp + (l.P + kBN - 1) / kBN;
  int4 *items_gu = items;
  int4 *items_dn = items + (size_t)tiles * mt_gu;

  // Every launch below is a programmatic dependent of the one before it (launch_pdl): set-up
  // overlaps the previous kernel's tail, and each kernel waits for that kernel's completion
  // before it reads or writes anything the chain shares.
  // router GEMM (an 8-bit router in its exact bf16 form, the token rows widened to match)
  const uint16_t *ra_a = L.router, *ra_b = x;
  if (router8(L)) {
    uint16_t *A = reinterpret_cast<uint16_t *>(b + l.off_r8a);
    uint16_t *B = reinterpret_cast<uint16_t *>(b + l.off_r8b);
    if (launch_pdl(router8_prep_a_kernel, dim3(E), dim3(256), 0, st, L.router_q8, E, H, l.Kr, A) !=
            cudaSuccess ||
        launch_pdl(router8_prep_b_kernel, dim3(T), dim3(256), 0, st, static_cast<const uint16_t *>(x),
                   H, l.Kr, B) != cudaSuccess)
      return LILY_Q4_ERR_CUDA;
    ra_a = A;
    ra_b = B;
  }
  GemmArgs ra{};
  ra.a_bf16 = ra_a;
  ra.a_rows = E;
  ra.K = l.Kr;
  ra.E = E;
  ra.b_src = ra_b;
  ra.mt_static = (E + kBM - 1) / kBM;
  ra.ksplit = kRouterSplit(H);
  ra.ksh = 1;
  ra.n_items_static = ra.mt_static * ((T + kBN - 1) / kBN) * ra.ksplit;
  ra.T = T;
  ra.logits = logits;  // partial logits [ksplit][T][E]
  ra.hdr = hdr;
  int rc = launch_gemm<kRouter>(ra, ra.n_items_static < sms ? ra.n_items_static : sms, st);
  if (rc != LILY_Q4_OK) return rc;

  const uint16_t *sgate = L.has_shared ? L.shared_gate : nullptr;
  TopkArgs ta{logits, L.router_bias, ra.ksplit, T, E, k, idx, p, ctab, topk_idx, topk_w,
              x, xperm, sgate, sigma, H};
  const dim3 tk_grid(nbk), tk_block(32 * kTopkTokens);
  cudaError_t ce = E <= 256   ? launch_pdl(topk_prefill_kernel<8>, tk_grid, tk_block, 0, st, ta)
                   : E <= 512 ? launch_pdl(topk_prefill_kernel<16>, tk_grid, tk_block, 0, st, ta)
                              : launch_pdl(topk_prefill_kernel<32>, tk_grid, tk_block, 0, st, ta);
  if (ce != cudaSuccess) return LILY_Q4_ERR_CUDA;

  ScanArgs sa{ctab, cpre, nbk, offsets, items_gu, items_dn, hdr, T, E, k, L.has_shared, mt_gu, mt_dn};
  if (launch_pdl(scan_items_kernel, dim3(1), dim3(1024), 0, st, sa) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;

  PermArgs pa{idx, p, sigma, offsets, ctab, cpre, nbk, perm, pw, inv, T, E, k, L.has_shared};
  const int nplace = nbk + (L.has_shared ? (T + kPlaceThreads - 1) / kPlaceThreads : 0);
  if (launch_pdl(place_kernel, dim3(nplace), dim3(kPlaceThreads), 0, st, pa) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;

  // an 8-bit shared expert as 4-bit codes of twice the width (its tiles run with K doubled)
  lily_q4_mat shg = L.sh_gate, shu = L.sh_up, shd = L.sh_down;
  const int ksh = shared8(L) ? 2 : 1;
  if (shared8(L)) {
    const Sh8Ptrs sp = sh8_ptrs(b + l.off_sh8, H, I);
    if ((rc = q8_to_q4x2(L.sh_gate, I, H, sp.gate, st)) != LILY_Q4_OK) return rc;
    if ((rc = q8_to_q4x2(L.sh_up, I, H, sp.up, st)) != LILY_Q4_OK) return rc;
    if ((rc = q8_to_q4x2(L.sh_down, H, I, sp.down, st)) != LILY_Q4_OK) return rc;
    shg = sp.gate;
    shu = sp.up;
    shd = sp.down;
  }
  GemmArgs ga{};
  ga.a0 = L.gate;
  ga.a1 = L.up;
  ga.sh0 = shg;
  ga.sh1 = shu;
  ga.ksh = ksh;
  ga.a_rows = I;
  ga.K = H;
  ga.E = E;
  ga.b_src = xperm;
  ga.perm = perm;
  ga.items = items_gu;
  ga.n_items_ptr = hdr + kHdrItemsGU;
  ga.h_out = h;
  ga.pw = pw;
  ga.P = l.P;
  ga.hdr = hdr;
  rc = launch_gemm<kGateUp>(ga, sms, st);
  if (rc != LILY_Q4_OK) return rc;

  GemmArgs da{};
  da.a0 = L.down;
  da.sh0 = shd;
  da.ksh = ksh;
  da.a_rows = H;
  da.K = I;
  da.E = E;
  da.b_src = h;
  da.P = l.P;
  da.items = items_dn;
  da.n_items_ptr = hdr + kHdrItemsDN;
  da.o_out = o;
  da.o_ld = H;
  da.hdr = hdr;
  rc = launch_gemm<kDown>(da, sms, st);
  if (rc != LILY_Q4_OK) return rc;

  const int cch = T * H / 8;
  const dim3 cb_grid((cch + 255) / 256 < 8 * sms ? (cch + 255) / 256 : 8 * sms), cb_block(256);
  const int nslots = k + L.has_shared;
  const uint16_t *oc = o;
  // h is dead after the down GEMM (the combine drops it, and the o lines it reads, from L2)
  const char *dead_h = b + l.off_h;
  const size_t dead_h_bytes = (sizeof(uint16_t) * (size_t)l.P * l.I) & ~(size_t)127;
  if ((nslots <= 9 ? launch_pdl(combine_kernel<9>, cb_grid, cb_block, 0, st, oc, inv, y, T, H, nslots, k + 1,
                                dead_h, dead_h_bytes)
                   : launch_pdl(combine_kernel<17>, cb_grid, cb_block, 0, st, oc, inv, y, T, H, nslots,
                                k + 1, dead_h, dead_h_bytes)) != cudaSuccess)
    return LILY_Q4_ERR_CUDA;
  return check_launch();
}

}  // namespace lq4
