// Device helpers shared by the kernels of the Q4 library (not by the oracle).
//
// In-register dequantisation of the MLX-affine 4-bit format with groups of 64 weights
// (Lily README, first paragraph and "Requirements").  For one group of 64
// weights with scale s and bias b:
//
//     sum_k (s*q_k + b) x_k  =  s * sum_k q_k x_k  +  b * sum_k x_k
//
// so the codes are multiplied with x as small integers and s, b are applied once
// per group.  Codes become floats with the bf16 magic-number trick: OR-ing a
// nibble into the low mantissa bits of bf16 128.0 (0x4300) gives exactly 128+q.
// One LOP3 turns nibbles j and j+4 of a word into such a bf16 pair.  The low half,
// moved to the high half, is the fp32 value 128+q_j exactly.  The word itself read as fp32 is
// 128.26171875 + q_{j+4} + q_j/65536; the q_j/65536 term is cancelled exactly by
// pre-subtracting x_{j+4}/65536 from the x that multiplies the low half.  Summing
// (w32 * x_hi + lo32 * x_lo') over the group therefore gives
//     sum q x + 128.259765625 * X_hi + 128 * X_lo
// where X_hi / X_lo are the sums of x over nibble positions 4..7 / 0..3; those two
// sums depend on x only and are computed once per lane.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace lq4 {

constexpr int kGroup = 64;
constexpr float kHiOffset = 128.259765625f;  // 128 + 17152/65536 - 128/65536
constexpr float kLoOffset = 128.0f;

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t f2bf16_rne(float f) {
  uint16_t r;  // round to nearest even (one conversion instruction)
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// L2 policy of the weight streams: evict first.  A layer's weights are read once per step and
// are far larger than L2; left at normal priority they would push out what is reused -- the
// kernels' code, activations, routing scratch.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Streaming 16-byte load: read-only, no L1 allocation, evict-first in L2 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(l2_evict_first()));
  return r;
}

// Programmatic dependent launch: let the next kernel on the stream be scheduled, and wait
// until the previous one has completed with its writes visible (a no-op for a kernel that
// was not launched as a programmatic dependent).
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_allow_next();
  pdl_wait_prev();
}

// 32 bytes (one 256-bit load; p 32-byte aligned) of a weight row that is read k-block by
// k-block: L2 fetches the surrounding 256 bytes (the row's next k-blocks) with it, at normal
// priority (the expert GEMMs re-read a tile's rows for each of its token tiles).
__device__ __forceinline__ void ld_stream32(const void *p, uint4 &lo, uint4 &hi) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z),
        "=r"(hi.w)
      : "l"(p));
}

__device__ __forceinline__ uint16_t ld_u16(const uint16_t *p) {
  uint16_t r;
  asm volatile("ld.global.nc.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(r) : "l"(p), "l"(l2_evict_first()));
  return r;
}

// 16- and 4-byte global -> shared copies of weights (cp.async), evict-first in L2.
__device__ __forceinline__ void cp_async16_stream(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(l2_evict_first())
               : "memory");
}
__device__ __forceinline__ void cp_async4_stream(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "l"(l2_evict_first())
               : "memory");
}

// One lane's share of an activation row for one 64-wide group, prepared for q4_group_dot.
struct XGroup {
  float2 xv[32];  // [4*m + j] = (x[8m+j+4], x[8m+j] - x[8m+j+4] * 2^-16), m = word, j = 0..3
  float C;        // 128.259765625 * X_hi + 128 * X_lo
  float X;        // sum of the 64 x values
};

// Build an XGroup from 64 fp32 values (in K order).
__device__ __forceinline__ void xgroup_from(XGroup &g, const float *v) {
  float xh = 0.f, xl = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float lo = v[8 * m + j], hi = v[8 * m + j + 4];
      g.xv[4 * m + j] = make_float2(hi, lo - hi * (1.0f / 65536.0f));
      xh += hi;
      xl += lo;
    }
  }
  g.C = kHiOffset * xh + kLoOffset * xl;
  g.X = xh + xl;
}

// 64 bf16 values (8 x 16-byte chunks in K order) -> XGroup.
__device__ __forceinline__ void xgroup_from_bf16(XGroup &g, const uint4 *chunks) {
  float v[64];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = chunks[c];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  xgroup_from(g, v);
}

// sum_k q_k * x_k + C for one group of 8 words (accumulation only, s/b not applied).
// Per word: three shifts and four LOP3 on the integer pipe; the low half of each pair is
// moved up with an integer multiply, which issues on the FMA pipe, leaving the integer
// pipe (the bottleneck of this loop) with under one operation per weight.
__device__ __forceinline__ float q4_group_raw(const uint4 w0, const uint4 w1, const XGroup &g) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t ws[4];
    ws[0] = w[m];
    asm("shr.b32 %0, %1, 4;" : "=r"(ws[1]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 8;" : "=r"(ws[2]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 12;" : "=r"(ws[3]) : "r"(w[m]));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v, lo;
      // v = (ws & 0x000F000F) | 0x43004300: the bf16 pair (128 + q_j, 128 + q_j+4)
      asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(v) : "r"(ws[j]));
      asm("mul.lo.u32 %0, %1, 65536;" : "=r"(lo) : "r"(v));
      const float2 xv = g.xv[4 * m + j];
      if (j & 1) {
        a0 = fmaf(__uint_as_float(v), xv.x, a0);
        a1 = fmaf(__uint_as_float(lo), xv.y, a1);
      } else {
        a2 = fmaf(__uint_as_float(v), xv.x, a2);
        a3 = fmaf(__uint_as_float(lo), xv.y, a3);
      }
    }
  }
  return (a0 + a2) + (a1 + a3);
}

// q4_group_raw with the two FMAs of a pair issued as one packed fp32x2 FMA: the pair
// (v as fp32, low half moved up) against the matching x pair.
__device__ __forceinline__ float q4_group_raw_x2(const uint4 w0, const uint4 w1, const XGroup &g) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t ws[4];
    ws[0] = w[m];
    asm("shr.b32 %0, %1, 4;" : "=r"(ws[1]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 8;" : "=r"(ws[2]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 12;" : "=r"(ws[3]) : "r"(w[m]));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v, lo;
      asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(v) : "r"(ws[j]));
      asm("mul.lo.u32 %0, %1, 65536;" : "=r"(lo) : "r"(v));
      const float2 xv = g.xv[4 * m + j];
      if (j & 1)
        asm("{\n.reg .b64 va, xa, acc;\nmov.b64 va, {%2, %3};\nmov.b64 xa, {%4, %5};\n"
            "mov.b64 acc, {%0, %1};\nfma.rn.f32x2 acc, va, xa, acc;\nmov.b64 {%0, %1}, acc;\n}"
            : "+f"(a0), "+f"(a1)
            : "r"(v), "r"(lo), "f"(xv.x), "f"(xv.y));
      else
        asm("{\n.reg .b64 va, xa, acc;\nmov.b64 va, {%2, %3};\nmov.b64 xa, {%4, %5};\n"
            "mov.b64 acc, {%0, %1};\nfma.rn.f32x2 acc, va, xa, acc;\nmov.b64 {%0, %1}, acc;\n}"
            : "+f"(a2), "+f"(a3)
            : "r"(v), "r"(lo), "f"(xv.x), "f"(xv.y));
    }
  }
  return (a0 + a2) + (a1 + a3);
}

__device__ __forceinline__ float q4_group_dot_x2(const uint4 w0, const uint4 w1, const XGroup &g,
                                                 float s, float b) {
  return fmaf(s, q4_group_raw_x2(w0, w1, g) - g.C, b * g.X);
}

// bf16 activations: one lane's 64 x values kept as the bf16 pairs (x_j, x_j+4) matching the
// code pairs an unpack produces, plus their sum.  Half the registers of XGroup.
struct XGroupB {
  uint32_t xp[32];  // [4*m + j] = x[8m+j] | x[8m+j+4] << 16 (bf16 bits)
  float X128;       // 128 * sum of the 64 x values
  float X;          // sum of the 64 x values
};

// 64 bf16 values (8 x 16-byte chunks in K order) -> XGroupB.
__device__ __forceinline__ void xgroupb_from_bf16(XGroupB &g, const uint4 *chunks) {
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t w[4] = {chunks[c].x, chunks[c].y, chunks[c].z, chunks[c].w};
    // w[i] holds x[8c+2i] (low) and x[8c+2i+1] (high)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu);          // x[8c+j]
      const uint32_t hi = (j & 1) ? (w[2 + (j >> 1)] >> 16) : (w[2 + (j >> 1)] & 0xFFFFu);  // x[8c+j+4]
      g.xp[4 * c + j] = lo | (hi << 16);
      sum += __uint_as_float(lo << 16) + __uint_as_float(hi << 16);
    }
  }
  g.X = sum;
  g.X128 = 128.0f * sum;
}

// sum_k (128 + q_k) x_k for one group: each bf16 pair (128 + q_j, 128 + q_j+4) from the
// unpack multiplies the matching bf16 x pair in mixed-precision FMAs (bf16 operands, fp32
// accumulation; the products are exact).  Per word: three shifts, four LOP3, eight FMAs.
__device__ __forceinline__ float q4_group_raw_b(const uint4 w0, const uint4 w1, const XGroupB &g) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    uint32_t ws[4];
    ws[0] = w[m];
    asm("shr.b32 %0, %1, 4;" : "=r"(ws[1]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 8;" : "=r"(ws[2]) : "r"(w[m]));
    asm("shr.b32 %0, %1, 12;" : "=r"(ws[3]) : "r"(w[m]));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v;
      asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(v) : "r"(ws[j]));
      if (j & 1)
        asm("{\n.reg .b16 vl, vh, xl, xh;\nmov.b32 {vl, vh}, %2;\nmov.b32 {xl, xh}, %3;\n"
            "fma.rn.f32.bf16 %0, vl, xl, %0;\nfma.rn.f32.bf16 %1, vh, xh, %1;\n}"
            : "+f"(a0), "+f"(a1)
            : "r"(v), "r"(g.xp[4 * m + j]));
      else
        asm("{\n.reg .b16 vl, vh, xl, xh;\nmov.b32 {vl, vh}, %2;\nmov.b32 {xl, xh}, %3;\n"
            "fma.rn.f32.bf16 %0, vl, xl, %0;\nfma.rn.f32.bf16 %1, vh, xh, %1;\n}"
            : "+f"(a2), "+f"(a3)
            : "r"(v), "r"(g.xp[4 * m + j]));
    }
  }
  return (a0 + a2) + (a1 + a3);
}

// s*(sum q x) + b*(sum x) for bf16 x.
__device__ __forceinline__ float q4_group_dot_b(const uint4 w0, const uint4 w1, const XGroupB &g,
                                                float s, float b) {
  return fmaf(s, q4_group_raw_b(w0, w1, g) - g.X128, b * g.X);
}

// ------------------------------------------------------------------ affine 8-bit codes
// Four 8-bit codes per uint32, lowest byte first.  bf16 holds 128 + n exactly only for a
// 4-bit n, so each code is taken as two nibbles, q = lo + 16 hi: one LOP3 with the magic
// 0x4300 turns the low (or, after a 4-bit shift, high) nibbles of bytes 0 and 2 (or, after
// an 8-bit shift, of bytes 1 and 3) into a bf16 pair, which multiplies the bf16 x pair
// (x_j, x_j+2) in mixed-precision FMAs.  sum q x = (A_lo - 128 X) + 16 (A_hi - 128 X).
// Per word (4 codes): three shifts, four LOP3, eight FMAs -- the 4-bit cost per code byte.

// bf16 activations for 8-bit codes: one lane's 64 x values as the pairs (x_4m+j, x_4m+j+2),
// j < 2, in word 2m + j, plus their sum.
struct XGroup8 {
  uint32_t xp[32];
  float X128;  // 128 * sum of the 64 x values
  float X;
};

// 64 bf16 values (8 x 16-byte chunks in K order) -> XGroup8.
__device__ __forceinline__ void xgroup8_from_bf16(XGroup8 &g, const uint4 *chunks) {
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t w[4] = {chunks[c].x, chunks[c].y, chunks[c].z, chunks[c].w};
    // w[i] = x[8c+2i] | x[8c+2i+1] << 16; word 2m+j of the group pairs x[4m+j] with x[4m+j+2]
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // the chunk's two 4-value words, m = 2c + h
      const uint32_t a = w[2 * h], b = w[2 * h + 1];
      g.xp[4 * c + 2 * h + 0] = (a & 0xFFFFu) | (b << 16);          // x[4m], x[4m+2]
      g.xp[4 * c + 2 * h + 1] = (a >> 16) | (b & 0xFFFF0000u);      // x[4m+1], x[4m+3]
      sum += __uint_as_float(a << 16) + __uint_as_float(a & 0xFFFF0000u) +
             __uint_as_float(b << 16) + __uint_as_float(b & 0xFFFF0000u);
    }
  }
  g.X = sum;
  g.X128 = 128.0f * sum;
}

// The same 64 x values re-paired for 8-bit codes from their 4-bit pairing: chunk c's words
// (x_8c+j, x_8c+j+4), j < 4, give (x_8c, x_8c+2), (x_8c+1, x_8c+3), (x_8c+4, x_8c+6),
// (x_8c+5, x_8c+7) by byte permutes.
__device__ __forceinline__ void xgroup8_from_b(XGroup8 &o, const XGroupB &g) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t b0 = g.xp[4 * c], b1 = g.xp[4 * c + 1], b2 = g.xp[4 * c + 2], b3 = g.xp[4 * c + 3];
    o.xp[4 * c + 0] = __byte_perm(b0, b2, 0x5410);
    o.xp[4 * c + 1] = __byte_perm(b1, b3, 0x5410);
    o.xp[4 * c + 2] = __byte_perm(b0, b2, 0x7632);
    o.xp[4 * c + 3] = __byte_perm(b1, b3, 0x7632);
  }
  o.X = g.X;
  o.X128 = g.X128;
}

// s*(sum q x) + b*(sum x) for one 64-group of 8-bit codes (16 words in w[0..3]) and bf16 x.
__device__ __forceinline__ float q8_group_dot_b(const uint4 (&wv)[4], const XGroup8 &g, float s,
                                                float b) {
  const uint32_t w[16] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w, wv[1].x, wv[1].y, wv[1].z, wv[1].w,
                          wv[2].x, wv[2].y, wv[2].z, wv[2].w, wv[3].x, wv[3].y, wv[3].z, wv[3].w};
  float l0 = 0.f, l1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    uint32_t ws[4];
    ws[0] = w[m];  // low nibbles of bytes 0, 2
    asm("shr.b32 %0, %1, 8;" : "=r"(ws[1]) : "r"(w[m]));   // low nibbles of bytes 1, 3
    asm("shr.b32 %0, %1, 4;" : "=r"(ws[2]) : "r"(w[m]));   // high nibbles of bytes 0, 2
    asm("shr.b32 %0, %1, 12;" : "=r"(ws[3]) : "r"(w[m]));  // high nibbles of bytes 1, 3
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v;
      asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(v) : "r"(ws[j]));
      const uint32_t xv = g.xp[2 * m + (j & 1)];
      if (j < 2)
        asm("{\n.reg .b16 vl, vh, xl, xh;\nmov.b32 {vl, vh}, %2;\nmov.b32 {xl, xh}, %3;\n"
            "fma.rn.f32.bf16 %0, vl, xl, %0;\nfma.rn.f32.bf16 %1, vh, xh, %1;\n}"
            : "+f"(l0), "+f"(l1)
            : "r"(v), "r"(xv));
      else
        asm("{\n.reg .b16 vl, vh, xl, xh;\nmov.b32 {vl, vh}, %2;\nmov.b32 {xl, xh}, %3;\n"
            "fma.rn.f32.bf16 %0, vl, xl, %0;\nfma.rn.f32.bf16 %1, vh, xh, %1;\n}"
            : "+f"(h0), "+f"(h1)
            : "r"(v), "r"(xv));
    }
  }
  const float lo = (l0 + l1) - g.X128, hi = (h0 + h1) - g.X128;
  return fmaf(s, fmaf(16.0f, hi, lo), b * g.X);
}

// s*(sum q v) + b*(sum v) for one 64-group of 8-bit codes (16 words in w[0..3]) and fp32
// activations v[0..63] in K order (the three-launch decode path keeps h in fp32).
__device__ __forceinline__ float q8_group_dot_f32(const uint4 (&wv)[4], const float *v, float s,
                                                  float b) {
  const uint32_t w[16] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w, wv[1].x, wv[1].y, wv[1].z, wv[1].w,
                          wv[2].x, wv[2].y, wv[2].z, wv[2].w, wv[3].x, wv[3].y, wv[3].z, wv[3].w};
  float a0 = 0.f, a1 = 0.f, x0 = 0.f, x1 = 0.f;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q = (float)((w[m] >> (8 * j)) & 0xFFu);
      if (j & 1) {
        a1 = fmaf(q, v[4 * m + j], a1);
        x1 += v[4 * m + j];
      } else {
        a0 = fmaf(q, v[4 * m + j], a0);
        x0 += v[4 * m + j];
      }
    }
  }
  return fmaf(s, a0 + a1, b * (x0 + x1));
}

// Dot product of one dequantised 64-group with the prepared x: s*(sum q x) + b*(sum x).
__device__ __forceinline__ float q4_group_dot(const uint4 w0, const uint4 w1, const XGroup &g,
                                              float s, float b) {
  const float A = q4_group_raw(w0, w1, g);
  return fmaf(s, A - g.C, b * g.X);
}

// Sum over the lanes of a segment of `width` consecutive lanes (width a power of two).
template <int W>
__device__ __forceinline__ float seg_sum(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp-wide exclusive scan of one int per lane; returns the lane's prefix, *total = sum.
__device__ __forceinline__ int warp_excl_scan(int v, int *total) {
  const int lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

// SiLU(g) * u.  The fast divide is within 2 ulp for denominators below 2^126 and gives 0 above
// (SiLU of a large negative g is 0 to fp32 precision anyway).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Candidate value for an argmax / top-k: NaN counts as -inf, so every candidate can win a
// round (candidates start at -inf and ties go to the lower index) and a selected index is
// always a real one, whatever the inputs.
__device__ __forceinline__ float cand(float v) { return v != v ? -INFINITY : v; }

// Order-preserving map of a float to uint32 (-0 is folded onto +0 first, so the two compare
// equal as floats do); and back.
__device__ __forceinline__ uint32_t f2key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp-wide argmax of (v, i): larger value first, ties to the lower index (NaN-free input);
// every lane gets the result.  Two single-instruction warp reductions.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
  const uint32_t key = f2key(v);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  i = (int)__reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)i : 0xffffffffu);
  v = key2f(kmax);
}

// Top-k of one row of logits by one warp: lane j holds logits j, j+32, ... as order-preserving
// keys (NaN counts as -inf); each of the k rounds takes the warp maximum of the keys (one
// reduction), then the lowest index holding it (a second reduction), and removes that entry.
// Lane i < k receives selection i (descending value, ties to the lower index): its index and
// value.  The lane's running maximum is a tree of max operations, so a round is a short chain.
// warp_topk_keys is the selection on keys the lanes already hold: key[j] of lane l is entry
// l + 32 j (f2key of the candidate value; 0 for no entry, which sorts below every real key);
// it consumes the keys.  warp_topk loads them from a row of logits first.
template <int EC>  // entries per lane: E <= 32 * EC
__device__ __forceinline__ void warp_topk_keys(uint32_t (&key)[EC], int k, int &my_e, float &my_v) {
  const int lane = threadIdx.x & 31;
  my_e = 0;
  my_v = 0.f;
#pragma unroll 1
  for (int i = 0; i < k; ++i) {
    uint32_t m[EC];
#pragma unroll
    for (int j = 0; j < EC; ++j) m[j] = key[j];
#pragma unroll
    for (int s = 1; s < EC; s *= 2) {
#pragma unroll
      for (int j = 0; j < EC; j += 2 * s) m[j] = max(m[j], m[j + s]);
    }
    const uint32_t M = __reduce_max_sync(0xffffffffu, m[0]);
    // the lane's lowest entry holding M: a mask of the equal entries (independent compares,
    // OR-ed as a tree), then its lowest set bit
    uint32_t bits[EC];
#pragma unroll
    for (int j = 0; j < EC; ++j) bits[j] = key[j] == M ? (1u << j) : 0u;
#pragma unroll
    for (int s = 1; s < EC; s *= 2) {
#pragma unroll
      for (int j = 0; j < EC; j += 2 * s) bits[j] |= bits[j + s];
    }
    const uint32_t ce = bits[0] ? (uint32_t)(lane + 32 * (__ffs(bits[0]) - 1)) : 0xffffffffu;
    const uint32_t be = __reduce_min_sync(0xffffffffu, ce);
    const bool mine = (int)(be & 31u) == lane;
    const int jw = (int)(be >> 5);
#pragma unroll
    for (int j = 0; j < EC; ++j) key[j] = (mine && jw == j) ? 0u : key[j];
    my_e = lane == i ? (int)be : my_e;
    my_v = lane == i ? key2f(M) : my_v;
  }
}

template <int EC>
__device__ __forceinline__ void warp_topk(const float *lg, int E, int k, int &my_e, float &my_v) {
  const int lane = threadIdx.x & 31;
  uint32_t key[EC];
#pragma unroll
  for (int j = 0; j < EC; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? f2key(cand(__ldcg(lg + e))) : 0u;
  }
  warp_topk_keys<EC>(key, k, my_e, my_v);
}

// (value, index) ordering used by every argmax / top-k: larger value first, then lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

}  // namespace lq4
