// Internal declarations shared by the library's translation units (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lily_q4.h"

namespace lq4 {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Every workspace starts with a 256-byte header of int32 words.
enum HeaderWord : int {
  kHdrError = 0,    // nonzero after a bounded device-side wait gave up
  kHdrCounterA = 1, // last-block-done counters (self-resetting)
  kHdrCounterB = 2,
  kHdrCounterC = 3,
  kHdrBarrier64 = 4,  // words 4-5: 64-bit grid-barrier arrival count
  kHdrArgmax64 = 6,   // words 6-7: the LM head's running (value, row) maximum, packed (self-resetting)
  kHdrWords = 64,
};

// ---------------------------------------------------------------- LM head
struct LmWsLayout {
  size_t off_partial_v, off_partial_i;
  size_t total_argmax;                  // bytes the argmax-only call needs
  size_t off_partial_m, off_partial_s;  // per-block (max, sum of exp) for the log-sum-exp
  size_t off_logits;                    // f32 [N]: logits of a log-sum-exp call without logprobs
  size_t total;                         // bytes either call needs
  int grid;
  int rows_per_block;  // streaming kernel (K >= 512): contiguous rows per block
};
LmWsLayout lm_ws_layout(int N, int K, int bits = 4);
// 8-bit codes (four per uint32): greedy token (and logits) for K = 512, 1024 or 2048.
int launch_q8_gemv_argmax(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                          float *logits, void *ws, cudaStream_t st, float *lse = nullptr);
// lse == nullptr: greedy token (and logits) only.  Otherwise also *lse = log sum_n exp(logit[n])
// and, with logits set, logits[n] - *lse in place of the logits (a second, elementwise launch).
int launch_gemv_argmax(const lily_q4_mat &W, int N, int K, const uint16_t *x, int32_t *token,
                       float *logits, void *ws, cudaStream_t st, float *lse = nullptr);

// ---------------------------------------------------------------- decode MoE
struct DecodeWsLayout {
  int T, E, k, I, H, P, Umax;
  size_t off_logits;    // f32 [T][E]
  size_t off_idx;       // i32 [T][k]
  size_t off_p;         // f32 [T][k]
  size_t off_sigma;     // f32 [T]
  size_t off_meta;      // i32: [0] = number of unique experts U, [1..Umax] expert ids, then ubase[Umax+1]
  size_t off_pair_tok;  // i32 [P]: token of each (unique expert, token) pair
  size_t off_pair_w;    // f32 [P]: its combine weight (p, or sigma for the shared expert)
  size_t off_h;         // f32 [P][I]: SwiGLU activations of each pair
  size_t total;
};
DecodeWsLayout decode_ws_layout(const lily_q4_moe_layer &L, int T);
int decode_launch_count(const lily_q4_moe_layer &L, int T);
// One block waiting on a grid barrier (which = 0) or an mbarrier (1) that never completes,
// until the bound; records the time-out in the workspace header.
int selftest_wait(void *ws, int which, cudaStream_t st);
// Device address, on the current device, of the fixed scratch of lily_q4_gemv_argmax_noalloc
// (a workspace header followed by the per-block argmax pairs).
int noalloc_scratch(void **out);
int launch_moe_decode(const lily_q4_moe_layer &L, const uint16_t *x, int T, uint16_t *y,
                      int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t st);

// ---------------------------------------------------------------- prefill MoE
struct PrefillWsLayout {
  int T, E, k, I, H, P, Tpad;
  size_t off_logits;    // f32 [T][E]
  size_t off_idx;       // i32 [T][k]
  size_t off_p;         // f32 [T][k]
  size_t off_sigma;     // f32 [T]
  size_t off_ctab;      // i32 [T/16 blocks][E]: each top-k block's count per expert
  size_t off_cpre;      // i32 [T/128][E]: exclusive prefix over the blocks before every 8th
  size_t off_offsets;   // i32 [E+2] exclusive prefix of counts
  size_t off_perm;      // i32 [P] token of each sorted pair
  size_t off_pw;        // f32 [P] combine weight of each sorted pair
  size_t off_inv;       // i32 [T][k+1] sorted position of (token, slot)
  size_t off_items;     // int4 work lists of the grouped GEMMs
  size_t off_xperm;     // bf16 [T][H] token rows in the permuted K order
  size_t off_h;         // bf16 [P][I] SwiGLU activations, sorted by expert
  size_t off_o;         // bf16 [P][H] weighted expert outputs, sorted by expert
  // affine 8-bit parts
  int Kr;               // reduction length of the router GEMM: H, or for an 8-bit router its
                        // exact bf16 form (2H + 3 H/64, rounded up to whole K-split blocks)
  size_t off_r8a;       // bf16 [E][Kr] the 8-bit router's exact bf16 form
  size_t off_r8b;       // bf16 [T][Kr] token rows widened to match
  size_t off_sh8;       // 8-bit shared expert as 4-bit codes of twice the width: gate, up, down
  size_t total;
  int max_items;
};
PrefillWsLayout prefill_ws_layout(const lily_q4_moe_layer &L, int T);
int prefill_launch_count(const lily_q4_moe_layer &L);
int launch_moe_prefill(const lily_q4_moe_layer &L, const uint16_t *x, int T, uint16_t *y,
                       int32_t *topk_idx, float *topk_w, void *ws, cudaStream_t st);

int sm_count();
int check_launch();

// Launch `fn` as a programmatic dependent of the previous kernel on `st`: its blocks may be
// scheduled while that kernel drains, and they wait (griddepcontrol.wait) for its completion
// before touching anything it wrote or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

}  // namespace lq4
