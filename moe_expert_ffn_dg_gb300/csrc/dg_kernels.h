// Launch parameters and host-side launchers of the block's kernels.  Shared
// by the kernel translation units and the C-ABI implementation.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_common.cuh"

namespace dg {

// Token rows per tile of the grouped GEMMs are bounded by BN (32 to 256);
// tiles are {group, feature tile, first row, rows}; group == E is the dense
// branch.
struct RouterParams {
  const uint16_t* h;             // bf16 [T, H]
  const void* wr;                // bf16 [E, H] or u8 codes [E, H]
  const uint16_t* wr_scales;     // bf16 [E, H/64] (8-bit router) or null
  const uint16_t* wr_biases;     // bf16 [E, H/64] (8-bit router) or null
  const uint16_t* router_scale;  // bf16 [H]
  const uint16_t* pes;           // bf16 [E]
  const uint16_t* w_pre_ff;      // bf16 [H]
  const float* router_bias;      // f32 [E] or null
  int T, H, E, K;
  int router_u8;
  float eps;
  // H^-1/2 rounded to fp32 and to fp64, computed on the host: square root
  // and division in double are slow on this part, and every thread needs them
  float cH;
  double cHd;
  float* r_out;      // [T] 1/rms(h)
  float* xnorm_out;  // [T] |router input|
  float* wnorm_out;  // [E] |router row|
  int32_t* idx;      // [T, K]
  float* w;          // [T, K]
  float* logits;     // [T, E] fp32 logits
  int32_t* chunk_counts;  // [nchunks, E] expert histogram per 256 tokens (zeroed)
  // [nchunks, E, 8]: per 256-token chunk and expert, a bit per token that
  // chose the expert (zeroed), or null
  uint32_t* chunk_masks;
  uint16_t* xd;      // bf16 [T, H]
  // Fused attention half of the decoder layer: with attn non-null, h is the
  // layer input (the attention residual) and the block input is built as
  // bf16(h + bf16(rms(attn) * w_post_attn)), written to h_out by the first
  // expert column (the later kernels then read h_out).
  const uint16_t* attn;         // bf16 [T, H] or null
  const uint16_t* w_post_attn;  // bf16 [H]
  uint16_t* h_out;              // bf16 [T, H]
  float* y_moe;      // [T, H], zeroed here (null: not zeroed)
  int* n_refined;    // counter of tokens whose top-k was re-checked exactly
  // Tensor-core logits (large batches): the prep kernel writes the router
  // rows times router_scale as two bf16 planes [E, 2H] (hi | lo, an exact
  // split for a bf16 router), r, xd, |W'_e| (wnorm) and r H^-1/2 |h_t|
  // (xnorm); the router GEMM then writes the logits, and the selection
  // bounds their error with the tensor-core bound.
  int logits_tc;
  uint16_t* planes;
  // Two-pass selection (large batches): the fast pass writes the outputs of
  // the tokens whose top-k is certain and lists the others (flagged [T],
  // count *n_flagged, zeroed); the re-check pass finishes those.  Null: one
  // pass does both.
  int32_t* flagged;
  int* n_flagged;
  // Split-K router GEMM: z_split K ranges (the bound depends on it); with
  // z_part non-null (z_split > 1) the logits come as z_split fp32 partial
  // sums [z_split, T, E] of sum_i W'_ei h_i, which the selection adds
  // (error-free) and scales by r H^-1/2 itself, writing the logits.
  const float* z_part;
  int z_split;
};

struct ScatterParams {
  const int32_t* idx;        // [T, K]
  const float* w;            // [T, K]
  const int32_t* chunk_counts;  // [nchunks, E]
  const uint32_t* chunk_masks;  // [nchunks, E, 8] token bits of each chunk and expert
  int T, K, E;
  int32_t* offsets;          // [E + 1]
  int32_t* perm;             // [T*K]
  int32_t* tok_perm;         // [T*K]
  float* w_perm;             // [T*K]
  int32_t* inv;              // [T*K] grouped row of assignment t*K + k, or null
  DevStatus* status;
};

struct GatherParams {
  const uint16_t* h;          // bf16 [T, H]
  const float* r;             // [T]
  const int32_t* tok_perm;    // [T*K]
  const uint16_t* w_pre_ff2;  // bf16 [H]
  int TK, H;
  uint16_t* xe_perm;          // bf16 [T*K, H]
};

struct GemmParams {
  // A side (weights), 64 K-columns per box, 128B swizzle:
  //  gate_up: wa_exp 5-D view of [E, 2I, H] whose 128-row box interleaves
  //           16 gate rows and the 16 matching up rows four times;
  //           dense: wa_d5 the same view over (dense_gate, dense_up) when up
  //           lies above gate in memory, else 16-row boxes of wa_d0 / wa_d1.
  //  down:    wa_exp [E*H, I] and wa_d0 [H, D], 128-row boxes.
  CUtensorMap wa_exp;
  CUtensorMap wa_d0;
  CUtensorMap wa_d1;
  CUtensorMap wa_d5;
  // B side (token rows), boxes of 64 and of 16 rows:
  //  gate_up: xe_perm [TKmax, H] and xd [Tmax, H]; down: act and act_d.
  CUtensorMap xb_exp64;
  CUtensorMap xb_exp16;
  CUtensorMap xb_d64;
  CUtensorMap xb_d16;
  // Boxes of a whole tile width (256 and 128 rows; 32 is encoded but measured
  // slower than two 16-row boxes) of the same tensors: a full token stage in
  // one copy
  CUtensorMap xb_exp256;
  CUtensorMap xb_d256;
  CUtensorMap xb_exp128;
  CUtensorMap xb_d128;
  CUtensorMap xb_exp32;
  CUtensorMap xb_d32;
  // Tiles, decoded in each CTA from the expert offsets: first the dense tiles
  // (ceil(T/bn) token tiles x mt_dense feature tiles), then per expert e
  // ceil(n_e/bn) token tiles x mt_exp feature tiles, feature tile fastest.
  const int32_t* offsets;  // [E + 1]
  int T, bn, mt_exp, mt_dense;
  int E, I, D, H;
  int kb_exp, kb_dense;  // 64-wide K blocks of an expert / a dense tile
  int dense_5d;          // gate_up: dense A tile through wa_d5
  uint16_t* act;         // gate_up out: bf16 [TK, I]
  uint16_t* act_d;       // gate_up out: bf16 [T, D]
  float* y_moe;          // down out: f32 [T, H] (accumulated), when y_perm is null
  float* y_perm;         // down out: f32 [T*K, H], w * expert output per grouped row, or null
  // NVFP4 matrix scales (fp32), applied to the accumulator: per expert, and
  // for the dense tensors (gate_up: gate and up; down: d0)
  const float* g_exp;
  const float* g_d0;
  const float* g_d1;
  float* y_dense;        // down out: f32 [T, H]
  const int32_t* tok_perm;
  const float* w_perm;
  DevStatus* status;
  // 4-bit group-64 affine weights (the wa_* maps then hold the u32 code words,
  // 8 codes a word, 128B swizzle, boxes of 32 words = 256 codes): bf16 scale
  // and bias rows [rows, K/64] of the expert stack and of the dense matrices
  // (gate_up: d0 = dense gate, d1 = dense up; down: d0 = dense down).
  const uint16_t* sc_exp;
  const uint16_t* bi_exp;
  const uint16_t* sc_d0;
  const uint16_t* bi_d0;
  const uint16_t* sc_d1;
  const uint16_t* bi_d1;
  int sc_slot_bytes;  // shared-memory bytes of one tile's scale (or bias) rows
  // Router GEMM (mode 2): logits [T, z_E] f32 = r[t] H^-1/2 (sum over the
  // eight accumulators) + bias[e]; with z_split > 1 the K blocks are split in
  // z_split ranges over as many CTAs (feature tile = expert tile * z_split +
  // range) and each writes its unscaled fp32 partial to z_part[range, T, E].
  float* z_out;
  float* z_part;
  int z_split;
  const float* z_r;
  const float* z_bias;
  int z_E;
  float z_cH;
  // Bounded-wait test: non-zero makes CTA 0's epilogue wait on a barrier
  // nothing arrives on until kTestStallNs runs out (status kDevTimeout at
  // kSiteGemmEpilogue, info kTestStallInfo); 0 in every ordinary launch.
  int test_stall;
};

struct CombineParams {
  const float* y_dense;
  const float* y_moe;   // [T, H], read when y_perm is null
  const float* y_perm;  // [T*K, H] weighted expert rows, or null
  const int32_t* inv;   // [T*K] grouped row of each assignment (with y_perm)
  int K;
  float* y_moe_out;     // with y_perm: the summed [T, H] rows written here, or null
  const uint16_t* w_next;  // bf16 [H]: the next layer's input norm weight, or null
  uint16_t* next_out;      // bf16 [T, H]: rms(out) * w_next, with w_next
  const uint16_t* h;
  const uint16_t* w_post1;
  const uint16_t* w_post2;
  const uint16_t* w_post;
  int T, H;
  float eps;
  float layer_scalar;
  uint16_t* out;
};

constexpr int kChunkTokens = 256;  // tokens per permutation chunk
// From this many tokens on, the down GEMM stores each assignment's weighted
// f32 row and the combine sums a token's K rows, instead of reducing into
// the per-token accumulator with global atomics (whose throughput, ~1.7 TB/s
// of payload on this part, bounds the down GEMM of large batches).
constexpr int kPartialRowsMinTokens = 1024;
// From this many tokens on, the logits come from the register-tiled kernel
// (64 tokens x 64 experts per block) instead of the 4-token one (measured:
// 4-token blocks are faster at 2048 tokens, 117 vs 195 us; the tiled kernel
// at 16384, 631 vs 802 us).
constexpr int kRouterTileMinTokens = 4096;

// Launch with programmatic stream serialization (the kernel pairs
// pdl_trigger / pdl_wait, see dg_common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raise the dynamic shared-memory limits of the kernels to what their
// launches may use (router and quantised GEMMs: the device's opt-in maximum
// smem_max, as their sizes depend on the shapes; bf16 GEMMs: their fixed
// tile sizes).  The limits belong to the current device; they are set once
// per handle at creation instead of before every launch.
cudaError_t prepare_router(int smem_max);
cudaError_t prepare_gemm_bf16();
cudaError_t prepare_gemm_affine(int smem_max);

cudaError_t launch_router(const RouterParams& p, cudaStream_t s);
cudaError_t launch_router_select(const RouterParams& p, int num_sms, cudaStream_t s);
// The grouping (offsets, perm, tok_perm, w_perm, inv) and the grouped expert
// rows in one token-major kernel.
cudaError_t launch_scatter_gather(const ScatterParams& sp, const GatherParams& gp,
                                  cudaStream_t s);
// From this many tokens on, the router logits come from the tensor cores
// (prep kernel + router GEMM) and the selection runs in two passes (a fast
// one, then the re-check of the tokens near a tie); below, from the
// CUDA-core logit kernel (which also serves the allocation-free entry point)
// and one selection pass.
constexpr int kRouterTcMinTokens = 1024;
// Token rows per tile of the router GEMM and its accumulators: a tile's K
// range is dealt to kRouterAcc TMEM accumulators in turn (kRouterAcc x 256
// columns), summed error-free in the epilogue.  Wide tiles keep the weight
// planes' re-reads low (each tile reads all of them); the K split over CTAs
// (router_split) keeps each accumulator's MMA count, and with it the error
// bound, small.
constexpr int kRouterBn = 256;
constexpr int kRouterAcc = 2;
cudaError_t launch_router_prep_tc(const RouterParams& p, cudaStream_t s);

// K ranges of the router GEMM (kb = 2H / 64 K blocks): the fewest that keep
// an accumulator to kRouterMaxAccMmas MMAs (the bound of the logits), none
// empty.  Fewer MMAs an accumulator tighten the bound, so fewer tokens take
// the exact re-check, but give more partial sums to write and add: of 44, 24
// and 12 (four, eight and fifteen ranges at H = 2816), 24 measured fastest
// at 1024, 2048 and 16 384 tokens.
constexpr int kRouterMaxAccMmas = 24;
inline int router_split(int T, int E, int kb) {
  (void)T;
  (void)E;
  const int kbs_max = kRouterAcc * (kRouterMaxAccMmas / 4);  // K blocks a range may hold
  int s = (kb + kbs_max - 1) / kbs_max;
  if (s < 1) s = 1;
  while (s > 1 && (s - 1) * ((kb + s - 1) / s) >= kb) --s;
  return s;
}

// CTAs of the bf16 projection GEMMs per SM (grid = SMs times this, for
// token tiles up to 128), each with its share of the 192 KB stage ring.
constexpr int kProjCtasPerSm = 2;

// mode 0: gate_up + GEGLU, mode 1: down + weighted scatter, mode 2: router
// logits (bn = kRouterBn)
cudaError_t launch_gemm(int mode, int bn, const GemmParams& p, int grid, cudaStream_t s);
size_t gemm_smem_bytes(int bn);
// Grouped GEMM over quantised weights, dequantised to bf16 in shared memory;
// same modes, bn 32, 64, 128 or 256.  qf 4 or 8 (group-64 affine codes of
// that many bits) or kQfNvfp4 (e2m1 codes, e4m3 scales per 16, fp32 matrix
// scales).
constexpr int kQfNvfp4 = 16;
cudaError_t launch_gemm_affine(int mode, int bn, int qf, const GemmParams& p, int grid,
                               cudaStream_t s);
size_t gemm_q4_smem_bytes(int bn, int sc_slot_bytes);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

}  // namespace dg
