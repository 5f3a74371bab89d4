// Launch parameters and host-side launchers of the block's kernels.  Shared
// by the kernel translation units and the C-ABI implementation.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_common.cuh"

namespace dg {

// Token rows per tile of the grouped GEMMs is bounded by BN (128 or 256);
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
  float* r_out;      // [T] 1/rms(h)
  int32_t* idx;      // [T, K]
  float* w;          // [T, K]
  float* logits;     // [T, E] or null
  uint16_t* xd;      // bf16 [T, H]
  float* y_moe;      // [T, H], zeroed here
  int* n_refined;    // counter of tokens re-checked in fp64
};

struct ScatterParams {
  const int32_t* idx;        // [T, K]
  const float* w;            // [T, K]
  const int32_t* chunk_counts;  // [nchunks, E]
  int T, K, E, H, I, D;
  int bn_exp, bn_dense;      // token rows per expert / dense tile
  int32_t* offsets;          // [E + 1]
  int32_t* perm;             // [T*K]
  int32_t* tok_perm;         // [T*K]
  float* w_perm;             // [T*K]
  int4* tiles_gu;            // gate_up tiles
  int4* tiles_dn;            // down tiles
  int* ntiles;               // [2]: gate_up, down
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
  CUtensorMap wa_exp;  // expert weights: gate_up [E*2I, H] or down [E*H, I]
  CUtensorMap wa_d0;   // dense gate [D, H] (gate_up) or dense down [H, D]
  CUtensorMap wa_d1;   // dense up [D, H] (gate_up only)
  CUtensorMap xb_exp;  // expert rows: xe_perm [TKmax, H] or act [TKmax, I]
  CUtensorMap xb_d;    // dense rows: xd [Tmax, H] or act_d [Tmax, D]
  const int4* tiles;
  const int* ntiles;
  int E, I, D, H;
  int kb_exp, kb_dense;  // 64-wide K blocks of an expert / a dense tile
  uint16_t* act;         // gate_up out: bf16 [TK, I]
  uint16_t* act_d;       // gate_up out: bf16 [T, D]
  float* y_moe;          // down out: f32 [T, H] (accumulated)
  float* y_dense;        // down out: f32 [T, H]
  const int32_t* tok_perm;
  const float* w_perm;
  DevStatus* status;
};

struct CombineParams {
  const float* y_dense;
  const float* y_moe;
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

cudaError_t launch_router(const RouterParams& p, cudaStream_t s);
cudaError_t launch_route_count(const int32_t* idx, int T, int K, int E, int32_t* chunk_counts,
                               cudaStream_t s);
cudaError_t launch_route_scatter(const ScatterParams& p, cudaStream_t s);
cudaError_t launch_gather(const GatherParams& p, int num_sms, cudaStream_t s);
// mode 0: gate_up + GEGLU, mode 1: down + weighted scatter
cudaError_t launch_gemm(int mode, int bn, const GemmParams& p, int grid, cudaStream_t s);
size_t gemm_smem_bytes(int bn);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

}  // namespace dg
