// Host-side helpers of the C-ABI implementations (the MoE block and the
// self-conditioning MLP): argument checks, token-tile widths and the TMA
// descriptors of the weights and activations.
#pragma once

#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/dg_moe.h"
#include "dg_kernels.h"

namespace dg {
namespace host {

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Token rows per GEMM tile: small canvases favour deep weight pipelines (more
// stages fit when the token slot is small), large batches favour wide N.
inline int pick_bn(int T) { return T <= 512 ? 64 : (T <= 2048 ? 128 : 256); }

// The same for the 4-bit GEMM: narrow tiles for one canvas keep many token
// stages in flight; 256-token tiles for large batches halve the weights to
// dequantise per MMA cycle.  The widest one whose shared memory fits.
inline int pick_bn_q4(int T, size_t slot_gu, size_t slot_dn, size_t smem_max) {
  int bn = T <= 256 ? 32 : (T <= 512 ? 64 : (T <= 2048 ? 128 : 256));
  while (bn > 32 && (gemm_q4_smem_bytes(bn, (int)slot_gu) > smem_max ||
                     gemm_q4_smem_bytes(bn, (int)slot_dn) > smem_max))
    bn /= 2;
  return bn;
}

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline dg_status_t check_qtensor(const dg_qtensor_t& t, dg_format_t fmt) {
  if (!t.q) return DG_ERR_INVALID_ARG;
  if (!aligned(t.q, 16)) return DG_ERR_ALIGNMENT;
  if (fmt == DG_FMT_NVFP4_G16) {
    // block scale rows are fetched with bulk copies; matrix scales are floats
    if (!t.scales || !t.biases) return DG_ERR_INVALID_ARG;
    if (!aligned(t.scales, 16) || !aligned(t.biases, 4)) return DG_ERR_ALIGNMENT;
    return DG_OK;
  }
  if (fmt != DG_FMT_BF16) {
    if (!t.scales || !t.biases) return DG_ERR_INVALID_ARG;
    // 4-bit scale rows are fetched with bulk copies (16-byte granules)
    const size_t a = fmt == DG_FMT_AFFINE_U4_G64 ? 16 : 2;
    if (!aligned(t.scales, a) || !aligned(t.biases, a)) return DG_ERR_ALIGNMENT;
  }
  return DG_OK;
}

// Configuration fields the routing kernels use (shared by the block's
// handle creation and the allocation-free routing entry point).
inline dg_status_t check_router_config(const dg_moe_config_t* c) {
  if (!c) return DG_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->rms_eps < 0.f || c->flags != 0)
    return DG_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return DG_ERR_INVALID_ARG;
  if (c->hidden % 128) return DG_ERR_UNSUPPORTED;
  if (c->hidden > 8192 || c->n_experts > 256 || c->top_k > 16) return DG_ERR_UNSUPPORTED;
  if (c->router_fmt != DG_FMT_BF16 && c->router_fmt != DG_FMT_AFFINE_U8_G64)
    return DG_ERR_UNSUPPORTED;
  return DG_OK;
}

// Weights the routing kernels read: the router matrix (and its 8-bit scales
// and biases), router_scale and w_pre_ff (16-byte vector loads),
// per_expert_scale (bf16 loads) and the optional f32 router_bias.
inline dg_status_t check_router_weights(const dg_moe_config_t& c, const dg_moe_weights_t* w) {
  if (!w) return DG_ERR_INVALID_ARG;
  dg_status_t s;
  if ((s = check_qtensor(w->router, c.router_fmt)) != DG_OK) return s;
  for (const void* v : {w->router_scale, w->w_pre_ff}) {
    if (!v) return DG_ERR_INVALID_ARG;
    if (!aligned(v, 16)) return DG_ERR_ALIGNMENT;
  }
  if (!w->per_expert_scale) return DG_ERR_INVALID_ARG;
  if (!aligned(w->per_expert_scale, 2)) return DG_ERR_ALIGNMENT;
  if (w->router_bias && !aligned(w->router_bias, 4)) return DG_ERR_ALIGNMENT;
  return DG_OK;
}

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Tiled TMA descriptor with the 128-byte swizzle the MMA descriptors expect.
// dims[0] is the contiguous dimension (elements); strides are in bytes for
// dims 1..rank-1.
inline bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i) gstride[i - 1] = strides[i - 1];
  }
  CUresult r = enc(map, dt, (cuuint32_t)rank, const_cast<void*>(base), gdim, gstride, bx, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, cols] read in boxes of box_rows x 64 columns.
inline bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box);
}

// Row-major affine code matrix [rows, K] (4-bit: u32 words of 8 codes;
// 8-bit: one byte a code) read as u32 words in boxes of box_rows x 32 words
// (128 bytes: 256 or 128 codes).
inline bool encode_q_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                          uint32_t box_rows, int bits) {
  const uint64_t dims[2] = {K * bits / 32, rows};
  const uint64_t strides[1] = {K * bits / 8};
  const uint32_t box[2] = {32, box_rows};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dims, strides, box);
}
inline bool encode_q4_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                           uint32_t box_rows) {
  return encode_q_rows(map, base, rows, K, box_rows, 4);
}

// gate_up weights as [groups][2 halves][n/16 chunks][16 rows][K]: one box of
// (128 bytes of K, 16, 2, 4, 1) is 128 rows that interleave 16 gate rows with
// the 16 matching up rows, four times.  half_stride is the byte distance from
// a gate row to its up row; group_stride the distance between groups.
// rank 5 (with a group dimension) for the expert stack, rank 4 for the
// dense pair.  qbits 4 or 8: affine code words (128 bytes of a row per box)
// instead of bf16 (qbits 0).
inline bool encode_gate_up(CUtensorMap* map, const void* gate, uint64_t K, uint64_t n,
                    uint64_t half_stride, int rank, uint64_t groups, uint64_t group_stride,
                    int qbits = 0) {
  const uint64_t row_bytes = qbits ? K * qbits / 8 : K * 2;
  const uint64_t dims[5] = {qbits ? K * qbits / 32 : K, 16, 2, n / 16, groups};
  const uint64_t strides[4] = {row_bytes, half_stride, 16 * row_bytes, group_stride};
  const uint32_t box[5] = {qbits ? 32u : 64u, 16, 2, 4, 1};
  return encode_tiled(map, qbits ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      rank, gate, dims, strides, box);
}

}  // namespace host
}  // namespace dg
