// Pieces shared by the grouped GEMM kernels (bf16 weights loaded into shared
// memory by TMA; quantised weights dequantised into shared memory): the
// persistent tile schedule, TMA loads of rank 4 and 5, the drain wait and the
// per-mode epilogue.
#pragma once

#include "dg_kernels.h"

namespace dg {
namespace gemm {

constexpr int kBoxRows = 16;  // token rows per small TMA box
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kMaxGroups = 256;
constexpr int kTileTableBytes = 2 * (kMaxGroups + 2) * 4;

// Tile t of the persistent schedule: dense tiles first, then the expert tiles
// (feature tile fastest).  s_start[e] = first expert tile of expert e
// (exclusive prefix of ceil(n_e / bn) * mt_exp), s_off = expert offsets.
// Returns {group, feature tile, first row, rows}; group == E is the dense
// branch.
__device__ __forceinline__ int4 decode_tile(const GemmParams& p, int t, int nd,
                                            const int* s_start, const int* s_off) {
  if (t < nd) {
    const int j = t / p.mt_dense, m = t - j * p.mt_dense;
    return make_int4(p.E, m, j * p.bn, min(p.bn, p.T - j * p.bn));
  }
  const int u = t - nd;
  int lo = 0, hi = p.E - 1;  // last e with s_start[e] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo, local = u - s_start[e];
  const int j = local / p.mt_exp, m = local - j * p.mt_exp;
  const int n = s_off[e + 1] - s_off[e];
  return make_int4(e, m, s_off[e] + j * p.bn, min(p.bn, n - j * p.bn));
}

// Fill the tile table from the expert offsets: s_off = offsets, s_start =
// exclusive prefix of the per-expert tile counts.  Called by 4 consecutive
// warps (tid 0..127); the prefix is taken by the first of them.
__device__ __forceinline__ void build_tile_table(const GemmParams& p, int tid, int* s_start,
                                                 int* s_off) {
  const int lane = tid & 31;
  for (int e = tid; e <= p.E; e += 128) s_off[e] = p.offsets[e];
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      int c = 0;
      if (e < p.E) {
        const int n = p.offsets[e + 1] - p.offsets[e];
        c = (n + p.bn - 1) / p.bn * p.mt_exp;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < p.E) s_start[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_start[p.E] = run;
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int c0, int c1, int c2, int c3, int c4,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4), "l"(policy)
      : "memory");
}

// Named barrier 1 between an MMA issuer warp and its waiter warp (64
// threads, both block), OR-reducing one predicate: returns true if either
// side passed true.
constexpr int kHandoffBarrier = 1;
__device__ __forceinline__ bool handoff(bool stop) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, %2, 64, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)stop), "n"(kHandoffBarrier)
      : "memory");
  return r != 0;
}
// The map whose box is a whole BN-row token stage (BN 32, 64, 128 or 256).
template <int BN>
__device__ __forceinline__ const CUtensorMap* full_stage_map(const GemmParams& p, bool dense) {
  if (BN == 256) return dense ? &p.xb_d256 : &p.xb_exp256;
  if (BN == 128) return dense ? &p.xb_d128 : &p.xb_exp128;
  if (BN == 64) return dense ? &p.xb_d64 : &p.xb_exp64;
  return dense ? &p.xb_d32 : &p.xb_exp32;
}

// Wait that ignores the abort flag (used to drain in-flight copies and MMAs
// before the CTA exits); bounded by kWaitLimitNs.
__device__ __forceinline__ bool wait_no_abort(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Epilogue of one tile from TMEM: warp quarter q reads its 32 lanes (the
// tile's 128 weight rows are the lanes), ncols token columns.
// MODE 0 (gate_up): lanes 32q..32q+15 hold gate and 32q+16..32q+31 up of the
// same 16 features; pair them with one shuffle and write
// act = bf16(gelu_tanh(gate) * up).
// g_lo / g_hi scale the accumulator first (NVFP4 matrix scales).
// MODE 1 (down): 128 output channels; the dense branch stores its f32
// output; experts either store w * y as the f32 row of the assignment
// (y_perm, summed per token later) or add it into the f32 per-token
// accumulator (y_moe).
// Expert tiles of the down GEMM: lane l holds the routing weight (and, for
// the reduction into y_moe, the token) of grouped row r0 + l of the tile.
__device__ __forceinline__ void fetch_tile_rows(const GemmParams& p, int4 td, int lane, int r0,
                                                float& w, int& t) {
  const int r = r0 + lane;
  w = 0.f;
  t = 0;
  if (r < td.w) {
    w = __ldg(p.w_perm + td.z + r);
    if (!p.y_perm) t = __ldg(p.tok_perm + td.z + r);
  }
}
// The first two blocks of 32 rows, fetched before the epilogue waits for the
// tile's accumulator so that their latency is hidden behind the wait.
struct EpiRows {
  float w[2];
  int t[2];
};
template <int MODE>
__device__ __forceinline__ EpiRows epilogue_rows(const GemmParams& p, int4 td, int lane) {
  EpiRows e{{0.f, 0.f}, {0, 0}};
  if (MODE == 1 && td.x != p.E) {
    fetch_tile_rows(p, td, lane, 0, e.w[0], e.t[0]);
    fetch_tile_rows(p, td, lane, 32, e.w[1], e.t[1]);
  }
  return e;
}

template <int MODE>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, int4 td, uint32_t tbase,
                                              int ncols, int q, int lane, const EpiRows& pre,
                                              float g_lo = 1.f, float g_hi = 1.f) {
  const bool dense = td.x == p.E;
  // scale of the accumulator (NVFP4 matrix scales; 1 otherwise): in gate_up
  // tiles lanes 0..15 of a quarter hold gate rows, 16..31 up rows
  const float gsc = (MODE == 0 && lane >= 16) ? g_hi : g_lo;
  // routing rows of the current and the next block of 32 grouped rows; the
  // block after next is fetched as a block is entered, so the loads overlap
  // the stores
  const bool rows = MODE == 1 && !dense;
  float w_cur = pre.w[0], w_nxt = pre.w[1];
  int t_cur = pre.t[0], t_nxt = pre.t[1];
  for (int c0 = 0; c0 < ncols; c0 += 16) {
    if (rows && c0 > 0 && (c0 & 31) == 0) {
      w_cur = w_nxt;
      t_cur = t_nxt;
      fetch_tile_rows(p, td, lane, c0 + 32, w_nxt, t_nxt);
    }
    __syncwarp();
    float v[16];
    tmem_ld16(tbase + (uint32_t)c0, v);
    if (gsc != 1.f) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] *= gsc;
    }
    if (MODE == 0) {
      const int ld = dense ? p.D : p.I;
      uint16_t* out = dense ? p.act_d : p.act;
      const int feat = td.y * 64 + 16 * q + (lane & 15);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = 2 * jj;
        const float send = lane < 16 ? v[j + 1] : v[j];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        const float g = lane < 16 ? v[j] : recv;
        const float u = lane < 16 ? recv : v[j + 1];
        const int col = c0 + j + (lane >> 4);
        if (col < td.w) {
          const size_t row = (size_t)(td.z + col);
          out[row * ld + feat] = f32_to_bf16_rne(gelu_tanh(g) * u);
        }
      }
    } else if (dense) {
      const int feat = td.y * 128 + 32 * q + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < td.w) p.y_dense[(size_t)(td.z + c0 + j) * p.H + feat] = v[j];
    } else if (p.y_perm) {
      // lane l holds channel 32q + l of 16 grouped rows: each store writes
      // 128 contiguous bytes of one row; streaming stores (the rows are read
      // once, by the combine) keep L2 for the token rows and weights
      const int feat = td.y * 128 + 32 * q + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w_cur, (c0 & 16) + j);
        if (c0 + j < td.w) __stcs(p.y_perm + (size_t)(td.z + c0 + j) * p.H + feat, wj * v[j]);
      }
    } else {
      // Routing-weighted add into the f32 per-token accumulator, four
      // features per vector reduction: transpose each 4 x 4 block of
      // (lane in quad) x (token) values across the quad, so lane 4i + r ends
      // up with features 4i..4i+3 of token 4m + r.
      const int r = lane & 3;
      float* ybase = p.y_moe + td.y * 128 + 32 * q + (lane & ~3);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float a[4] = {v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]};
#pragma unroll
        for (int j2 = 0; j2 < 2; ++j2) {  // swap the off-diagonal 2 x 2 blocks
          const float send = (r & 2) ? a[j2] : a[j2 + 2];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
          if (r & 2) a[j2] = recv;
          else a[j2 + 2] = recv;
        }
#pragma unroll
        for (int j = 0; j < 4; j += 2) {  // transpose inside each 2 x 2 block
          const float send = (r & 1) ? a[j] : a[j + 1];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
          if (r & 1) a[j] = recv;
          else a[j + 1] = recv;
        }
        const int tj = __shfl_sync(0xffffffffu, t_cur, (c0 & 16) + 4 * m + r);
        const float wj = __shfl_sync(0xffffffffu, w_cur, (c0 & 16) + 4 * m + r);
        if (c0 + 4 * m + r < td.w) {
          float* dst = ybase + (size_t)tj * p.H;
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(wj * a[0]),
                       "f"(wj * a[1]), "f"(wj * a[2]), "f"(wj * a[3])
                       : "memory");
        }
      }
    }
  }
}

// Router GEMM tiles: feature tile y = expert tile * z_split + K range.
__device__ __forceinline__ int router_etile(const GemmParams& p, int y) {
  return p.z_split > 1 ? y / p.z_split : y;
}
// K blocks [x, y) of the range of feature tile y (ranges of equal length,
// the last one shorter).
__device__ __forceinline__ int2 router_krange(const GemmParams& p, int y, int kbn) {
  if (p.z_split <= 1) return make_int2(0, kbn);
  const int r = y % p.z_split, len = (kbn + p.z_split - 1) / p.z_split;
  const int lo = r * len < kbn ? r * len : kbn;
  return make_int2(lo, lo + len < kbn ? lo + len : kbn);
}

// Router logits (mode 2) from the kRouterAcc accumulators of one tile:
// lane = expert row of the tile (32q + lane), column = token.  The
// accumulators are summed as an error-free fp32 pair (hi, lo) (TwoSum), then
// z = hi rc + (lo rc + bias) with rc = r[t] H^-1/2 in fp32 (two fused
// multiply-adds: a few units of fp32 rounding, inside the bound's 2^-17).
// With a K split the pair's sum is rounded once to fp32 and stored unscaled
// as the range's partial; the selection adds the ranges.
template <int BN>
__device__ __forceinline__ void epilogue_router(const GemmParams& p, int4 td, uint32_t tbase,
                                                int ncols, int q, int lane) {
  const int e = router_etile(p, td.y) * 128 + 32 * q + lane;
  const int2 kr = router_krange(p, td.y, p.kb_dense);
  const int nacc = kr.y - kr.x < kRouterAcc ? kr.y - kr.x : kRouterAcc;
  float* part = p.z_split > 1 ? p.z_part + (size_t)(td.y % p.z_split) * p.T * p.z_E : nullptr;
  const float bias = (p.z_bias && e < p.z_E) ? __ldg(p.z_bias + e) : 0.f;
  for (int c0 = 0; c0 < ncols; c0 += 16) {
    float hi[16], lo[16];
    __syncwarp();
    tmem_ld16(tbase + (uint32_t)c0, hi);
#pragma unroll
    for (int j = 0; j < 16; ++j) lo[j] = 0.f;
    for (int a = 1; a < nacc; ++a) {
      float v[16];
      tmem_ld16(tbase + (uint32_t)(a * BN + c0), v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float s = __fadd_rn(hi[j], v[j]);
        const float bb = __fsub_rn(s, hi[j]);
        const float err = __fadd_rn(__fsub_rn(hi[j], __fsub_rn(s, bb)), __fsub_rn(v[j], bb));
        hi[j] = s;
        lo[j] = __fadd_rn(lo[j], err);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = td.z + c0 + j;
      if (c0 + j < td.w && e < p.z_E) {
        if (part) {
          part[(size_t)t * p.z_E + e] = __fadd_rn(hi[j], lo[j]);
        } else {
          const float rc = __ldg(p.z_r + t) * p.z_cH;
          p.z_out[(size_t)t * p.z_E + e] = fmaf(hi[j], rc, fmaf(lo[j], rc, bias));
        }
      }
    }
  }
}

}  // namespace gemm
}  // namespace dg
