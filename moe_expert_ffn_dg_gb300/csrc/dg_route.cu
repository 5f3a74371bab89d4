// Routing of the MoE FFN block on sm_103a.
//
// k_router_logits / k_router_select: per token, RMS of the residual stream,
//   router input x = h / rms(h) * router_scale * H^-1/2 (two literal steps,
//   "DiffusionGemma port — plan & parity strategy", Reference dossier §2
//   Router and the D1 finding), E fp32 logits, top-k with ties to the lower
//   expert index ("diffgemma — architecture & implemented contract", Part II
//   §2.1 MoE order), weights = softmax over the k selected logits times
//   per_expert_scale (equal to the renormalised softmax over all E,
//   "DiffusionGemma Explained", MOEBlock.forward).  The fp32 logits carry a
//   rigorous error bound; a token whose top-k boundary is closer than the
//   bound gets exact logits for its candidate experts, so the selected set is
//   the one exact arithmetic gives.  The logits kernel also writes the dense
//   branch input xd = bf16(h / rms(h) * w_pre_ff) and zeroes the token's row
//   of the f32 expert-sum accumulator; the select kernel also counts the
//   per-chunk expert histogram and token bit masks.
// k_scatter_gather: token -> expert grouping from the per-chunk histograms
//   (prefix sum, stable positions: assignments sorted by expert, then token)
//   and the expert input rows xe = bf16(h / rms(h) * w_pre_ff2) in grouped
//   order, the B operand of the gate_up GEMM.
#include <math.h>

#include "dg_kernels.h"

namespace dg {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxSlots = 8;  // experts per lane: E <= 256

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
// Warp-wide arg-max under the order (value desc, index asc); every lane gets
// the winner.
template <typename T>
__device__ __forceinline__ void warp_argmax(T& v, int& e) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    T ov = __shfl_xor_sync(kFull, v, o);
    int oe = __shfl_xor_sync(kFull, e, o);
    if (ov > v || (ov == v && oe < e)) {
      v = ov;
      e = oe;
    }
  }
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  return (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(b) << 16);
}

// The attention half of the decoder layer ends with h = residual +
// post_attention_layernorm(attn) ("DiffusionGemma port — plan & parity
// strategy", Reference dossier §2 DecoderLayer), both bf16 planes: the normed
// attention n = bf16(attn * ra * w) and h = bf16(x + n), each rounded once
// (x + n is exact in fp32 whenever it can change the bf16 result).  Eight
// elements; ra = 1/rms of the token's attention row.
__device__ __forceinline__ uint4 attn_residual8(const uint4& xv, const uint4& av, const uint4& wv,
                                                float ra) {
  float x[8], a[8], w[8];
  unpack8(xv, x);
  unpack8(av, a);
  unpack8(wv, w);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float n0 = __uint_as_float((uint32_t)f32_to_bf16_rne(a[2 * i] * ra * w[2 * i]) << 16);
    const float n1 =
        __uint_as_float((uint32_t)f32_to_bf16_rne(a[2 * i + 1] * ra * w[2 * i + 1]) << 16);
    o[i] = pack2_bf16(x[2 * i] + n0, x[2 * i + 1] + n1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 1/rms of a bf16 row (fp32 rsqrt and one Newton step), summed by one warp.
__device__ __forceinline__ float row_rinv(const uint4* row, int nvec, int H, float eps, int lane) {
  float ss = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    float f[8];
    unpack8(__ldg(row + v), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = warp_sum_f(ss);
  const float msq = ss / (float)H + eps;
  float r = rsqrtf(msq);
  return r * (1.5f - 0.5f * msq * r * r);
}

// Error-free transformations in fp32 (Knuth's TwoSum; Dekker's product via
// FMA).  A pair (hi, lo) carries a sum whose rounding error is second order
// (~n u^2 of the magnitudes), which keeps fp64 (slow on this part) out of
// the loops.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void df_add(float& hi, float& lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo = __fadd_rn(lo, e);
}
// (hi, lo) += (hi2, lo2)
__device__ __forceinline__ void df_add2(float& hi, float& lo, float hi2, float lo2) {
  float s, e;
  two_sum(hi, hi2, s, e);
  hi = s;
  lo = __fadd_rn(__fadd_rn(lo, lo2), e);
}
__device__ __forceinline__ double df_value(float hi, float lo) { return (double)hi + (double)lo; }

// Error bound of the fp32 logits, relative to |W_e| |x| + |bias_e| (u is the
// fp32 unit roundoff 2^-24).  A computed logit is (1 + d) z_e + err_e with
// |err_e| <= ~22 u sum_i |W_ei x_i| <= 22 u |W_e| |x|: 3 u from the three
// fp32 products of the router input, 16 u from each 16-term fp32 chunk sum
// (chunk sums are accumulated as error-free fp32 pairs), a few u from the
// final rounding; and d (~50 u) is the error of the fp32 1/rms, a factor
// common to all logits of the token.  Without a router bias the common
// factor cannot change the order, so 2^-18 = 64 u bounds err_e with a factor
// of about 3; with a bias d acts like a per-expert error (|d| |z_e - b_e|),
// and 2^-16 = 256 u covers 22 u + 50 u + the bias rounding.
constexpr float kLogitBoundNoBias = 3.814697265625e-06f;  // 2^-18
constexpr float kLogitBoundBias = 1.52587890625e-05f;     // 2^-16

// Error bound of the tensor-core logits (router GEMM), relative to
// r H^-1/2 |h_t| |W'_e| + |bias_e| with W'_e = W_e * router_scale.  A
// tensor-core MMA adds 16 exact products of bf16 operands to its fp32
// accumulator; its rounding is not specified, so each MMA is allowed an
// error of up to 17 units in the last place of the largest magnitude among
// its addends and the accumulator (every addend truncated after alignment),
// which the accumulator's running sum of |terms| bounds.  Each of the
// kRouterAcc accumulators adds 2H / (16 kRouterAcc) MMAs, so the products
// carry at most 17 (2H / 128) 2^-23 sum_i |W'_ei h_i| (x 1.3 margin); the
// two-plane split of W' (exact for a bf16 router, 2^-18 for the decoded
// 8-bit one) and the final rounding add 2^-17.  The factor r H^-1/2 is
// common to the token's logits (it cannot change their order); with a bias
// its error acts per expert and 2^-16 is added, as for the CUDA-core logits.
// With the K blocks split in S ranges (split-K over CTAs) an accumulator
// adds the MMAs of ceil(range / kRouterAcc) K blocks; each range's sum is
// rounded once to fp32 (2^-24 of the sum of |terms|) and the ranges are
// added error-free.
__host__ __device__ inline float tc_logit_bound(int H, int S, bool bias) {
  const int kb = 2 * H / 64, len = (kb + S - 1) / S;
  const int mmas = 4 * ((len + kRouterAcc - 1) / kRouterAcc);
  return 17.0f * (float)mmas * 1.1920928955078125e-07f * 1.3f + 7.62939453125e-06f +
         (S > 1 ? 5.9604644775390625e-08f : 0.0f) + (bias ? kLogitBoundBias : 0.0f);
}

// Prep of the tensor-core logits.  Warp per token (blocks [0, nbt)): 1/rms
// (fp32 rsqrt and one Newton step), r H^-1/2 |h_t| (rounded up: a bound),
// xd = bf16(h / rms(h) * w_pre_ff), the zeroed y_moe row when the down GEMM
// reduces with atomics, and with the fused attention half the block input
// built and published.  Warp per expert (the blocks after): W' = W * router_scale
// in fp32 (exact for bf16 weights: 8 + 8 significant bits; one rounding
// after the exact 8-bit decode s q + b otherwise), split into the bf16
// planes hi = bf16(W') and lo = bf16(W' - hi) of row e of [E, 2H], and
// |W'_e| rounded up.
template <bool U8, bool FUSED>
__global__ void __launch_bounds__(256) k_router_prep_tc(const RouterParams p, int nbt) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, nvec = H >> 3;
  const float cH = p.cH;
  if ((int)blockIdx.x < nbt) {
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    const uint4* hrow = reinterpret_cast<const uint4*>(p.h + (size_t)t * H);
    const uint4* arow = reinterpret_cast<const uint4*>(FUSED ? p.attn + (size_t)t * H : p.h);
    const uint4* wav = reinterpret_cast<const uint4*>(p.w_post_attn);
    const float ra = FUSED ? row_rinv(arow, nvec, H, p.eps, lane) : 0.f;
    auto hvec = [&](int v) {
      return FUSED ? attn_residual8(__ldg(hrow + v), __ldg(arow + v), __ldg(wav + v), ra)
                   : __ldg(hrow + v);
    };
    float ss = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(hvec(v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum_f(ss);
    const float msq = ss / (float)H + p.eps;
    float rf = rsqrtf(msq);
    rf = rf * (1.5f - 0.5f * msq * rf * rf);
    uint4* xdrow = reinterpret_cast<uint4*>(p.xd + (size_t)t * H);
    uint4* hout = reinterpret_cast<uint4*>(FUSED ? p.h_out + (size_t)t * H : p.xd);
    const uint4* wpv = reinterpret_cast<const uint4*>(p.w_pre_ff);
    for (int v = lane; v < nvec; v += 32) {
      float f[8], wp[8];
      const uint4 hv = hvec(v);
      if (FUSED) hout[v] = hv;
      unpack8(hv, f);
      unpack8(__ldg(wpv + v), wp);
      uint4 o;
      o.x = pack2_bf16(f[0] * rf * wp[0], f[1] * rf * wp[1]);
      o.y = pack2_bf16(f[2] * rf * wp[2], f[3] * rf * wp[3]);
      o.z = pack2_bf16(f[4] * rf * wp[4], f[5] * rf * wp[5]);
      o.w = pack2_bf16(f[6] * rf * wp[6], f[7] * rf * wp[7]);
      xdrow[v] = o;
    }
    if (lane == 0) {
      p.r_out[t] = rf;
      p.xnorm_out[t] = rf * cH * sqrtf(ss) * 1.001f;  // rounded up: used in a bound
    }
    if (p.y_moe) {
      float4* yr = reinterpret_cast<float4*>(p.y_moe + (size_t)t * H);
      for (int v = lane; v < (H >> 2); v += 32) yr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int e = ((int)blockIdx.x - nbt) * 8 + warp;
  if (e >= p.E) return;
  const int ngroups = H >> 6;
  const uint4* sv = reinterpret_cast<const uint4*>(p.router_scale);
  uint4* phi = reinterpret_cast<uint4*>(p.planes + (size_t)e * 2 * H);
  uint4* plo = reinterpret_cast<uint4*>(p.planes + (size_t)e * 2 * H + H);
  float wsq = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    float w[8], sc[8];
    unpack8(__ldg(sv + v), sc);
    if constexpr (!U8) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                   (size_t)e * H) + v), w);
    } else {
      const uint2 q2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.wr) +
                                                            (size_t)e * H) + v);
      const int g = (8 * v) >> 6;
      const float gs = bf16_to_f32(p.wr_scales[(size_t)e * ngroups + g]);
      const float gb = bf16_to_f32(p.wr_biases[(size_t)e * ngroups + g]);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = fmaf(gs, (float)((((i < 4) ? q2.x : q2.y) >> (8 * (i & 3))) & 0xffu), gb);
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = w[2 * i] * sc[2 * i], b = w[2 * i + 1] * sc[2 * i + 1];
      wsq = fmaf(a, a, fmaf(b, b, wsq));
      const uint16_t ah = f32_to_bf16_rne(a), bh = f32_to_bf16_rne(b);
      hw[i] = (uint32_t)ah | ((uint32_t)bh << 16);
      lw[i] = pack2_bf16(a - bf16_to_f32(ah), b - bf16_to_f32(bh));
    }
    phi[v] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    plo[v] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  wsq = warp_sum_f(wsq);
  if (lane == 0) p.wnorm_out[e] = sqrtf(wsq) * 1.001f;  // rounded up: a bound
}

constexpr int kLogitEPT = 2;                    // experts per thread of k_router_logits
constexpr int kLogitExperts = 32 * kLogitEPT;  // experts per block of k_router_logits
constexpr int kLogitSlices = 8;    // K slices per expert (lanes of one warp)

// Logits for TB tokens x 64 experts.  Thread (el, slice j) handles experts
// el and el + 32 of the block's column and sums the 16-element runs
// k = 16 (8 q + j) .. + 15 of the hidden dimension, so the eight slices of an
// expert read one contiguous 256-byte run of its router row; every router
// input value read from shared memory serves both experts.  The h rows of the block and the per-channel vectors are loaded into
// shared memory in one round; the router input is built there, laid out
// [token][slice][H/8 + 4] (the padding puts the eight slices of a warp on
// distinct banks).  Blocks of the first expert column also write r, |x|,
// xd and zero the y_moe rows.
template <int TB, bool U8>
__global__ void __launch_bounds__(256) k_router_logits(const RouterParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int H = p.H, E = p.E;
  const int L = H / kLogitSlices;   // K elements per slice (multiple of 16)
  const int LS = L + 4;             // padded slice stride (floats)
  float* xs = reinterpret_cast<float*>(sm);                                   // [TB][8][LS]
  uint4* hs = reinterpret_cast<uint4*>(xs + (size_t)TB * kLogitSlices * LS);  // [TB][H/8]
  uint4* rss = hs + (size_t)TB * (H >> 3);                                    // router_scale
  uint4* wps = rss + (H >> 3);                                                // w_pre_ff
  uint4* was = wps + (H >> 3);                   // w_post_attn (fused neighbour only)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TB;
  const bool first_col = blockIdx.y == 0;
  const int nvec = H >> 3;
  const float cH = p.cH;
  const int ngroups = H >> 6;

  // thread (expert el, slice j); its first weight runs are requested before
  // the dependency wait and the router input is built (the router weights
  // are constant), so their latency overlaps both
  pdl_trigger();
  constexpr int EPT = kLogitEPT;
  const int el = threadIdx.x >> 3, j = threadIdx.x & 7;
  int ee[EPT];
  bool evalid[EPT];
#pragma unroll
  for (int q = 0; q < EPT; ++q) {
    const int er = blockIdx.y * kLogitExperts + el + 32 * q;
    evalid[q] = er < E;
    ee[q] = er < E ? er : E - 1;
  }
  // router weights of one 16-run for this thread's experts
  auto load_run = [&](int c, uint4 (&raw)[EPT][2]) {
    if (c < L) {
      const int k0 = ((c >> 4) * kLogitSlices + j) * 16;  // interleaved 16-runs
#pragma unroll
      for (int q = 0; q < EPT; ++q) {
        if constexpr (!U8) {
          const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                              (size_t)ee[q] * H + k0);
          raw[q][0] = __ldg(wrow);
          raw[q][1] = __ldg(wrow + 1);
        } else {
          raw[q][0] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.wr) +
                                                           (size_t)ee[q] * H + k0));
        }
      }
    }
  };
  // kRuns runs in flight (a register ring; run c + 16 kRuns is requested as
  // run c is consumed)
  constexpr int kRuns = 4;
  uint4 ring[kRuns][EPT][2];
#pragma unroll
  for (int r = 0; r < kRuns; ++r) load_run(16 * r, ring[r]);
  pdl_wait();

  // ---- phase 1: h rows and vectors in one round of loads, router input, xd
  for (int i = threadIdx.x; i < TB * nvec; i += blockDim.x) {
    const int tl = i / nvec, v = i - tl * nvec;
    const int t = t0 + tl;
    hs[i] = t < p.T ? __ldg(reinterpret_cast<const uint4*>(p.h + (size_t)t * H) + v)
                    : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    rss[v] = __ldg(reinterpret_cast<const uint4*>(p.router_scale) + v);
    if (first_col) wps[v] = __ldg(reinterpret_cast<const uint4*>(p.w_pre_ff) + v);
    if (p.attn) was[v] = __ldg(reinterpret_cast<const uint4*>(p.w_post_attn) + v);
  }
  __syncthreads();
  if (p.attn) {
    // the block input from the attention half, in place of the residual
    // rows; the first expert column publishes it
    for (int tl = warp; tl < TB; tl += 8) {
      const int t = t0 + tl;
      if (t >= p.T) continue;
      const uint4* arow = reinterpret_cast<const uint4*>(p.attn + (size_t)t * H);
      const float ra = row_rinv(arow, nvec, H, p.eps, lane);
      uint4* hrow = hs + (size_t)tl * nvec;
      uint4* hout = reinterpret_cast<uint4*>(p.h_out + (size_t)t * H);
      for (int v = lane; v < nvec; v += 32) {
        const uint4 hv = attn_residual8(hrow[v], __ldg(arow + v), was[v], ra);
        hrow[v] = hv;
        if (first_col) hout[v] = hv;
      }
    }
    __syncthreads();
  }

  for (int tl = warp; tl < TB; tl += 8) {
    const int t = t0 + tl;
    float* xrow = xs + (size_t)tl * kLogitSlices * LS;
    const uint4* hrow = hs + (size_t)tl * nvec;
    float ss = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(hrow[v], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum_f(ss);
    // 1/rms in fp32 (rsqrt and one Newton step); its error is a factor
    // common to all logits of the token
    const float msq = ss / (float)H + p.eps;
    float rf = rsqrtf(msq);
    rf = rf * (1.5f - 0.5f * msq * rf * rf);
    float xnl = 0.f;
    uint4* xdrow = reinterpret_cast<uint4*>(p.xd + (size_t)t * H);
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
      float f[8], sc[8];
      unpack8(hrow[v], f);
      unpack8(rss[v], sc);
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = f[i] * rf * sc[i] * cH;
        xnl = fmaf(x[i], x[i], xnl);
      }
      // element k goes to slice (k / 16) % 8 at position (k / 128) * 16 + k % 16
      const int k = 8 * v, sl = (k >> 4) & 7, off = ((k >> 7) << 4) + (k & 15);
      float4* xo = reinterpret_cast<float4*>(xrow + sl * LS + off);
      xo[0] = make_float4(x[0], x[1], x[2], x[3]);
      xo[1] = make_float4(x[4], x[5], x[6], x[7]);
      if (first_col && t < p.T) {
        float wp[8];
        unpack8(wps[v], wp);
        uint4 o;
        o.x = pack2_bf16(f[0] * rf * wp[0], f[1] * rf * wp[1]);
        o.y = pack2_bf16(f[2] * rf * wp[2], f[3] * rf * wp[3]);
        o.z = pack2_bf16(f[4] * rf * wp[4], f[5] * rf * wp[5]);
        o.w = pack2_bf16(f[6] * rf * wp[6], f[7] * rf * wp[7]);
        xdrow[v] = o;
      }
    }
    if (first_col && t < p.T) {
      const float xnd = warp_sum_f(xnl);
      if (lane == 0) {
        p.r_out[t] = rf;
        p.xnorm_out[t] = sqrtf(xnd) * 1.001f;  // rounded up: used in a bound
      }
      if (p.y_moe) {
        float4* yr = reinterpret_cast<float4*>(p.y_moe + (size_t)t * H);
        for (int v = lane; v < (H >> 2); v += 32) yr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  __syncthreads();

  // ---- phase 2: 16-term chunk sums (two 8-term fp32x2 halves, even and odd
  // elements), accumulated over the slice as error-free fp32 pairs; the
  // eight slices of an expert are then summed with shuffles.  Weights two
  // runs ahead are loaded while the current run computes.
  float acc_hi[EPT][TB], acc_lo[EPT][TB];
  float2 wsq2[EPT];
#pragma unroll
  for (int q = 0; q < EPT; ++q) {
    wsq2[q] = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      acc_hi[q][t] = 0.f;
      acc_lo[q][t] = 0.f;
    }
  }
  const bool need_norm = blockIdx.x == 0;
  for (int c = 0; c < L; c += 16) {
    const int k0 = ((c >> 4) * kLogitSlices + j) * 16;
    float2 w2[EPT][8];
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
      if constexpr (!U8) {
        const uint32_t wd[8] = {ring[0][q][0].x, ring[0][q][0].y, ring[0][q][0].z,
                                ring[0][q][0].w, ring[0][q][1].x, ring[0][q][1].y,
                                ring[0][q][1].z, ring[0][q][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w2[q][i] = make_float2(__uint_as_float(wd[i] << 16), __uint_as_float(wd[i] & 0xffff0000u));
      } else {
        // a 16-run never straddles a 64-group (16 | k0)
        const float gs = bf16_to_f32(p.wr_scales[(size_t)ee[q] * ngroups + (k0 >> 6)]);
        const float gb = bf16_to_f32(p.wr_biases[(size_t)ee[q] * ngroups + (k0 >> 6)]);
        const uint32_t wd[4] = {ring[0][q][0].x, ring[0][q][0].y, ring[0][q][0].z,
                                ring[0][q][0].w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w2[q][i] = make_float2(fmaf(gs, (float)((wd[i >> 1] >> (16 * (i & 1))) & 0xffu), gb),
                                 fmaf(gs, (float)((wd[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu), gb));
      }
      if (need_norm) {
#pragma unroll
        for (int i = 0; i < 8; ++i) wsq2[q] = __ffma2_rn(w2[q][i], w2[q][i], wsq2[q]);
      }
    }
#pragma unroll
    for (int r = 0; r + 1 < kRuns; ++r)
#pragma unroll
      for (int q = 0; q < EPT; ++q) {
        ring[r][q][0] = ring[r + 1][q][0];
        ring[r][q][1] = ring[r + 1][q][1];
      }
    load_run(c + 16 * kRuns, ring[kRuns - 1]);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const float4* xv =
          reinterpret_cast<const float4*>(xs + ((size_t)t * kLogitSlices + j) * LS + c);
      float4 xa[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) xa[r] = xv[r];
#pragma unroll
      for (int q = 0; q < EPT; ++q) {
        float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          a2 = __ffma2_rn(w2[q][2 * r], make_float2(xa[r].x, xa[r].y), a2);
          b2 = __ffma2_rn(w2[q][2 * r + 1], make_float2(xa[r].z, xa[r].w), b2);
        }
        df_add(acc_hi[q][t], acc_lo[q][t],
               __fadd_rn(__fadd_rn(a2.x, a2.y), __fadd_rn(b2.x, b2.y)));
      }
    }
  }
#pragma unroll
  for (int q = 0; q < EPT; ++q) {
    float wsq = wsq2[q].x + wsq2[q].y;
#pragma unroll
    for (int o = 1; o < kLogitSlices; o <<= 1) {
      wsq += __shfl_xor_sync(kFull, wsq, o);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const float h2 = __shfl_xor_sync(kFull, acc_hi[q][t], o);
        const float l2 = __shfl_xor_sync(kFull, acc_lo[q][t], o);
        df_add2(acc_hi[q][t], acc_lo[q][t], h2, l2);
      }
    }
    if (j == 0 && evalid[q]) {
      const int e = ee[q];
      const double bias = p.router_bias ? (double)p.router_bias[e] : 0.0;
#pragma unroll
      for (int t = 0; t < TB; ++t)
        if (t0 + t < p.T)
          p.logits[(size_t)(t0 + t) * E + e] = (float)(df_value(acc_hi[q][t], acc_lo[q][t]) + bias);
      if (need_norm) p.wnorm_out[e] = sqrtf(wsq) * 1.001f;  // rounded up: a bound
    }
  }
}

// Logits for large batches: a register-tiled product of 64 tokens x 64
// experts per block, K in chunks of 32 staged in shared memory (router input
// and decoded weights as fp32, K-major).  Thread (ty, tx) accumulates the
// 4 x 4 tile tokens 4ty.., experts 4tx..; each 32-term chunk sum (sequential
// fp32 FMAs, error <= 32 u of the chunk's sum of |terms|) is folded into an
// error-free fp32 pair, so the logits carry the same bound as the
// small-batch kernel.  The raw inputs of the next chunk are loaded into
// registers while the current chunk computes.  The router weights are read
// once per 64 tokens; the per-token work (1/rms, and in the first expert
// column |x|, xd and the y_moe zeroing) once per token and column.
constexpr int kRT = 64;   // tokens per block
constexpr int kRE = 64;   // experts per block
constexpr int kRK = 32;   // K per staged chunk
constexpr int kXS = kRT + 4;
constexpr int kWS = kRE + 4;

template <bool U8, bool FUSED>
__global__ void __launch_bounds__(256, 3) k_router_logits_tile(const RouterParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  float* xT = reinterpret_cast<float*>(sm);           // [2][kRK][kXS]
  float* wT = xT + 2 * kRK * kXS;                     // [2][kRK][kWS]
  float* rs = wT + 2 * kRK * kWS;                     // [kRT] 1/rms
  float* ras = rs + kRT;                              // [kRT] 1/rms of attn (fused)
  uint16_t* sc_s = reinterpret_cast<uint16_t*>(ras + kRT);  // [H] router_scale
  uint16_t* wa_s = sc_s + p.H;                        // [H] w_post_attn (fused)
  const int H = p.H, E = p.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int t0 = blockIdx.x * kRT, e0 = blockIdx.y * kRE;
  const bool first_col = blockIdx.y == 0;
  const float cH = p.cH;
  const int nvec = H >> 3;
  pdl_trigger();
  pdl_wait();

  constexpr bool fused = FUSED;
  for (int v = tid; v < nvec; v += 256) {
    reinterpret_cast<uint4*>(sc_s)[v] = __ldg(reinterpret_cast<const uint4*>(p.router_scale) + v);
    if (fused)
      reinterpret_cast<uint4*>(wa_s)[v] = __ldg(reinterpret_cast<const uint4*>(p.w_post_attn) + v);
  }
  __syncthreads();

  // ---- per token: 1/rms (and, in the first expert column, |x|, xd, y_moe = 0;
  // with the fused attention half, the block input is rebuilt from the
  // residual and attention rows wherever it is read, and published here)
  for (int tl = warp; tl < kRT; tl += 8) {
    const int t = t0 + tl;
    if (t >= p.T) {
      if (lane == 0) rs[tl] = 0.f;
      if (lane == 0) ras[tl] = 0.f;
      continue;
    }
    const uint4* hrow = reinterpret_cast<const uint4*>(p.h + (size_t)t * H);
    const uint4* arow = reinterpret_cast<const uint4*>(fused ? p.attn + (size_t)t * H : p.h);
    const float ra = fused ? row_rinv(arow, nvec, H, p.eps, lane) : 0.f;
    if (lane == 0) ras[tl] = ra;
    auto hvec = [&](int v) {
      return fused ? attn_residual8(__ldg(hrow + v), __ldg(arow + v),
                                    reinterpret_cast<const uint4*>(wa_s)[v], ra)
                   : __ldg(hrow + v);
    };
    float ss = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(hvec(v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum_f(ss);
    const float msq = ss / (float)H + p.eps;
    float rf = rsqrtf(msq);
    rf = rf * (1.5f - 0.5f * msq * rf * rf);
    if (lane == 0) rs[tl] = rf;
    if (first_col) {
      float xnl = 0.f;
      uint4* xdrow = reinterpret_cast<uint4*>(p.xd + (size_t)t * H);
      uint4* hout = reinterpret_cast<uint4*>(fused ? p.h_out + (size_t)t * H : p.xd);
      for (int v = lane; v < nvec; v += 32) {
        float f[8], sc[8], wp[8];
        const uint4 hv = hvec(v);
        if (fused) hout[v] = hv;
        unpack8(hv, f);
        unpack8(reinterpret_cast<const uint4*>(sc_s)[v], sc);
        unpack8(__ldg(reinterpret_cast<const uint4*>(p.w_pre_ff) + v), wp);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x = f[i] * rf * sc[i] * cH;
          xnl = fmaf(x, x, xnl);
        }
        uint4 o;
        o.x = pack2_bf16(f[0] * rf * wp[0], f[1] * rf * wp[1]);
        o.y = pack2_bf16(f[2] * rf * wp[2], f[3] * rf * wp[3]);
        o.z = pack2_bf16(f[4] * rf * wp[4], f[5] * rf * wp[5]);
        o.w = pack2_bf16(f[6] * rf * wp[6], f[7] * rf * wp[7]);
        xdrow[v] = o;
      }
      const float xnd = warp_sum_f(xnl);
      if (lane == 0) {
        p.r_out[t] = rf;
        p.xnorm_out[t] = sqrtf(xnd) * 1.001f;  // rounded up: used in a bound
      }
      if (p.y_moe) {
        float4* yr = reinterpret_cast<float4*>(p.y_moe + (size_t)t * H);
        for (int v = lane; v < (H >> 2); v += 32) yr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  __syncthreads();

  // ---- staging: thread (row, octet) moves 8 K values of token row xt and of
  // expert row we; the raw values of the next chunk wait in registers
  const int xt = tid & 63, oc = tid >> 6;
  const int we = tid & 63;
  const int e_load = e0 + we < E ? e0 + we : E - 1;
  const bool need_norm = blockIdx.x == 0;
  const bool tok_ok = t0 + xt < p.T;
  const float rx = rs[xt];
  const float rax = ras[xt];
  float wsq = 0.f;
  uint4 hv;   // next chunk: 8 h values of token xt (the residual, when fused)
  uint4 av;   // next chunk: 8 attention values of token xt (fused only)
  uint4 wv;   // next chunk: 8 router weights of expert we (bf16, or 8 codes in .x/.y)
  auto fetch = [&](int k0) {
    const int k = k0 + 8 * oc;
    hv = tok_ok ? __ldg(reinterpret_cast<const uint4*>(p.h + (size_t)(t0 + xt) * H + k))
                : make_uint4(0u, 0u, 0u, 0u);
    if (fused)
      av = tok_ok ? __ldg(reinterpret_cast<const uint4*>(p.attn + (size_t)(t0 + xt) * H + k))
                  : make_uint4(0u, 0u, 0u, 0u);
    if constexpr (!U8) {
      wv = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                (size_t)e_load * H + k));
    } else {
      const uint2 q2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.wr) +
                                                            (size_t)e_load * H + k));
      wv = make_uint4(q2.x, q2.y, 0u, 0u);
    }
  };
  auto store = [&](int buf, int k0) {
    const int k = k0 + 8 * oc;
    float* xb = xT + buf * kRK * kXS + (8 * oc) * kXS + xt;
    float* wb = wT + buf * kRK * kWS + (8 * oc) * kWS + we;
    float f[8], sc[8];
    unpack8(fused ? attn_residual8(hv, av, reinterpret_cast<const uint4*>(wa_s)[k >> 3], rax) : hv,
            f);
    unpack8(reinterpret_cast<const uint4*>(sc_s)[k >> 3], sc);
#pragma unroll
    for (int i = 0; i < 8; ++i) xb[i * kXS] = f[i] * rx * sc[i] * cH;
    float w[8];
    if constexpr (!U8) {
      unpack8(wv, w);
    } else {
      const int g = k >> 6;
      const float gs = bf16_to_f32(p.wr_scales[(size_t)e_load * (H >> 6) + g]);
      const float gb = bf16_to_f32(p.wr_biases[(size_t)e_load * (H >> 6) + g]);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = fmaf(gs, (float)((((i < 4) ? wv.x : wv.y) >> (8 * (i & 3))) & 0xffu), gb);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      wb[i * kWS] = w[i];
      if (need_norm) wsq = fmaf(w[i], w[i], wsq);
    }
  };

  // ---- tiled product
  const int ty = tid >> 4, tx = tid & 15;
  float hi[4][4], lo[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      hi[a][b] = 0.f;
      lo[a][b] = 0.f;
    }
  const int nch = H / kRK;
  fetch(0);
  store(0, 0);
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    const int cur = c & 1;
    if (c + 1 < nch) fetch((c + 1) * kRK);
    const float* xb = xT + cur * kRK * kXS + 4 * ty;
    const float* wb = wT + cur * kRK * kWS + 4 * tx;
    float2 acc[4][2];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      acc[a][0] = make_float2(0.f, 0.f);
      acc[a][1] = make_float2(0.f, 0.f);
    }
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float4 xa = *reinterpret_cast<const float4*>(xb + kk * kXS);
      const float4 w4 = *reinterpret_cast<const float4*>(wb + kk * kWS);
      const float xs[4] = {xa.x, xa.y, xa.z, xa.w};
      const float2 w01 = make_float2(w4.x, w4.y), w23 = make_float2(w4.z, w4.w);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        acc[a][0] = __ffma2_rn(make_float2(xs[a], xs[a]), w01, acc[a][0]);
        acc[a][1] = __ffma2_rn(make_float2(xs[a], xs[a]), w23, acc[a][1]);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      df_add(hi[a][0], lo[a][0], acc[a][0].x);
      df_add(hi[a][1], lo[a][1], acc[a][0].y);
      df_add(hi[a][2], lo[a][2], acc[a][1].x);
      df_add(hi[a][3], lo[a][3], acc[a][1].y);
    }
    if (c + 1 < nch) store(cur ^ 1, (c + 1) * kRK);
    __syncthreads();
  }

  // ---- |W_e| from the first token block; logits
  if (need_norm) {
    float* red = xT;  // staging buffers are free now
    red[tid] = wsq;
    __syncthreads();
    if (tid < kRE && e0 + tid < E)
      p.wnorm_out[e0 + tid] =
          sqrtf(red[tid] + red[tid + 64] + red[tid + 128] + red[tid + 192]) * 1.001f;
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int e = e0 + 4 * tx + b;
    if (e >= E) continue;
    const double bias = p.router_bias ? (double)p.router_bias[e] : 0.0;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int t = t0 + 4 * ty + a;
      if (t < p.T) p.logits[(size_t)t * E + e] = (float)(df_value(hi[a][b], lo[a][b]) + bias);
    }
  }
}

size_t router_tile_smem(int H) {
  return sizeof(float) * (2 * kRK * kXS + 2 * kRK * kWS + 2 * kRT) + (size_t)H * 4;
}

template <bool U8, bool FUSED>
cudaError_t launch_router_tile_f(const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_tile_smem(p.H);
  const dim3 grid((p.T + kRT - 1) / kRT, (p.E + kRE - 1) / kRE);
  return launch_pdl(k_router_logits_tile<U8, FUSED>, grid, dim3(256), smem, s, p);
}
template <bool U8>
cudaError_t launch_router_tile(const RouterParams& p, cudaStream_t s) {
  return p.attn ? launch_router_tile_f<U8, true>(p, s) : launch_router_tile_f<U8, false>(p, s);
}

// Exact logits: sum_i W_ei (router_scale_i h_i) with every term exact in
// fp32 (a bf16 triple product has at most 24 significant bits; an 8-bit
// affine weight is first split into two exact fp32 parts), summed as
// error-free fp32 pairs; 1/rms from the exact sum of squares (bf16 squares
// are exact).
__device__ __forceinline__ void exact_terms_bf16(const uint4& hv, const uint4& sv, const uint4& wv,
                                                 float& hi, float& lo) {
  float hf[8], sf[8], wf[8];
  unpack8(hv, hf);
  unpack8(sv, sf);
  unpack8(wv, wf);
#pragma unroll
  for (int i = 0; i < 8; ++i) df_add(hi, lo, __fmul_rn(wf[i], __fmul_rn(sf[i], hf[i])));
}
__device__ __forceinline__ void exact_terms_u8(const uint4& hv, const uint4& sv, uint32_t qx,
                                               uint32_t qy, float gs, float gb, float& hi,
                                               float& lo) {
  float hf[8], sf[8];
  unpack8(hv, hf);
  unpack8(sv, sf);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t code = ((i < 4 ? qx : qy) >> (8 * (i & 3))) & 0xffu;
    float wh, wl;
    two_sum(__fmul_rn(gs, (float)code), gb, wh, wl);  // W = wh + wl exactly
    const float sh = __fmul_rn(sf[i], hf[i]);           // exact (16 bits)
    const float p1 = __fmul_rn(wh, sh);
    df_add(hi, lo, p1);
    df_add(hi, lo, fmaf(wh, sh, -p1));                  // exact product error
    df_add(hi, lo, __fmul_rn(wl, sh));
  }
}
__device__ __forceinline__ void exact_squares(const uint4& hv, float& hi, float& lo) {
  float hf[8];
  unpack8(hv, hf);
#pragma unroll
  for (int i = 0; i < 8; ++i) df_add(hi, lo, __fmul_rn(hf[i], hf[i]));
}

constexpr int kSelTokens = 8;

// Order-preserving map of a float (no NaN) to an unsigned key, and back; -0
// and +0 compare equal as floats, so -0 is first made +0.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}


// Eight tokens per block, warp per token: top-k of the fp32 logits; where
// the k-th / (k+1)-th boundary is closer than the error bound, the candidate
// experts get exact logits; then reselection, softmax of the k selected
// logits times per_expert_scale, outputs in ascending expert order and the
// per-chunk expert histogram.  For the exact logits, warp w owns the slice
// [w H/8, (w+1) H/8) of the hidden dimension and walks every (token,
// candidate) job of the block four at a time; the eight partial sums of a
// job are combined in a fixed order.
template <bool U8, int SLOTS, int MODE>
__global__ void __launch_bounds__(256) k_router_select(const RouterParams p) {
  __shared__ int s_cand[kSelTokens][256];
  __shared__ int s_ncand[kSelTokens];
  __shared__ double s_zx[kSelTokens][256];
  __shared__ double s_ss[kSelTokens];
  __shared__ int s_tok[kSelTokens];
  const int H = p.H, E = p.E, K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  // groups of eight tokens: consecutive ones (modes 0, 1), or the tokens the
  // fast pass flagged (mode 2, a persistent loop over the list)
  // (mode 2: G flagged tokens a group, as many as spread the list over the
  // grid, so a short list still uses every block and a token's exact jobs
  // spread over all eight warps)
  const int nflag = MODE == 2 ? *p.n_flagged : 0;
  const int G = MODE == 2 ? min(kSelTokens, max(1, (nflag + (int)gridDim.x - 1) / (int)gridDim.x))
                          : kSelTokens;
  const int ngrp = MODE == 2 ? (nflag + G - 1) / G : (int)gridDim.x;
  for (int grp = blockIdx.x; grp < ngrp; grp += (MODE == 2 ? (int)gridDim.x : ngrp)) {
  int t;
  bool valid;
  if (MODE == 2) {
    const int i = grp * G + warp;
    valid = warp < G && i < nflag;
    t = valid ? p.flagged[i] : 0;
  } else {
    t = grp * kSelTokens + warp;
    valid = t < p.T;
  }
  if (lane == 0) s_tok[warp] = t;

  // ---- A: selection on the fp32 logits, candidate list if near a tie
  float zl[SLOTS];
  uint32_t taken = 0, certain = 0;  // slot masks of this lane
  int ncand = 0;
  if (valid) {
    const float* z = p.logits + (size_t)t * E;
    const float xnt = p.xnorm_out[t];
    const float bound = p.logits_tc ? tc_logit_bound(H, p.z_split > 1 ? p.z_split : 1,
                                                     p.router_bias != nullptr)
                                    : (p.router_bias ? kLogitBoundBias : kLogitBoundNoBias);
    // split-K logits: the partial sums added error-free (hi, lo), then
    // z = hi rc + (lo rc + bias) in fp32, as the unsplit epilogue does; the
    // logits are written for the record
    const float rc = p.z_part ? p.r_out[t] * p.cH : 0.f;
    float el[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int e = 32 * s + lane;
      if (e < E) {
        float v;
        if (p.z_part) {
          float hi = 0.f, lo = 0.f;
          for (int r = 0; r < p.z_split; ++r)
            df_add(hi, lo, p.z_part[((size_t)r * p.T + t) * E + e]);
          v = fmaf(hi, rc, fmaf(lo, rc, p.router_bias ? p.router_bias[e] : 0.f));
          if (MODE != 2) p.logits[(size_t)t * E + e] = v;
        } else {
          v = z[e];
        }
        zl[s] = isnan(v) ? -INFINITY : v;
        const float b = p.router_bias ? fabsf(p.router_bias[e]) : 0.f;
        el[s] = bound * (p.wnorm_out[e] * xnt + b) + 1e-30f;
      } else {
        zl[s] = -INFINITY;
        el[s] = 0.f;
      }
    }
    // k rounds: each lane's best untaken slot (ties to the lower expert),
    // then the warp's largest key and, among lanes holding it, the lowest
    // expert index (two integer reductions per round)
    uint32_t zk[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) zk[s] = order_key(zl[s]);
    for (int k = 0; k < K; ++k) {
      uint32_t bk = 0;
      uint32_t be = 0xffffffffu;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int e = 32 * s + lane;
        if (e < E && !((taken >> s) & 1u) && zk[s] > bk) {  // slots ascend in e
          bk = zk[s];
          be = (uint32_t)e;
        }
      }
      const uint32_t wk = __reduce_max_sync(kFull, bk);
      const uint32_t we = __reduce_min_sync(kFull, bk == wk ? be : 0xffffffffu);
      if ((int)(we & 31) == lane) taken |= 1u << (we >> 5);
    }
    uint32_t lk = 0xffffffffu, uk = 0u;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      if (32 * s + lane >= E) continue;
      if ((taken >> s) & 1u) lk = min(lk, order_key(zl[s] - el[s]));
      else uk = max(uk, order_key(zl[s] + el[s]));
    }
    const float L = key_value(__reduce_min_sync(kFull, lk));
    const uint32_t ukw = __reduce_max_sync(kFull, uk);
    const float U = ukw == 0u ? -INFINITY : key_value(ukw);  // 0: every expert taken
    if (!(L > U)) {
      // A selected expert whose lower bound is above every unselected upper
      // bound beats every unselected expert exactly, so at most k - 1 others
      // can beat it: it is certainly in the exact top-k.  The other m' = k - m
      // places go to the exact top-m' of the rest.  Let L2 be the smallest
      // lower bound of the uncertain selected experts: the m' of them have
      // exact logits >= L2, so every member of that exact top-m' has an upper
      // bound >= L2.  Those are the candidates (ascending expert order); they
      // get exact logits.
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if (((taken >> s) & 1u) && zl[s] - el[s] > U) certain |= 1u << s;
      uint32_t l2k = 0xffffffffu;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if (((taken & ~certain) >> s) & 1u) l2k = min(l2k, order_key(zl[s] - el[s]));
      const float L2 = key_value(__reduce_min_sync(kFull, l2k));
      const unsigned lt = (1u << lane) - 1u;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const bool c = 32 * s + lane < E && !((certain >> s) & 1u) && zl[s] + el[s] >= L2;
        const unsigned ms = __ballot_sync(kFull, c);
        if (c) s_cand[warp][ncand + __popc(ms & lt)] = 32 * s + lane;
        ncand += __popc(ms);
      }
    }
  }
  if (MODE == 1 && ncand > 0) {
    // near a tie: left to the re-check pass, which writes this token's outputs
    if (lane == 0) p.flagged[atomicAdd(p.n_flagged, 1)] = t;
    valid = false;
    ncand = 0;
  }
  if (lane == 0) s_ncand[warp] = ncand;
  __syncthreads();

  // ---- B: exact logits.  Jobs of a near-tie token: its sum of squares
  // (c = -1), then its candidates (c = 0 .. ncand-1).  One warp per job: the
  // whole dot product over H, its loads issued in batches, lanes strided over
  // the 8-element vectors, then a fixed shuffle tree.
  int njobs = 0, first[kSelTokens + 1];
#pragma unroll
  for (int w = 0; w < kSelTokens; ++w) {
    first[w] = njobs;
    njobs += s_ncand[w] > 0 ? s_ncand[w] + 1 : 0;
  }
  first[kSelTokens] = njobs;
  if (MODE != 1 && njobs > 0) {
    const int nvec = H >> 3;
    const int ngroups = H >> 6;
    const uint4* sv = reinterpret_cast<const uint4*>(p.router_scale);
    for (int job = warp; job < njobs; job += kSelTokens) {
      int w = 0;
#pragma unroll
      for (int q = 1; q < kSelTokens; ++q)
        if (job >= first[q]) w = q;
      const int c = job - first[w] - 1;
      const int e = c >= 0 ? s_cand[w][c] : -1;
      const int tt = s_tok[w];
      const uint4* hrow = reinterpret_cast<const uint4*>(p.h + (size_t)tt * H);
      // kB independent (hi, lo) chains, one per vector of a batch
      constexpr int kB = 4;  // vectors per lane in flight
      float hi4[kB], lo4[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        hi4[u] = 0.f;
        lo4[u] = 0.f;
      }
      for (int v0 = lane; v0 < nvec; v0 += 32 * kB) {
        uint4 rh[kB], rs[kB], rw[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int v = v0 + 32 * u;
          if (v < nvec) {
            rh[u] = __ldg(hrow + v);
            if (e >= 0) {
              rs[u] = __ldg(sv + v);
              if constexpr (!U8) {
                rw[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                             (size_t)e * H) + v);
              } else {
                const uint2 q2 = __ldg(reinterpret_cast<const uint2*>(
                                           static_cast<const uint8_t*>(p.wr) + (size_t)e * H) + v);
                rw[u] = make_uint4(q2.x, q2.y, 0u, 0u);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int v = v0 + 32 * u;
          if (v >= nvec) continue;
          if (e < 0) {
            exact_squares(rh[u], hi4[u], lo4[u]);
          } else if constexpr (!U8) {
            exact_terms_bf16(rh[u], rs[u], rw[u], hi4[u], lo4[u]);
          } else {
            const int gi = (8 * v) >> 6;
            exact_terms_u8(rh[u], rs[u], rw[u].x, rw[u].y,
                           bf16_to_f32(p.wr_scales[(size_t)e * ngroups + gi]),
                           bf16_to_f32(p.wr_biases[(size_t)e * ngroups + gi]), hi4[u], lo4[u]);
          }
        }
      }
      float hi = hi4[0], lo = lo4[0];
#pragma unroll
      for (int u = 1; u < kB; ++u) df_add2(hi, lo, hi4[u], lo4[u]);
#pragma unroll
      for (int o = 16; o; o >>= 1)
        df_add2(hi, lo, __shfl_xor_sync(kFull, hi, o), __shfl_xor_sync(kFull, lo, o));
      if (lane == 0) {
        if (c < 0) s_ss[w] = df_value(hi, lo);
        else s_zx[w][c] = df_value(hi, lo);
      }
    }
    __syncthreads();
    // exact logit = dot * (1/rms) * H^-1/2 + bias
    const double cHd = p.cHd;
    for (int i = threadIdx.x; i < kSelTokens * 256; i += blockDim.x) {
      const int w = i >> 8, c = i & 255;
      if (c < s_ncand[w]) {
        const double r64 = 1.0 / sqrt(s_ss[w] / (double)H + (double)p.eps);
        const int e = s_cand[w][c];
        s_zx[w][c] = s_zx[w][c] * r64 * cHd + (p.router_bias ? (double)p.router_bias[e] : 0.0);
      }
    }
  }
  __syncthreads();
  if (valid) {
  // ---- C: reselection among the candidates, weights, outputs
  if (ncand > 0) {
    if (lane == 0) atomicAdd(p.n_refined, 1);
    // candidate c = lane + 32 q is held by this lane; bit q of usedc marks it
    // taken.  The certain experts stay; the rest of the k come from the
    // candidates by exact logit (ties to the lower index).
    int ncert = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) ncert += __popc(__ballot_sync(kFull, (certain >> s) & 1u));
    taken = certain;
    uint32_t usedc = 0;
    for (int k = ncert; k < K; ++k) {
      double bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < SLOTS; ++q) {
        const int c = lane + 32 * q;
        if (c < ncand && !((usedc >> q) & 1u)) {
          const int e = s_cand[warp][c];
          const double v = s_zx[warp][c];
          if (v > bv || (v == bv && e < be)) {
            bv = v;
            be = e;
          }
        }
      }
      warp_argmax(bv, be);
      if (be == 0x7fffffff) break;
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
#pragma unroll
      for (int q = 0; q < SLOTS; ++q) {
        const int c = lane + 32 * q;
        if (c < ncand && s_cand[warp][c] == be) usedc |= 1u << q;
      }
    }
  }
  float zmax = -INFINITY;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s)
    if ((taken >> s) & 1u) zmax = fmaxf(zmax, zl[s]);
  zmax = warp_max_f(zmax);
  float ex[SLOTS];
  float se = 0.f;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    ex[s] = ((taken >> s) & 1u) ? expf(zl[s] - zmax) : 0.f;
    se += ex[s];
  }
  se = warp_sum_f(se);
  int running = 0;
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const unsigned ms = __ballot_sync(kFull, (taken >> s) & 1u);
    if ((taken >> s) & 1u) {
      const int e = 32 * s + lane;
      const int rank = running + __popc(ms & lt);
      p.idx[(size_t)t * K + rank] = e;
      p.w[(size_t)t * K + rank] = ex[s] / se * bf16_to_f32(p.pes[e]);
      atomicAdd(&p.chunk_counts[(size_t)(t / kChunkTokens) * E + e], 1);
      if (p.chunk_masks)
        atomicOr(&p.chunk_masks[((size_t)(t / kChunkTokens) * E + e) * (kChunkTokens / 32) +
                                ((t % kChunkTokens) >> 5)],
                 1u << (t & 31));
    }
    running += __popc(ms);
  }
  }  // valid
  __syncthreads();  // the next group reuses the shared arrays
  }  // groups
}

// Exclusive scan over the 256 threads of a block; returns the exclusive
// prefix of v and leaves the total in *total.
__device__ int block_excl_scan256(int v, int* tmp, int* total) {
  const int tid = threadIdx.x;
  tmp[tid] = v;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    const int x = tid >= off ? tmp[tid - off] : 0;
    __syncthreads();
    tmp[tid] += x;
    __syncthreads();
  }
  const int incl = tmp[tid];
  *total = tmp[255];
  __syncthreads();
  return incl - v;
}

// Grouping and expert rows in one pass, token-major.  A block of 256 threads
// takes TPB consecutive tokens (one 256-token chunk holds them all) with
// 8 / TPB warps per token.  It rebuilds from the per-chunk histograms what
// it needs: the expert offsets (exclusive scan of the totals; block 0
// publishes them) and per expert the assignments in earlier chunks.  The
// stable position of assignment (t, j) with expert e is then offset[e] +
// earlier chunks' count + the chunk's tokens before t that chose e, counted
// in the chunk's token bit mask of e that the selection wrote (assignments
// sorted by expert, then token).  Each token's row of h is read once; xe = bf16(h / rms(h) *
// w_pre_ff2) is formed once and stored at its K grouped rows.
template <int TPB>
__global__ void __launch_bounds__(256) k_scatter_gather(const ScatterParams sp,
                                                        const GatherParams gp) {
  __shared__ int s_tmp[256];
  __shared__ int s_base[256];
  __shared__ int s_pos[TPB][16];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = sp.E, K = sp.K, T = sp.T;
  const int t0 = blockIdx.x * TPB;
  const int chunk = t0 / kChunkTokens, c0 = chunk * kChunkTokens;
  const int nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  int tot = 0, bef = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = sp.chunk_counts[(size_t)c * E + tid];
      tot += v;
      if (c < chunk) bef += v;
    }
  }
  int total;
  const int base = block_excl_scan256(tot, s_tmp, &total);
  s_base[tid] = base + bef;
  if (blockIdx.x == 0) {
    if (tid < E) sp.offsets[tid] = base;
    if (tid == 0) sp.offsets[E] = total;
  }
  __syncthreads();
  if (tid < TPB * K) {
    const int tt = tid / K, j = tid - tt * K, t = t0 + tt;
    if (t < T) {
      const int e = sp.idx[(size_t)t * K + j];
      int pos = 0;
      if ((unsigned)e < (unsigned)E) {
        const int tl = t - c0;
        const uint32_t* m = sp.chunk_masks + ((size_t)chunk * E + e) * (kChunkTokens / 32);
        int rank = __popc(__ldg(m + (tl >> 5)) & ((1u << (tl & 31)) - 1u));
        for (int w = 0; w < (tl >> 5); ++w) rank += __popc(__ldg(m + w));
        pos = s_base[e] + rank;
        sp.perm[pos] = t * K + j;
        sp.tok_perm[pos] = t;
        sp.w_perm[pos] = sp.w[(size_t)t * K + j];
        if (sp.inv) sp.inv[t * K + j] = pos;
      } else {
        report(sp.status, kDevBounds, kSiteScatter, (unsigned)t, (unsigned)e);
      }
      s_pos[tt][j] = pos;  // an out-of-range expert was reported; its row is not read
    }
  }
  __syncthreads();
  constexpr int WPT = 8 / TPB;  // warps per token
  const int tt = warp / WPT, part = warp - tt * WPT, t = t0 + tt;
  if (t >= T) return;
  const int nvec = gp.H >> 3;
  const float r = gp.r[t];
  const uint4* hrow = reinterpret_cast<const uint4*>(gp.h + (size_t)t * gp.H);
  const uint4* wv = reinterpret_cast<const uint4*>(gp.w_pre_ff2);
  int pos[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) pos[j] = j < K ? s_pos[tt][j] : 0;
  for (int v = part * 32 + lane; v < nvec; v += 32 * WPT) {
    float f[8], w[8];
    unpack8(__ldg(hrow + v), f);
    unpack8(__ldg(wv + v), w);
    uint4 o;
    o.x = pack2_bf16(f[0] * r * w[0], f[1] * r * w[1]);
    o.y = pack2_bf16(f[2] * r * w[2], f[3] * r * w[3]);
    o.z = pack2_bf16(f[4] * r * w[4], f[5] * r * w[5]);
    o.w = pack2_bf16(f[6] * r * w[6], f[7] * r * w[7]);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < K) reinterpret_cast<uint4*>(gp.xe_perm + (size_t)pos[j] * gp.H)[v] = o;
  }
}


template <int TB>
size_t router_smem(int H) {
  return sizeof(float) * (size_t)TB * kLogitSlices * (H / kLogitSlices + 4) +
         (size_t)(TB + 3) * H * 2;
}

template <int TB, bool U8>
cudaError_t launch_router_tb(const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_smem<TB>(p.H);
  const dim3 grid((p.T + TB - 1) / TB, (p.E + kLogitExperts - 1) / kLogitExperts);
  return launch_pdl(k_router_logits<TB, U8>, grid, dim3(256), smem, s, p);
}

}  // namespace

cudaError_t prepare_router(int smem_max) {
  cudaError_t e = cudaSuccess;
  auto one = [&](auto kernel) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  };
  one(k_router_logits<4, false>);
  one(k_router_logits<4, true>);
  one(k_router_logits_tile<false, false>);
  one(k_router_logits_tile<false, true>);
  one(k_router_logits_tile<true, false>);
  one(k_router_logits_tile<true, true>);
  return e;
}

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  // four tokens per block give a single canvas enough blocks; from a few
  // canvases on, the register-tiled kernel reads the router weights once per
  // 64 tokens and does the per-token work once
  if (p.T >= kRouterTileMinTokens) {
    return p.router_u8 ? launch_router_tile<true>(p, s) : launch_router_tile<false>(p, s);
  }
  return p.router_u8 ? launch_router_tb<4, true>(p, s) : launch_router_tb<4, false>(p, s);
}

cudaError_t launch_router_prep_tc(const RouterParams& p, cudaStream_t s) {
  const int nbt = (p.T + 7) / 8, nbe = (p.E + 7) / 8;
  const dim3 grid(nbt + nbe);
  if (p.attn)
    return p.router_u8 ? launch_pdl(k_router_prep_tc<true, true>, grid, dim3(256), 0, s, p, nbt)
                       : launch_pdl(k_router_prep_tc<false, true>, grid, dim3(256), 0, s, p, nbt);
  return p.router_u8 ? launch_pdl(k_router_prep_tc<true, false>, grid, dim3(256), 0, s, p, nbt)
                     : launch_pdl(k_router_prep_tc<false, false>, grid, dim3(256), 0, s, p, nbt);
}

template <bool U8, int SLOTS>
cudaError_t launch_select_slots(const RouterParams& p, int num_sms, cudaStream_t s) {
  const int grid = (p.T + kSelTokens - 1) / kSelTokens;
  if (!p.flagged) return launch_pdl(k_router_select<U8, SLOTS, 0>, dim3(grid), dim3(256), 0, s, p);
  // large batches: a fast pass over all tokens, then the near-tie tokens
  cudaError_t err = launch_pdl(k_router_select<U8, SLOTS, 1>, dim3(grid), dim3(256), 0, s, p);
  if (err != cudaSuccess) return err;
  const int g2 = grid < 2 * num_sms ? grid : 2 * num_sms;
  return launch_pdl(k_router_select<U8, SLOTS, 2>, dim3(g2), dim3(256), 0, s, p);
}

cudaError_t launch_router_select(const RouterParams& p, int num_sms, cudaStream_t s) {
  if (p.E <= 128)
    return p.router_u8 ? launch_select_slots<true, 4>(p, num_sms, s)
                       : launch_select_slots<false, 4>(p, num_sms, s);
  return p.router_u8 ? launch_select_slots<true, 8>(p, num_sms, s)
                     : launch_select_slots<false, 8>(p, num_sms, s);
}

cudaError_t launch_scatter_gather(const ScatterParams& sp, const GatherParams& gp,
                                  cudaStream_t s) {
  // small batches: two tokens a block (four warps each) for enough blocks;
  // large ones: eight (a warp each)
  if (sp.T < kRouterTcMinTokens)
    return launch_pdl(k_scatter_gather<2>, dim3((sp.T + 1) / 2), dim3(256), 0, s, sp, gp);
  return launch_pdl(k_scatter_gather<8>, dim3((sp.T + 7) / 8), dim3(256), 0, s, sp, gp);
}

}  // namespace dg
