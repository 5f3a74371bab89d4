// Routing of the MoE FFN block on sm_103a.
//
// k_router_logits / k_router_select: per token, RMS of the residual stream, router input
//   x = h / rms(h) * router_scale * H^-1/2 (two literal steps, "DiffusionGemma
//   port — plan & parity strategy", Reference dossier §2 Router and the D1
//   finding), E fp32 logits, top-k with ties to the lower expert index
//   ("diffgemma — architecture & implemented contract", Part II §2.1 MoE
//   order), weights = softmax over the k selected logits times
//   per_expert_scale (equal to the renormalised softmax over all E,
//   "DiffusionGemma Explained", MOEBlock.forward).  The fp32 logits carry a
//   rigorous error bound; a token whose top-k boundary is closer than the
//   bound is re-checked with fp64 logits of the candidate experts, so the
//   selected set is the one exact arithmetic gives.  Also writes the dense
//   branch input xd = bf16(h / rms(h) * w_pre_ff) and zeroes the token's row
//   of the f32 expert-sum accumulator.
// k_route_scatter: token -> expert grouping from the per-chunk histogram
//   (counted by k_router_select), prefix sum and a stable scatter
//   (assignments sorted by expert, then token).
// k_gather_xe: expert input rows xe = bf16(h / rms(h) * w_pre_ff2) in
//   grouped order, the B operand of the gate_up GEMM.
#include <math.h>

#include "dg_kernels.h"

namespace dg {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxSlots = 8;  // experts per lane: E <= 256

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
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
// Error-free transformations in fp32 (Knuth's TwoSum; Dekker's product via
// FMA).  A pair (hi, lo) carries a sum whose rounding error is second order
// (~n u^2 of the magnitudes), which makes fp64 unnecessary in the loops.
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

__device__ __forceinline__ void unpack8p(const uint4& u, float* f) {
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

// Error bound of the fp32 logits, relative to |W_e| |x| + |bias_e|.  The
// computed logit differs from the exact one by at most ~70 unit roundoffs
// times sum_i |W_ei x_i| (<= |W_e| |x|): 48 from the router input (fp64
// rms, three fp32 products), 16 from each 16-term fp32 chunk sum (chunk sums
// are accumulated as error-free fp32 pairs), a few from the final rounding
// and the bias add.  2^-16 = 256 unit roundoffs leaves a factor of 3.6.
constexpr float kLogitBound = 1.52587890625e-05f;  // 2^-16

constexpr int kLogitExperts = 32;  // experts per block of k_router_logits
constexpr int kLogitSlices = 8;    // K slices per expert (lanes of one warp)

// Logits for TB tokens x 32 experts.  Every block recomputes the router input
// of its tokens into shared memory, laid out [token][slice][H/8 + 4] so that
// the eight K-slices of a warp read distinct banks; blocks of the first
// expert column also write r, xd and zero the y_moe rows.
template <int TB>
__global__ void __launch_bounds__(256) k_router_logits(const RouterParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int H = p.H, E = p.E;
  const int L = H / kLogitSlices;   // K elements per slice (multiple of 16)
  const int LS = L + 4;             // padded slice stride (floats)
  float* xs = reinterpret_cast<float*>(sm);  // [TB][8][LS]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TB;
  const bool first_col = blockIdx.y == 0;
  const int nvec = H >> 3;
  const float cH = (float)(1.0 / sqrt((double)H));
  const uint4* rsv = reinterpret_cast<const uint4*>(p.router_scale);
  const uint4* wpv = reinterpret_cast<const uint4*>(p.w_pre_ff);

  for (int tl = warp; tl < TB; tl += 8) {
    const int t = t0 + tl;
    float* xrow = xs + (size_t)tl * kLogitSlices * LS;
    if (t >= p.T) {
      for (int i = lane; i < kLogitSlices * LS; i += 32) xrow[i] = 0.f;
      continue;
    }
    const uint4* hrow = reinterpret_cast<const uint4*>(p.h + (size_t)t * H);
    float ss = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(__ldg(hrow + v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    const double ssd = warp_sum_d((double)ss);
    const double r64 = 1.0 / sqrt(ssd / (double)H + (double)p.eps);
    const float rf = (float)r64;
    float xnl = 0.f;
    uint4* xdrow = reinterpret_cast<uint4*>(p.xd + (size_t)t * H);
    for (int v = lane; v < nvec; v += 32) {
      float f[8], sc[8];
      unpack8(__ldg(hrow + v), f);
      unpack8(__ldg(rsv + v), sc);
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = f[i] * rf * sc[i] * cH;
        xnl = fmaf(x[i], x[i], xnl);
      }
      const int k = 8 * v, sl = k / L, off = k - sl * L;  // 8 | L: a vector never straddles
      float4* xo = reinterpret_cast<float4*>(xrow + sl * LS + off);
      xo[0] = make_float4(x[0], x[1], x[2], x[3]);
      xo[1] = make_float4(x[4], x[5], x[6], x[7]);
      if (first_col) {
        float wp[8];
        unpack8(__ldg(wpv + v), wp);
        uint4 o;
        o.x = pack2_bf16(f[0] * rf * wp[0], f[1] * rf * wp[1]);
        o.y = pack2_bf16(f[2] * rf * wp[2], f[3] * rf * wp[3]);
        o.z = pack2_bf16(f[4] * rf * wp[4], f[5] * rf * wp[5]);
        o.w = pack2_bf16(f[6] * rf * wp[6], f[7] * rf * wp[7]);
        xdrow[v] = o;
      }
    }
    if (first_col) {
      const double xnd = warp_sum_d((double)xnl);
      if (lane == 0) {
        p.r_out[t] = rf;
        p.r64_out[t] = r64;
        p.xnorm_out[t] = (float)sqrt(xnd);
      }
      float4* yr = reinterpret_cast<float4*>(p.y_moe + (size_t)t * H);
      for (int v = lane; v < (H >> 2); v += 32) yr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();

  // thread (expert el, slice j): 16-term fp32 chunk sums over its K slice,
  // added in fp64, then the 8 slices of a warp are summed with shuffles
  const int el = threadIdx.x >> 3, j = threadIdx.x & 7;
  const int e_raw = blockIdx.y * kLogitExperts + el;
  const int e = e_raw < E ? e_raw : E - 1;
  float acc_hi[TB], acc_lo[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    acc_hi[t] = 0.f;
    acc_lo[t] = 0.f;
  }
  float wsq = 0.f;
  const int ngroups = H >> 6;
  for (int c = 0; c < L; c += 16) {
    const int k0 = j * L + c;
    float wv[16];
    if (!p.router_u8) {
      const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                          (size_t)e * H + k0);
      unpack8p(__ldg(wrow), wv);
      unpack8p(__ldg(wrow + 1), wv + 8);
    } else {
      // a 16-run never straddles a 64-group (16 | k0)
      const float gs = bf16_to_f32(p.wr_scales[(size_t)e * ngroups + (k0 >> 6)]);
      const float gb = bf16_to_f32(p.wr_biases[(size_t)e * ngroups + (k0 >> 6)]);
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.wr) +
                                                           (size_t)e * H + k0));
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = fmaf(gs, (float)((wd[i >> 2] >> (8 * (i & 3))) & 0xffu), gb);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) wsq = fmaf(wv[i], wv[i], wsq);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const float4* xv = reinterpret_cast<const float4*>(xs + ((size_t)t * kLogitSlices + j) * LS + c);
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = xv[q];
        s = fmaf(wv[4 * q + 0], a.x, s);
        s = fmaf(wv[4 * q + 1], a.y, s);
        s = fmaf(wv[4 * q + 2], a.z, s);
        s = fmaf(wv[4 * q + 3], a.w, s);
      }
      df_add(acc_hi[t], acc_lo[t], s);
    }
  }
#pragma unroll
  for (int o = 1; o < kLogitSlices; o <<= 1) {
    wsq += __shfl_xor_sync(kFull, wsq, o);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      const float h2 = __shfl_xor_sync(kFull, acc_hi[t], o);
      const float l2 = __shfl_xor_sync(kFull, acc_lo[t], o);
      df_add2(acc_hi[t], acc_lo[t], h2, l2);
    }
  }
  if (j == 0 && e_raw < E) {
    const double bias = p.router_bias ? (double)p.router_bias[e] : 0.0;
#pragma unroll
    for (int t = 0; t < TB; ++t)
      if (t0 + t < p.T)
        p.logits[(size_t)(t0 + t) * E + e] = (float)(df_value(acc_hi[t], acc_lo[t]) + bias);
    if (blockIdx.x == 0) p.wnorm_out[e] = sqrtf(wsq) * 1.001f;  // rounded up: a bound
  }
}

// Warp per token: top-k of the fp32 logits, an fp64 re-check of the
// candidates when the k-th / (k+1)-th boundary is closer than the error
// bound, softmax of the k selected logits times per_expert_scale, outputs in
// ascending expert order.
__global__ void __launch_bounds__(256) k_router_select(const RouterParams p) {
  const int H = p.H, E = p.E, K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= p.T) return;
  const float* z = p.logits + (size_t)t * E;
  const int ngroups = H >> 6;
  const double cHd = 1.0 / sqrt((double)H);
  float zl[kMaxSlots], el[kMaxSlots];
  const float xnt = p.xnorm_out[t];
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    const int e = 32 * s + lane;
    if (e < E) {
      const float v = z[e];
      zl[s] = isnan(v) ? -INFINITY : v;
      const float b = p.router_bias ? fabsf(p.router_bias[e]) : 0.f;
      el[s] = kLogitBound * (p.wnorm_out[e] * xnt + b) + 1e-30f;
    } else {
      zl[s] = -INFINITY;
      el[s] = 0.f;
    }
  }
  uint32_t taken = 0;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s) {
      const int e = 32 * s + lane;
      if (e < E && !((taken >> s) & 1u) && (zl[s] > bv || (zl[s] == bv && e < be))) {
        bv = zl[s];
        be = e;
      }
    }
    warp_argmax(bv, be);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
  }
  float L = INFINITY, U = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    if (32 * s + lane >= E) continue;
    if ((taken >> s) & 1u) L = fminf(L, zl[s] - el[s]);
    else U = fmaxf(U, zl[s] + el[s]);
  }
  L = warp_min_f(L);
  U = warp_max_f(U);
  if (!(L > U)) {
    // Candidates that may belong to the exact top-k: z + bound >= L, where L
    // is the smallest lower bound among the k chosen (at least k experts have
    // exact logits >= L, so every exact top-k member passes).
    uint32_t cand = 0;
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s)
      if (32 * s + lane < E && zl[s] + el[s] >= L) cand |= 1u << s;
    const double r64 = p.r64_out[t];
    const uint16_t* hrow = p.h + (size_t)t * H;
    double zx[kMaxSlots];
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s) {
      zx[s] = -INFINITY;
      uint32_t m = __ballot_sync(kFull, (cand >> s) & 1u);
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int e = 32 * s + src;
        // exact terms W_ei * (router_scale_i * h_i) summed as an fp32 pair:
        // a bf16 triple product has at most 24 significant bits, and an
        // 8-bit affine weight is split into two exact fp32 parts first
        float hi = 0.f, lo = 0.f;
        const uint4* hv = reinterpret_cast<const uint4*>(hrow);
        const uint4* sv = reinterpret_cast<const uint4*>(p.router_scale);
        for (int v = lane; v < (H >> 3); v += 32) {
          float hf[8], sf[8], wf[8];
          unpack8p(__ldg(hv + v), hf);
          unpack8p(__ldg(sv + v), sf);
          if (!p.router_u8) {
            unpack8p(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) +
                                                          (size_t)e * H) + v), wf);
#pragma unroll
            for (int i = 0; i < 8; ++i) df_add(hi, lo, __fmul_rn(wf[i], __fmul_rn(sf[i], hf[i])));
          } else {
            const int g = (8 * v) >> 6;
            const float gs = bf16_to_f32(p.wr_scales[(size_t)e * ngroups + g]);
            const float gb = bf16_to_f32(p.wr_biases[(size_t)e * ngroups + g]);
            const uint2 q = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.wr) +
                                                                 (size_t)e * H) + v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t code = ((i < 4 ? q.x : q.y) >> (8 * (i & 3))) & 0xffu;
              float wh, wl;
              two_sum(__fmul_rn(gs, (float)code), gb, wh, wl);   // W = wh + wl exactly
              const float sh = __fmul_rn(sf[i], hf[i]);           // exact (16 bits)
              const float p1 = __fmul_rn(wh, sh);
              const float p1e = fmaf(wh, sh, -p1);                // exact product error
              df_add(hi, lo, p1);
              df_add(hi, lo, p1e);
              df_add(hi, lo, __fmul_rn(wl, sh));
            }
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float h2 = __shfl_xor_sync(kFull, hi, o);
          const float l2 = __shfl_xor_sync(kFull, lo, o);
          df_add2(hi, lo, h2, l2);
        }
        const double part = df_value(hi, lo);
        const double zz = part * r64 * cHd + (p.router_bias ? (double)p.router_bias[e] : 0.0);
        if (lane == src) zx[s] = zz;
      }
    }
    taken = 0;
    for (int k = 0; k < K; ++k) {
      double bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s) {
        const int e = 32 * s + lane;
        if (((cand >> s) & 1u) && !((taken >> s) & 1u) && (zx[s] > bv || (zx[s] == bv && e < be))) {
          bv = zx[s];
          be = e;
        }
      }
      warp_argmax(bv, be);
      if (be != 0x7fffffff && (be & 31) == lane) taken |= 1u << (be >> 5);
    }
    if (lane == 0) atomicAdd(p.n_refined, 1);
  }
  float zmax = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s)
    if ((taken >> s) & 1u) zmax = fmaxf(zmax, zl[s]);
  zmax = warp_max_f(zmax);
  float ex[kMaxSlots];
  float se = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    ex[s] = ((taken >> s) & 1u) ? expf(zl[s] - zmax) : 0.f;
    se += ex[s];
  }
  se = warp_sum_f(se);
  int running = 0;
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    const unsigned ms = __ballot_sync(kFull, (taken >> s) & 1u);
    if ((taken >> s) & 1u) {
      const int e = 32 * s + lane;
      const int rank = running + __popc(ms & lt);
      p.idx[(size_t)t * K + rank] = e;
      p.w[(size_t)t * K + rank] = ex[s] / se * bf16_to_f32(p.pes[e]);
      atomicAdd(&p.chunk_counts[(size_t)(t / kChunkTokens) * E + e], 1);
    }
    running += __popc(ms);
  }
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

__global__ void __launch_bounds__(256) k_route_scatter(const ScatterParams p) {
  __shared__ int s_tmp[256];
  __shared__ int s_base[256];
  __shared__ int s_before[256];
  __shared__ unsigned s_wmask[8][256];
  __shared__ int s_wbase[8][256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x, nchunks = gridDim.x;
  const int E = p.E, K = p.K, T = p.T;

  int tot = 0, bef = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = p.chunk_counts[(size_t)c * E + tid];
      tot += v;
      if (c < chunk) bef += v;
    }
  }
  int total;
  const int base = block_excl_scan256(tot, s_tmp, &total);
  s_base[tid] = base;
  s_before[tid] = bef;

  if (chunk == 0) {
    if (tid < E) p.offsets[tid] = base;
    if (tid == 0) p.offsets[E] = total;
  }

  // stable ranks inside the chunk: per warp, one ballot per expert
  const int t = chunk * kChunkTokens + tid;
  const bool valid = t < T;
  int ex[16];
  unsigned bits[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) bits[w] = 0u;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    ex[j] = -1;
    if (j < K && valid) {
      const int e = p.idx[(size_t)t * K + j];
      if ((unsigned)e < (unsigned)E) {
        ex[j] = e;
#pragma unroll
        for (int w = 0; w < 8; ++w)
          if ((e >> 5) == w) bits[w] |= 1u << (e & 31);
      } else {
        report(p.status, kDevBounds, kSiteScatter, (unsigned)t, (unsigned)e);
      }
    }
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    if (32 * w >= E) break;
    for (int b = 0; b < 32; ++b) {
      const int e = 32 * w + b;
      if (e >= E) break;
      const unsigned m = __ballot_sync(kFull, (bits[w] >> b) & 1u);
      if (lane == 0) s_wmask[warp][e] = m;
    }
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < 8; ++w) {
      s_wbase[w][tid] = run;
      run += __popc(s_wmask[w][tid]);
    }
  }
  __syncthreads();
  if (valid) {
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= K) break;
      const int e = ex[j];
      if (e < 0) continue;
      const int pos = s_base[e] + s_before[e] + s_wbase[warp][e] + __popc(s_wmask[warp][e] & lt);
      p.perm[pos] = t * K + j;
      p.tok_perm[pos] = t;
      p.w_perm[pos] = p.w[(size_t)t * K + j];
    }
  }
}

__global__ void __launch_bounds__(256) k_gather_xe(const GatherParams p) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = p.H >> 3;
  const uint4* wv = reinterpret_cast<const uint4*>(p.w_pre_ff2);
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < p.TK; row += nwarps) {
    const int t = p.tok_perm[row];
    const float r = p.r[t];
    const uint4* hrow = reinterpret_cast<const uint4*>(p.h + (size_t)t * p.H);
    uint4* orow = reinterpret_cast<uint4*>(p.xe_perm + (size_t)row * p.H);
    for (int v = lane; v < nvec; v += 32) {
      float f[8], w[8];
      unpack8(__ldg(hrow + v), f);
      unpack8(__ldg(wv + v), w);
      uint4 o;
      o.x = pack2_bf16(f[0] * r * w[0], f[1] * r * w[1]);
      o.y = pack2_bf16(f[2] * r * w[2], f[3] * r * w[3]);
      o.z = pack2_bf16(f[4] * r * w[4], f[5] * r * w[5]);
      o.w = pack2_bf16(f[6] * r * w[6], f[7] * r * w[7]);
      orow[v] = o;
    }
  }
}

template <int TB>
size_t router_smem(int H) {
  return sizeof(float) * (size_t)TB * kLogitSlices * (H / kLogitSlices + 4);
}

template <int TB>
cudaError_t launch_router_tb(const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_smem<TB>(p.H);
  cudaError_t err = cudaFuncSetAttribute(k_router_logits<TB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const dim3 grid((p.T + TB - 1) / TB, (p.E + kLogitExperts - 1) / kLogitExperts);
  k_router_logits<TB><<<grid, 256, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  // eight tokens per block amortise the router-weight reads; four when the
  // staged router input of eight would not fit
  if (router_smem<8>(p.H) <= 160 * 1024) return launch_router_tb<8>(p, s);
  return launch_router_tb<4>(p, s);
}

cudaError_t launch_router_select(const RouterParams& p, cudaStream_t s) {
  k_router_select<<<(p.T + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_route_scatter(const ScatterParams& p, cudaStream_t s) {
  const int grid = (p.T + kChunkTokens - 1) / kChunkTokens;
  k_route_scatter<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams& p, int num_sms, cudaStream_t s) {
  const int rows_per_block = 8;
  int grid = (p.TK + rows_per_block - 1) / rows_per_block;
  grid = grid < num_sms * 8 ? grid : num_sms * 8;
  if (grid < 1) grid = 1;
  k_gather_xe<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dg
