// Routing of the MoE FFN block on sm_103a.
//
// k_router: per token, RMS of the residual stream, router input
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
// k_route_count / k_route_scatter: token -> expert grouping by per-chunk
//   histogram, prefix sum and a stable scatter (assignments sorted by expert,
//   then token), plus the tile lists of the two grouped GEMMs.
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
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  return (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(b) << 16);
}

// Error bound of the fp32 logits, relative to |W_e| |x| + |bias_e|.  The
// computed logit differs from the exact one by at most ~114 unit roundoffs
// times sum_i |W_ei x_i| (<= |W_e| |x|): 48 from the router input (fp64 rms,
// three fp32 products), 64 from each 64-term fp32 chunk sum (chunks are then
// added in fp64), 2 from the final rounding and bias add.  2^-15 = 512 unit
// roundoffs leaves a factor 4.5.
constexpr float kLogitBound = 3.0517578125e-05f;  // 2^-15

template <int TB>
__global__ void __launch_bounds__(128) k_router(const RouterParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int H = p.H, E = p.E, K = p.K;
  double* r64s = reinterpret_cast<double*>(sm);        // [TB]
  float* xn = reinterpret_cast<float*>(r64s + TB);     // [TB]
  float* wn = xn + ((TB + 3) & ~3);                    // [E] row norms of Wr
  float* zs = wn + ((E + 3) & ~3);                     // [TB][E]
  float* xs = zs + ((TB * E + 3) & ~3);                // [TB][H]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TB;
  const int nvec = H >> 3;
  const float cH = (float)(1.0 / sqrt((double)H));
  const uint4* rsv = reinterpret_cast<const uint4*>(p.router_scale);
  const uint4* wpv = reinterpret_cast<const uint4*>(p.w_pre_ff);

  // ---- 1. norms, router input (fp32, smem), dense input xd, zero y_moe row
  for (int tl = warp; tl < TB; tl += 4) {
    const int t = t0 + tl;
    float* xrow = xs + (size_t)tl * H;
    if (t >= p.T) {
      for (int i = lane; i < H; i += 32) xrow[i] = 0.f;
      if (lane == 0) {
        r64s[tl] = 0.0;
        xn[tl] = 0.f;
      }
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
      float f[8], sc[8], wp[8];
      unpack8(__ldg(hrow + v), f);
      unpack8(__ldg(rsv + v), sc);
      unpack8(__ldg(wpv + v), wp);
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = f[i] * rf * sc[i] * cH;
        xnl = fmaf(x[i], x[i], xnl);
      }
      float4* xo = reinterpret_cast<float4*>(xrow + 8 * v);
      xo[0] = make_float4(x[0], x[1], x[2], x[3]);
      xo[1] = make_float4(x[4], x[5], x[6], x[7]);
      uint4 o;
      o.x = pack2_bf16(f[0] * rf * wp[0], f[1] * rf * wp[1]);
      o.y = pack2_bf16(f[2] * rf * wp[2], f[3] * rf * wp[3]);
      o.z = pack2_bf16(f[4] * rf * wp[4], f[5] * rf * wp[5]);
      o.w = pack2_bf16(f[6] * rf * wp[6], f[7] * rf * wp[7]);
      xdrow[v] = o;
    }
    const double xnd = warp_sum_d((double)xnl);
    if (lane == 0) {
      r64s[tl] = r64;
      xn[tl] = (float)sqrt(xnd);
      p.r_out[t] = rf;
    }
    float4* yr = reinterpret_cast<float4*>(p.y_moe + (size_t)t * H);
    for (int v = lane; v < (H >> 2); v += 32) yr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();

  // ---- 2. logits: thread per expert, 64-term fp32 chunks added in fp64
  const int ngroups = H >> 6;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.0;
    double wsq = 0.0;
    for (int c = 0; c < ngroups; ++c) {
      float part[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) part[t] = 0.f;
      float wsqp = 0.f;
      if (!p.router_u8) {
        const uint4* wrow =
            reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.wr) + (size_t)e * H) +
            c * 8;
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          float wv[8];
          unpack8(__ldg(wrow + j), wv);
#pragma unroll
          for (int i = 0; i < 8; ++i) wsqp = fmaf(wv[i], wv[i], wsqp);
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            const float4* xv = reinterpret_cast<const float4*>(xs + (size_t)t * H + c * 64 + 8 * j);
            const float4 a = xv[0], b = xv[1];
            float s = part[t];
            s = fmaf(wv[0], a.x, s); s = fmaf(wv[1], a.y, s);
            s = fmaf(wv[2], a.z, s); s = fmaf(wv[3], a.w, s);
            s = fmaf(wv[4], b.x, s); s = fmaf(wv[5], b.y, s);
            s = fmaf(wv[6], b.z, s); s = fmaf(wv[7], b.w, s);
            part[t] = s;
          }
        }
      } else {
        const float gs = bf16_to_f32(p.wr_scales[(size_t)e * ngroups + c]);
        const float gb = bf16_to_f32(p.wr_biases[(size_t)e * ngroups + c]);
        const uint4* qrow =
            reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.wr) + (size_t)e * H) + c * 4;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const uint4 u = __ldg(qrow + j);
          const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int hq = 0; hq < 4; ++hq) {
            float wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              wv[i] = fmaf(gs, (float)((wd[hq] >> (8 * i)) & 0xffu), gb);
              wsqp = fmaf(wv[i], wv[i], wsqp);
            }
#pragma unroll
            for (int t = 0; t < TB; ++t) {
              const float4 a =
                  *reinterpret_cast<const float4*>(xs + (size_t)t * H + c * 64 + 16 * j + 4 * hq);
              float s = part[t];
              s = fmaf(wv[0], a.x, s); s = fmaf(wv[1], a.y, s);
              s = fmaf(wv[2], a.z, s); s = fmaf(wv[3], a.w, s);
              part[t] = s;
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] += (double)part[t];
      wsq += (double)wsqp;
    }
    const double bias = p.router_bias ? (double)p.router_bias[e] : 0.0;
#pragma unroll
    for (int t = 0; t < TB; ++t) zs[t * E + e] = (float)(acc[t] + bias);
    wn[e] = (float)sqrt(wsq);
  }
  __syncthreads();

  // ---- 3. selection, exact re-check near the boundary, weights
  const double cHd = 1.0 / sqrt((double)H);
  for (int tl = warp; tl < TB; tl += 4) {
    const int t = t0 + tl;
    if (t >= p.T) continue;
    const float* z = zs + tl * E;
    float zl[kMaxSlots], el[kMaxSlots];
    const float xnt = xn[tl];
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s) {
      const int e = 32 * s + lane;
      if (e < E) {
        const float v = z[e];
        zl[s] = isnan(v) ? -INFINITY : v;
        const float b = p.router_bias ? fabsf(p.router_bias[e]) : 0.f;
        el[s] = kLogitBound * (wn[e] * xnt + b) + 1e-30f;
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
      // Candidates that may belong to the exact top-k: z + bound >= L, where
      // L is the smallest lower bound among the k chosen (at least k experts
      // have exact logits >= L, so every exact top-k member passes).
      uint32_t cand = 0;
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s)
        if (32 * s + lane < E && zl[s] + el[s] >= L) cand |= 1u << s;
      double zx[kMaxSlots];
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s) {
        zx[s] = -INFINITY;
        uint32_t m = __ballot_sync(kFull, (cand >> s) & 1u);
        while (m) {
          const int src = __ffs(m) - 1;
          m &= m - 1;
          const int e = 32 * s + src;
          double part = 0.0;
          const uint16_t* hrow = p.h + (size_t)t * H;
          if (!p.router_u8) {
            const uint16_t* wrow = static_cast<const uint16_t*>(p.wr) + (size_t)e * H;
            for (int i = lane; i < H; i += 32)
              part = fma((double)bf16_to_f32(wrow[i]),
                         (double)bf16_to_f32(p.router_scale[i]) * (double)bf16_to_f32(hrow[i]),
                         part);
          } else {
            const uint8_t* qrow = static_cast<const uint8_t*>(p.wr) + (size_t)e * H;
            for (int i = lane; i < H; i += 32) {
              const double w = (double)bf16_to_f32(p.wr_scales[(size_t)e * ngroups + (i >> 6)]) *
                                   (double)qrow[i] +
                               (double)bf16_to_f32(p.wr_biases[(size_t)e * ngroups + (i >> 6)]);
              part = fma(w,
                         (double)bf16_to_f32(p.router_scale[i]) * (double)bf16_to_f32(hrow[i]),
                         part);
            }
          }
          const double tot = warp_sum_d(part);
          const double zz =
              tot * r64s[tl] * cHd + (p.router_bias ? (double)p.router_bias[e] : 0.0);
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
    // weights: softmax over the k selected fp32 logits, times per_expert_scale
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
    // outputs in ascending expert order: rank = selected experts below e
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
      }
      running += __popc(ms);
    }
    if (p.logits) {
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s)
        if (32 * s + lane < E) p.logits[(size_t)t * E + 32 * s + lane] = z[32 * s + lane];
    }
  }
}

// Per-chunk expert histogram.
__global__ void __launch_bounds__(256) k_route_count(const int32_t* __restrict__ idx, int T, int K,
                                                     int E, int32_t* __restrict__ chunk_counts) {
  __shared__ int cnt[256];
  cnt[threadIdx.x] = 0;
  __syncthreads();
  const int t = blockIdx.x * kChunkTokens + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < K; ++j) {
      const int e = idx[(size_t)t * K + j];
      if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  if ((int)threadIdx.x < E) chunk_counts[(size_t)blockIdx.x * E + threadIdx.x] = cnt[threadIdx.x];
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
    // tile lists: dense tiles first, then per expert (token tile, feature tile)
    const int BN = p.bn_exp, BNd = p.bn_dense;
    const int mt_gu = p.I / 64, mt_dn = p.H / 128, mt_dgu = p.D / 64;
    const int ndt = (T + BNd - 1) / BNd;
    const int nd_gu = ndt * mt_dgu, nd_dn = ndt * mt_dn;
    const int nj = tid < E ? (tot + BN - 1) / BN : 0;
    int tot_gu, tot_dn;
    const int st_gu = block_excl_scan256(nj * mt_gu, s_tmp, &tot_gu);
    const int st_dn = block_excl_scan256(nj * mt_dn, s_tmp, &tot_dn);
    for (int j = 0; j < nj; ++j) {
      const int r0 = base + j * BN;
      const int nr = min(BN, tot - j * BN);
      for (int m = 0; m < mt_gu; ++m)
        p.tiles_gu[nd_gu + st_gu + j * mt_gu + m] = make_int4(tid, m, r0, nr);
      for (int m = 0; m < mt_dn; ++m)
        p.tiles_dn[nd_dn + st_dn + j * mt_dn + m] = make_int4(tid, m, r0, nr);
    }
    for (int i = tid; i < nd_gu; i += 256) {
      const int j = i / mt_dgu, m = i % mt_dgu;
      p.tiles_gu[i] = make_int4(E, m, j * BNd, min(BNd, T - j * BNd));
    }
    for (int i = tid; i < nd_dn; i += 256) {
      const int j = i / mt_dn, m = i % mt_dn;
      p.tiles_dn[i] = make_int4(E, m, j * BNd, min(BNd, T - j * BNd));
    }
    if (tid == 0) {
      p.ntiles[0] = nd_gu + tot_gu;
      p.ntiles[1] = nd_dn + tot_dn;
    }
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
size_t router_smem(int H, int E) {
  return sizeof(double) * TB + sizeof(float) * (((TB + 3) & ~3) + ((E + 3) & ~3) +
                                                ((TB * E + 3) & ~3) + (size_t)TB * H);
}

template <int TB>
cudaError_t launch_router_tb(const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_smem<TB>(p.H, p.E);
  cudaError_t err = cudaFuncSetAttribute(k_router<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (p.T + TB - 1) / TB;
  k_router<TB><<<grid, 128, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  // more tokens per block amortise the router-weight reads; few tokens per
  // block keep enough blocks in flight for a single canvas
  if (p.T >= 2048 && router_smem<8>(p.H, p.E) <= 160 * 1024) return launch_router_tb<8>(p, s);
  return launch_router_tb<2>(p, s);
}

cudaError_t launch_route_count(const int32_t* idx, int T, int K, int E, int32_t* chunk_counts,
                               cudaStream_t s) {
  const int grid = (T + kChunkTokens - 1) / kChunkTokens;
  k_route_count<<<grid, 256, 0, s>>>(idx, T, K, E, chunk_counts);
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
