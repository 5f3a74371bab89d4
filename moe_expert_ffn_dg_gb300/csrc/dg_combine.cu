// FFN norm sandwich and residual of the MoE block, one CTA per token:
//   h1  = rms(y_dense) * w_post_ff1,   h2 = rms(y_moe) * w_post_ff2
//   out = bf16((h + rms(h1 + h2) * w_post_ff) * layer_scalar)
// ("DiffusionGemma port — plan & parity strategy", Reference dossier §2
// DecoderLayer; "DiffusionGemma Explained", MOEBlock.forward and the layer
// scalar; "diffgemma — architecture & implemented contract", Part II §2.1:
// seven norms, weight multiplied directly, layer_scalar on the whole output).
// Every input of the token is loaded up front (one round of memory latency),
// then two block reductions.  h and out may alias: each element of h is read
// by the thread that writes the same element of out, before it writes.
// y_moe is either read as the accumulated [T, H] rows or summed here from
// the token's K weighted expert rows (large batches).  Optionally the next
// layer's input norm of the output plane is written beside it.
#include "dg_kernels.h"

namespace dg {
namespace {

constexpr int kThreads = 256;

template <int NV>
__device__ __forceinline__ void block_sum2(float& x, float& y, float2* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = make_float2(x, y);
  __syncthreads();
  float sx = 0.f, sy = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    sx += red[w].x;
    sy += red[w].y;
  }
  x = sx;
  y = sy;
}

__device__ __forceinline__ void bf16x4(const uint16_t* p, float (&f)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}

// NV: groups of four elements per thread (H <= 4 * NV * 256).  Thread x
// owns elements 4v..4v+3 for v = x + 256 j: every access is a 16-byte (f32)
// or 8-byte (bf16) vector.
template <int NV>
__global__ void __launch_bounds__(kThreads) k_combine(const CombineParams p) {
  __shared__ float2 red[kThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int H = p.H, nq = H >> 2;
  const float4* yd = reinterpret_cast<const float4*>(p.y_dense + (size_t)t * H);
  const uint16_t* hrow = p.h + (size_t)t * H;
  float a[NV][4], b[NV][4], hv[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int v = threadIdx.x + j * kThreads;
    if (v < nq) {
      const float4 d = yd[v];
      a[j][0] = d.x, a[j][1] = d.y, a[j][2] = d.z, a[j][3] = d.w;
      bf16x4(hrow + 4 * v, hv[j]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) a[j][e] = hv[j][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) b[j][e] = 0.f;
  }
  if (p.y_perm) {
    // y_moe = sum over the token's K assignments of their weighted expert
    // rows, in slot order (deterministic); four rows' loads in flight
    const int32_t* inv = p.inv + (size_t)t * p.K;
    for (int k0 = 0; k0 < p.K; k0 += 4) {
      const float4* rows[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        rows[u] = k0 + u < p.K ? reinterpret_cast<const float4*>(p.y_perm + (size_t)inv[k0 + u] * H)
                               : nullptr;
      float4 g[4][NV];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const int v = threadIdx.x + j * kThreads;
          g[u][j] = rows[u] && v < nq ? rows[u][v] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          b[j][0] += g[u][j].x;
          b[j][1] += g[u][j].y;
          b[j][2] += g[u][j].z;
          b[j][3] += g[u][j].w;
        }
    }
    if (p.y_moe_out) {
      float4* yo = reinterpret_cast<float4*>(p.y_moe_out + (size_t)t * H);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int v = threadIdx.x + j * kThreads;
        if (v < nq) yo[v] = make_float4(b[j][0], b[j][1], b[j][2], b[j][3]);
      }
    }
  } else {
    const float4* ym = reinterpret_cast<const float4*>(p.y_moe + (size_t)t * H);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = threadIdx.x + j * kThreads;
      if (v < nq) {
        const float4 m = ym[v];
        b[j][0] = m.x, b[j][1] = m.y, b[j][2] = m.z, b[j][3] = m.w;
      }
    }
  }
  float sd = 0.f, sm = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sd = fmaf(a[j][e], a[j][e], sd);
      sm = fmaf(b[j][e], b[j][e], sm);
    }
  block_sum2<NV>(sd, sm, red);
  const float rd = 1.0f / sqrtf(sd / (float)H + p.eps);
  const float rm = 1.0f / sqrtf(sm / (float)H + p.eps);
  float ss = 0.f, dummy = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int v = threadIdx.x + j * kThreads;
    float w1[4], w2[4];
    if (v < nq) {
      bf16x4(p.w_post1 + 4 * v, w1);
      bf16x4(p.w_post2 + 4 * v, w2);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) w1[e] = w2[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[j][e] = a[j][e] * rd * w1[e] + b[j][e] * rm * w2[e];
      ss = fmaf(a[j][e], a[j][e], ss);
    }
  }
  block_sum2<NV>(ss, dummy, red);
  const float rs = 1.0f / sqrtf(ss / (float)H + p.eps);
  uint16_t* orow = p.out + (size_t)t * H;
  uint2 ov[NV];
  float sn = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int v = threadIdx.x + j * kThreads;
    ov[j] = make_uint2(0u, 0u);
    if (v < nq) {
      float w3[4];
      bf16x4(p.w_post + 4 * v, w3);
      uint2 o;
      o.x = (uint32_t)f32_to_bf16_rne((hv[j][0] + a[j][0] * rs * w3[0]) * p.layer_scalar) |
            ((uint32_t)f32_to_bf16_rne((hv[j][1] + a[j][1] * rs * w3[1]) * p.layer_scalar) << 16);
      o.y = (uint32_t)f32_to_bf16_rne((hv[j][2] + a[j][2] * rs * w3[2]) * p.layer_scalar) |
            ((uint32_t)f32_to_bf16_rne((hv[j][3] + a[j][3] * rs * w3[3]) * p.layer_scalar) << 16);
      ov[j] = o;
    }
  }
  if (p.w_next) {
    // the next layer's input_layernorm on the bf16 output plane ("DiffusionGemma
    // port — plan & parity strategy", Reference dossier §2 DecoderLayer:
    // input_layernorm opens the next layer), fused here
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float o4[4] = {__uint_as_float(ov[j].x << 16), __uint_as_float(ov[j].x & 0xffff0000u),
                           __uint_as_float(ov[j].y << 16), __uint_as_float(ov[j].y & 0xffff0000u)};
#pragma unroll
      for (int e = 0; e < 4; ++e) sn = fmaf(o4[e], o4[e], sn);
    }
    block_sum2<NV>(sn, dummy, red);
  }
  // every input of the token is read by now: out may alias h
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int v = threadIdx.x + j * kThreads;
    if (v < nq) *reinterpret_cast<uint2*>(orow + 4 * v) = ov[j];
  }
  if (p.w_next) {
    const float rn = 1.0f / sqrtf(sn / (float)H + p.eps);
    uint16_t* nrow = p.next_out + (size_t)t * H;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = threadIdx.x + j * kThreads;
      if (v < nq) {
        float w4[4];
        bf16x4(p.w_next + 4 * v, w4);
        const float o4[4] = {__uint_as_float(ov[j].x << 16), __uint_as_float(ov[j].x & 0xffff0000u),
                             __uint_as_float(ov[j].y << 16), __uint_as_float(ov[j].y & 0xffff0000u)};
        uint2 q;
        q.x = (uint32_t)f32_to_bf16_rne(o4[0] * rn * w4[0]) |
              ((uint32_t)f32_to_bf16_rne(o4[1] * rn * w4[1]) << 16);
        q.y = (uint32_t)f32_to_bf16_rne(o4[2] * rn * w4[2]) |
              ((uint32_t)f32_to_bf16_rne(o4[3] * rn * w4[3]) << 16);
        *reinterpret_cast<uint2*>(nrow + 4 * v) = q;
      }
    }
  }
}

template <int NV>
cudaError_t launch_nv(const CombineParams& p, cudaStream_t s) {
  return launch_pdl(k_combine<NV>, dim3(p.T), dim3(kThreads), 0, s, p);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const int nv = (p.H / 4 + kThreads - 1) / kThreads;
  if (nv <= 1) return launch_nv<1>(p, s);
  if (nv <= 2) return launch_nv<2>(p, s);
  if (nv <= 3) return launch_nv<3>(p, s);
  if (nv <= 4) return launch_nv<4>(p, s);
  return launch_nv<8>(p, s);
}

}  // namespace dg
