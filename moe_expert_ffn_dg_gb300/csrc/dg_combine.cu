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

// NPT: elements per thread (H <= NPT * 256)
template <int NPT>
__global__ void __launch_bounds__(kThreads) k_combine(const CombineParams p) {
  __shared__ float2 red[kThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int H = p.H;
  const float* yd = p.y_dense + (size_t)t * H;
  const float* ym = p.y_moe + (size_t)t * H;
  const uint16_t* hrow = p.h + (size_t)t * H;
  float a[NPT], b[NPT], hv[NPT], w1[NPT], w2[NPT], w3[NPT];
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int i = threadIdx.x + j * kThreads;
    const bool in = i < H;
    a[j] = in ? yd[i] : 0.f;
    b[j] = in ? ym[i] : 0.f;
    hv[j] = in ? bf16_to_f32(hrow[i]) : 0.f;
    w1[j] = in ? bf16_to_f32(p.w_post1[i]) : 0.f;
    w2[j] = in ? bf16_to_f32(p.w_post2[i]) : 0.f;
    w3[j] = in ? bf16_to_f32(p.w_post[i]) : 0.f;
  }
  float sd = 0.f, sm = 0.f;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    sd = fmaf(a[j], a[j], sd);
    sm = fmaf(b[j], b[j], sm);
  }
  block_sum2<NPT>(sd, sm, red);
  const float rd = 1.0f / sqrtf(sd / (float)H + p.eps);
  const float rm = 1.0f / sqrtf(sm / (float)H + p.eps);
  float ss = 0.f, dummy = 0.f;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    a[j] = a[j] * rd * w1[j] + b[j] * rm * w2[j];
    ss = fmaf(a[j], a[j], ss);
  }
  block_sum2<NPT>(ss, dummy, red);
  const float rs = 1.0f / sqrtf(ss / (float)H + p.eps);
  uint16_t* orow = p.out + (size_t)t * H;
#pragma unroll
  for (int j = 0; j < NPT; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < H) orow[i] = f32_to_bf16_rne((hv[j] + a[j] * rs * w3[j]) * p.layer_scalar);
  }
}

template <int NPT>
cudaError_t launch_npt(const CombineParams& p, cudaStream_t s) {
  return launch_pdl(k_combine<NPT>, dim3(p.T), dim3(kThreads), 0, s, p);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const int npt = (p.H + kThreads - 1) / kThreads;
  if (npt <= 4) return launch_npt<4>(p, s);
  if (npt <= 8) return launch_npt<8>(p, s);
  if (npt <= 12) return launch_npt<12>(p, s);
  if (npt <= 16) return launch_npt<16>(p, s);
  return launch_npt<32>(p, s);
}

}  // namespace dg
