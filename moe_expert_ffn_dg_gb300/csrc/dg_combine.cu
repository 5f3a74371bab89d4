// FFN norm sandwich and residual of the MoE block, one CTA per token:
//   h1  = rms(y_dense) * w_post_ff1,   h2 = rms(y_moe) * w_post_ff2
//   out = bf16((h + rms(h1 + h2) * w_post_ff) * layer_scalar)
// ("DiffusionGemma port — plan & parity strategy", Reference dossier §2
// DecoderLayer; "DiffusionGemma Explained", MOEBlock.forward and the layer
// scalar; "diffgemma — architecture & implemented contract", Part II §2.1:
// seven norms, weight multiplied directly, layer_scalar on the whole output).
// h and out may alias: each element of h is read by the thread that writes
// the same element of out, before it writes.
#include "dg_kernels.h"

namespace dg {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPerThread = 32;  // H <= 8192

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

__global__ void __launch_bounds__(kThreads) k_combine(const CombineParams p) {
  __shared__ float red[kThreads / 32];
  const int t = blockIdx.x;
  const int H = p.H;
  const float* yd = p.y_dense + (size_t)t * H;
  const float* ym = p.y_moe + (size_t)t * H;
  float a[kMaxPerThread], b[kMaxPerThread];
  float sd = 0.f, sm = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerThread; ++j) {
    const int i = threadIdx.x + j * kThreads;
    a[j] = 0.f;
    b[j] = 0.f;
    if (i < H) {
      a[j] = yd[i];
      b[j] = ym[i];
      sd = fmaf(a[j], a[j], sd);
      sm = fmaf(b[j], b[j], sm);
    }
  }
  sd = block_sum(sd, red);
  sm = block_sum(sm, red);
  const float rd = 1.0f / sqrtf(sd / (float)H + p.eps);
  const float rm = 1.0f / sqrtf(sm / (float)H + p.eps);
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerThread; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < H) {
      a[j] = a[j] * rd * bf16_to_f32(p.w_post1[i]) + b[j] * rm * bf16_to_f32(p.w_post2[i]);
      ss = fmaf(a[j], a[j], ss);
    }
  }
  ss = block_sum(ss, red);
  const float rs = 1.0f / sqrtf(ss / (float)H + p.eps);
  const uint16_t* hrow = p.h + (size_t)t * H;
  uint16_t* orow = p.out + (size_t)t * H;
#pragma unroll
  for (int j = 0; j < kMaxPerThread; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < H) {
      const float hv = bf16_to_f32(hrow[i]);
      orow[i] = f32_to_bf16_rne((hv + a[j] * rs * bf16_to_f32(p.w_post[i])) * p.layer_scalar);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  k_combine<<<p.T, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dg
