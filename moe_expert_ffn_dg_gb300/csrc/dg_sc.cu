// Self-conditioning MLP on sm_103a: a pre-normed GEGLU MLP of the dense FFN's
// shape on the soft signal, added to the token embeddings, then RMS-normalised
// without a weight ("DiffusionGemma port — plan & parity strategy", Reference
// dossier §3 SelfConditioning; "diffgemma — architecture & implemented
// contract", Part II §2.1 SC injection).
//
// Four launches: k_sc_prenorm (x = bf16(rms(signal) * pre_norm)), the grouped
// GEMMs of the block with no experts (the dense tiles only: gate_up + GEGLU,
// then down into an f32 buffer), and k_sc_post (out = bf16 of the weightless
// RMSNorm of embeds + s).
#include <stdio.h>

#include <new>

#include "../../include/dg_moe.h"
#include "dg_host.h"
#include "dg_kernels.h"

using namespace dg;
using namespace dg::host;

namespace {

constexpr int kScThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red reuse across calls
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kScThreads / 32; ++w) s += red[w];
  return s;
}

__device__ __forceinline__ void unpack8f(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(b) << 16);
}

// One token per block: x = bf16(signal / sqrt(mean(signal^2) + eps) * pre_norm).
__global__ void __launch_bounds__(kScThreads) k_sc_prenorm(const uint16_t* __restrict__ signal,
                                                           const uint16_t* __restrict__ w,
                                                           int H, float eps,
                                                           uint16_t* __restrict__ x) {
  __shared__ float red[kScThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, nvec = H >> 3;
  const uint4* row = reinterpret_cast<const uint4*>(signal + (size_t)t * H);
  float ss = 0.f;
  for (int v = threadIdx.x; v < nvec; v += kScThreads) {
    float f[8];
    unpack8f(row[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  uint4* out = reinterpret_cast<uint4*>(x + (size_t)t * H);
  for (int v = threadIdx.x; v < nvec; v += kScThreads) {
    float f[8], g[8];
    unpack8f(row[v], f);
    unpack8f(reinterpret_cast<const uint4*>(w)[v], g);
    uint4 o;
    o.x = pack2(f[0] * r * g[0], f[1] * r * g[1]);
    o.y = pack2(f[2] * r * g[2], f[3] * r * g[3]);
    o.z = pack2(f[4] * r * g[4], f[5] * r * g[5]);
    o.w = pack2(f[6] * r * g[6], f[7] * r * g[7]);
    out[v] = o;
  }
}

// One token per block: out = bf16(v / sqrt(mean(v^2) + eps)), v = embeds + s.
// The row is read fully before it is written, so out may alias embeds.
__global__ void __launch_bounds__(kScThreads) k_sc_post(const uint16_t* embeds,
                                                        const float* __restrict__ s, int H,
                                                        float eps, uint16_t* out) {
  __shared__ float red[kScThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, nvec = H >> 3;
  constexpr int kMaxVec = 8;  // H <= 8 * 8 * 256
  float v[kMaxVec][8];
  float ss = 0.f;
  const uint4* er = reinterpret_cast<const uint4*>(embeds + (size_t)t * H);
  const float4* sr = reinterpret_cast<const float4*>(s + (size_t)t * H);
#pragma unroll
  for (int j = 0; j < kMaxVec; ++j) {
    const int vi = threadIdx.x + j * kScThreads;
    if (vi < nvec) {
      float e[8];
      unpack8f(er[vi], e);
      const float4 a = sr[2 * vi], b = sr[2 * vi + 1];
      const float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[j][i] = e[i] + y[i];
        ss = fmaf(v[j][i], v[j][i], ss);
      }
    }
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  uint4* orow = reinterpret_cast<uint4*>(out + (size_t)t * H);
#pragma unroll
  for (int j = 0; j < kMaxVec; ++j) {
    const int vi = threadIdx.x + j * kScThreads;
    if (vi < nvec) {
      uint4 o;
      o.x = pack2(v[j][0] * r, v[j][1] * r);
      o.y = pack2(v[j][2] * r, v[j][3] * r);
      o.z = pack2(v[j][4] * r, v[j][5] * r);
      o.w = pack2(v[j][6] * r, v[j][7] * r);
      orow[vi] = o;
    }
  }
}

constexpr int kScKernels = 4;
const char* const kScKernelNames[kScKernels] = {"sc_prenorm", "gemm_gate_up", "gemm_down",
                                                 "sc_post"};

struct ScLayout {
  size_t status, zero, x, act, y, total;
};

ScLayout sc_layout(const dg_sc_mlp_config_t& c) {
  ScLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  const size_t T = (size_t)c.max_tokens, H = c.hidden, D = c.inter;
  L.status = take(sizeof(DevStatus));
  L.zero = take(16);  // expert offsets of a launch with no experts: {0}
  L.x = take(T * H * 2);
  L.act = take(T * D * 2);
  L.y = take(T * H * 4);
  L.total = off;
  return L;
}

dg_status_t sc_check_config(const dg_sc_mlp_config_t* c) {
  if (!c) return DG_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->inter <= 0 || c->max_tokens <= 0 || c->rms_eps < 0.f || c->flags != 0)
    return DG_ERR_INVALID_ARG;
  if (c->hidden % 128 || c->inter % 64 || c->hidden > 8 * 8 * kScThreads)
    return DG_ERR_UNSUPPORTED;
  if (c->max_tokens > (1 << 20)) return DG_ERR_UNSUPPORTED;
  if (c->fmt != DG_FMT_BF16 && c->fmt != DG_FMT_AFFINE_U4_G64 && c->fmt != DG_FMT_AFFINE_U8_G64)
    return DG_ERR_UNSUPPORTED;
  if (c->fmt != DG_FMT_BF16 && (c->hidden > 2944 || c->inter > 2944)) return DG_ERR_UNSUPPORTED;
  return DG_OK;
}

}  // namespace

struct dg_sc_mlp {
  dg_sc_mlp_config_t cfg;
  dg_sc_mlp_weights_t w;
  uint8_t* ws;
  ScLayout L;
  int num_sms;
  size_t smem_optin;
  bool q4;    // group-64 affine weights (the quantised GEMM)
  int qbits;  // their code width: 4 or 8
  GemmParams gu, dn;
  dg_event_t* prof = nullptr;
};

extern "C" {

dg_status_t dg_sc_mlp_workspace_size(const dg_sc_mlp_config_t* cfg, size_t* bytes) {
  if (!bytes) return DG_ERR_INVALID_ARG;
  const dg_status_t s = sc_check_config(cfg);
  if (s != DG_OK) return s;
  *bytes = sc_layout(*cfg).total;
  return DG_OK;
}

dg_status_t dg_sc_mlp_create(const dg_sc_mlp_config_t* cfg, const dg_sc_mlp_weights_t* weights,
                             void* workspace, size_t workspace_bytes, dg_sc_mlp_t** out) {
  if (!out) return DG_ERR_INVALID_ARG;
  *out = nullptr;
  dg_status_t s = sc_check_config(cfg);
  if (s != DG_OK) return s;
  if (!weights) return DG_ERR_INVALID_ARG;
  if ((s = check_qtensor(weights->gate, cfg->fmt)) != DG_OK) return s;
  if ((s = check_qtensor(weights->up, cfg->fmt)) != DG_OK) return s;
  if ((s = check_qtensor(weights->down, cfg->fmt)) != DG_OK) return s;
  if (!weights->pre_norm) return DG_ERR_INVALID_ARG;
  if (!aligned(weights->pre_norm, 16)) return DG_ERR_ALIGNMENT;
  const ScLayout L = sc_layout(*cfg);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 1024)) return DG_ERR_WORKSPACE;

  dg_sc_mlp* m = new (std::nothrow) dg_sc_mlp();
  if (!m) return DG_ERR_CUDA;
  m->cfg = *cfg;
  if (m->cfg.rms_eps == 0.f) m->cfg.rms_eps = 1e-6f;
  m->w = *weights;
  m->ws = static_cast<uint8_t*>(workspace);
  m->L = L;
  m->q4 = cfg->fmt != DG_FMT_BF16;
  m->qbits = cfg->fmt == DG_FMT_AFFINE_U8_G64 ? 8 : 4;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  m->smem_optin = (size_t)optin;
  if ((m->q4 ? prepare_gemm_affine(optin) : prepare_gemm_bf16()) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  const uint64_t H = cfg->hidden, D = cfg->inter, T = cfg->max_tokens;
  uint8_t* ws = m->ws;
  const bool q4 = m->q4;
  const int qb = m->qbits;
  bool ok = true;
  // gate_up: the dense pair (4-D interleaving view when up lies above gate)
  if (q4) {
    ok = ok && encode_q_rows(&m->gu.wa_d0, weights->gate.q, D, H, 16, qb);
    ok = ok && encode_q_rows(&m->gu.wa_d1, weights->up.q, D, H, 16, qb);
  } else {
    ok = ok && encode_bf16_rows(&m->gu.wa_d0, weights->gate.q, D, H, 16);
    ok = ok && encode_bf16_rows(&m->gu.wa_d1, weights->up.q, D, H, 16);
  }
  {
    const uintptr_t g = (uintptr_t)weights->gate.q, u = (uintptr_t)weights->up.q;
    m->gu.dense_5d = u > g && ((u - g) % 16) == 0 && (u - g) < (1ull << 40) &&
                     encode_gate_up(&m->gu.wa_d5, weights->gate.q, H, D, u - g, 4, 1, 0, q4 ? qb : 0);
    if (!m->gu.dense_5d) m->gu.wa_d5 = m->gu.wa_d0;
  }
  ok = ok && encode_bf16_rows(&m->gu.xb_d64, ws + L.x, T, H, 64);
  ok = ok && encode_bf16_rows(&m->gu.xb_d16, ws + L.x, T, H, 16);
  ok = ok && encode_bf16_rows(&m->gu.xb_d256, ws + L.x, T, H, 256);
  ok = ok && encode_bf16_rows(&m->gu.xb_d128, ws + L.x, T, H, 128);
  ok = ok && encode_bf16_rows(&m->gu.xb_d32, ws + L.x, T, H, 32);
  // down: [H, D] in 128-row boxes over act
  if (q4) ok = ok && encode_q_rows(&m->dn.wa_d0, weights->down.q, H, D, 128, qb);
  else ok = ok && encode_bf16_rows(&m->dn.wa_d0, weights->down.q, H, D, 128);
  ok = ok && encode_bf16_rows(&m->dn.xb_d64, ws + L.act, T, D, 64);
  ok = ok && encode_bf16_rows(&m->dn.xb_d16, ws + L.act, T, D, 16);
  ok = ok && encode_bf16_rows(&m->dn.xb_d256, ws + L.act, T, D, 256);
  ok = ok && encode_bf16_rows(&m->dn.xb_d128, ws + L.act, T, D, 128);
  ok = ok && encode_bf16_rows(&m->dn.xb_d32, ws + L.act, T, D, 32);
  if (!ok) {
    delete m;
    return DG_ERR_CUDA;
  }
  // no experts: the expert-side maps are copies of valid ones (never used)
  m->gu.wa_exp = m->gu.wa_d0;
  m->gu.xb_exp64 = m->gu.xb_d64;
  m->gu.xb_exp16 = m->gu.xb_d16;
  m->gu.xb_exp256 = m->gu.xb_d256;
  m->gu.xb_exp128 = m->gu.xb_d128;
  m->gu.xb_exp32 = m->gu.xb_d32;
  m->dn.wa_exp = m->dn.wa_d0;
  m->dn.wa_d1 = m->dn.wa_d0;
  m->dn.wa_d5 = m->dn.wa_d0;
  m->dn.dense_5d = 0;
  m->dn.xb_exp64 = m->dn.xb_d64;
  m->dn.xb_exp16 = m->dn.xb_d16;
  m->dn.xb_exp256 = m->dn.xb_d256;
  m->dn.xb_exp128 = m->dn.xb_d128;
  m->dn.xb_exp32 = m->dn.xb_d32;
  if (cudaMemset(ws + L.status, 0, sizeof(DevStatus)) != cudaSuccess ||
      cudaMemset(ws + L.zero, 0, 16) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  auto u16 = [](const void* v) { return static_cast<const uint16_t*>(v); };
  for (GemmParams* g : {&m->gu, &m->dn}) {
    g->offsets = reinterpret_cast<const int32_t*>(ws + L.zero);
    g->E = 0;
    g->I = 0;
    g->D = (int)D;
    g->H = (int)H;
    g->mt_exp = 0;
    g->kb_exp = 0;
    g->act = nullptr;
    g->act_d = reinterpret_cast<uint16_t*>(ws + L.act);
    g->y_moe = nullptr;
    g->y_perm = nullptr;
    g->y_dense = reinterpret_cast<float*>(ws + L.y);
    g->tok_perm = nullptr;
    g->w_perm = nullptr;
    g->status = reinterpret_cast<DevStatus*>(ws + L.status);
  }
  m->gu.kb_dense = (int)(H / 64);
  m->gu.mt_dense = (int)(D / 64);
  m->dn.kb_dense = (int)(D / 64);
  m->dn.mt_dense = (int)(H / 128);
  m->gu.sc_d0 = u16(weights->gate.scales);
  m->gu.bi_d0 = u16(weights->gate.biases);
  m->gu.sc_d1 = u16(weights->up.scales);
  m->gu.bi_d1 = u16(weights->up.biases);
  m->gu.sc_exp = m->gu.sc_d0;
  m->gu.bi_exp = m->gu.bi_d0;
  m->dn.sc_d0 = m->dn.sc_d1 = m->dn.sc_exp = u16(weights->down.scales);
  m->dn.bi_d0 = m->dn.bi_d1 = m->dn.bi_exp = u16(weights->down.biases);
  m->gu.sc_slot_bytes = (int)round_up(128 * (H / 64) * 2, 128);
  m->dn.sc_slot_bytes = (int)round_up(128 * (D / 64) * 2, 128);
  if (q4 && (gemm_q4_smem_bytes(32, m->gu.sc_slot_bytes) > m->smem_optin ||
             gemm_q4_smem_bytes(32, m->dn.sc_slot_bytes) > m->smem_optin)) {
    delete m;
    return DG_ERR_UNSUPPORTED;
  }
  *out = m;
  return DG_OK;
}

dg_status_t dg_sc_mlp_forward(dg_sc_mlp_t* m, const void* embeds, const void* signal, void* out,
                              int n_tokens, dg_stream_t stream) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_tokens > m->cfg.max_tokens) return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!embeds || !signal || !out) return DG_ERR_INVALID_ARG;
  if (!aligned(embeds, 16) || !aligned(signal, 16) || !aligned(out, 16)) return DG_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = n_tokens, H = m->cfg.hidden;
  const float eps = m->cfg.rms_eps;
  uint8_t* ws = m->ws;
  const ScLayout& L = m->L;
  cudaError_t err = cudaSuccess;
  auto mark = [&](int i) {
    if (m->prof && err == cudaSuccess)
      err = cudaEventRecord(reinterpret_cast<cudaEvent_t>(m->prof[i]), s);
  };
  mark(0);
  if (err == cudaSuccess)
    err = launch_pdl(k_sc_prenorm, dim3(T), dim3(kScThreads), 0, s,
                     static_cast<const uint16_t*>(signal),
                     static_cast<const uint16_t*>(m->w.pre_norm), H, eps,
                     reinterpret_cast<uint16_t*>(ws + L.x));
  mark(1);
  GemmParams gu = m->gu, dn = m->dn;
  gu.T = dn.T = T;
  const int bn = m->q4 ? pick_bn_q4(T, gu.sc_slot_bytes, dn.sc_slot_bytes, m->smem_optin)
                       : pick_bn(T);
  gu.bn = dn.bn = bn;
  if (err == cudaSuccess)
    err = m->q4 ? launch_gemm_affine(0, bn, m->qbits, gu, m->num_sms, s)
                : launch_gemm(0, bn, gu, m->num_sms, s);
  mark(2);
  if (err == cudaSuccess)
    err = m->q4 ? launch_gemm_affine(1, bn, m->qbits, dn, m->num_sms, s)
                : launch_gemm(1, bn, dn, m->num_sms, s);
  mark(3);
  if (err == cudaSuccess)
    err = launch_pdl(k_sc_post, dim3(T), dim3(kScThreads), 0, s,
                     static_cast<const uint16_t*>(embeds),
                     reinterpret_cast<const float*>(ws + L.y), H, eps,
                     static_cast<uint16_t*>(out));
  mark(4);
  return err == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status_t dg_sc_mlp_last_device_status(dg_sc_mlp_t* m, dg_stream_t stream) {
  if (!m) return DG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
  DevStatus st;
  if (cudaMemcpy(&st, m->ws + m->L.status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaMemset(m->ws + m->L.status, 0, sizeof(st)) != cudaSuccess) return DG_ERR_CUDA;
  if (st.code == kDevTimeout) return DG_ERR_TIMEOUT;
  if (st.code == kDevBounds) return DG_ERR_DEVICE_CHECK;
  return DG_OK;
}

dg_status_t dg_sc_mlp_kernel_names(const dg_sc_mlp_t* m, const char** names, int* n) {
  if (!m || !n) return DG_ERR_INVALID_ARG;
  *n = kScKernels;
  if (names)
    for (int i = 0; i < kScKernels; ++i) names[i] = kScKernelNames[i];
  return DG_OK;
}

dg_status_t dg_sc_mlp_set_profile_events(dg_sc_mlp_t* m, dg_event_t* events, int n_events) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (events && n_events != kScKernels + 1) return DG_ERR_INVALID_ARG;
  m->prof = events;
  return DG_OK;
}

dg_status_t dg_sc_mlp_destroy(dg_sc_mlp_t* m) {
  delete m;
  return DG_OK;
}

}  // extern "C"
