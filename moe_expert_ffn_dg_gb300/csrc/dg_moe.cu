// C-ABI implementation of the MoE FFN block: argument validation, workspace
// layout, TMA descriptors and the launch sequence of one forward.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "../../include/dg_moe.h"
#include "dg_host.h"
#include "dg_kernels.h"

using namespace dg;
using namespace dg::host;

namespace {

constexpr int kNumKernels = 6;
const char* const kKernelNames[kNumKernels] = {
    "router_logits", "router_select", "scatter_gather", "gemm_gate_up", "gemm_down", "combine"};



struct Layout {
  size_t status, counters, r, xnorm, wnorm, logits, idx, w, chunk_counts, chunk_masks, offsets, perm,
      tok_perm, w_perm, inv, zero16, planes, flagged, zpart;
  size_t xd, xe_perm, act, act_d, y_moe, y_dense, y_perm, hmid, stage_in, stage_out;
  size_t zero_begin, zero_end;  // counters, chunk counts and masks, cleared per forward
  size_t total;
};


Layout make_layout(const dg_moe_config_t& c) {
  Layout L;
  const size_t T = (size_t)c.max_tokens, H = c.hidden, E = c.n_experts, K = c.top_k;
  const size_t I = c.expert_inter, D = c.dense_inter, TK = T * K;
  const size_t nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  L.status = take(sizeof(DevStatus));
  L.counters = take(16 * sizeof(int));  // [0] n_refined, [1] flagged tokens
  L.chunk_counts = take(nchunks * E * 4);
  L.chunk_masks = take(nchunks * E * (kChunkTokens / 32) * 4);
  L.zero_begin = L.counters;
  L.zero_end = L.chunk_masks + nchunks * E * (kChunkTokens / 32) * 4;
  L.r = take(T * 4);
  L.xnorm = take(T * 4);
  L.wnorm = take(E * 4);
  L.logits = take(T * E * 4);
  L.idx = take(TK * 4);
  L.w = take(TK * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(TK * 4);
  L.tok_perm = take(TK * 4);
  L.w_perm = take(TK * 4);
  L.inv = take(TK * 4);
  L.zero16 = take(16);  // expert offsets {0} of a launch with no experts
  // router rows times router_scale as bf16 planes (hi | lo), for the
  // tensor-core logits of large batches
  const bool tc = T >= (size_t)kRouterTcMinTokens;
  L.planes = tc ? take(E * 2 * H * 2) : 0;
  // split-K partial logits: the largest split times tokens over the batch
  // sizes the handle accepts
  {
    const int kb = (int)(2 * H / 64);
    size_t most = 0;
    for (size_t n = kRouterTcMinTokens / kRouterBn; tc && n <= (T + kRouterBn - 1) / kRouterBn;
         ++n) {
      const size_t t = n * kRouterBn < T ? n * kRouterBn : T;
      const size_t sp = (size_t)router_split((int)t, (int)E, kb);
      if (sp > 1 && sp * t > most) most = sp * t;
    }
    L.zpart = take(most * E * 4);
  }
  // tokens left to the re-check pass of the two-pass selection
  L.flagged = T >= (size_t)kRouterTcMinTokens ? take(T * 4) : 0;
  L.xd = take(T * H * 2);
  L.hmid = take(T * H * 2);  // the block input built by the fused attention half
  L.xe_perm = take(TK * H * 2);
  L.act = take(TK * I * 2);
  L.act_d = take(T * D * 2);
  L.y_moe = take(T * H * 4);
  L.y_dense = take(T * H * 4);
  // weighted expert rows, for batches that avoid the atomic reduction
  L.y_perm = T >= (size_t)kPartialRowsMinTokens ? take(TK * H * 4) : 0;
  L.stage_in = take(T * H * 2);
  L.stage_out = take(T * H * 2);
  L.total = off;
  return L;
}


dg_status_t check_config(const dg_moe_config_t* c) {
  dg_status_t s = check_router_config(c);
  if (s != DG_OK) return s;
  if (c->expert_inter <= 0 || c->dense_inter <= 0 || c->max_tokens <= 0) return DG_ERR_INVALID_ARG;
  if (c->expert_inter % 64 || c->dense_inter % 64) return DG_ERR_UNSUPPORTED;
  if (c->max_tokens > (1 << 20)) return DG_ERR_UNSUPPORTED;
  // expert and dense weights: both bf16, or 4-bit group-64 affine experts
  // with a 4- or 8-bit dense branch
  const bool bf16w = c->expert_fmt == DG_FMT_BF16 && c->dense_fmt == DG_FMT_BF16;
  const bool q4w = (c->expert_fmt == DG_FMT_AFFINE_U4_G64 &&
                    (c->dense_fmt == DG_FMT_AFFINE_U4_G64 || c->dense_fmt == DG_FMT_AFFINE_U8_G64)) ||
                   (c->expert_fmt == DG_FMT_NVFP4_G16 && c->dense_fmt == DG_FMT_NVFP4_G16);
  if (!bf16w && !q4w) return DG_ERR_UNSUPPORTED;
  // 4-bit: one tile's scale and bias rows (128 x K/64 each, twice) must fit
  // in shared memory beside the narrowest tiles' pipelines
  if (q4w && (c->hidden > 2944 || c->expert_inter > 2944 || c->dense_inter > 2944))
    return DG_ERR_UNSUPPORTED;
  return DG_OK;
}


dg_status_t check_weights(const dg_moe_config_t& c, const dg_moe_weights_t* w) {
  dg_status_t s;
  if ((s = check_router_weights(c, w)) != DG_OK) return s;
  if ((s = check_qtensor(w->gate_up, c.expert_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->down, c.expert_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_gate, c.dense_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_up, c.dense_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_down, c.dense_fmt)) != DG_OK) return s;
  const void* vecs[] = {w->w_pre_ff2, w->w_post_ff1, w->w_post_ff2, w->w_post_ff};
  for (const void* v : vecs) {
    if (!v) return DG_ERR_INVALID_ARG;
    if (!aligned(v, 16)) return DG_ERR_ALIGNMENT;
  }
  return DG_OK;
}

}  // namespace

struct dg_moe {
  dg_moe_config_t cfg;
  dg_moe_weights_t w;
  uint8_t* ws;
  size_t ws_bytes;
  Layout L;
  int device;
  int num_sms;
  GemmParams gu;
  GemmParams dn;
  bool q4;  // quantised expert weights (4-bit affine or NVFP4) and dense
  int qf_exp;         // expert code format: 4 or kQfNvfp4 (with q4)
  int dense_bits;     // dense code format: 4, 8 or kQfNvfp4 (with q4)
  GemmParams gu_d;    // dense-only launches when the dense bits differ (8-bit)
  GemmParams dn_d;
  GemmParams gr;      // router logits on the tensor cores (large batches)
  size_t smem_optin;  // largest dynamic shared memory a block may opt into
  dg_event_t* prof;
  int n_prof;
  int stall_armed;  // the next forward runs the bounded-wait test
  char last_error[256];
};

namespace {
// Record the failing CUDA call in the handle and map it to DG_ERR_CUDA.
dg_status_t cuda_fail(dg_moe* m, const char* what, cudaError_t e) {
  if (m) snprintf(m->last_error, sizeof(m->last_error), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  return DG_ERR_CUDA;
}
}  // namespace

extern "C" {

const char* dg_moe_status_string(dg_status_t s) {
  switch (s) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument";
    case DG_ERR_ALIGNMENT: return "pointer misaligned";
    case DG_ERR_UNSUPPORTED: return "unsupported shape or format";
    case DG_ERR_CUDA: return "CUDA error";
    case DG_ERR_TIMEOUT: return "device wait timed out";
    case DG_ERR_DEVICE_CHECK: return "device range check failed";
    case DG_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

dg_status_t dg_moe_workspace_size(const dg_moe_config_t* cfg, size_t* bytes) {
  if (!bytes) return DG_ERR_INVALID_ARG;
  dg_status_t s = check_config(cfg);
  if (s != DG_OK) return s;
  *bytes = make_layout(*cfg).total;
  return DG_OK;
}

dg_status_t dg_moe_create(const dg_moe_config_t* cfg, const dg_moe_weights_t* weights,
                          void* workspace, size_t workspace_bytes, dg_moe_t** out) {
  if (!out) return DG_ERR_INVALID_ARG;
  *out = nullptr;
  dg_status_t s = check_config(cfg);
  if (s != DG_OK) return s;
  s = check_weights(*cfg, weights);
  if (s != DG_OK) return s;
  const Layout L = make_layout(*cfg);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 1024)) return DG_ERR_WORKSPACE;

  dg_moe* m = new (std::nothrow) dg_moe();
  if (!m) return DG_ERR_CUDA;
  m->cfg = *cfg;
  if (m->cfg.rms_eps == 0.f) m->cfg.rms_eps = 1e-6f;
  m->w = *weights;
  m->ws = static_cast<uint8_t*>(workspace);
  m->ws_bytes = workspace_bytes;
  m->L = L;
  m->prof = nullptr;
  m->n_prof = 0;
  m->last_error[0] = 0;
  int optin = 0;
  if (cudaGetDevice(&m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, m->device) !=
          cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  m->smem_optin = (size_t)optin;
  const dg_moe_config_t& c = m->cfg;
  const bool quantised = c.expert_fmt != DG_FMT_BF16;
  // the bf16 GEMM kernels serve the router logits of large batches in every
  // weight format
  if (prepare_router(optin) != cudaSuccess || prepare_gemm_bf16() != cudaSuccess ||
      (quantised && prepare_gemm_affine(optin) != cudaSuccess)) {
    delete m;
    return DG_ERR_CUDA;
  }
  const uint64_t H = c.hidden, E = c.n_experts, I = c.expert_inter, D = c.dense_inter;
  const uint64_t T = c.max_tokens, TK = T * c.top_k;
  uint8_t* ws = m->ws;
  bool ok = true;
  // gate_up A: experts through the interleaving 5-D view; the dense pair the
  // same way when dense_up lies above dense_gate, else 16-row boxes of each
  const bool nvfp4 = c.expert_fmt == DG_FMT_NVFP4_G16;
  const bool q4 = c.expert_fmt == DG_FMT_AFFINE_U4_G64 || nvfp4;
  m->q4 = q4;
  m->qf_exp = nvfp4 ? kQfNvfp4 : 4;
  // dense code bits in the slabs (NVFP4 codes are 4-bit, in the affine layout)
  const int db = c.dense_fmt == DG_FMT_AFFINE_U8_G64 ? 8 : 4;
  m->dense_bits = !q4 ? 0 : (c.dense_fmt == DG_FMT_NVFP4_G16 ? kQfNvfp4 : db);
  const uint64_t wb2 = q4 ? 1 : 4;  // bytes of two weights
  ok = ok && encode_gate_up(&m->gu.wa_exp, weights->gate_up.q, H, I, I * H * wb2 / 2, 5, E,
                            2 * I * H * wb2 / 2, q4 ? 4 : 0);
  if (q4) {
    ok = ok && encode_q_rows(&m->gu.wa_d0, weights->dense_gate.q, D, H, 16, db);
    ok = ok && encode_q_rows(&m->gu.wa_d1, weights->dense_up.q, D, H, 16, db);
  } else {
    ok = ok && encode_bf16_rows(&m->gu.wa_d0, weights->dense_gate.q, D, H, 16);
    ok = ok && encode_bf16_rows(&m->gu.wa_d1, weights->dense_up.q, D, H, 16);
  }
  {
    const uintptr_t g = (uintptr_t)weights->dense_gate.q, u = (uintptr_t)weights->dense_up.q;
    m->gu.dense_5d = u > g && ((u - g) % 16) == 0 && (u - g) < (1ull << 40) &&
                     encode_gate_up(&m->gu.wa_d5, weights->dense_gate.q, H, D, u - g, 4, 1, 0,
                                    q4 ? db : 0);
    if (!m->gu.dense_5d) m->gu.wa_d5 = m->gu.wa_d0;
  }
  // gate_up B: xe_perm / xd rows
  ok = ok && encode_bf16_rows(&m->gu.xb_exp64, ws + L.xe_perm, TK, H, 64);
  ok = ok && encode_bf16_rows(&m->gu.xb_exp16, ws + L.xe_perm, TK, H, 16);
  ok = ok && encode_bf16_rows(&m->gu.xb_d64, ws + L.xd, T, H, 64);
  ok = ok && encode_bf16_rows(&m->gu.xb_d16, ws + L.xd, T, H, 16);
  for (const uint32_t br : {256u, 128u, 32u}) {
    CUtensorMap* me = br == 256 ? &m->gu.xb_exp256 : br == 128 ? &m->gu.xb_exp128 : &m->gu.xb_exp32;
    CUtensorMap* md = br == 256 ? &m->gu.xb_d256 : br == 128 ? &m->gu.xb_d128 : &m->gu.xb_d32;
    ok = ok && encode_bf16_rows(me, ws + L.xe_perm, TK, H, br);
    ok = ok && encode_bf16_rows(md, ws + L.xd, T, H, br);
  }
  // down A: [E*H, I] and [H, D] in 128-row boxes; B: act / act_d rows
  if (q4) {
    ok = ok && encode_q4_rows(&m->dn.wa_exp, weights->down.q, E * H, I, 128);
    ok = ok && encode_q_rows(&m->dn.wa_d0, weights->dense_down.q, H, D, 128, db);
  } else {
    ok = ok && encode_bf16_rows(&m->dn.wa_exp, weights->down.q, E * H, I, 128);
    ok = ok && encode_bf16_rows(&m->dn.wa_d0, weights->dense_down.q, H, D, 128);
  }
  m->dn.wa_d1 = m->dn.wa_d0;
  m->dn.wa_d5 = m->dn.wa_d0;
  m->dn.dense_5d = 0;
  ok = ok && encode_bf16_rows(&m->dn.xb_exp64, ws + L.act, TK, I, 64);
  ok = ok && encode_bf16_rows(&m->dn.xb_exp16, ws + L.act, TK, I, 16);
  ok = ok && encode_bf16_rows(&m->dn.xb_d64, ws + L.act_d, T, D, 64);
  ok = ok && encode_bf16_rows(&m->dn.xb_d16, ws + L.act_d, T, D, 16);
  for (const uint32_t br : {256u, 128u, 32u}) {
    CUtensorMap* me = br == 256 ? &m->dn.xb_exp256 : br == 128 ? &m->dn.xb_exp128 : &m->dn.xb_exp32;
    CUtensorMap* md = br == 256 ? &m->dn.xb_d256 : br == 128 ? &m->dn.xb_d128 : &m->dn.xb_d32;
    ok = ok && encode_bf16_rows(me, ws + L.act, TK, I, br);
    ok = ok && encode_bf16_rows(md, ws + L.act_d, T, D, br);
  }
  if (!ok) {
    delete m;
    return DG_ERR_CUDA;
  }
  // the device status word starts clear
  if (cudaMemset(ws + L.status, 0, sizeof(DevStatus)) != cudaSuccess ||
      cudaMemset(ws + L.zero16, 0, 16) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  for (GemmParams* g : {&m->gu, &m->dn}) {
    g->offsets = reinterpret_cast<const int32_t*>(ws + L.offsets);
    g->E = (int)E;
    g->I = (int)I;
    g->D = (int)D;
    g->H = (int)H;
    g->act = reinterpret_cast<uint16_t*>(ws + L.act);
    g->act_d = reinterpret_cast<uint16_t*>(ws + L.act_d);
    g->y_moe = reinterpret_cast<float*>(ws + L.y_moe);
    g->y_dense = reinterpret_cast<float*>(ws + L.y_dense);
    g->tok_perm = reinterpret_cast<const int32_t*>(ws + L.tok_perm);
    g->w_perm = reinterpret_cast<const float*>(ws + L.w_perm);
    g->status = reinterpret_cast<DevStatus*>(ws + L.status);
  }
  m->gu.kb_exp = (int)(H / 64);
  m->gu.kb_dense = (int)(H / 64);
  m->gu.mt_exp = (int)(I / 64);
  m->gu.mt_dense = (int)(D / 64);
  m->dn.kb_exp = (int)(I / 64);
  m->dn.kb_dense = (int)(D / 64);
  m->dn.mt_exp = (int)(H / 128);
  m->dn.mt_dense = (int)(H / 128);
  // scale and bias rows of the 4-bit weights (unused for bf16)
  auto u16 = [](const void* v) { return static_cast<const uint16_t*>(v); };
  m->gu.sc_exp = u16(weights->gate_up.scales);
  m->gu.bi_exp = u16(weights->gate_up.biases);
  m->gu.sc_d0 = u16(weights->dense_gate.scales);
  m->gu.bi_d0 = u16(weights->dense_gate.biases);
  m->gu.sc_d1 = u16(weights->dense_up.scales);
  m->gu.bi_d1 = u16(weights->dense_up.biases);
  m->dn.sc_exp = u16(weights->down.scales);
  m->dn.bi_exp = u16(weights->down.biases);
  m->dn.sc_d0 = m->dn.sc_d1 = u16(weights->dense_down.scales);
  m->dn.bi_d0 = m->dn.bi_d1 = u16(weights->dense_down.biases);
  // NVFP4 matrix scales (the biases slot of its tensors)
  auto f32p = [](const void* v) { return static_cast<const float*>(v); };
  m->gu.g_exp = f32p(weights->gate_up.biases);
  m->gu.g_d0 = f32p(weights->dense_gate.biases);
  m->gu.g_d1 = f32p(weights->dense_up.biases);
  m->dn.g_exp = f32p(weights->down.biases);
  m->dn.g_d0 = m->dn.g_d1 = f32p(weights->dense_down.biases);
  // one tile's scales: affine s and b (bf16 per 64) or NVFP4 e4m3 per 16,
  // both 128 x K/16 bytes over the slot pair
  m->gu.sc_slot_bytes = (int)round_up(128 * (H / 64) * 2, 128);
  m->dn.sc_slot_bytes = (int)round_up(128 * (I > D ? I : D) / 64 * 2, 128);
  if (q4 && (gemm_q4_smem_bytes(32, m->gu.sc_slot_bytes) > m->smem_optin ||
             gemm_q4_smem_bytes(32, m->dn.sc_slot_bytes) > m->smem_optin)) {
    delete m;
    return DG_ERR_UNSUPPORTED;
  }
  if (T >= (uint64_t)kRouterTcMinTokens) {
    // router GEMM: the planes [E, 2H] are the weight side (M = 128 experts a
    // tile), the token rows of the block input the other; no expert groups
    GemmParams& g = m->gr;
    if (!encode_bf16_rows(&g.wa_d0, ws + L.planes, E, 2 * H, 128)) {
      delete m;
      return DG_ERR_CUDA;
    }
    g.wa_exp = g.wa_d1 = g.wa_d5 = g.wa_d0;
    g.offsets = reinterpret_cast<const int32_t*>(ws + L.zero16);
    g.E = 0;
    g.H = (int)H;
    g.mt_exp = 0;
    g.kb_exp = 0;
    g.mt_dense = (int)((E + 127) / 128);
    g.kb_dense = (int)(2 * H / 64);
    g.z_out = reinterpret_cast<float*>(ws + L.logits);
    g.z_part = reinterpret_cast<float*>(ws + L.zpart);
    g.z_r = reinterpret_cast<const float*>(ws + L.r);
    g.z_bias = weights->router_bias;
    g.z_E = (int)E;
    g.z_cH = (float)(1.0 / sqrt((double)H));
    g.status = reinterpret_cast<DevStatus*>(ws + L.status);
  }
  if (q4 && m->dense_bits != m->qf_exp) {
    // the dense branch in launches of its own (no expert tiles), the expert
    // launches without dense tiles
    m->gu_d = m->gu;
    m->dn_d = m->dn;
    for (GemmParams* g : {&m->gu_d, &m->dn_d}) {
      g->E = 0;
      g->mt_exp = 0;
      g->offsets = reinterpret_cast<const int32_t*>(ws + L.zero16);
      g->wa_exp = g->wa_d0;  // valid maps, never read
    }
    m->gu.mt_dense = 0;
    m->dn.mt_dense = 0;
  }
  *out = m;
  return DG_OK;
}

const char* dg_moe_last_error(const dg_moe_t* m) {
  if (!m) return "no handle";
  return m->last_error;
}

dg_status_t dg_moe_destroy(dg_moe_t* m) {
  delete m;
  return DG_OK;
}

dg_status_t dg_moe_kernel_names(const dg_moe_t* m, const char** names, int* n) {
  if (!m || !n) return DG_ERR_INVALID_ARG;
  *n = kNumKernels;
  if (names)
    for (int i = 0; i < kNumKernels; ++i) names[i] = kKernelNames[i];
  return DG_OK;
}

dg_status_t dg_moe_arm_wait_timeout_test(dg_moe_t* m) {
  if (!m) return DG_ERR_INVALID_ARG;
  m->stall_armed = 1;
  return DG_OK;
}

dg_status_t dg_moe_set_profile_events(dg_moe_t* m, dg_event_t* events, int n_events) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (events && n_events != kNumKernels + 1) return DG_ERR_INVALID_ARG;
  m->prof = events;
  m->n_prof = events ? n_events : 0;
  return DG_OK;
}

namespace {
// One forward; nb (may be null) fuses the decoder layer's neighbours.
dg_status_t forward_impl(dg_moe_t* m, const void* h_in, void* h_out, int n_tokens,
                         float layer_scalar, dg_stream_t stream, const dg_moe_debug_t* dbg,
                         const dg_moe_neighbours_t* nb) {
  const dg_moe_config_t& c = m->cfg;
  const Layout& L = m->L;
  uint8_t* ws = m->ws;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = n_tokens, H = c.hidden, E = c.n_experts, K = c.top_k;
  const int TK = T * K;
  const int bn = m->q4 ? pick_bn_q4(T, m->gu.sc_slot_bytes, m->dn.sc_slot_bytes, m->smem_optin)
                      : pick_bn(T);
  int* counters = reinterpret_cast<int*>(ws + L.counters);
  DevStatus* status = reinterpret_cast<DevStatus*>(ws + L.status);
  cudaError_t err = cudaSuccess;
  const char* failed = "";
  auto mark = [&](int i) {
    if (err != cudaSuccess && !failed[0]) failed = i > 0 ? kKernelNames[i - 1] : "event";
    if (m->prof && err == cudaSuccess) {
      err = cudaEventRecord(reinterpret_cast<cudaEvent_t>(m->prof[i]), s);
      if (err != cudaSuccess) failed = "profile event record";
    }
  };
  if ((err = cudaMemsetAsync(ws + L.zero_begin, 0, L.zero_end - L.zero_begin, s)) != cudaSuccess)
    return cuda_fail(m, "memset counters", err);

  RouterParams rp{};
  rp.h = static_cast<const uint16_t*>(h_in);
  rp.wr = m->w.router.q;
  rp.wr_scales = static_cast<const uint16_t*>(m->w.router.scales);
  rp.wr_biases = static_cast<const uint16_t*>(m->w.router.biases);
  rp.router_scale = static_cast<const uint16_t*>(m->w.router_scale);
  rp.pes = static_cast<const uint16_t*>(m->w.per_expert_scale);
  rp.w_pre_ff = static_cast<const uint16_t*>(m->w.w_pre_ff);
  rp.router_bias = m->w.router_bias;
  rp.T = T;
  rp.H = H;
  rp.cHd = 1.0 / sqrt((double)H);
  rp.cH = (float)rp.cHd;
  rp.E = E;
  rp.K = K;
  rp.router_u8 = c.router_fmt == DG_FMT_AFFINE_U8_G64;
  rp.eps = c.rms_eps;
  rp.r_out = reinterpret_cast<float*>(ws + L.r);
  rp.xnorm_out = reinterpret_cast<float*>(ws + L.xnorm);
  rp.wnorm_out = reinterpret_cast<float*>(ws + L.wnorm);
  rp.idx = reinterpret_cast<int32_t*>(ws + L.idx);
  rp.w = reinterpret_cast<float*>(ws + L.w);
  rp.logits = reinterpret_cast<float*>(ws + L.logits);
  rp.chunk_counts = reinterpret_cast<int32_t*>(ws + L.chunk_counts);
  rp.chunk_masks = reinterpret_cast<uint32_t*>(ws + L.chunk_masks);
  rp.xd = reinterpret_cast<uint16_t*>(ws + L.xd);
  // large batches: weighted expert rows summed by the combine, no
  // accumulator to clear; small ones: atomic adds into the cleared y_moe
  const bool partials = T >= kPartialRowsMinTokens;
  rp.y_moe = partials ? nullptr : reinterpret_cast<float*>(ws + L.y_moe);
  rp.n_refined = counters;
  // the block input: h_in itself, or built by the router from the residual
  // h_in and the attention output
  const uint16_t* hb = rp.h;
  if (nb) {
    rp.attn = static_cast<const uint16_t*>(nb->attn_out);
    rp.w_post_attn = static_cast<const uint16_t*>(nb->w_post_attn);
    rp.h_out = static_cast<uint16_t*>(nb->h_mid ? nb->h_mid : ws + L.hmid);
    hb = rp.h_out;
  }
  mark(0);
  if (T >= kRouterTcMinTokens) {
    // tensor-core logits: prep (r, xd, planes, norms), then the router GEMM
    // over the block input (split over K ranges while the token tiles alone
    // would leave most SMs idle), and the selection in two passes
    const int split = router_split(T, E, 2 * H / 64);
    rp.logits_tc = 1;
    rp.planes = reinterpret_cast<uint16_t*>(ws + L.planes);
    rp.z_split = split;
    rp.z_part = split > 1 ? reinterpret_cast<const float*>(ws + L.zpart) : nullptr;
    rp.flagged = reinterpret_cast<int32_t*>(ws + L.flagged);
    rp.n_flagged = counters + 1;
    if (err == cudaSuccess) err = launch_router_prep_tc(rp, s);
    GemmParams gr = m->gr;
    gr.T = T;
    gr.bn = kRouterBn;
    gr.z_split = split;
    gr.mt_dense *= split;
    if (err == cudaSuccess &&
        !(encode_bf16_rows(&gr.xb_d64, hb, (uint64_t)T, (uint64_t)H, 64) &&
          encode_bf16_rows(&gr.xb_d16, hb, (uint64_t)T, (uint64_t)H, 16)))
      return cuda_fail(m, "router token map", cudaErrorInvalidValue);
    gr.xb_exp64 = gr.xb_d64;
    gr.xb_exp16 = gr.xb_d16;
    // (whole-tile maps are not used by the router GEMM)
    gr.xb_exp256 = gr.xb_d256 = gr.xb_exp128 = gr.xb_d128 = gr.xb_exp32 = gr.xb_d32 = gr.xb_d64;
    if (err == cudaSuccess) err = launch_gemm(2, kRouterBn, gr, m->num_sms, s);
  } else if (err == cudaSuccess) {
    // small batches: the CUDA-core logit kernel (latency-bound either way,
    // and it keeps the tighter bound), one selection pass
    err = launch_router(rp, s);
  }
  rp.h = hb;
  rp.attn = nullptr;
  mark(1);
  if (err == cudaSuccess) err = launch_router_select(rp, m->num_sms, s);
  ScatterParams sp{};
  sp.idx = rp.idx;
  sp.w = rp.w;
  sp.chunk_counts = reinterpret_cast<const int32_t*>(ws + L.chunk_counts);
  sp.chunk_masks = reinterpret_cast<const uint32_t*>(ws + L.chunk_masks);
  sp.T = T;
  sp.K = K;
  sp.E = E;
  sp.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  sp.perm = reinterpret_cast<int32_t*>(ws + L.perm);
  sp.tok_perm = reinterpret_cast<int32_t*>(ws + L.tok_perm);
  sp.w_perm = reinterpret_cast<float*>(ws + L.w_perm);
  sp.inv = partials ? reinterpret_cast<int32_t*>(ws + L.inv) : nullptr;
  sp.status = status;

  GatherParams gp{};
  gp.h = hb;
  gp.r = rp.r_out;
  gp.tok_perm = sp.tok_perm;
  gp.w_pre_ff2 = static_cast<const uint16_t*>(m->w.w_pre_ff2);
  gp.TK = TK;
  gp.H = H;
  gp.xe_perm = reinterpret_cast<uint16_t*>(ws + L.xe_perm);
  mark(2);
  if (err == cudaSuccess) err = launch_scatter_gather(sp, gp, s);
  GemmParams gu = m->gu, dn = m->dn;
  gu.test_stall = m->stall_armed;
  m->stall_armed = 0;
  gu.T = dn.T = T;
  gu.bn = dn.bn = bn;
  dn.y_perm = partials ? reinterpret_cast<float*>(ws + L.y_perm) : nullptr;
  // 8-bit dense weights beside 4-bit experts: a dense-only launch after each
  // expert launch (the same profiling slot)
  const bool split = m->q4 && m->dense_bits != m->qf_exp;
  GemmParams gu_d = m->gu_d, dn_d = m->dn_d;
  gu_d.T = dn_d.T = T;
  gu_d.bn = dn_d.bn = bn;
  dn_d.y_perm = dn.y_perm;
  mark(3);
  if (err == cudaSuccess)
    err = m->q4 ? launch_gemm_affine(0, bn, m->qf_exp, gu, m->num_sms, s)
                : launch_gemm(0, bn, gu, m->num_sms, s);
  if (err == cudaSuccess && split) err = launch_gemm_affine(0, bn, m->dense_bits, gu_d, m->num_sms, s);
  mark(4);
  if (err == cudaSuccess)
    err = m->q4 ? launch_gemm_affine(1, bn, m->qf_exp, dn, m->num_sms, s)
                : launch_gemm(1, bn, dn, m->num_sms, s);
  if (err == cudaSuccess && split) err = launch_gemm_affine(1, bn, m->dense_bits, dn_d, m->num_sms, s);

  CombineParams cp{};
  cp.y_dense = reinterpret_cast<const float*>(ws + L.y_dense);
  cp.y_moe = reinterpret_cast<const float*>(ws + L.y_moe);
  cp.y_perm = dn.y_perm;
  cp.inv = sp.inv;
  cp.K = K;
  cp.y_moe_out = partials && dbg && dbg->y_moe ? reinterpret_cast<float*>(ws + L.y_moe) : nullptr;
  cp.h = hb;
  if (nb && nb->w_next_in) {
    cp.w_next = static_cast<const uint16_t*>(nb->w_next_in);
    cp.next_out = static_cast<uint16_t*>(nb->next_in);
  }
  cp.w_post1 = static_cast<const uint16_t*>(m->w.w_post_ff1);
  cp.w_post2 = static_cast<const uint16_t*>(m->w.w_post_ff2);
  cp.w_post = static_cast<const uint16_t*>(m->w.w_post_ff);
  cp.T = T;
  cp.H = H;
  cp.eps = c.rms_eps;
  cp.layer_scalar = layer_scalar;
  cp.out = static_cast<uint16_t*>(h_out);
  mark(5);
  if (err == cudaSuccess) err = launch_combine(cp, s);
  mark(6);
  if (err != cudaSuccess) return cuda_fail(m, failed[0] ? failed : "launch", err);

  if (dbg) {
    struct Copy { void* dst; size_t off; size_t bytes; };
    const Copy copies[] = {
        {dbg->idx, L.idx, (size_t)TK * 4},
        {dbg->w, L.w, (size_t)TK * 4},
        {dbg->logits, L.logits, (size_t)T * E * 4},
        {dbg->offsets, L.offsets, (size_t)(E + 1) * 4},
        {dbg->perm, L.perm, (size_t)TK * 4},
        {dbg->xd, L.xd, (size_t)T * H * 2},
        {dbg->xe_perm, L.xe_perm, (size_t)TK * H * 2},
        {dbg->y_moe, L.y_moe, (size_t)T * H * 4},
        {dbg->y_dense, L.y_dense, (size_t)T * H * 4},
        {dbg->n_refined, L.counters, 4},
    };
    for (const Copy& cp2 : copies)
      if (cp2.dst && (err = cudaMemcpyAsync(cp2.dst, ws + cp2.off, cp2.bytes,
                                            cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return cuda_fail(m, "debug copy", err);
  }
  return DG_OK;
}

}  // namespace

dg_status_t dg_moe_forward(dg_moe_t* m, const void* h_in, void* h_out, int n_tokens,
                           float layer_scalar, dg_stream_t stream, const dg_moe_debug_t* dbg) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_tokens > m->cfg.max_tokens) return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!h_in || !h_out) return DG_ERR_INVALID_ARG;
  if (!aligned(h_in, 16) || !aligned(h_out, 16)) return DG_ERR_ALIGNMENT;
  return forward_impl(m, h_in, h_out, n_tokens, layer_scalar, stream, dbg, nullptr);
}

dg_status_t dg_moe_forward_neighbours(dg_moe_t* m, const void* x, const dg_moe_neighbours_t* nb,
                                      void* out, int n_tokens, float layer_scalar,
                                      dg_stream_t stream, const dg_moe_debug_t* dbg) {
  if (!m || !nb) return DG_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_tokens > m->cfg.max_tokens) return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!x || !out || !nb->attn_out || !nb->w_post_attn) return DG_ERR_INVALID_ARG;
  if (nb->w_next_in && !nb->next_in) return DG_ERR_INVALID_ARG;
  const void* ptrs[] = {x, out, nb->attn_out, nb->w_post_attn, nb->w_next_in, nb->next_in,
                        nb->h_mid};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return DG_ERR_ALIGNMENT;
  return forward_impl(m, x, out, n_tokens, layer_scalar, stream, dbg, nb);
}

dg_status_t dg_moe_forward_host(dg_moe_t* m, const void* h_in_host, void* h_out_host, int n_tokens,
                                float layer_scalar, dg_stream_t stream) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_tokens > m->cfg.max_tokens) return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!h_in_host || !h_out_host) return DG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)n_tokens * m->cfg.hidden * 2;
  void* din = m->ws + m->L.stage_in;
  void* dout = m->ws + m->L.stage_out;
  cudaError_t err;
  if ((err = cudaMemcpyAsync(din, h_in_host, bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(m, "copy in", err);
  dg_status_t st = dg_moe_forward(m, din, dout, n_tokens, layer_scalar, stream, nullptr);
  if (st != DG_OK) return st;
  if ((err = cudaMemcpyAsync(h_out_host, dout, bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(m, "copy out", err);
  if ((err = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(m, "synchronize", err);
  return DG_OK;
}

dg_status_t dg_moe_last_device_status(dg_moe_t* m, dg_stream_t stream, unsigned int* where,
                                      unsigned int* info) {
  if (!m) return DG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if ((err = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(m, "synchronize", err);
  DevStatus st;
  if ((err = cudaMemcpy(&st, m->ws + m->L.status, sizeof(st), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(m, "read status", err);
  if ((err = cudaMemset(m->ws + m->L.status, 0, sizeof(st))) != cudaSuccess)
    return cuda_fail(m, "clear status", err);
  if (where) *where = st.where;
  if (info) *info = st.info0;
  if (st.code == kDevTimeout) return DG_ERR_TIMEOUT;
  if (st.code == kDevBounds) return DG_ERR_DEVICE_CHECK;
  return DG_OK;
}

}  // extern "C"
