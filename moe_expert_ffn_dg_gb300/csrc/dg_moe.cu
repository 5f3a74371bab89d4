// C-ABI implementation of the MoE FFN block: argument validation, workspace
// layout, TMA descriptors and the launch sequence of one forward.
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "../../include/dg_moe.h"
#include "dg_kernels.h"

using namespace dg;

namespace {

constexpr int kNumKernels = 7;
const char* const kKernelNames[kNumKernels] = {
    "router", "route_count", "route_scatter", "gather_xe",
    "gemm_gate_up", "gemm_down", "combine"};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t status, counters, r, idx, w, chunk_counts, offsets, perm, tok_perm, w_perm;
  size_t xd, xe_perm, act, act_d, y_moe, y_dense, tiles_gu, tiles_dn, stage_in, stage_out;
  size_t total;
  int max_tiles_gu, max_tiles_dn;
};

// Smallest token-tile height the kernels use; it bounds the tile counts.
constexpr int kMinBN = 128;

Layout make_layout(const dg_moe_config_t& c) {
  Layout L;
  const size_t T = (size_t)c.max_tokens, H = c.hidden, E = c.n_experts, K = c.top_k;
  const size_t I = c.expert_inter, D = c.dense_inter, TK = T * K;
  const size_t nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  const size_t exp_tok_tiles = E + (TK + kMinBN - 1) / kMinBN;
  const size_t dense_tok_tiles = (T + kMinBN - 1) / kMinBN;
  L.max_tiles_gu = (int)(exp_tok_tiles * (I / 64) + dense_tok_tiles * (D / 64));
  L.max_tiles_dn = (int)(exp_tok_tiles * (H / 128) + dense_tok_tiles * (H / 128));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  L.status = take(sizeof(DevStatus));
  L.counters = take(16 * sizeof(int));  // [0] n_refined, [1..2] tile counts
  L.r = take(T * 4);
  L.idx = take(TK * 4);
  L.w = take(TK * 4);
  L.chunk_counts = take(nchunks * E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(TK * 4);
  L.tok_perm = take(TK * 4);
  L.w_perm = take(TK * 4);
  L.xd = take(T * H * 2);
  L.xe_perm = take(TK * H * 2);
  L.act = take(TK * I * 2);
  L.act_d = take(T * D * 2);
  L.y_moe = take(T * H * 4);
  L.y_dense = take(T * H * 4);
  L.tiles_gu = take((size_t)L.max_tiles_gu * 16);
  L.tiles_dn = take((size_t)L.max_tiles_dn * 16);
  L.stage_in = take(T * H * 2);
  L.stage_out = take(T * H * 2);
  L.total = off;
  return L;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

dg_status_t check_config(const dg_moe_config_t* c) {
  if (!c) return DG_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->expert_inter <= 0 ||
      c->dense_inter <= 0 || c->max_tokens <= 0 || c->rms_eps < 0.f || c->flags != 0)
    return DG_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return DG_ERR_INVALID_ARG;
  if (c->hidden % 128 || c->expert_inter % 64 || c->dense_inter % 64) return DG_ERR_UNSUPPORTED;
  if (c->hidden > 8192 || c->n_experts > 256 || c->top_k > 16) return DG_ERR_UNSUPPORTED;
  if (c->max_tokens > (1 << 20)) return DG_ERR_UNSUPPORTED;
  if (c->expert_fmt != DG_FMT_BF16 || c->dense_fmt != DG_FMT_BF16) return DG_ERR_UNSUPPORTED;
  if (c->router_fmt != DG_FMT_BF16 && c->router_fmt != DG_FMT_AFFINE_U8_G64)
    return DG_ERR_UNSUPPORTED;
  return DG_OK;
}

dg_status_t check_qtensor(const dg_qtensor_t& t, dg_format_t fmt) {
  if (!t.q) return DG_ERR_INVALID_ARG;
  if (!aligned(t.q, 16)) return DG_ERR_ALIGNMENT;
  if (fmt != DG_FMT_BF16) {
    if (!t.scales || !t.biases) return DG_ERR_INVALID_ARG;
    if (!aligned(t.scales, 2) || !aligned(t.biases, 2)) return DG_ERR_ALIGNMENT;
  }
  return DG_OK;
}

dg_status_t check_weights(const dg_moe_config_t& c, const dg_moe_weights_t* w) {
  if (!w) return DG_ERR_INVALID_ARG;
  dg_status_t s;
  if ((s = check_qtensor(w->router, c.router_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->gate_up, c.expert_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->down, c.expert_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_gate, c.dense_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_up, c.dense_fmt)) != DG_OK) return s;
  if ((s = check_qtensor(w->dense_down, c.dense_fmt)) != DG_OK) return s;
  const void* vecs[] = {w->router_scale, w->w_pre_ff, w->w_pre_ff2, w->w_post_ff1,
                        w->w_post_ff2, w->w_post_ff};
  for (const void* v : vecs) {
    if (!v) return DG_ERR_INVALID_ARG;
    if (!aligned(v, 16)) return DG_ERR_ALIGNMENT;
  }
  if (!w->per_expert_scale) return DG_ERR_INVALID_ARG;
  if (!aligned(w->per_expert_scale, 2)) return DG_ERR_ALIGNMENT;
  if (w->router_bias && !aligned(w->router_bias, 4)) return DG_ERR_ALIGNMENT;
  return DG_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// Row-major bf16 matrix [rows, cols] read in boxes of 16 rows x 64 columns
// with the 128-byte swizzle the MMA descriptors expect.
bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
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
  dg_event_t* prof;
  int n_prof;
};

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
  if (cudaGetDevice(&m->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  const dg_moe_config_t& c = m->cfg;
  const uint64_t H = c.hidden, E = c.n_experts, I = c.expert_inter, D = c.dense_inter;
  const uint64_t T = c.max_tokens, TK = T * c.top_k;
  uint8_t* ws = m->ws;
  bool ok = true;
  // gate_up: weights [E*2I, H], dense gate/up [D, H]; rows xe_perm / xd
  ok = ok && encode_bf16_rows(&m->gu.wa_exp, weights->gate_up.q, E * 2 * I, H);
  ok = ok && encode_bf16_rows(&m->gu.wa_d0, weights->dense_gate.q, D, H);
  ok = ok && encode_bf16_rows(&m->gu.wa_d1, weights->dense_up.q, D, H);
  ok = ok && encode_bf16_rows(&m->gu.xb_exp, ws + L.xe_perm, TK, H);
  ok = ok && encode_bf16_rows(&m->gu.xb_d, ws + L.xd, T, H);
  // down: weights [E*H, I], dense down [H, D]; rows act / act_d
  ok = ok && encode_bf16_rows(&m->dn.wa_exp, weights->down.q, E * H, I);
  ok = ok && encode_bf16_rows(&m->dn.wa_d0, weights->dense_down.q, H, D);
  ok = ok && encode_bf16_rows(&m->dn.wa_d1, weights->dense_down.q, H, D);
  ok = ok && encode_bf16_rows(&m->dn.xb_exp, ws + L.act, TK, I);
  ok = ok && encode_bf16_rows(&m->dn.xb_d, ws + L.act_d, T, D);
  if (!ok) {
    delete m;
    return DG_ERR_CUDA;
  }
  // the device status word starts clear
  if (cudaMemset(ws + L.status, 0, sizeof(DevStatus)) != cudaSuccess) {
    delete m;
    return DG_ERR_CUDA;
  }
  for (GemmParams* g : {&m->gu, &m->dn}) {
    g->ntiles = nullptr;
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
  m->gu.tiles = reinterpret_cast<const int4*>(ws + L.tiles_gu);
  m->gu.ntiles = reinterpret_cast<const int*>(ws + L.counters) + 1;
  m->gu.kb_exp = (int)(H / 64);
  m->gu.kb_dense = (int)(H / 64);
  m->dn.tiles = reinterpret_cast<const int4*>(ws + L.tiles_dn);
  m->dn.ntiles = reinterpret_cast<const int*>(ws + L.counters) + 2;
  m->dn.kb_exp = (int)(I / 64);
  m->dn.kb_dense = (int)(D / 64);
  *out = m;
  return DG_OK;
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

dg_status_t dg_moe_set_profile_events(dg_moe_t* m, dg_event_t* events, int n_events) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (events && n_events != kNumKernels + 1) return DG_ERR_INVALID_ARG;
  m->prof = events;
  m->n_prof = events ? n_events : 0;
  return DG_OK;
}

dg_status_t dg_moe_forward(dg_moe_t* m, const void* h_in, void* h_out, int n_tokens,
                           float layer_scalar, dg_stream_t stream, const dg_moe_debug_t* dbg) {
  if (!m) return DG_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_tokens > m->cfg.max_tokens) return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!h_in || !h_out) return DG_ERR_INVALID_ARG;
  if (!aligned(h_in, 16) || !aligned(h_out, 16)) return DG_ERR_ALIGNMENT;
  const dg_moe_config_t& c = m->cfg;
  const Layout& L = m->L;
  uint8_t* ws = m->ws;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = n_tokens, H = c.hidden, E = c.n_experts, K = c.top_k;
  const int I = c.expert_inter, D = c.dense_inter, TK = T * K;
  const int bn = T <= 1024 ? 128 : 256;
  int* counters = reinterpret_cast<int*>(ws + L.counters);
  DevStatus* status = reinterpret_cast<DevStatus*>(ws + L.status);
  cudaError_t err = cudaSuccess;
  auto mark = [&](int i) {
    if (m->prof && err == cudaSuccess) err = cudaEventRecord(reinterpret_cast<cudaEvent_t>(m->prof[i]), s);
  };
  if (cudaMemsetAsync(counters, 0, 16 * sizeof(int), s) != cudaSuccess) return DG_ERR_CUDA;

  RouterParams rp;
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
  rp.E = E;
  rp.K = K;
  rp.router_u8 = c.router_fmt == DG_FMT_AFFINE_U8_G64;
  rp.eps = c.rms_eps;
  rp.r_out = reinterpret_cast<float*>(ws + L.r);
  rp.idx = reinterpret_cast<int32_t*>(ws + L.idx);
  rp.w = reinterpret_cast<float*>(ws + L.w);
  rp.logits = dbg ? dbg->logits : nullptr;
  rp.xd = reinterpret_cast<uint16_t*>(ws + L.xd);
  rp.y_moe = reinterpret_cast<float*>(ws + L.y_moe);
  rp.n_refined = counters;
  mark(0);
  if (err == cudaSuccess) err = launch_router(rp, s);
  mark(1);
  if (err == cudaSuccess)
    err = launch_route_count(rp.idx, T, K, E, reinterpret_cast<int32_t*>(ws + L.chunk_counts), s);

  ScatterParams sp;
  sp.idx = rp.idx;
  sp.w = rp.w;
  sp.chunk_counts = reinterpret_cast<const int32_t*>(ws + L.chunk_counts);
  sp.T = T;
  sp.K = K;
  sp.E = E;
  sp.H = H;
  sp.I = I;
  sp.D = D;
  sp.bn_exp = bn;
  sp.bn_dense = bn;
  sp.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  sp.perm = reinterpret_cast<int32_t*>(ws + L.perm);
  sp.tok_perm = reinterpret_cast<int32_t*>(ws + L.tok_perm);
  sp.w_perm = reinterpret_cast<float*>(ws + L.w_perm);
  sp.tiles_gu = reinterpret_cast<int4*>(ws + L.tiles_gu);
  sp.tiles_dn = reinterpret_cast<int4*>(ws + L.tiles_dn);
  sp.ntiles = counters + 1;
  sp.status = status;
  mark(2);
  if (err == cudaSuccess) err = launch_route_scatter(sp, s);

  GatherParams gp;
  gp.h = rp.h;
  gp.r = rp.r_out;
  gp.tok_perm = sp.tok_perm;
  gp.w_pre_ff2 = static_cast<const uint16_t*>(m->w.w_pre_ff2);
  gp.TK = TK;
  gp.H = H;
  gp.xe_perm = reinterpret_cast<uint16_t*>(ws + L.xe_perm);
  mark(3);
  if (err == cudaSuccess) err = launch_gather(gp, m->num_sms, s);
  mark(4);
  if (err == cudaSuccess) err = launch_gemm(0, bn, m->gu, m->num_sms, s);
  mark(5);
  if (err == cudaSuccess) err = launch_gemm(1, bn, m->dn, m->num_sms, s);

  CombineParams cp;
  cp.y_dense = reinterpret_cast<const float*>(ws + L.y_dense);
  cp.y_moe = reinterpret_cast<const float*>(ws + L.y_moe);
  cp.h = rp.h;
  cp.w_post1 = static_cast<const uint16_t*>(m->w.w_post_ff1);
  cp.w_post2 = static_cast<const uint16_t*>(m->w.w_post_ff2);
  cp.w_post = static_cast<const uint16_t*>(m->w.w_post_ff);
  cp.T = T;
  cp.H = H;
  cp.eps = c.rms_eps;
  cp.layer_scalar = layer_scalar;
  cp.out = static_cast<uint16_t*>(h_out);
  mark(6);
  if (err == cudaSuccess) err = launch_combine(cp, s);
  mark(7);
  if (err != cudaSuccess) return DG_ERR_CUDA;

  if (dbg) {
    struct Copy { void* dst; size_t off; size_t bytes; };
    const Copy copies[] = {
        {dbg->idx, L.idx, (size_t)TK * 4},
        {dbg->w, L.w, (size_t)TK * 4},
        {dbg->offsets, L.offsets, (size_t)(E + 1) * 4},
        {dbg->perm, L.perm, (size_t)TK * 4},
        {dbg->xd, L.xd, (size_t)T * H * 2},
        {dbg->xe_perm, L.xe_perm, (size_t)TK * H * 2},
        {dbg->y_moe, L.y_moe, (size_t)T * H * 4},
        {dbg->y_dense, L.y_dense, (size_t)T * H * 4},
        {dbg->n_refined, L.counters, 4},
    };
    for (const Copy& cp2 : copies)
      if (cp2.dst && cudaMemcpyAsync(cp2.dst, ws + cp2.off, cp2.bytes, cudaMemcpyDeviceToDevice, s) !=
                         cudaSuccess)
        return DG_ERR_CUDA;
  }
  return DG_OK;
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
  if (cudaMemcpyAsync(din, h_in_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DG_ERR_CUDA;
  dg_status_t st = dg_moe_forward(m, din, dout, n_tokens, layer_scalar, stream, nullptr);
  if (st != DG_OK) return st;
  if (cudaMemcpyAsync(h_out_host, dout, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}

dg_status_t dg_moe_last_device_status(dg_moe_t* m, dg_stream_t stream, unsigned int* where,
                                      unsigned int* info) {
  if (!m) return DG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
  DevStatus st;
  if (cudaMemcpy(&st, m->ws + m->L.status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaMemset(m->ws + m->L.status, 0, sizeof(st)) != cudaSuccess) return DG_ERR_CUDA;
  if (where) *where = st.where;
  if (info) *info = st.info0;
  if (st.code == kDevTimeout) return DG_ERR_TIMEOUT;
  if (st.code == kDevBounds) return DG_ERR_DEVICE_CHECK;
  return DG_OK;
}

}  // extern "C"
