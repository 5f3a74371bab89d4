// Routing for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside an
// allocator hook or an arena that owns every byte of the device, plug-ins
// that are handed raw pointers by a host framework that forbids allocation
// on its hot path, or a routing query made while the caller is itself in the
// middle of managing memory.  For them dg_moe_route_noalloc runs the same
// two routing kernels as dg_moe_forward (logits, then selection), with the
// kernels' scratch in a fixed array that lives in this library's device
// memory for as long as the library is loaded, on every GPU that loads it.
// The caller passes only the inputs and the two outputs.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/dg_moe.h"
#include "dg_host.h"
#include "dg_kernels.h"

using namespace dg;
using namespace dg::host;

namespace {

// Fixed device scratch for the allocation-free routing entry point.
constexpr size_t kRouteScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets inside the scratch array for T tokens, hidden H, E experts.
struct RouteScratch {
  size_t r, xnorm, wnorm, logits, counts, nref, xd, total;
};
RouteScratch route_scratch_layout(size_t T, size_t H, size_t E) {
  RouteScratch s;
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off = up256(off + b);
    return o;
  };
  s.counts = take(((T + kChunkTokens - 1) / kChunkTokens) * E * 4);  // cleared per call
  s.nref = take(4);                                                  // cleared per call
  s.r = take(T * 4);
  s.xnorm = take(T * 4);
  s.wnorm = take(E * 4);
  s.logits = take(T * E * 4);
  s.xd = take(T * H * 2);
  s.total = off;
  return s;
}

// The scratch array's device address belongs to a CUDA context: a device's
// primary context, or a context the caller created, and a new context
// (after cudaDeviceReset, say) loads the library's device code again at
// another address.  So the address is looked up once per context and cached
// under the context's unique id, which the driver never reuses; the kernels'
// shared-memory limits are raised in the same set-up.
struct ScratchEntry {
  unsigned long long ctx_id;
  void* ptr;
};
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxContexts];
int g_n_scratch = 0;

PFN_cuCtxGetCurrent_v4000 g_get_ctx = nullptr;
PFN_cuCtxGetId_v12000 g_get_ctx_id = nullptr;

bool driver_fns() {
  if (g_get_ctx && g_get_ctx_id) return true;
  void* a = nullptr;
  void* b = nullptr;
  cudaDriverEntryPointQueryResult qa, qb;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) !=
          cudaSuccess ||
      qa != cudaDriverEntryPointSuccess ||
      cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
          cudaSuccess ||
      qb != cudaDriverEntryPointSuccess)
    return false;
  g_get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
  g_get_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
  return true;
}

// Device address of the scratch array in the current context (the array's
// name is only a host-side stand-in for it).
dg_status_t scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!driver_fns()) return DG_ERR_CUDA;
  CUcontext ctx = nullptr;
  void* p = nullptr;
  if (g_get_ctx(&ctx) != CUDA_SUCCESS) return DG_ERR_CUDA;
  if (!ctx) {
    // no context yet: the runtime query sets up the device's primary one
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return DG_ERR_CUDA;
    if (g_get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return DG_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_get_ctx_id(ctx, &id) != CUDA_SUCCESS) return DG_ERR_CUDA;
  for (int i = 0; i < g_n_scratch; ++i)
    if (g_scratch[i].ctx_id == id) {
      *out = g_scratch[i].ptr;
      return DG_OK;
    }
  int dev = 0, optin = 0;
  if (!p && (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p)) return DG_ERR_CUDA;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      prepare_router(optin) != cudaSuccess)
    return DG_ERR_CUDA;
  if (g_n_scratch < kMaxContexts) g_scratch[g_n_scratch++] = {id, p};
  *out = p;
  return DG_OK;
}

}  // namespace

extern "C" dg_status_t dg_moe_route_noalloc(const dg_moe_config_t* cfg,
                                            const dg_moe_weights_t* weights, const void* h_in,
                                            int n_tokens, int32_t* idx_out, float* w_out,
                                            dg_stream_t stream) {
  // the same checks as handle creation applies to the fields routing uses
  dg_status_t st = check_router_config(cfg);
  if (st != DG_OK) return st;
  if ((st = check_router_weights(*cfg, weights)) != DG_OK) return st;
  if (n_tokens < 0) return DG_ERR_INVALID_ARG;
  const int H = cfg->hidden, E = cfg->n_experts, K = cfg->top_k;
  const bool u8 = cfg->router_fmt == DG_FMT_AFFINE_U8_G64;
  if (n_tokens == 0) return DG_OK;
  if (!h_in || !idx_out || !w_out) return DG_ERR_INVALID_ARG;
  if (!aligned(h_in, 16) || !aligned(idx_out, 4) || !aligned(w_out, 4)) return DG_ERR_ALIGNMENT;
  const RouteScratch L = route_scratch_layout((size_t)n_tokens, (size_t)H, (size_t)E);
  if (L.total > kRouteScratchBytes) return DG_ERR_UNSUPPORTED;  // beyond the fixed scratch

  void* base = nullptr;
  st = scratch_address(&base);
  if (st != DG_OK) return st;
  uint8_t* sc = static_cast<uint8_t*>(base);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the histogram and the re-check counter must start at zero on every call
  if (cudaMemsetAsync(sc + L.counts, 0, L.r - L.counts, s) != cudaSuccess) return DG_ERR_CUDA;

  RouterParams rp{};
  rp.h = static_cast<const uint16_t*>(h_in);
  rp.wr = weights->router.q;
  rp.wr_scales = static_cast<const uint16_t*>(weights->router.scales);
  rp.wr_biases = static_cast<const uint16_t*>(weights->router.biases);
  rp.router_scale = static_cast<const uint16_t*>(weights->router_scale);
  rp.pes = static_cast<const uint16_t*>(weights->per_expert_scale);
  rp.w_pre_ff = static_cast<const uint16_t*>(weights->w_pre_ff);
  rp.router_bias = weights->router_bias;
  rp.T = n_tokens;
  rp.H = H;
  rp.cHd = 1.0 / sqrt((double)H);
  rp.cH = (float)rp.cHd;
  rp.E = E;
  rp.K = K;
  rp.router_u8 = u8 ? 1 : 0;
  rp.eps = cfg->rms_eps == 0.f ? 1e-6f : cfg->rms_eps;
  rp.r_out = reinterpret_cast<float*>(sc + L.r);
  rp.xnorm_out = reinterpret_cast<float*>(sc + L.xnorm);
  rp.wnorm_out = reinterpret_cast<float*>(sc + L.wnorm);
  rp.idx = idx_out;
  rp.w = w_out;
  rp.logits = reinterpret_cast<float*>(sc + L.logits);
  rp.chunk_counts = reinterpret_cast<int32_t*>(sc + L.counts);
  rp.xd = reinterpret_cast<uint16_t*>(sc + L.xd);
  rp.y_moe = nullptr;  // no accumulator to clear: routing only
  rp.n_refined = reinterpret_cast<int*>(sc + L.nref);
  if (launch_router(rp, s) != cudaSuccess) return DG_ERR_CUDA;
  if (launch_router_select(rp, 0, s) != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}
