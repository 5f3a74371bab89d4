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
#include <mutex>

#include "../../include/dg_moe.h"
#include "dg_kernels.h"

using namespace dg;

namespace {

// Fixed device scratch for the allocation-free routing entry point.
constexpr size_t kRouteScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

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

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Device address of the scratch array on the current device, looked up once
// per device (the array's name is only a host-side stand-in).
dg_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return DG_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DG_OK;
}

}  // namespace

extern "C" dg_status_t dg_moe_route_noalloc(const dg_moe_config_t* cfg,
                                            const dg_moe_weights_t* weights, const void* h_in,
                                            int n_tokens, int32_t* idx_out, float* w_out,
                                            dg_stream_t stream) {
  if (!cfg || !weights) return DG_ERR_INVALID_ARG;
  const int H = cfg->hidden, E = cfg->n_experts, K = cfg->top_k;
  if (H <= 0 || E <= 0 || K <= 0 || K > E || n_tokens < 0) return DG_ERR_INVALID_ARG;
  if (H % 128 || H > 8192 || E > 256 || K > 16) return DG_ERR_UNSUPPORTED;
  if (cfg->router_fmt != DG_FMT_BF16 && cfg->router_fmt != DG_FMT_AFFINE_U8_G64)
    return DG_ERR_UNSUPPORTED;
  const bool u8 = cfg->router_fmt == DG_FMT_AFFINE_U8_G64;
  if (!weights->router.q || !weights->router_scale || !weights->per_expert_scale ||
      !weights->w_pre_ff || (u8 && (!weights->router.scales || !weights->router.biases)))
    return DG_ERR_INVALID_ARG;
  if (n_tokens == 0) return DG_OK;
  if (!h_in || !idx_out || !w_out) return DG_ERR_INVALID_ARG;
  if (!aligned_to(weights->router.q, 16) || !aligned_to(weights->router_scale, 16) ||
      !aligned_to(weights->w_pre_ff, 16) || !aligned_to(h_in, 16) || !aligned_to(idx_out, 4) ||
      !aligned_to(w_out, 4))
    return DG_ERR_ALIGNMENT;
  const RouteScratch L = route_scratch_layout((size_t)n_tokens, (size_t)H, (size_t)E);
  if (L.total > kRouteScratchBytes) return DG_ERR_UNSUPPORTED;  // beyond the fixed scratch

  void* base = nullptr;
  dg_status_t st = scratch_address(&base);
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
  if (launch_router_select(rp, s) != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}
