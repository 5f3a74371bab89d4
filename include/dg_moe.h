/*
 * dg_moe.h — C ABI of the GB300 (sm_103a) routed-MoE feed-forward block.
 *
 * The block is the FFN half of a DiffusionGemma decoder layer, run over a
 * whole [T, H] activation (one or several 256-token canvases):
 *
 *   r       = 1 / sqrt(mean(h^2) + eps)                       per token
 *   z       = (h r router_scale H^-1/2) Wr^T (+ router_bias)  E logits
 *   S, w    = top-k of z (ties to the lower expert index); softmax over
 *             all E, the k selected renormalised to sum 1, times
 *             per_expert_scale
 *   xe, xd  = h r w_pre_ff2,  h r w_pre_ff                    (bf16)
 *   y_moe   = sum_k w_k down_e(gelu_tanh(gate_e xe) * up_e xe), e = S_k
 *   y_dense = down_d(gelu_tanh(gate_d xd) * up_d xd)
 *   out     = (h + rms(rms(y_dense) w_post1 + rms(y_moe) w_post2) w_post)
 *             * layer_scalar                                   (bf16)
 *
 * Where this comes from:
 *  - router order, renormalisation, per_expert_scale, tie-break, fused
 *    gate_up [gate || up], GELU-tanh, dense MLP as the always-on path,
 *    RMSNorm x / sqrt(mean(x^2) + eps) * w with eps 1e-6, layer_scalar:
 *    "diffgemma — architecture & implemented contract", Part II §1 (model
 *    constants) and §2.1 (forward-pass details);
 *  - MOEBlock.forward, MLP, the routed combine and the layer scalar:
 *    "DiffusionGemma Explained", sections "MLP and mixture-of-experts block"
 *    and "Complete DiffusionGemma model";
 *  - DecoderLayer FFN sandwich, Router (norm before the projection, two
 *    literal steps), Experts, tensor shapes and the group-64 affine quant:
 *    "DiffusionGemma port — plan & parity strategy", Reference dossier §1
 *    (weight schema & quant map) and §2 (decoder architecture), and the D1
 *    router-norm finding;
 *  - precision policy (bf16 activations, f32 router logits and MoE scratch):
 *    "diffgemma — architecture & implemented contract", Part III (precision
 *    policy).
 *
 * Conventions
 *  - All tensor pointers are device pointers unless a function says "host".
 *    Weights are borrowed: the library reads them for the handle's lifetime
 *    and never frees or writes them.  The workspace is owned by the caller;
 *    its size comes from dg_moe_workspace_size().  The handle owns only host
 *    memory (TMA descriptors, launch parameters).
 *  - Layouts are row-major; [a, b] means b is contiguous.  bf16 tensors are
 *    passed as the 16-bit patterns.  Expert weights keep the checkpoint
 *    orientation [E, out, in]: gate_up [E, 2I, H] (rows 0..I-1 gate, I..2I-1
 *    up), down [E, H, I]; dense gate/up [D, H], down [H, D]; router [E, H].
 *  - Group-wise affine tensors (DG_FMT_AFFINE_U4_G64 / _U8_G64): W = s q + b
 *    per group of 64 along the input dimension K.  q: 4-bit codes packed 8
 *    per uint32 word, element k at bits 4 (k % 8) of word k / 8, [.., K/8];
 *    or uint8 [.., K]; scales and biases bf16 [.., K/64].
 *  - NVFP4 tensors (DG_FMT_NVFP4_G16; "diffgemma — architecture & implemented
 *    contract", §8: the nvfp4 expert profile, K a multiple of 16):
 *    W = e2m1(q) * e4m3(scale) * global.  q: two e2m1 codes a byte, element
 *    k in the low nibble of byte k / 2 for even k, [.., K/2] (the same nibble
 *    order as the 4-bit affine words); scales: one fp8 e4m3 byte per 16
 *    consecutive elements along K, [.., K/16]; biases: the fp32 matrix
 *    scales, one per expert of a stack [E], or one [1] for a 2-D tensor.
 *  - Every call is asynchronous on the given stream (a cudaStream_t) unless
 *    it says otherwise; nothing synchronises the host, and routing counts
 *    stay on the device.
 *  - Errors: host-detectable problems return a status and launch nothing.
 *    Kernels never trap: a bounded wait that runs out or a failed device
 *    check records itself in a status word in the workspace, read (and
 *    cleared) by dg_moe_last_device_status().
 */
#ifndef DG_MOE_H
#define DG_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dg_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st* dg_event_t;   /* same type as cudaEvent_t */

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,  /* NULL pointer, negative or zero size, T > max_tokens */
  DG_ERR_ALIGNMENT = 2,    /* a pointer below the alignment it must have */
  DG_ERR_UNSUPPORTED = 3,  /* shape or format combination not implemented */
  DG_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed */
  DG_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out */
  DG_ERR_DEVICE_CHECK = 6, /* a device-side range check failed */
  DG_ERR_WORKSPACE = 7     /* workspace NULL, too small or misaligned */
} dg_status_t;

typedef enum {
  DG_FMT_BF16 = 0,
  DG_FMT_AFFINE_U4_G64 = 1,
  DG_FMT_AFFINE_U8_G64 = 2,
  DG_FMT_NVFP4_G16 = 3
} dg_format_t;

/* Shape and format of one layer.  Supported: hidden % 128 == 0,
 * expert_inter % 64 == 0, dense_inter % 64 == 0, 1 <= top_k <= 16,
 * top_k <= n_experts <= 256, hidden <= 8192, max_tokens >= 1.  gate_up and
 * down share expert_fmt (one format per expert stack, as a step-block
 * profile requires in "diffgemma — architecture & implemented contract",
 * Part II §8).  rms_eps 0 means the model's 1e-6. */
typedef struct {
  int hidden;        /* H */
  int n_experts;     /* E */
  int top_k;         /* K */
  int expert_inter;  /* I */
  int dense_inter;   /* D */
  int max_tokens;    /* largest T a forward may be called with */
  dg_format_t expert_fmt;
  dg_format_t dense_fmt;
  dg_format_t router_fmt;
  float rms_eps;
  unsigned int flags; /* reserved, must be 0 */
} dg_moe_config_t;

/* A weight tensor: bf16 uses q only (the bf16 array); affine formats use all
 * three (NVFP4: codes, block scales, fp32 matrix scales).  All pointers
 * 16-byte aligned (NVFP4 matrix scales: 4-byte aligned).  Supported format
 * pairs (expert, dense): bf16 + bf16, 4-bit affine + 4- or 8-bit affine,
 * NVFP4 + NVFP4. */
typedef struct {
  const void* q;
  const void* scales;
  const void* biases;
} dg_qtensor_t;

typedef struct {
  dg_qtensor_t router;     /* [E, H] */
  dg_qtensor_t gate_up;    /* [E, 2I, H] */
  dg_qtensor_t down;       /* [E, H, I] */
  dg_qtensor_t dense_gate; /* [D, H] */
  dg_qtensor_t dense_up;   /* [D, H] */
  dg_qtensor_t dense_down; /* [H, D] */
  const void* router_scale;     /* bf16 [H] */
  const void* per_expert_scale; /* bf16 [E] */
  const void* w_pre_ff;         /* bf16 [H], dense-branch input norm */
  const void* w_pre_ff2;        /* bf16 [H], expert input norm */
  const void* w_post_ff1;       /* bf16 [H], dense-branch output norm */
  const void* w_post_ff2;       /* bf16 [H], expert-sum output norm */
  const void* w_post_ff;        /* bf16 [H], norm of the branch sum */
  const float* router_bias;     /* f32 [E] added to the logits, or NULL
                                   (an extension for skewed-load workloads;
                                   the model itself has no router bias) */
} dg_moe_weights_t;

/* Optional device outputs of a forward, for stage-wise checking.  Any field
 * may be NULL.  Filled by device-to-device copies on the forward's stream. */
typedef struct {
  int32_t* idx;      /* [T, K] selected experts, ascending per token */
  float* w;          /* [T, K] routing weights, same order as idx */
  float* logits;     /* [T, E] fp32 router logits */
  int32_t* offsets;  /* [E + 1] exclusive prefix sum of per-expert counts */
  int32_t* perm;     /* [T*K] assignment ids t*K + j sorted by (expert, token) */
  uint16_t* xd;      /* bf16 [T, H] dense-branch input */
  uint16_t* xe_perm; /* bf16 [T*K, H] expert input rows in perm order */
  float* y_moe;      /* [T, H] routing-weighted expert sum */
  float* y_dense;    /* [T, H] dense-branch output */
  int32_t* n_refined;/* [1] tokens whose top-k was re-checked in fp64 */
} dg_moe_debug_t;

typedef struct dg_moe dg_moe_t;

/* Bytes of device workspace a handle with this config needs.  Host only. */
dg_status_t dg_moe_workspace_size(const dg_moe_config_t* cfg, size_t* bytes);

/* Validate cfg and weights, and build the handle: TMA descriptors for the
 * weights and for workspace buffers, launch shapes.  workspace: device
 * memory of at least dg_moe_workspace_size() bytes, 1024-byte aligned,
 * used only by this handle, or shared by handles of one shape whose
 * forwards run one after another on one stream (a layer stack).  Allocates no device memory and launches no
 * kernel; clears the workspace's status word with one blocking memset.
 * Validation errors are returned before any CUDA call.  On error *out is
 * set to NULL. */
dg_status_t dg_moe_create(const dg_moe_config_t* cfg, const dg_moe_weights_t* weights,
                          void* workspace, size_t workspace_bytes, dg_moe_t** out);

/* One forward of the block.  h_in: bf16 [n_tokens, H]; h_out: bf16
 * [n_tokens, H] (may alias h_in: h_in is last read by the final kernel,
 * element by element before it writes).  Both 16-byte aligned.
 * 0 <= n_tokens <= max_tokens (0 launches nothing).  dbg may be NULL. */
dg_status_t dg_moe_forward(dg_moe_t* m, const void* h_in, void* h_out, int n_tokens,
                           float layer_scalar, dg_stream_t stream, const dg_moe_debug_t* dbg);

/* The block fused with its neighbours in the decoder layer ("DiffusionGemma
 * port — plan & parity strategy", Reference dossier §2 DecoderLayer): the
 * attention half's last step and the next layer's first one.
 *
 *   h       = x + post_attention_layernorm(attn_out)   (bf16 planes:
 *             n = bf16(rms(attn_out) * w_post_attn), h = bf16(x + n))
 *   out     = the block on h                           (as dg_moe_forward)
 *   next_in = bf16(rms(out) * w_next_in)              (the next layer's
 *             input_layernorm, optional)
 *
 * The router's prep kernel builds h from x and attn_out and publishes it (in
 * h_mid or the workspace) for the later kernels; the combine writes next_in
 * beside out.  x is the
 * decoder layer's input (the attention residual). */
typedef struct {
  const void* attn_out;     /* bf16 [n_tokens, H]: self-attention output (o_proj), before its norm */
  const void* w_post_attn;  /* bf16 [H]: post_attention_layernorm weight of this layer */
  const void* w_next_in;    /* bf16 [H]: the next layer's input_layernorm weight, or NULL */
  void* next_in;            /* bf16 [n_tokens, H]: receives next_in; required with w_next_in */
  void* h_mid;              /* bf16 [n_tokens, H]: receives h, or NULL (kept in the workspace) */
} dg_moe_neighbours_t;

/* x: bf16 [n_tokens, H]; out: bf16 [n_tokens, H] and may alias x (x is read
 * only by the first kernel) or attn_out; next_in may alias x or attn_out but
 * not out; h_mid aliases nothing.  All 16-byte aligned.  Otherwise as
 * dg_moe_forward (dbg sees h as the block input). */
dg_status_t dg_moe_forward_neighbours(dg_moe_t* m, const void* x, const dg_moe_neighbours_t* nb,
                                      void* out, int n_tokens, float layer_scalar,
                                      dg_stream_t stream, const dg_moe_debug_t* dbg);

/* End-to-end forward with HOST buffers: copies h_in (host, bf16
 * [n_tokens, H]) into the workspace, runs dg_moe_forward, copies the result
 * to h_out (host) and synchronises the stream before returning.  Page-locked
 * host memory gives asynchronous copies; pageable memory also works. */
dg_status_t dg_moe_forward_host(dg_moe_t* m, const void* h_in_host, void* h_out_host,
                                int n_tokens, float layer_scalar, dg_stream_t stream);

/* Release the handle (host memory only).  NULL is accepted. */
dg_status_t dg_moe_destroy(dg_moe_t* m);

/* Synchronise `stream`, read the device status word, clear it.  Returns
 * DG_OK, DG_ERR_TIMEOUT or DG_ERR_DEVICE_CHECK; *where / *info (optional)
 * receive the reporting site and its detail. */
dg_status_t dg_moe_last_device_status(dg_moe_t* m, dg_stream_t stream, unsigned int* where,
                                      unsigned int* info);

/* Number of profiling slots of one forward, and their names (static
 * strings): router_logits (prep + router GEMM), router_select (one pass, or
 * the fast pass and the re-check pass from 1024 tokens), scatter_gather,
 * gemm_gate_up, gemm_down (each with a dense-only launch after it when an
 * 8-bit dense branch sits beside 4-bit experts), combine.  names may be
 * NULL; *n receives the count. */
dg_status_t dg_moe_kernel_names(const dg_moe_t* m, const char** names, int* n);

/* Profiling: when events is non-NULL, every later forward records events[i]
 * on its stream just before the launches of slot i and events[n_slots] after
 * the last one; n_events must be n_slots + 1.  The events separate the
 * launches, which then no longer overlap their neighbours' start and end.  NULL switches it off.  Events are
 * borrowed (created and destroyed by the caller). */
dg_status_t dg_moe_set_profile_events(dg_moe_t* m, dg_event_t* events, int n_events);

/* Test of the bounded device waits.  Arms the next forward of this handle
 * (one forward only): in its gate_up GEMM, block 0's epilogue waits on a
 * shared-memory barrier that nothing ever arrives on.  After 10 ms the wait
 * gives up as every wait of the kernels does when its limit runs out: it
 * records a timeout in the workspace status word (site 3, the GEMM
 * epilogue; info 0x57A11), the block stops its copy and MMA roles, waits for
 * the copies and MMAs already in flight and releases its tensor memory; the
 * other blocks finish normally.  That forward's output is not meaningful.
 * dg_moe_last_device_status then returns DG_ERR_TIMEOUT (and clears the
 * word); the handle and the CUDA context stay usable, and the next forward
 * runs normally.  Nothing faults, traps or hangs. */
dg_status_t dg_moe_arm_wait_timeout_test(dg_moe_t* m);

/* Text of the last CUDA failure seen by this handle (the call and the CUDA
 * error), "" if none.  Owned by the handle; valid until the next call. */
const char* dg_moe_last_error(const dg_moe_t* m);

/* Routing only, for callers that may not allocate device memory.  The
 * pages have no counterpart: this is a library convenience.  Some callers
 * cannot call cudaMalloc (an allocator hook or arena that owns all device
 * memory, a host framework that forbids allocation on its hot path); this
 * entry point needs no handle and no workspace.  It computes the same
 * routing as dg_moe_forward (the same selection, exact re-check included;
 * its logits come from the CUDA-core logit kernels, which need no weight
 * planes) on h_in (bf16 [n_tokens, H]) with the router
 * weights of `weights` (router, router_scale, per_expert_scale, w_pre_ff,
 * router_bias; cfg gives H, E, K, router_fmt and rms_eps) and writes
 * idx_out (int32 [n_tokens, K], ascending experts per token) and w_out
 * (f32 [n_tokens, K]), asynchronously on `stream`.
 * Scratch: a fixed 8 MiB array in the library's device memory, held on
 * every GPU that loads the library until the process exits.  It needs
 * about n_tokens * (2 H + 4 E + 8) bytes; larger calls return
 * DG_ERR_UNSUPPORTED (a 256-token canvas at H 2816 needs 1.6 MB).  The
 * array's device address belongs to the CUDA context current at the call
 * (normally the device's primary context): the first call in each context
 * looks it up and raises the routing kernels' shared-memory limits (CUDA
 * runtime queries and attributes, no allocation) and caches it under the
 * context's unique id, so a context created later (after cudaDeviceReset,
 * say) gets its own lookup.  Make that first call before any stream
 * capture.  Every call in a context shares the one array and finds the
 * previous call's contents in it (the parts that must start at zero are
 * cleared on the stream): calls that can overlap on the GPU (different
 * streams without ordering) race.  The same argument checks as
 * dg_moe_create applies to the routing fields (cfg: hidden, n_experts,
 * top_k, router_fmt, rms_eps >= 0, flags == 0; weights: router tensor and
 * its 8-bit scales and biases, router_scale, w_pre_ff, per_expert_scale,
 * router_bias alignment), then h_in 16-byte and the outputs 4-byte aligned.
 * Allocates nothing. */
dg_status_t dg_moe_route_noalloc(const dg_moe_config_t* cfg, const dg_moe_weights_t* weights,
                                 const void* h_in, int n_tokens, int32_t* idx_out, float* w_out,
                                 dg_stream_t stream);

/* ------------------------------------------------------------------------
 * Self-conditioning MLP (before layer 0 of a decode step):
 *
 *   x   = rms(signal) * pre_norm                        (bf16)
 *   s   = down(gelu_tanh(gate x) * up x)                dense-FFN shapes
 *   out = (embeds + s) / sqrt(mean((embeds + s)^2) + eps)   (bf16, no weight)
 *
 * "DiffusionGemma port — plan & parity strategy", Reference dossier §3
 * (SelfConditioning: pre_norm, gate/up/down, post_norm = RMSNormNoScale);
 * "diffgemma — architecture & implemented contract", Part II §2.1 (SC
 * injection) and Part I §4 (SC MLP, q8/4-bit gate/up/down);
 * "DiffusionGemma Explained", MLP (conditioning_mlp) and the note that the
 * MLP maps 0 to 0 on the first decode step.  The signal is the soft
 * embedding of the previous step (probabilities times the embedding table
 * times sqrt(hidden)), computed by the caller.
 * Runs on the same grouped GEMM kernels as the dense branch of the block.
 * ------------------------------------------------------------------------ */
typedef struct dg_sc_mlp dg_sc_mlp_t;

typedef struct {
  int hidden;         /* H, multiple of 128 */
  int inter;          /* gate/up rows, multiple of 64 */
  int max_tokens;     /* largest n_tokens of a forward */
  dg_format_t fmt;    /* gate, up, down: DG_FMT_BF16, DG_FMT_AFFINE_U4_G64 or
                         DG_FMT_AFFINE_U8_G64 (q8); quantised: H and inter <= 2944 */
  float rms_eps;      /* 0 means 1e-6 */
  unsigned flags;     /* must be 0 */
} dg_sc_mlp_config_t;

typedef struct {
  dg_qtensor_t gate;     /* [inter, H] */
  dg_qtensor_t up;       /* [inter, H] */
  dg_qtensor_t down;     /* [H, inter] */
  const void* pre_norm;  /* bf16 [H] */
} dg_sc_mlp_weights_t;

/* Bytes of workspace a handle of this configuration needs. */
dg_status_t dg_sc_mlp_workspace_size(const dg_sc_mlp_config_t* cfg, size_t* bytes);

/* Create a handle: validates the configuration and the weights (device
 * pointers, 16-byte aligned; borrowed), lays out the caller's workspace
 * (1024-byte aligned, at least dg_sc_mlp_workspace_size bytes) and builds
 * the TMA descriptors.  Allocates no device memory. */
dg_status_t dg_sc_mlp_create(const dg_sc_mlp_config_t* cfg, const dg_sc_mlp_weights_t* weights,
                             void* workspace, size_t workspace_bytes, dg_sc_mlp_t** out);

/* out = the self-conditioning MLP of (embeds, signal), all bf16 [n_tokens, H]
 * device tensors, 16-byte aligned; out may alias embeds or signal.  n_tokens
 * in [0, max_tokens]; asynchronous on `stream`.  Device-side failures are
 * read with dg_sc_mlp_last_device_status. */
dg_status_t dg_sc_mlp_forward(dg_sc_mlp_t* m, const void* embeds, const void* signal, void* out,
                              int n_tokens, dg_stream_t stream);

/* Synchronise `stream`, read and clear the handle's device status word
 * (DG_OK, DG_ERR_TIMEOUT or DG_ERR_DEVICE_CHECK). */
dg_status_t dg_sc_mlp_last_device_status(dg_sc_mlp_t* m, dg_stream_t stream);

/* Number of kernels one forward launches and their names, as
 * dg_moe_kernel_names. */
dg_status_t dg_sc_mlp_kernel_names(const dg_sc_mlp_t* m, const char** names, int* n);

/* Profiling events around each kernel of later forwards, as
 * dg_moe_set_profile_events (n_events = number of kernels + 1, NULL off). */
dg_status_t dg_sc_mlp_set_profile_events(dg_sc_mlp_t* m, dg_event_t* events, int n_events);

/* Free the handle (NULL is accepted). */
dg_status_t dg_sc_mlp_destroy(dg_sc_mlp_t* m);

/* Static string for a status code. */
const char* dg_moe_status_string(dg_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* DG_MOE_H */
