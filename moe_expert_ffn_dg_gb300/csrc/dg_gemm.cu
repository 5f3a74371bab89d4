// Grouped tcgen05 GEMMs of the MoE FFN block (sm_103a).
//
// One persistent kernel per projection, one CTA per SM, warp-specialised:
//   warp 0  TMA producer: weight tile (128 rows x 64 K, bf16, 128B swizzle)
//           and token tile (up to BN rows x 64 K) into a STAGES-deep ring;
//   warp 1  allocates TMEM (two BN-column fp32 accumulators) and issues the
//           tcgen05.mma (M = 128 weight rows, N = token rows rounded to 16,
//           K = 16 per instruction) from a single thread;
//   warps 2-5 epilogue: TMEM -> registers, fused per-mode output.
// Weights are the M side ("swap AB"): a canvas gives ~16 tokens per expert,
// so the 128-row side of the MMA is filled by output features and the token
// count only sets N.
//
// mode 0 (gate_up): an A tile interleaves 16 gate rows and the 16 matching
// up rows four times, so TMEM lanes 32q..32q+15 hold gate and 32q+16..32q+31
// up of the same 16 features; the epilogue pairs them with one shuffle and
// writes act = bf16(gelu_tanh(gate) * up) ("diffgemma — architecture &
// implemented contract", Part II §2.1: fused [gate || up], GELU-tanh;
// "DiffusionGemma Explained", MLP).
// mode 1 (down): 128 output channels per tile; experts add w * y into the f32
// per-token accumulator (the routing-weighted combine, "DiffusionGemma
// Explained", MOEBlock.forward), or, from 1024 tokens, store it as the
// assignment's f32 row for the combine to sum; the dense branch stores its f32
// output.
//
// Tiles {group, feature tile, first row, rows} (group == E is the dense
// branch) are decoded from the expert offsets in each CTA and dealt
// round-robin to the CTAs.
// Every wait is bounded; a wait that runs out records itself in the status
// word and the CTA winds down (its TMA copies and MMAs are drained before
// TMEM is released).
#include "dg_gemm_common.cuh"

namespace dg {
namespace {

using namespace gemm;

// Warps 0 producer, 1 MMA issuer, 2-5 epilogue; the router mode adds warp 6,
// which waits on the stage barriers for the issuer (see the waiter below).
constexpr int kThreads = 192;
template <int MODE>
constexpr int threads_of() { return MODE == 2 ? kThreads + 32 : kThreads; }
constexpr int kATileBytes = 128 * 128;  // 128 rows x 64 bf16

// CTAs an SM and the stage ring of each: the projections run kProjCtasPerSm
// CTAs an SM, each with its share of the 192 KB ring (measured: one CTA
// streams weights at only ~45 GB/s, and two an SM lift one canvas's gate_up
// from 180 to 164 us); the router GEMM and 256-token tiles keep one CTA an SM
// (their accumulators fill the TMEM) and the whole ring.
constexpr int kRingBytes = 192 * 1024;
template <int MODE, int BN>
constexpr int ctas_of() { return (MODE == 2 || BN == 256) ? 1 : kProjCtasPerSm; }
template <int MODE, int BN>
constexpr int ring_of() { return kRingBytes / ctas_of<MODE, BN>(); }

template <int BN, int RING>
struct Cfg {
  static constexpr int kBTileBytes = BN * 128;
  static constexpr int kStages = RING / (kATileBytes + kBTileBytes);
  static constexpr int kTmemCols = 2 * BN;
  static constexpr size_t kSmem =
      1024 + (size_t)kStages * (kATileBytes + kBTileBytes) + 256 + kTileTableBytes;
};

template <int MODE, int BN>
__global__ void __launch_bounds__(threads_of<MODE>(), ctas_of<MODE, BN>())
    k_grouped_gemm(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN, ring_of<MODE, BN>()>;
  constexpr int S = C::kStages;
  // router logits: one set of kRouterAcc accumulators (the whole TMEM);
  // the projections: two accumulators, so an epilogue overlaps the next tile
  constexpr uint32_t kTmemCols = MODE == 2 ? 512u : (uint32_t)C::kTmemCols;
  static_assert(MODE != 2 || BN * kRouterAcc == 512, "router accumulators fill TMEM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)S * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)S * C::kBTileBytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* stall = drain + 1;  // bounded-wait test: never arrived on
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(stall + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_start = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + 256);  // [E + 1]
  int* s_off = s_start + kMaxGroups + 2;                                            // [E + 1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.wa_exp);
    tma_prefetch_map(&p.wa_d0);
    if (MODE == 0) {
      tma_prefetch_map(&p.wa_d1);
      tma_prefetch_map(&p.wa_d5);
    }
    tma_prefetch_map(&p.xb_exp64);
    tma_prefetch_map(&p.xb_exp16);
    tma_prefetch_map(&p.xb_d64);
    tma_prefetch_map(&p.xb_d16);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  // everything above touches only this CTA's resources; from here on the
  // kernel reads what earlier kernels wrote
  pdl_wait();
  if (warp >= 2 && warp < 6) build_tile_table(p, threadIdx.x - 64, s_start, s_off);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int nd = (p.T + p.bn - 1) / p.bn * p.mt_dense;
  const int ntiles = nd + s_start[p.E];
  // deal the tiles to only as many CTAs as keep the number of rounds, so that
  // the last round is full (no lone CTAs streaming one more tile at the end)
  const int rounds = (ntiles + (int)gridDim.x - 1) / (int)gridDim.x;
  const int nct = rounds > 0 ? (ntiles + rounds - 1) / rounds : 1;
  const int first = (int)blockIdx.x < nct ? (int)blockIdx.x : ntiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // weights are read once per forward (evict first) and token rows reused
      // by the feature tiles (evict last); the router's two weight planes are
      // read by every token tile and its token rows once: the other way round
      const uint64_t pol_w = MODE == 2 ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_x = MODE == 2 ? l2_policy_evict_first() : l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = first; tile < ntiles && ok; tile += nct) {
        const int4 td = decode_tile(p, tile, nd, s_start, s_off);
        const bool dense = td.x == p.E;
        const int kbn = dense ? p.kb_dense : p.kb_exp;
        // router: this tile's K range (split-K) and expert tile
        const int2 kr = MODE == 2 ? router_krange(p, td.y, kbn) : make_int2(0, kbn);
        // a full token tile of 128 or 256 rows in one box (projections), else
        // 64-row then 16-row boxes
        const bool whole = MODE != 2 && BN >= 128 && td.w == BN;
        const int nb64 = whole ? 0 : td.w / 64;
        const int nb16 = whole ? 0 : (td.w - 64 * nb64 + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes =
            kATileBytes + (whole ? BN * 128u : nb64 * 64 * 128 + nb16 * kBoxBytes);
        const CUtensorMap* mbf = full_stage_map<BN>(p, dense);
        const CUtensorMap* mb64 = dense ? &p.xb_d64 : &p.xb_exp64;
        const CUtensorMap* mb16 = dense ? &p.xb_d16 : &p.xb_exp16;
        for (int kb = kr.x; kb < kr.y; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            report(p.status, kDevTimeout, kSiteGemmProducer, (unsigned)tile, (unsigned)kb);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t* a_dst = sA + (size_t)stage * kATileBytes;
          uint8_t* b_dst = sB + (size_t)stage * C::kBTileBytes;
          const int x = kb * 64;
          if (MODE == 0) {
            if (!dense) {
              // rows e*2I + half*I + 16*(4m + c) + r, box (64, 16, 2, 4, 1)
              tma_load_5d(&p.wa_exp, &full[stage], a_dst, x, 0, 0, 4 * td.y, td.x, pol_w);
            } else if (p.dense_5d) {
              tma_load_4d(&p.wa_d5, &full[stage], a_dst, x, 0, 0, 4 * td.y, pol_w);
            } else {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int yg = td.y * 64 + 16 * c;
                tma_load_2d_hint(&p.wa_d0, &full[stage], a_dst + (2 * c) * kBoxBytes, x, yg, pol_w);
                tma_load_2d_hint(&p.wa_d1, &full[stage], a_dst + (2 * c + 1) * kBoxBytes, x, yg,
                                 pol_w);
              }
            }
          } else if (MODE == 1) {
            const CUtensorMap* ma = dense ? &p.wa_d0 : &p.wa_exp;
            tma_load_2d_hint(ma, &full[stage], a_dst, x, (dense ? 0 : td.x * p.H) + td.y * 128,
                             pol_w);
          } else {
            // router: 128 rows of the [E, 2H] planes (hi | lo)
            tma_load_2d_hint(&p.wa_d0, &full[stage], a_dst, x, router_etile(p, td.y) * 128, pol_w);
          }
          // router: the token rows [h | h] along K against the planes (hi | lo)
          const int xb = MODE == 2 ? x % p.H : x;
          if (whole) tma_load_2d_hint(mbf, &full[stage], b_dst, xb, td.z, pol_x);
          for (int j = 0; j < nb64; ++j)
            tma_load_2d_hint(mb64, &full[stage], b_dst + j * 64 * 128, xb, td.z + 64 * j, pol_x);
          for (int j = 0; j < nb16; ++j)
            tma_load_2d_hint(mb16, &full[stage], b_dst + (64 * nb64 + kBoxRows * j) * 128, xb,
                             td.z + 64 * nb64 + kBoxRows * j, pol_x);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (int s = 0; s < S; ++s)
        if ((armed >> s) & 1u)
          if (!wait_no_abort(&full[s], (armed_par >> s) & 1u))
            report(p.status, kDevTimeout, kSiteGemmDrain, (unsigned)s, 0u);
    }
  } else if (MODE == 2 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (router) The router GEMM is bound by MMA issue, not by memory: its
    // issuer learns that a stage is ready only through handoff() with the
    // waiter warp, as a shared-memory poll by a thread with MMAs in flight
    // waits for them to complete.
    int stage = 0;
    bool stop = false, issued = false;
    for (int tile = first; tile < ntiles && !stop; tile += nct) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const int nb = (td.w + kBoxRows - 1) / kBoxRows;
      const int2 kr = router_krange(p, td.y, p.kb_dense);
      const uint32_t idesc = idesc_bf16_f32(128, nb * kBoxRows);
      for (int kb = kr.x; kb < kr.y; ++kb) {
        if (handoff(false)) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sA + (size_t)stage * kATileBytes);
          const uint32_t b0 = smem_u32(sB + (size_t)stage * C::kBTileBytes);
          const uint32_t dk = tmem_base + (uint32_t)(((kb - kr.x) % kRouterAcc) * BN);
          const bool fresh = kb - kr.x < kRouterAcc;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(dk, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k), idesc,
                      (!fresh || k != 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (kb == kr.y - 1) umma_commit(&acc_full[0]);
        }
        issued = true;
        if (++stage == S) stage = 0;
        __syncwarp();
      }
    }
    if (lane == 0 && issued) {
      umma_commit(drain);
      if (!wait_no_abort(drain, 0u)) report(p.status, kDevTimeout, kSiteGemmDrain, 99u, 0u);
    }
  } else if (MODE == 2 && warp == 6) {
    // ------------------------------------------------------------ waiter
    // (router) the bounded waits of the issuer: the accumulators free before
    // a tile's first stage, each stage's operands landed; "stop" (a wait
    // that ran out) travels in the reduced predicate, so both warps leave
    // on the same round
    int stage = 0, local = 0;
    uint32_t phase = 0;
    bool stop = false;
    for (int tile = first; tile < ntiles && !stop; tile += nct, ++local) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const int2 kr = router_krange(p, td.y, p.kb_dense);
      for (int kb = kr.x; kb < kr.y; ++kb) {
        bool ok = true;
        unsigned what = 0;
        if (kb == kr.x && !mbar_wait(&acc_empty[0], ((uint32_t)local & 1u) ^ 1u, abort_flag)) {
          ok = false;
          what = 0xffffffffu;
        }
        if (ok && !mbar_wait(&full[stage], phase, abort_flag)) {
          ok = false;
          what = (unsigned)kb;
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
        if (!ok) {
          if (lane == 0) report(p.status, kDevTimeout, kSiteGemmMma, (unsigned)tile, what);
          *abort_flag = 1;
        }
        if (handoff(!ok)) {
          stop = true;
          break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true, issued = false;
      for (int tile = first; tile < ntiles && ok; tile += nct, ++local) {
        const int4 td = decode_tile(p, tile, nd, s_start, s_off);
        const bool dense = td.x == p.E;
        const int nb = (td.w + kBoxRows - 1) / kBoxRows;
        const int kbn = dense ? p.kb_dense : p.kb_exp;
        // router: this tile's K range (split-K) and expert tile
        const int2 kr = MODE == 2 ? router_krange(p, td.y, kbn) : make_int2(0, kbn);
        const int acc = MODE == 2 ? 0 : (local & 1);
        const uint32_t use = MODE == 2 ? (uint32_t)local : (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[acc], (use & 1u) ^ 1u, abort_flag)) {
          report(p.status, kDevTimeout, kSiteGemmMma, (unsigned)tile, 0xffffffffu);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const uint32_t idesc = idesc_bf16_f32(128, nb * kBoxRows);
        for (int kb = kr.x; kb < kr.y; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            report(p.status, kDevTimeout, kSiteGemmMma, (unsigned)tile, (unsigned)kb);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + (size_t)stage * kATileBytes);
          const uint32_t b0 = smem_u32(sB + (size_t)stage * C::kBTileBytes);
          // router: K block kb goes to accumulator kb mod kRouterAcc
          const uint32_t dk =
              MODE == 2 ? d_tmem + (uint32_t)(((kb - kr.x) % kRouterAcc) * BN) : d_tmem;
          const bool fresh = MODE == 2 ? kb - kr.x < kRouterAcc : kb == 0;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(dk, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k), idesc,
                      (!fresh || k != 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          issued = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&acc_full[acc]);
      }
      // every MMA issued here must have completed before TMEM is released
      if (issued) {
        umma_commit(drain);
        if (!wait_no_abort(drain, 0u)) report(p.status, kDevTimeout, kSiteGemmDrain, 99u, 0u);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int local = 0;
    bool stalled = false;
    if (p.test_stall && blockIdx.x == 0 && !mbar_wait_for(stall, 0u, abort_flag, kTestStallNs)) {
      if (lane == 0) report(p.status, kDevTimeout, kSiteGemmEpilogue, kTestStallInfo, 0u);
      *abort_flag = 1;
      stalled = true;
    }
    for (int tile = first; tile < ntiles && !stalled; tile += nct, ++local) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const int nb = (td.w + kBoxRows - 1) / kBoxRows;
      const int acc = MODE == 2 ? 0 : (local & 1);
      const uint32_t use = MODE == 2 ? (uint32_t)local : (uint32_t)(local >> 1);
      const EpiRows pre = epilogue_rows<MODE>(p, td, lane);  // requested before the wait
      if (!mbar_wait(&acc_full[acc], use & 1u, abort_flag)) {
        if (lane == 0) report(p.status, kDevTimeout, kSiteGemmEpilogue, (unsigned)tile, 0u);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if constexpr (MODE == 2)
        epilogue_router<BN>(p, td, tbase, nb * kBoxRows, q, lane);
      else
        epilogue_tile<MODE>(p, td, tbase, nb * kBoxRows, q, lane, pre);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE, int BN>
cudaError_t launch_mode_bn(const GemmParams& p, int grid, cudaStream_t s) {
  return launch_pdl(k_grouped_gemm<MODE, BN>, dim3(grid * ctas_of<MODE, BN>()),
                    dim3(threads_of<MODE>()), Cfg<BN, ring_of<MODE, BN>()>::kSmem,
                    s, p);
}

template <int MODE, int BN>
cudaError_t allow_smem() {
  static_assert(MODE != 2 || BN == kRouterBn, "router tiles");
  return cudaFuncSetAttribute(k_grouped_gemm<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)Cfg<BN, ring_of<MODE, BN>()>::kSmem);
}

}  // namespace

cudaError_t prepare_gemm_bf16() {
  cudaError_t e;
  if ((e = allow_smem<2, kRouterBn>()) != cudaSuccess) return e;
  if ((e = allow_smem<0, 64>()) != cudaSuccess || (e = allow_smem<0, 128>()) != cudaSuccess ||
      (e = allow_smem<0, 256>()) != cudaSuccess || (e = allow_smem<1, 64>()) != cudaSuccess ||
      (e = allow_smem<1, 128>()) != cudaSuccess || (e = allow_smem<1, 256>()) != cudaSuccess)
    return e;
  return cudaSuccess;
}

size_t gemm_smem_bytes(int bn) {
  return bn == 256   ? Cfg<256, ring_of<0, 256>()>::kSmem
         : bn == 128 ? Cfg<128, ring_of<0, 128>()>::kSmem
                     : Cfg<64, ring_of<0, 64>()>::kSmem;
}

cudaError_t launch_gemm(int mode, int bn, const GemmParams& p, int grid, cudaStream_t s) {
  if (mode == 2) return launch_mode_bn<2, kRouterBn>(p, grid, s);
  if (mode == 0) {
    if (bn == 256) return launch_mode_bn<0, 256>(p, grid, s);
    if (bn == 128) return launch_mode_bn<0, 128>(p, grid, s);
    return launch_mode_bn<0, 64>(p, grid, s);
  }
  if (bn == 256) return launch_mode_bn<1, 256>(p, grid, s);
  if (bn == 128) return launch_mode_bn<1, 128>(p, grid, s);
  return launch_mode_bn<1, 64>(p, grid, s);
}

}  // namespace dg
