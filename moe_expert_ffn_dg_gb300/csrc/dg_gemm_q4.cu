// Grouped tcgen05 GEMMs over 4- or 8-bit group-64 affine weights (sm_103a).
//
// The weight format is the one of "DiffusionGemma port — plan & parity
// strategy", Reference dossier §1 (OptiQ affine quantisation, group size 64,
// 4-bit experts, 8-bit where its predicate keeps 8 bits, as for the dense
// MLP): per row, code words of 8 four-bit codes (code k of a word at bits 4k)
// or bytes of 8-bit codes, and per group of 64 codes a bf16 scale s and bias
// b; the weight is s * q + b.  The same kernel takes NVFP4 weights ("diffgemma
// — architecture & implemented contract", §8 nvfp4 expert profile): e2m1
// codes in the 4-bit slab layout, an e4m3 scale per 16 codes and an fp32
// scale per matrix; a code times its block scale is exact in bf16, and the
// matrix scale multiplies the fp32 accumulator in the epilogue.  "Independent
// GGUF Forward Pass and Bit-Identical Cross-Backend Consistency for a 26B
// Text-Diffusion Model" (§1 contribution 6, §4 bottleneck ablation) names the
// per-expert 4-bit dequantisation as the cost that dominates; here it runs
// beside the tensor core instead of in front of it.
//
// Dataflow of one tile (128 weight rows x up to BN token rows), in stages of
// one group (64 along K):
//   warp 0   TMA: code slabs (128 rows x 128 bytes = 16 KB, 128B swizzle:
//            256 four-bit or 128 eight-bit codes a row) into a ring, and per
//            tile the rows' scales and
//            biases (bulk copies; the rows are 2K/64 bytes, not TMA-able);
//   warp 1   TMA: the tokens of each stage (BN rows x 64 bf16) into a ring;
//   warp 2   TMEM owner and MMA issuer: four tcgen05.mma (K = 16) per stage,
//            both operands in shared memory;
//   warp 3   waits, for the issuer, until a stage's operands are ready and
//            hands it over through a named barrier (see below);
//   warps 4..  dequantise, in NT teams of four warps (one warp per 32 weight
//            rows): stage s of the CTA's sequence belongs to team s mod NT,
//            whose threads expand one row's 64 codes each to bf16 (exact
//            s * q + b, one rounding) into one of the team's own A stages, in
//            the 128B-swizzled K-major layout the MMA reads;
//   last 4   epilogue, as for bf16 weights (GEGLU or the weighted rows).
// Dequantised weights go to shared memory rather than TMEM: concurrent
// tcgen05.st traffic slows A-from-TMEM MMAs about threefold on this part,
// while shared-memory stores (and proxy fences) at the full store rate leave
// shared-memory MMAs at their unloaded cost (55 cycles for N <= 128, 128 for
// N = 256).  TMEM then holds only the two fp32 accumulators, so token tiles
// go up to 256.  Every ring slot has one consumer group that takes its uses
// in order (the A stages belong to one team each), so an mbarrier parity
// wait can never be two phases ahead of its slot.
//
// Why the issuer does not wait on mbarriers itself: on sm_103a, a shared-
// memory access (an mbarrier poll or a plain load) by a thread that has
// tcgen05.mma in flight stalls until those MMAs complete, so one poll per
// stage costs the MMA pipeline latency (measured ~700 cycles against ~55
// cycles per M=128, K=16 MMA).  Another warp's polls are not affected, and a
// named CTA barrier is not a memory access.  So warp 3 does the bounded
// mbarrier waits and meets the issuer at a barrier.red.or once per stage; the
// reduced predicate carries "stop" (a wait that ran out), so both warps leave
// on the same round and the barrier can never be left half-arrived.
//
// Every wait is bounded; a wait that runs out records itself in the status
// word and the CTA winds down (copies and MMAs in flight are drained before
// TMEM is released).
#include "dg_gemm_common.cuh"

// Cycle accounting of the pipeline roles, compiled in only with
// -DDG_Q4_TIMING=1 (off by default: it adds clock reads and atomics).
// Slots (cycles summed over the warps that record them; [15] counts
// stages): 0 dequant waits for its scales, 1 for a code slab, 2 for its A
// slot (the MMAs of its previous stage), 3 dequantising and storing a stage,
// 4 fence and arrive; 5 waiter on the accumulators, 6 on an A stage, 7 on a
// token stage; 8 issuer at the hand-off barrier.  Read with
// dg_q4_timing_read() (exported only in such a build).
#ifndef DG_Q4_TIMING
#define DG_Q4_TIMING 0
#endif
#if DG_Q4_TIMING
__device__ unsigned long long g_q4_timing[16];
#define DG_T0(v) const long long v = clock64()
#define DG_TADD(slot, v) atomicAdd(&g_q4_timing[slot], (unsigned long long)(clock64() - (v)))
#else
#define DG_T0(v)
#define DG_TADD(slot, v)
#endif

namespace dg {
namespace {

using namespace gemm;

constexpr int kSlabWords = 32;                 // 32-bit code words per row of a slab
constexpr int kQSlabBytes = 128 * kSlabWords * 4;  // 16 KB
constexpr int kAGroupBytes = 128 * 128;        // 128 rows x 64 bf16
constexpr int kDequantWarp0 = 4;
// Completion of stage s (its four MMAs) is signalled on sdone[s mod
// kStageRing], one commit per stage: a tcgen05.commit costs about as much as
// a quarter of a stage's MMAs, so the token and A slots freed by one stage
// share it.  A slot's next writer waits for the stage that last used it,
// NB (tokens) or M * NT (A) stages back; with the ring longer than both, no
// parity wait can alias.
constexpr int kStageRing = 32;

// Per token-tile width: groups of 64 along K per stage (GPS: one stage is
// 4 * GPS MMAs, one hand-off and one commit; narrow tiles take two groups, as
// each stage's fixed cost is then shared by twice the MMAs of ~55 cycles),
// dequantising teams (NT), A stages per team (M; GPS x 16 KB each), code
// slabs in flight (SQ) and token stages in flight (NB, GPS x BN x 128 bytes
// each), beside double-buffered per-tile scales and biases.  The token ring
// covers the L2 latency plus the MMA time of a stage; a team refills its A
// stage while the other teams' stages are multiplied.  With K up to 2944
// (46 groups) every width fits.
template <int BN>
struct CfgQ {
  static constexpr int kGPS = BN <= 64 ? 2 : 1;
  static constexpr int kNT = BN == 128 ? 4 : 3;
  static constexpr int kM = 1;
  static constexpr int kNA = kNT * kM;
  static constexpr int kSQ = 2;
  static constexpr int kNB = BN == 256 ? 3 : BN == 128 ? 5 : BN == 64 ? 3 : 6;
  static constexpr int kAStageBytes = kGPS * kAGroupBytes;
  static constexpr int kBGroupBytes = BN * 128;
  static constexpr int kBStageBytes = kGPS * kBGroupBytes;
  static constexpr int kNumDequantWarps = 4 * kNT;
  static constexpr int kEpilogueWarp0 = kDequantWarp0 + kNumDequantWarps;
  static constexpr int kThreads = 32 * (kEpilogueWarp0 + 4);
  static constexpr int kBarBytes = 1024;
  static_assert(kNB < kStageRing && kM * kNT < kStageRing, "stage ring too short");
  // mbarriers (qfull, qempty, bfull, afull, sdone, sfull, sempty, acc_full,
  // acc_empty, drain, stall), then the TMEM address and the abort flag
  static_assert(8 * (2 * kSQ + kNB + kNA + kStageRing + 10) + 8 <= kBarBytes, "barrier area");
  static constexpr size_t kFixed = 1024 + (size_t)kSQ * kQSlabBytes +
                                   (size_t)kNB * kBStageBytes + (size_t)kNA * kAStageBytes +
                                   kBarBytes + kTileTableBytes;
};

// Per-team stage counters in one register (16 bits each; only their low
// bits matter, for the slot and the parity): the issuer must not touch local
// memory while its MMAs are in flight.
__device__ __forceinline__ uint32_t team_count(uint64_t packed, int team) {
  return (uint32_t)(packed >> (16 * team)) & 0xFFFFu;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Store 16 bytes at a shared-memory address.
__device__ __forceinline__ void sts_u32x4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void lds_u32x4(const uint8_t* p, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(smem_u32(p))
               : "memory");
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
  __nv_bfloat162 r;
  memcpy(&r, &u, 4);
  return r;
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) {
  uint32_t r;
  memcpy(&r, &v, 4);
  return r;
}

// 16 eight-bit codes (four words, code k at byte k) -> 8 bf16 pairs in K
// order, w = s * q + b rounded once to bf16.  q = 16 hi + lo with the two
// nibbles exact as in dequant32 below, q itself exact in bf16 (8 bits), then
// the group's fused multiply-add.
__device__ __forceinline__ void dequant16_u8(const uint32_t (&w)[4], uint32_t s2, uint32_t b2,
                                             uint32_t (&o)[8]) {
  const __nv_bfloat162 s = as_bf162(s2), b = as_bf162(b2), m = as_bf162(0x43004300u),
                       sixteen = as_bf162(0x41804180u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u = w[j] >> 4;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      // bytes 2pp and 2pp+1 of the word -> codes (low, high) of the pair
      // result bytes [w byte 2pp, 0, w byte 2pp+1, 0] (selector 4 = a zero byte)
      const uint32_t sel = 0x4140u + 0x0202u * pp;
      const uint32_t lo = (__byte_perm(w[j], 0u, sel) & 0x000F000Fu) | 0x43004300u;
      const uint32_t hi = (__byte_perm(u, 0u, sel) & 0x000F000Fu) | 0x43004300u;
      const __nv_bfloat162 q = __hfma2(__hsub2(as_bf162(hi), m), sixteen, __hsub2(as_bf162(lo), m));
      o[2 * j + pp] = as_u32(__hfma2(q, s, b));
    }
  }
}

// NVFP4: 32 e2m1 codes (four words, two a byte, low nibble first) of two
// blocks of 16 -> 16 bf16 pairs in K order, each code times its block's
// e4m3 scale (exact: at most 6 significant bits).  The hardware converts a
// byte's two codes to f16 exactly; the products are formed in fp32 and packed.
__device__ __forceinline__ void dequant32_nvfp4(const uint32_t (&w)[4], float s_a, float s_b,
                                                uint32_t (&o)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float sc = j < 2 ? s_a : s_b;  // words 0-1: block a, 2-3: block b
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w[j]));
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      __half2 hv;
      memcpy(&hv, &h[pp], 4);
      const float2 f = __half22float2(hv);
      o[4 * j + pp] = as_u32(__floats2bfloat162_rn(f.x * sc, f.y * sc));
    }
  }
}

// e4m3 byte (non-negative) -> float: the 7 magnitude bits placed at float
// bits 20..26 read as 2^(e-127) (1 + m/8) (or m 2^-129 for e = 0), times 2^120.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  return __uint_as_float((c & 0x7Fu) << 20) * 0x1p120f;
}

// 32 codes (four words) -> 16 bf16 pairs in K order, w = s * q + b rounded
// once to bf16.  A code q sits in the low mantissa bits of the bf16 128 + q
// (0x4300 | q, exact); subtracting 128 leaves q exactly, then one fused
// multiply-add applies the group's scale and bias.
__device__ __forceinline__ void dequant32(const uint32_t (&w)[4], uint32_t s2, uint32_t b2,
                                          uint32_t (&o)[16]) {
  const __nv_bfloat162 s = as_bf162(s2), b = as_bf162(b2), m = as_bf162(0x43004300u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u = w[j] >> 4;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      // bytes: [w.byte pp, -, u.byte pp, -] -> codes 2pp (low) and 2pp+1 (high)
      uint32_t t = __byte_perm(w[j], u, 0x4400u + 0x1111u * pp);
      t = (t & 0x000F000Fu) | 0x43004300u;
      const __nv_bfloat162 qv = __hsub2(as_bf162(t), m);
      o[4 * j + pp] = as_u32(__hfma2(qv, s, b));
    }
  }
}

template <int MODE, int BN, int QF>
__global__ void __launch_bounds__(CfgQ<BN>::kThreads, 1)
    k_grouped_gemm_q4(const __grid_constant__ GemmParams p) {
  using C = CfgQ<BN>;
  constexpr int SQ = C::kSQ, NB = C::kNB, NA = C::kNA, NT = C::kNT, GPS = C::kGPS;
  constexpr bool NVFP4 = QF == kQfNvfp4;
  constexpr int GPSL = QF == 8 ? 2 : 4;  // groups of 64 per code slab
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sB = sQ + (size_t)SQ * kQSlabBytes;
  uint8_t* sA = sB + (size_t)NB * C::kBStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + (size_t)NA * C::kAStageBytes);
  uint64_t* qfull = bars;
  uint64_t* qempty = qfull + SQ;
  uint64_t* bfull = qempty + SQ;
  uint64_t* afull = bfull + NB;
  uint64_t* sdone = afull + NA;
  uint64_t* sfull = sdone + kStageRing;
  uint64_t* sempty = sfull + 2;
  uint64_t* acc_full = sempty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* stall = drain + 1;  // bounded-wait test: never arrived on
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(stall + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_start = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + C::kBarBytes);
  int* s_off = s_start + kMaxGroups + 2;
  uint8_t* sScale = reinterpret_cast<uint8_t*>(bars) + C::kBarBytes + kTileTableBytes;
  const int slot_bytes = p.sc_slot_bytes;  // scales of one tile; biases follow

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < SQ; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], C::kNumDequantWarps);
    }
    for (int s = 0; s < NB; ++s) mbar_init(&bfull[s], 1);
    for (int a = 0; a < NA; ++a) mbar_init(&afull[a], 4);  // the four warps of one team
    for (int r = 0; r < kStageRing; ++r) mbar_init(&sdone[r], 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sfull[a], 1);
      mbar_init(&sempty[a], C::kNumDequantWarps);
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
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&p.xb_exp64);
    tma_prefetch_map(&p.xb_exp16);
    tma_prefetch_map(&p.xb_d64);
    tma_prefetch_map(&p.xb_d16);
    tma_prefetch_map(full_stage_map<BN>(p, false));
    tma_prefetch_map(full_stage_map<BN>(p, true));
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  // everything above touches only this CTA's resources; from here on the
  // kernel reads what earlier kernels wrote
  pdl_wait();
  if (warp >= C::kEpilogueWarp0)
    build_tile_table(p, threadIdx.x - 32 * C::kEpilogueWarp0, s_start, s_off);
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
    // ------------------------------------------------- weight codes + scales
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      int qs = 0;
      uint32_t qph = 0, qarmed = 0, qarmed_par = 0, sarmed = 0, sarmed_par = 0;
      bool ok = true;
      int local = 0;
      for (int tile = first; tile < ntiles && ok; tile += nct, ++local) {
        const int4 td = decode_tile(p, tile, nd, s_start, s_off);
        const bool dense = td.x == p.E;
        const int ng = dense ? p.kb_dense : p.kb_exp;  // groups of 64 per row
        // scale bytes per row: affine bf16 s (and b, in the second half of
        // the slot); NVFP4 one e4m3 per 16 codes, across the whole slot
        const uint32_t rowb = NVFP4 ? 4u * (uint32_t)ng : 2u * (uint32_t)ng;
        const int ss = local & 1;
        const uint32_t sph = (uint32_t)(local >> 1) & 1u;
        if (!mbar_wait(&sempty[ss], sph ^ 1u, abort_flag)) {
          report(p.status, kDevTimeout, kSiteGemmProducer, (unsigned)tile, 0xfffffffeu);
          *abort_flag = 1;
          break;
        }
        uint8_t* dsc = sScale + (size_t)ss * 2 * slot_bytes;
        uint8_t* dbi = dsc + slot_bytes;
        mbar_arrive_expect_tx(&sfull[ss], (NVFP4 ? 1u : 2u) * 128u * rowb);
        if (MODE == 0) {
          // 16-row blocks in the order of the interleaved slab: block 2c+h
          // holds gate (h = 0) or up (h = 1) rows 16c..16c+15 of the tile
#pragma unroll 1
          for (int blk = 0; blk < 8; ++blk) {
            const int c4 = blk >> 1, h = blk & 1;
            size_t src_row;
            const uint16_t *sc, *bi;
            if (dense) {
              src_row = (size_t)(64 * td.y + 16 * c4);
              sc = h ? p.sc_d1 : p.sc_d0;
              bi = h ? p.bi_d1 : p.bi_d0;
            } else {
              src_row = (size_t)td.x * 2 * p.I + (size_t)h * p.I + 64 * td.y + 16 * c4;
              sc = p.sc_exp;
              bi = p.bi_exp;
            }
            if (NVFP4) {
              bulk_g2s(dsc + (size_t)16 * blk * rowb,
                       reinterpret_cast<const uint8_t*>(sc) + src_row * rowb, 16 * rowb,
                       &sfull[ss], pol_w);
            } else {
              bulk_g2s(dsc + (size_t)16 * blk * rowb, sc + src_row * ng, 16 * rowb, &sfull[ss],
                       pol_w);
              bulk_g2s(dbi + (size_t)16 * blk * rowb, bi + src_row * ng, 16 * rowb, &sfull[ss],
                       pol_w);
            }
          }
        } else {
          const size_t src_row = (dense ? (size_t)0 : (size_t)td.x * p.H) + 128 * (size_t)td.y;
          const uint16_t* sc = dense ? p.sc_d0 : p.sc_exp;
          const uint16_t* bi = dense ? p.bi_d0 : p.bi_exp;
          if (NVFP4) {
            bulk_g2s(dsc, reinterpret_cast<const uint8_t*>(sc) + src_row * rowb, 128 * rowb,
                     &sfull[ss], pol_w);
          } else {
            bulk_g2s(dsc, sc + src_row * ng, 128 * rowb, &sfull[ss], pol_w);
            bulk_g2s(dbi, bi + src_row * ng, 128 * rowb, &sfull[ss], pol_w);
          }
        }
        sarmed |= 1u << ss;
        sarmed_par = (sarmed_par & ~(1u << ss)) | (sph << ss);
        const int nsl = (ng + GPSL - 1) / GPSL;
        for (int sl = 0; sl < nsl; ++sl) {
          if (!mbar_wait(&qempty[qs], qph ^ 1u, abort_flag)) {
            report(p.status, kDevTimeout, kSiteGemmProducer, (unsigned)tile, (unsigned)sl);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&qfull[qs], kQSlabBytes);
          uint8_t* dst = sQ + (size_t)qs * kQSlabBytes;
          const int x = sl * kSlabWords;
          if (MODE == 0) {
            if (!dense) {
              tma_load_5d(&p.wa_exp, &qfull[qs], dst, x, 0, 0, 4 * td.y, td.x, pol_w);
            } else if (p.dense_5d) {
              tma_load_4d(&p.wa_d5, &qfull[qs], dst, x, 0, 0, 4 * td.y, pol_w);
            } else {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int yg = td.y * 64 + 16 * c;
                tma_load_2d_hint(&p.wa_d0, &qfull[qs], dst + (2 * c) * kBoxBytes, x, yg, pol_w);
                tma_load_2d_hint(&p.wa_d1, &qfull[qs], dst + (2 * c + 1) * kBoxBytes, x, yg, pol_w);
              }
            }
          } else {
            const CUtensorMap* ma = dense ? &p.wa_d0 : &p.wa_exp;
            tma_load_2d_hint(ma, &qfull[qs], dst, x, (dense ? 0 : td.x * p.H) + td.y * 128, pol_w);
          }
          qarmed |= 1u << qs;
          qarmed_par = (qarmed_par & ~(1u << qs)) | (qph << qs);
          if (++qs == SQ) {
            qs = 0;
            qph ^= 1u;
          }
        }
      }
      for (int s = 0; s < SQ; ++s)
        if ((qarmed >> s) & 1u)
          if (!wait_no_abort(&qfull[s], (qarmed_par >> s) & 1u))
            report(p.status, kDevTimeout, kSiteGemmDrain, (unsigned)s, 1u);
      for (int s = 0; s < 2; ++s)
        if ((sarmed >> s) & 1u)
          if (!wait_no_abort(&sfull[s], (sarmed_par >> s) & 1u))
            report(p.status, kDevTimeout, kSiteGemmDrain, (unsigned)s, 2u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------- token stages
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_last();
      int bs = 0;
      uint32_t bph = 0, armed = 0, armed_par = 0, st = 0;  // st: global stage index
      bool ok = true;
      for (int tile = first; tile < ntiles && ok; tile += nct) {
        const int4 td = decode_tile(p, tile, nd, s_start, s_off);
        const bool dense = td.x == p.E;
        const int ng = dense ? p.kb_dense : p.kb_exp;
        // a full stage of 128 or 256 rows in one box (measured: faster there,
        // slower than two 16-row boxes at 32), else 64-row then 16-row boxes
        const bool full = BN >= 128 && td.w == BN;
        const int nb64 = full ? 0 : td.w / 64;
        const int nb16 = full ? 0 : (td.w - 64 * nb64 + kBoxRows - 1) / kBoxRows;
        const uint32_t group_bytes = full ? BN * 128u : nb64 * 64 * 128 + nb16 * kBoxBytes;
        const CUtensorMap* mbf = full_stage_map<BN>(p, dense);
        const CUtensorMap* mb64 = dense ? &p.xb_d64 : &p.xb_exp64;
        const CUtensorMap* mb16 = dense ? &p.xb_d16 : &p.xb_exp16;
        const int nst = (ng + GPS - 1) / GPS;
        for (int k = 0; k < nst; ++k, ++st) {
          // the slot's previous stage, NB back, must have been multiplied
          const uint32_t w = st - (uint32_t)NB;
          if (st >= (uint32_t)NB &&
              !mbar_wait(&sdone[w % kStageRing], (w / kStageRing) & 1u, abort_flag)) {
            report(p.status, kDevTimeout, kSiteGemmTokens, (unsigned)tile, (unsigned)k);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const int ngk = min(GPS, ng - GPS * k);
          mbar_arrive_expect_tx(&bfull[bs], group_bytes * (uint32_t)ngk);
          for (int gi = 0; gi < ngk; ++gi) {
            uint8_t* b_dst = sB + (size_t)bs * C::kBStageBytes + (size_t)gi * C::kBGroupBytes;
            const int x = 64 * (GPS * k + gi);
            if (full) tma_load_2d_hint(mbf, &bfull[bs], b_dst, x, td.z, pol_x);
            for (int r = 0; r < nb64; ++r)
              tma_load_2d_hint(mb64, &bfull[bs], b_dst + r * 64 * 128, x, td.z + 64 * r, pol_x);
            for (int r = 0; r < nb16; ++r)
              tma_load_2d_hint(mb16, &bfull[bs], b_dst + (64 * nb64 + kBoxRows * r) * 128, x,
                               td.z + 64 * nb64 + kBoxRows * r, pol_x);
          }
          armed |= 1u << bs;
          armed_par = (armed_par & ~(1u << bs)) | (bph << bs);
          if (++bs == NB) {
            bs = 0;
            bph ^= 1u;
          }
        }
      }
      for (int s = 0; s < NB; ++s)
        if ((armed >> s) & 1u)
          if (!wait_no_abort(&bfull[s], (armed_par >> s) & 1u))
            report(p.status, kDevTimeout, kSiteGemmDrain, (unsigned)s, 3u);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- MMA issuer
    // Learns that a stage's operands are ready only through handoff(): it
    // touches no mbarrier while its MMAs are in flight.
    int bs = 0, local = 0;
    uint32_t st = 0;  // global stage index
    uint64_t cnt = 0;
    bool stop = false, issued = false;
    for (int tile = first; tile < ntiles && !stop; tile += nct, ++local) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const bool dense = td.x == p.E;
      const int ng = dense ? p.kb_dense : p.kb_exp;
      const int nb = (td.w + kBoxRows - 1) / kBoxRows;
      const int acc = local & 1;
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      const uint32_t idesc = idesc_bf16_f32(128, nb * kBoxRows);
      const int nst = (ng + GPS - 1) / GPS;
      for (int k = 0; k < nst; ++k, ++st) {
        DG_T0(t_ho);
        const bool ho_stop = handoff(false);
        if (lane == 0) DG_TADD(8, t_ho);
        if (ho_stop) {
          stop = true;
          break;
        }
        tc_fence_after();
        const int team = (int)(st % NT);
        const uint32_t as = (uint32_t)team + NT * (team_count(cnt, team) % C::kM);
        cnt += 1ull << (16 * team);
        if (lane == 0) {
          // descriptors of the stage's first K step; each further step of 16
          // (32 bytes) adds 2 to the address field
          // (a group further: 16 KB of A, BN x 128 bytes of B)
          const uint64_t da = sw128_kmajor_desc(smem_u32(sA + (size_t)as * C::kAStageBytes));
          const uint64_t db = sw128_kmajor_desc(smem_u32(sB + (size_t)bs * C::kBStageBytes));
          const int ngk = min(GPS, ng - GPS * k);
          umma_bf16(d_tmem, da, db, idesc, k != 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) umma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, 1u);
          if (GPS == 2 && ngk == 2) {
            const uint64_t da1 = da + (kAGroupBytes >> 4), db1 = db + (C::kBGroupBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(d_tmem, da1 + 2 * kk, db1 + 2 * kk, idesc, 1u);
          }
          umma_commit(&sdone[st % kStageRing]);
          if (k == nst - 1) umma_commit(&acc_full[acc]);
        }
        issued = true;
        if (++bs == NB) bs = 0;
        __syncwarp();
      }
    }
    // every MMA issued here must have completed before TMEM is released
    if (lane == 0 && issued) {
      umma_commit(drain);
      if (!wait_no_abort(drain, 0u)) report(p.status, kDevTimeout, kSiteGemmDrain, 99u, 0u);
    }
  } else if (warp == 3) {
    // ------------------------------------------------- waiter for the issuer
    int bs = 0, local = 0;
    uint32_t bph = 0, st = 0;
    uint64_t cnt = 0;
    bool stop = false;
    for (int tile = first; tile < ntiles && !stop; tile += nct, ++local) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const bool dense = td.x == p.E;
      const int ng = dense ? p.kb_dense : p.kb_exp;
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const int nst = (ng + GPS - 1) / GPS;
      for (int k = 0; k < nst; ++k, ++st) {
        bool ok = true;
        unsigned what = 0;
        const int team = (int)(st % NT);
        const uint32_t n = team_count(cnt, team);
        const uint32_t as = (uint32_t)team + NT * (n % C::kM);
        const uint32_t aph = (n / C::kM) & 1u;
        cnt += 1ull << (16 * team);
        DG_T0(t_w0);
        if (k == 0 && !mbar_wait(&acc_empty[acc], (use & 1u) ^ 1u, abort_flag)) {
          ok = false;
          what = 0xffffffffu;
        }
        if (lane == 0) DG_TADD(5, t_w0);
        DG_T0(t_w1);
        if (ok && !mbar_wait(&afull[as], aph, abort_flag)) {
          ok = false;
          what = 0x10000u + k;
        }
        if (lane == 0) DG_TADD(6, t_w1);
        DG_T0(t_w2);
        if (ok && !mbar_wait(&bfull[bs], bph, abort_flag)) {
          ok = false;
          what = 0x20000u + k;
        }
        if (lane == 0) DG_TADD(7, t_w2);
        if (++bs == NB) {
          bs = 0;
          bph ^= 1u;
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
  } else if (warp < C::kEpilogueWarp0) {
    // ------------------------------------------------- dequantise into A stages
    const int q = warp & 3;                        // 32-row quarter of the tile
    const int team = (warp - kDequantWarp0) >> 2;
    const int row = 32 * q + lane;                 // weight row of the tile
    // this thread's row in an A stage (128B-swizzled K-major: 8-row atoms of
    // 1024 bytes, 16-byte chunk c of row r at chunk c ^ (r & 7)); the code
    // slabs use the same swizzle on 128-byte rows
    const uint32_t a_row = smem_u32(sA) + (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    const int rsw = row & 7;
    int qs = 0, local = 0;
    uint32_t qph = 0, s0 = 0, j = 0;  // stage base of the tile; own stages so far
    bool ok = true;
    for (int tile = first; tile < ntiles && ok; tile += nct, ++local) {
      const int4 td = decode_tile(p, tile, nd, s_start, s_off);
      const bool dense = td.x == p.E;
      const int ng = dense ? p.kb_dense : p.kb_exp;
      const int nsl = (ng + GPSL - 1) / GPSL;
      const int ss = local & 1;
      const uint32_t sph = (uint32_t)(local >> 1) & 1u;
      DG_T0(t_sf);
      const bool sf_ok = mbar_wait(&sfull[ss], sph, abort_flag);
      if (lane == 0) DG_TADD(0, t_sf);
      if (!sf_ok) {
        if (lane == 0) report(p.status, kDevTimeout, kSiteGemmDequant, (unsigned)tile, 0xffffu);
        *abort_flag = 1;
        break;
      }
      const uint16_t* sc_row =
          reinterpret_cast<const uint16_t*>(sScale + (size_t)ss * 2 * slot_bytes) + row * ng;
      const uint16_t* bi_row = sc_row + slot_bytes / 2;
      // NVFP4: this row's e4m3 block scales, 4 per group
      const uint8_t* e4_row = sScale + (size_t)ss * 2 * slot_bytes + (size_t)row * 4 * ng;
      for (int sl = 0; sl < nsl && ok; ++sl) {
        DG_T0(t_qf);
        const bool qf_ok = mbar_wait(&qfull[qs], qph, abort_flag);
        if (lane == 0) DG_TADD(1, t_qf);
        if (!qf_ok) {
          if (lane == 0) report(p.status, kDevTimeout, kSiteGemmDequant, (unsigned)tile, (unsigned)sl);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const uint8_t* qrow = sQ + (size_t)qs * kQSlabBytes + row * 128;
        // the slab's stages (GPSL / GPS of them, fewer at the tile's end)
#pragma unroll 1
        for (int k = (GPSL * sl) / GPS; k < (GPSL * sl + GPSL) / GPS && GPS * k < ng; ++k) {
          const uint32_t stg = s0 + (uint32_t)k;  // global stage index
          if ((int)(stg % NT) != team) continue;
          const uint32_t as = (uint32_t)team + NT * (j % C::kM);
          // the slot's previous stage (this team's, M own stages back)
          const uint32_t w = stg - (uint32_t)(C::kM * NT);
          const bool first_use = j < (uint32_t)C::kM;
          ++j;
          DG_T0(t_sd);
          const bool sd_ok =
              first_use || mbar_wait(&sdone[w % kStageRing], (w / kStageRing) & 1u, abort_flag);
          if (lane == 0) DG_TADD(2, t_sd);
          DG_T0(t_dq);
          if (!sd_ok) {
            if (lane == 0)
              report(p.status, kDevTimeout, kSiteGemmDequant, (unsigned)tile, 0x10000u + k);
            *abort_flag = 1;
            ok = false;
            break;  // the code slab is still released below so the producer drains
          }
          const int ngk = min(GPS, ng - GPS * k);
#pragma unroll 1
          for (int gi = 0; gi < ngk; ++gi) {
            const int g = GPS * k + gi, gs = g % GPSL;  // group in the tile, in the slab
            uint32_t o[32];
            if (NVFP4) {  // the group's 32 bytes: chunks 2gs, 2gs + 1; 4 blocks of 16
              uint32_t w0[4], w1[4];
              lds_u32x4(qrow + (((2 * gs) ^ rsw) << 4), w0);
              lds_u32x4(qrow + (((2 * gs + 1) ^ rsw) << 4), w1);
              const uint32_t e4 = *reinterpret_cast<const uint32_t*>(e4_row + 4 * g);
              dequant32_nvfp4(w0, e4m3_to_f32(e4 & 0xFFu), e4m3_to_f32((e4 >> 8) & 0xFFu),
                              *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
              dequant32_nvfp4(w1, e4m3_to_f32((e4 >> 16) & 0xFFu), e4m3_to_f32(e4 >> 24),
                              *reinterpret_cast<uint32_t(*)[16]>(&o[16]));
            } else if (QF == 4) {  // the group's 32 bytes: chunks 2gs, 2gs + 1
              const uint32_t s = sc_row[g], b = bi_row[g];
              const uint32_t s2 = s | (s << 16), b2 = b | (b << 16);
              uint32_t w0[4], w1[4];
              lds_u32x4(qrow + (((2 * gs) ^ rsw) << 4), w0);
              lds_u32x4(qrow + (((2 * gs + 1) ^ rsw) << 4), w1);
              dequant32(w0, s2, b2, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
              dequant32(w1, s2, b2, *reinterpret_cast<uint32_t(*)[16]>(&o[16]));
            } else {  // 64 bytes: chunks 4gs .. 4gs + 3
              const uint32_t s = sc_row[g], b = bi_row[g];
              const uint32_t s2 = s | (s << 16), b2 = b | (b << 16);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t wv[4];
                lds_u32x4(qrow + (((4 * gs + c) ^ rsw) << 4), wv);
                dequant16_u8(wv, s2, b2, *reinterpret_cast<uint32_t(*)[8]>(&o[8 * c]));
              }
            }
            const uint32_t dst = a_row + as * (uint32_t)C::kAStageBytes + gi * (uint32_t)kAGroupBytes;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              sts_u32x4(dst + (uint32_t)((ch ^ rsw) << 4), o[4 * ch], o[4 * ch + 1],
                        o[4 * ch + 2], o[4 * ch + 3]);
          }
          if (lane == 0) DG_TADD(3, t_dq);
          DG_T0(t_fa);
          // make the generic-proxy stores visible to the tensor core
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[as]);
          if (lane == 0) DG_TADD(4, t_fa);
#if DG_Q4_TIMING
          if (lane == 0) atomicAdd(&g_q4_timing[15], 1ull);
#endif
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qs]);
        if (++qs == SQ) {
          qs = 0;
          qph ^= 1u;
        }
      }
      s0 += (uint32_t)((ng + GPS - 1) / GPS);
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&sempty[ss]);
    }
  } else {
    // ------------------------------------------------- epilogue
    const int q = warp & 3;
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
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      // per-tile values the epilogue needs, requested before the wait
      float g_lo = 1.f, g_hi = 1.f;  // NVFP4 matrix scales (gate / up lanes)
      if (NVFP4) {
        if (td.x != p.E) {
          g_lo = g_hi = __ldg(p.g_exp + td.x);
        } else {
          g_lo = __ldg(p.g_d0);
          g_hi = MODE == 0 ? __ldg(p.g_d1) : g_lo;
        }
      }
      const EpiRows pre = epilogue_rows<MODE>(p, td, lane);
      if (!mbar_wait(&acc_full[acc], use & 1u, abort_flag)) {
        if (lane == 0) report(p.status, kDevTimeout, kSiteGemmEpilogue, (unsigned)tile, 0u);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      epilogue_tile<MODE>(p, td, tbase, nb * kBoxRows, q, lane, pre, g_lo, g_hi);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE, int BN, int QF>
cudaError_t launch_q4(const GemmParams& p, int grid, cudaStream_t s) {
  const size_t smem = CfgQ<BN>::kFixed + 4 * (size_t)p.sc_slot_bytes;
  return launch_pdl(k_grouped_gemm_q4<MODE, BN, QF>, dim3(grid), dim3(CfgQ<BN>::kThreads), smem,
                    s, p);
}

// The scale slots depend on the shapes, so every instance may use up to the
// device's opt-in maximum; launches that would exceed it are refused at
// handle creation.
template <int QF>
cudaError_t allow_smem_q4(int smem_max) {
  cudaError_t e = cudaSuccess;
  auto one = [&](auto kernel) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  };
  one(k_grouped_gemm_q4<0, 32, QF>);
  one(k_grouped_gemm_q4<0, 64, QF>);
  one(k_grouped_gemm_q4<0, 128, QF>);
  one(k_grouped_gemm_q4<0, 256, QF>);
  one(k_grouped_gemm_q4<1, 32, QF>);
  one(k_grouped_gemm_q4<1, 64, QF>);
  one(k_grouped_gemm_q4<1, 128, QF>);
  one(k_grouped_gemm_q4<1, 256, QF>);
  return e;
}

template <int BITS>
cudaError_t launch_bits(int mode, int bn, const GemmParams& p, int grid, cudaStream_t s) {
  if (mode == 0) {
    if (bn == 256) return launch_q4<0, 256, BITS>(p, grid, s);
    if (bn == 128) return launch_q4<0, 128, BITS>(p, grid, s);
    if (bn == 64) return launch_q4<0, 64, BITS>(p, grid, s);
    return launch_q4<0, 32, BITS>(p, grid, s);
  }
  if (bn == 256) return launch_q4<1, 256, BITS>(p, grid, s);
  if (bn == 128) return launch_q4<1, 128, BITS>(p, grid, s);
  if (bn == 64) return launch_q4<1, 64, BITS>(p, grid, s);
  return launch_q4<1, 32, BITS>(p, grid, s);
}

}  // namespace

size_t gemm_q4_smem_bytes(int bn, int sc_slot_bytes) {
  const size_t fixed = bn == 256   ? CfgQ<256>::kFixed
                       : bn == 128 ? CfgQ<128>::kFixed
                       : bn == 64  ? CfgQ<64>::kFixed
                                   : CfgQ<32>::kFixed;
  return fixed + 4 * (size_t)sc_slot_bytes;
}

cudaError_t prepare_gemm_affine(int smem_max) {
  cudaError_t e;
  if ((e = allow_smem_q4<4>(smem_max)) != cudaSuccess) return e;
  if ((e = allow_smem_q4<8>(smem_max)) != cudaSuccess) return e;
  return allow_smem_q4<kQfNvfp4>(smem_max);
}

cudaError_t launch_gemm_affine(int mode, int bn, int qf, const GemmParams& p, int grid,
                               cudaStream_t s) {
  if (qf == kQfNvfp4) return launch_bits<kQfNvfp4>(mode, bn, p, grid, s);
  return qf == 8 ? launch_bits<8>(mode, bn, p, grid, s) : launch_bits<4>(mode, bn, p, grid, s);
}

}  // namespace dg

#if DG_Q4_TIMING
extern "C" int dg_q4_timing_read(unsigned long long* out16, int reset) {
  if (cudaMemcpyFromSymbol(out16, g_q4_timing, 16 * sizeof(unsigned long long)) != cudaSuccess)
    return 1;
  if (reset) {
    static const unsigned long long zero[16] = {};
    if (cudaMemcpyToSymbol(g_q4_timing, zero, sizeof(zero)) != cudaSuccess) return 1;
  }
  return 0;
}
#endif
