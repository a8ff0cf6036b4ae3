// pre_stats.cu -- the stats half of mhc_pre and of mhc_hc_head on GB300: per
// row, the projections of the flattened residual on the 5th-generation tensor
// cores, the row's sum of squares, and the gates (plus, for the pre pass, the
// Sinkhorn mix).
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre:
// hc_pre_torch_impl (rsqrt of mean(x^2) + rms_eps; mixes = (x @ fn^T) * rsqrt)
// and hc_split_sinkhorn (gates and the 4x4 Sinkhorn); deepseek_v4.py,
// hc_head_torch (4 mixes, pre = sigmoid(mix * scale + base) + hc_eps).
//
// Two builds of one kernel: NM = 24 mixes (the pre pass) and NM = 4 (hc_head).
//
// Decomposition.  A cluster of 16 CTAs owns a 128-row tile at a time; CTA s
// owns hidden columns [320 s, 320 s + 320) of all four streams, i.e. 1280 of a
// row's 20480 k.  fn's NM x 1280 slice of the CTA, split into bf16 hi (B rows
// [0, NM)) and lo (rows [NM, 2 NM)) halves, zero-padded to the MMA's N, stays
// in shared memory for the whole kernel (120 KB for 24 mixes), so each product
// is exact and the dot products carry ~2^-17 relative error per term.  Per
// tile and CTA:
//   * warp 0 streams R[128 rows, 64 k] boxes (128-byte swizzle) with TMA
//     through a 5-stage ring -- R is read from HBM exactly once;
//   * one thread of warp 1 issues tcgen05.mma (M=128 rows, N = 48 or 16,
//     K=16, bf16 -> fp32) into one of two accumulators in tensor memory;
//   * row warps 4..7 (one thread per tile row) accumulate sum x^2 from the
//     same stages (per 16-byte chunk an 8-square chain added to one of eight
//     accumulators, summed in a fixed tree);
//   * readout warps 8..11 load the accumulator (tcgen05.ld) and push each
//     row's NM mix partials and its sum of squares into the receive buffer of
//     the CTA that finalises the row (CTA s owns tile rows 8s..8s+7), then
//     signal all 16 CTAs with one cluster fence and relaxed remote arrives;
//   * owner warps 2, 3, 12, 13 reduce the 16 partials of a row in CTA order,
//     compute rsqrt, the mixes and the gates (and, for the pre pass, the 16
//     comb logits) and write them.
// The combine (x_norm, or hc_head's y) runs as a second, streaming launch
// (pre_simt.cu, combine_norm_kernel) that reads the pre gates this kernel
// writes; for the pre pass a fifth warp per row there runs the 4x4 Sinkhorn
// on the comb logits.
//
// Every row is reduced in one fixed order that depends only on its own data
// (same MMA sequence, same lanes, CTA-ordered cross-CTA sums), so any row
// range gives the whole-chunk bits.
//
// Every wait is bounded (~2 s of wall time); on expiry a CTA raises an abort
// flag, records which wait expired, drains its in-flight MMAs and copies,
// frees its TMEM and returns.
#include <cuda.h>

#include <mutex>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

// Bit s set: a bounded wait at site s expired; g_fused_where[s] holds
// (tile << 8) | cluster rank of the last one.  Bit 16 + s: a wait at site s
// gave up because its CTA had already aborted (g_fused_where_aborted[s]).
__device__ unsigned int g_fused_error;
__device__ unsigned int g_fused_where[32];
__device__ unsigned int g_fused_where_aborted[32];

namespace {
using namespace ptx;

// ---- geometry -------------------------------------------------------------
constexpr int kCl = 16;                       // CTAs per cluster (K split)
constexpr int kTile = 128;                    // rows per tile = UMMA M
constexpr int kHs = kH / kCl;                 // 320 hidden columns per CTA
constexpr int kBk = 64;                       // k per stage: 128-byte rows
constexpr int kHb = kHs / kBk;                // 5 column blocks per stream
constexpr int kKb = kHC * kHb;                // 20 k-blocks per tile per CTA
constexpr int kStages = 5;
constexpr int kStageBytes = kTile * kBk * 2;  // 16384
constexpr int kOwn = kTile / kCl;             // 8 rows finalised per CTA
constexpr int kHeadMix = kHC;                 // hc_head: one mix per stream
constexpr int kTmemCols = 128;                // two 48-column accumulators at 0 and 64

static_assert(kHs % kBk == 0 && kTile % kCl == 0, "");

// ---- warp roles -------------------------------------------------------------
// warp 0 producer, 1 MMA; 4..7 row warps and 8..11 readout warps (warp & 3 =
// the TMEM lane quarter, one thread per tile row); 2, 3, 12, 13 owners
constexpr int kProducerWarp = 0, kMmaWarp = 1;
constexpr int kRow0 = 4, kRowN = 4;           // sum x^2 from the stages
constexpr int kRead0 = 8, kReadN = 4;         // accumulator readout + push
constexpr int kOwnerN = 4;
constexpr int kOwnerLead = 2;                 // owner warp that broadcasts PFREE
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;         // 448
__device__ __forceinline__ int owner_index(int warp) {   // -1: not an owner warp
  return warp == 2 || warp == 3 ? warp - 2 : (warp == 12 || warp == 13 ? warp - 10 : -1);
}

// mbarrier slots (arrays are given explicit, non-overlapping ranges)
enum Bar : int {
  B_FULL = 0,                    // [kStages] TMA landed
  B_EMPTY = B_FULL + kStages,    // [kStages] MMA commit + 4 row warps done with the stage
  B_TFULL = B_EMPTY + kStages,   // [2] accumulator complete
  B_TEMPTY = B_TFULL + 2,        // [2] accumulator and sum x^2 read by the readout warps
  B_PREADY = B_TEMPTY + 2,       // all 16 CTAs pushed partials to us (remote)
  B_PFREE = B_PREADY + 1,        // all 16 owners consumed our previous push (remote)
  B_GALL = B_PFREE + 1,          // the readout warps pushed their partials
  B_OPULL = B_GALL + 1,          // 4 owner warps read the receive buffer
  B_DRAIN = B_OPULL + 1,         // final MMA drain
  B_FNREADY = B_DRAIN + 1,       // fn hi/lo tiles written (all warps but the producer)
  B_SSREADY = B_FNREADY + 1,     // [2] the row warps wrote a tile's sum x^2
  B_COUNT = B_SSREADY + 2
};
static_assert(B_COUNT == 2 * kStages + 2 + 2 + 6 + 2, "barrier slots overlap");

// Per-variant layout.  NM = 24: the pre pass (24 mixes); NM = 4: hc_head (4
// mixes).  B holds fn hi in rows [0, NM), fn lo in [NM, 2 NM), zero padding
// up to the MMA's N (a multiple of 16).  Shared memory offsets are from a
// 1024-byte aligned base.
template <int NM>
struct Cfg {
  static constexpr int kN = (2 * NM + 15) / 16 * 16;           // 48 / 16
  static constexpr int kFnBlkBytes = kN * kBk * 2;               // 6144 / 2048
  static constexpr int kRw = (NM + 1 + 3) / 4 * 4;               // NM dots, sum x^2, pad
  static constexpr int kOffFn = 0;
  static constexpr int kOffStage = kOffFn + kKb * kFnBlkBytes;
  static constexpr int kOffRecv = kOffStage + kStages * kStageBytes;   // [16 src][8 rows][kRw]
  static constexpr int kOffRed = kOffRecv + kCl * kOwn * kRw * 4;      // [8 rows][kRw]
  static constexpr int kOffSs = kOffRed + kOwn * kRw * 4;              // [2][128 rows] sum x^2
  static constexpr int kOffBar = kOffSs + 2 * kTile * 4;
  static constexpr int kOffMisc = kOffBar + B_COUNT * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // slack to align the base
  // instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, N, M = 128
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kTile >> 4) << 24);
  static_assert(NM == kMix || NM == kHeadMix, "two variants");
  static_assert(kN <= 64, "an accumulator holds 64 columns");
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
  static_assert(kOffStage % 1024 == 0 && kFnBlkBytes % 1024 == 0, "SW128 tiles need 1024-B alignment");
  static_assert(kOffRecv % 16 == 0 && (kRw * 4) % 16 == 0, "receive rows must take 16-byte stores");
  static_assert(NM % 4 == 0 && (2 * NM) % 8 == 0, "pushes of 4 mixes; padding starts on an 8-row group");
};

// fn's 8 consecutive k of mix c -> the bf16 hi and lo halves (hi = bf16(f),
// lo = bf16(f - hi), both round-to-nearest-even), written as two 16-byte
// chunks q of B-tile rows c and c + NM (K-major, 128-byte swizzle).  The
// stats kernel's loaders and the prepared-weights image use this one routine,
// so both give the same bits.
template <int NM>
__device__ __forceinline__ void fn_item_to_tile(const float4 &f0, const float4 &f1, int c, int q,
                                                uint8_t *tile) {
  const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * e]);
    const __nv_bfloat16 h1 = __float2bfloat16_rn(f[2 * e + 1]);
    hw[e] = pack2_rn(__bfloat162float(h0), __bfloat162float(h1));
    lw[e] = pack2_rn(f[2 * e] - __bfloat162float(h0), f[2 * e + 1] - __bfloat162float(h1));
  }
  const int nh = c, nlo = c + NM;
  *reinterpret_cast<uint4 *>(tile + (nh >> 3) * 1024 + (nh & 7) * 128 + ((q ^ (nh & 7)) << 4)) =
      make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4 *>(tile + (nlo >> 3) * 1024 + (nlo & 7) * 128 + ((q ^ (nlo & 7)) << 4)) =
      make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

struct StatsArgs {
  const float *fn;
  const uint8_t *fn_img;   // pre pass only, or NULL: fn already in this kernel's B-tile image
  const float *scale;
  const float *base;
  float *pre_ws;     // [rows, 4] pre gates for the combine launch
  float *post;       // pre pass only
  float *logit_ws;   // pre pass only: [rows, 16] comb logits for the combine launch
  float *pre_out;
  float *mix_out;
  int64_t rows;
  int num_tiles;
  float rms_eps, pre_eps, sink_eps, post_mult;
  int iters;
};

template <int NM>
__global__ void __launch_bounds__(kThreads, 1)
pre_stats_kernel(const __grid_constant__ CUtensorMap tmap, const StatsArgs a) {
  using C = Cfg<NM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;   // our tiles
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kOffMisc);
  Abort ab{reinterpret_cast<volatile int *>(sm + C::kOffMisc + 4), crank, &g_fused_error,
           g_fused_where, g_fused_where_aborted};

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *ab.flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1 + kRowN);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_TFULL + b), 1);
      mbar_init(bar(B_TEMPTY + b), kReadN);
      mbar_init(bar(B_SSREADY + b), kRowN);
    }
    mbar_init(bar(B_PREADY), kCl);
    mbar_init(bar(B_PFREE), kCl);
    mbar_init(bar(B_GALL), kReadN);
    mbar_init(bar(B_OPULL), kOwnerN);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_FNREADY), a.fn_img ? 1 : kWarps - 1 - kRowN);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  // fn columns of this CTA -> bf16 hi/lo B tiles (K-major, 128-byte swizzle),
  // written by the MMA, readout and owner warps while the producer starts
  // streaming R and the row warps wait for it:
  // k-block j covers k = (j%4)*5120 + 320*crank + 64*(j/4) + [0, 64)
  // With prepared weights the same bytes come from the image, in four bulk
  // copies.
  if (a.fn_img) {
    if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t kImg = kKb * C::kFnBlkBytes, kPart = kImg / 4;
      static_assert(kImg % 64 == 0 && kImg < (1u << 20), "bulk copies of 16-byte multiples");
      mbar_expect_tx(bar(B_FNREADY), kImg);
      const uint8_t *src = a.fn_img + (size_t)crank * kImg;
      for (int i = 0; i < 4; ++i)
        bulk_load(sb + C::kOffFn + i * kPart, src + i * kPart, kPart, bar(B_FNREADY));
    }
  } else if (warp != kProducerWarp && !(warp >= kRow0 && warp < kRow0 + kRowN)) {
    // 10 loader warps; loads of 8 items are issued before any is converted
    const int loader = warp == kMmaWarp ? 0 : (warp < kRow0 ? warp - 1 : warp - kRowN - 1);
    const int lt = loader * 32 + lane, nl = (kWarps - 1 - kRowN) * 32;
    if constexpr (C::kN > 2 * NM) {
      // zero the padding rows [2 NM, kN) of every k-block (whole 8-row groups)
      constexpr int kPadRows = C::kN - 2 * NM, kPadChunks = kKb * kPadRows * 8;
      for (int i = lt; i < kPadChunks; i += nl) {
        const int j = i / (kPadRows * 8), r = 2 * NM + (i >> 3) % kPadRows, q = i & 7;
        *reinterpret_cast<uint4 *>(sm + C::kOffFn + j * C::kFnBlkBytes + (r >> 3) * 1024 +
                                   (r & 7) * 128 + (q << 4)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    constexpr int kItems = NM * kKb * 8;       // items of 8 consecutive k (3840 for 24 mixes)
    for (int base = lt; base < kItems; base += 8 * nl) {
      float4 f0[8], f1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int item = base + u * nl;
        if (item < kItems) {
          const int q = item & 7, j = (item >> 3) % kKb, c = item / (8 * kKb);
          const int k0 = (j & 3) * kH + (int)crank * kHs + (j >> 2) * kBk + 8 * q;
          f0[u] = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + k0));
          f1[u] = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + k0 + 4));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int item = base + u * nl;
        if (item >= kItems) continue;
        const int q = item & 7, j = (item >> 3) % kKb, c = item / (8 * kKb);
        fn_item_to_tile<NM>(f0[u], f1[u], c, q, sm + C::kOffFn + j * C::kFnBlkBytes);
      }
    }
    // generic-proxy writes -> visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_FNREADY));
  }

  // ---- roles -------------------------------------------------------------------
  if (warp == kProducerWarp) {
    // the whole warp walks the loop (waits are warp-collective); lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    int last[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last[s] = -1;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int y = (cid + it * ncl) * kTile;
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_EMPTY + stage), phase ^ 1, false, ab, 1, it)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(bar(B_FULL + stage), kStageBytes);
          const int x = (j & 3) * kH + (int)crank * kHs + (j >> 2) * kBk;
          tma_load_2d(sb + C::kOffStage + stage * kStageBytes, &tmap, x, y, bar(B_FULL + stage));
        }
        __syncwarp();
        last[stage] = (int)phase;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    // every copy issued must have landed before the CTA may exit
    for (int s = 0; s < kStages; ++s)
      if (last[s] >= 0) drain1(bar(B_FULL + s), (uint32_t)last[s]);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    int stage = 0;
    uint32_t phase = 0;
    bool ok = waitw(bar(B_FNREADY), 0, false, ab, 0, 0);
    for (int it = 0; it < T && ok; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!waitw(bar(B_TEMPTY + buf), (use & 1) ^ 1, false, ab, 2, it)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * 64);
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_FULL + stage), phase, false, ab, 3, it)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t ad = sw128_desc(sb + C::kOffStage + stage * kStageBytes);
          const uint64_t bd = sw128_desc(sb + C::kOffFn + j * C::kFnBlkBytes);
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk)
            tc_mma(d, ad + 2 * kk, bd + 2 * kk, C::kIdesc, (j | kk) != 0);
          tc_commit(bar(B_EMPTY + stage));
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(B_TFULL + buf));
      __syncwarp();
    }
    // all issued MMAs complete before TMEM is freed
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    // the fn image copies have landed before the CTA may leave
    if (a.fn_img) drain1(bar(B_FNREADY), 0);
    __syncwarp();
  } else if (warp >= kRow0 && warp < kRow0 + kRowN) {
    // ---- row warps: one thread per tile row; sum x^2 from every stage -------
    const int row = 32 * (warp & 3) + lane;     // tile row
    const int sw = row & 7;
    float *ssbuf = reinterpret_cast<float *>(sm + C::kOffSs);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      // one accumulator per 16-byte chunk of the 128-byte row slice, one add
      // per stage of that chunk's 8 squares (short chains, summed in a fixed
      // tree at the end)
      float ssq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) ssq[q] = 0.f;
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_FULL + stage), phase, false, ab, 4, it)) { ok = false; break; }
        const uint8_t *st = sm + C::kOffStage + stage * kStageBytes + row * 128;
        uint4 cq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) cq[q] = *reinterpret_cast<const uint4 *>(st + ((q ^ sw) << 4));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          // the chunk's 8 squares in a short chain, then one add per stage
          const uint32_t w4[4] = {cq[q].x, cq[q].y, cq[q].z, cq[q].w};
          float c8 = lo_bf(w4[0]) * lo_bf(w4[0]);
          c8 = fmaf(hi_bf(w4[0]), hi_bf(w4[0]), c8);
#pragma unroll
          for (int e = 1; e < 4; ++e) {
            c8 = fmaf(lo_bf(w4[e]), lo_bf(w4[e]), c8);
            c8 = fmaf(hi_bf(w4[e]), hi_bf(w4[e]), c8);
          }
          ssq[q] += c8;
        }
        // the stage is released only after every lane has used its data
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + stage));
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      // hand the row's sum x^2 to the readout warps (slot free once tile it-2
      // was read out)
      const int buf = it & 1;
      if (!waitw(bar(B_TEMPTY + buf), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 10, it)) break;
      const float ss = ((ssq[0] + ssq[1]) + (ssq[2] + ssq[3])) + ((ssq[4] + ssq[5]) + (ssq[6] + ssq[7]));
      ssbuf[buf * kTile + row] = ss;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SSREADY + buf));
    }
  } else if (warp >= kRead0 && warp < kRead0 + kReadN) {
    // ---- readout warps: one thread per tile row (= TMEM lane) ---------------
    // accumulator + sum x^2 of tile t -> the owner CTA's receive buffer
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = 32 * quarter + lane;
    const float *ssbuf = reinterpret_cast<const float *>(sm + C::kOffSs);
    for (int t = 0; t < T; ++t) {
      const int buf = t & 1;
      const uint32_t use = (uint32_t)(t >> 1);
      if (!waitw(bar(B_TFULL + buf), use & 1, false, ab, 5, t)) break;
      if (!waitw(bar(B_SSREADY + buf), use & 1, false, ab, 11, t)) break;
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * 64);
      float mix[NM];                            // hi + lo of the NM dots
      float ss;
      if constexpr (NM == kMix) {
        float a0[16], a1[16], a2[16];           // columns 0..47: hi 0..23, lo 24..47
        tc_ld16(ta + 0, a0);
        tc_ld16(ta + 16, a1);
        tc_ld16(ta + 32, a2);
        tc_wait_ld();
        ss = ssbuf[buf * kTile + row];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TEMPTY + buf));
#pragma unroll
        for (int c = 0; c < 8; ++c) mix[c] = a0[c] + a1[c + 8];
#pragma unroll
        for (int c = 8; c < 16; ++c) mix[c] = a0[c] + a2[c - 8];
#pragma unroll
        for (int c = 16; c < 24; ++c) mix[c] = a1[c - 16] + a2[c - 8];
      } else {
        float a0[16];                           // columns 0..NM-1 hi, NM..2NM-1 lo
        tc_ld16(ta + 0, a0);
        tc_wait_ld();
        ss = ssbuf[buf * kTile + row];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TEMPTY + buf));
#pragma unroll
        for (int c = 0; c < NM; ++c) mix[c] = a0[c] + a0[c + NM];
      }
      // slot [our rank][row % 8] of the owner CTA (row / 8)
      if (!waitw(bar(B_PFREE), (uint32_t)(t & 1) ^ 1, true, ab, 6, t)) break;
      const uint32_t dm = mapa(sb + C::kOffRecv + (uint32_t)(((crank * kOwn + (row & 7)) * C::kRw) * 4),
                               (uint32_t)(row >> 3));
#pragma unroll
      for (int v = 0; v < NM / 4; ++v)
        st_cluster_v4(dm + 16 * v, mix[4 * v], mix[4 * v + 1], mix[4 * v + 2], mix[4 * v + 3]);
      st_cluster_f32(dm + 4 * NM, ss);
      // make the stores visible cluster-wide, then count this warp in
      fence_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_GALL));
      if (warp == kRead0) {
        // all readout warps pushed tile t: tell all 16 owners
        if (!waitw(bar(B_GALL), (uint32_t)(t & 1), false, ab, 7, t)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PREADY), kCl);
        __syncwarp();
      }
    }
  } else {
    // ---- owner warps: finalise 8 rows of each tile --------------------------
    const int o = owner_index(warp) * 32 + lane;   // 0..127
    const int q = o >> 4, e = o & 15;           // row of 8, lane of 16
    const int row_t = (int)crank * kOwn + q;
    const float *recv = reinterpret_cast<const float *>(sm + C::kOffRecv);
    float *red = reinterpret_cast<float *>(sm + C::kOffRed);
    // the pre pass reads scale[3] and base[24]; hc_head scale[1] and base[4]
    const float sc0 = __ldg(a.scale);
    const float sc1 = NM == kMix ? __ldg(a.scale + 1) : 0.f;
    const float sc2 = NM == kMix ? __ldg(a.scale + 2) : 0.f;
    const float bcomb = NM == kMix ? __ldg(a.base + 8 + e) : 0.f;
    const float bgate = e < (NM == kMix ? 8 : kHC) ? __ldg(a.base + e) : 0.f;
    const unsigned full = 0xffffffffu;          // a row's 16 lanes are half the warp
    const int gb = lane & 16;
    for (int it = 0; it < T; ++it) {
      const int64_t grow = (int64_t)(cid + it * ncl) * kTile + row_t;
      if (!waitw(bar(B_PREADY), (uint32_t)(it & 1), true, ab, 8, it)) break;
      // this row's 25 partials from the 16 CTAs, summed in CTA order
      float acc0 = 0.f, acc1 = 0.f;
      if (e <= NM) {
#pragma unroll
        for (int src = 0; src < kCl; ++src) acc0 += recv[(src * kOwn + q) * C::kRw + e];
      }
      if (e + 16 <= NM) {
#pragma unroll
        for (int src = 0; src < kCl; ++src) acc1 += recv[(src * kOwn + q) * C::kRw + e + 16];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OPULL));
      if (warp == kOwnerLead) {
        if (!waitw(bar(B_OPULL), (uint32_t)(it & 1), false, ab, 9, it)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PFREE), kCl);
        __syncwarp();
      }
      float *rq = red + q * C::kRw;
      if (e <= NM) rq[e] = acc0;
      if (e + 16 <= NM) rq[e + 16] = acc1;
      __syncwarp();
      const float rsq = 1.0f / sqrtf(rq[NM] / (float)kK + a.rms_eps);
      if constexpr (NM == kHeadMix) {
        // hc_head: lanes 0..3 hold pre_i = sigmoid(mix_i * scale + base_i) + hc_eps
        if (grow < a.rows && e < kHC) {
          const float mx = rq[e] * rsq;
          const float sg = 1.0f / (1.0f + expf(-fmaf(mx, sc0, bgate)));
          a.pre_ws[grow * kHC + e] = sg + a.pre_eps;
          if (a.pre_out) a.pre_out[grow * kHC + e] = sg + a.pre_eps;
          if (a.mix_out) a.mix_out[grow * NM + e] = mx;
        }
        (void)sc1; (void)sc2; (void)bcomb; (void)full;
      } else {
        // gates: lanes 0..3 pre, 4..7 post; lane e's comb logit (the combine
        // launch runs the Sinkhorn on them)
        float gate = 0.f;
        if (e < 8) {
          const float l = fmaf(rq[e] * rsq, e < 4 ? sc0 : sc1, bgate);
          const float sg = 1.0f / (1.0f + expf(-l));
          gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
        }
        const float lc = fmaf(rq[8 + e] * rsq, sc2, bcomb);
        if (grow < a.rows) {
          a.logit_ws[grow * 16 + e] = lc;
          if (e < 4) a.pre_ws[grow * kHC + e] = gate;
          if (e >= 4 && e < 8) a.post[grow * kHC + (e - 4)] = gate;
          if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
          if (a.mix_out) {
            a.mix_out[grow * NM + e] = rq[e] * rsq;
            if (e < 8) a.mix_out[grow * NM + 16 + e] = rq[16 + e] * rsq;
          }
        }
        (void)full;
      }
      (void)gb;
      __syncwarp();
    }
  }

  // this CTA's work is done: the next launch may start scheduling (earlier,
  // its waiting CTAs would sit beside this persistent grid for its whole run)
  pdl_trigger();

  // ---- teardown: no CTA leaves while its shared memory may still be addressed
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  __syncwarp();
  cluster_sync_all();
}

// ---- host side -------------------------------------------------------------------
constexpr int kMaxDev = 64;
std::mutex g_dev_mu;
template <int NM>
int g_max_clusters[kMaxDev];   // 0: not yet configured on that device

template <int NM>
cudaError_t configure(int dev, int *max_clusters) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_max_clusters<NM>[dev] > 0) {
    *max_clusters = g_max_clusters<NM>[dev];
    return cudaSuccess;
  }
  constexpr int kSmemBytes = Cfg<NM>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(pre_stats_kernel<NM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pre_stats_kernel<NM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  cfg.gridDim = dim3(kCl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, pre_stats_kernel<NM>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_max_clusters<NM>[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

template <int NM>
cudaError_t launch_stats(const uint16_t *R, const StatsArgs &a, int64_t logical_rows,
                         cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  int max_clusters = 0;
  e = configure<NM>(dev, &max_clusters);
  if (e != cudaSuccess) return e;

  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)kK, (cuuint64_t)a.rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)kK * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBk, (cuuint32_t)kTile};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(R), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // grid: as many clusters as fit at once, never more than the whole chunk's
  // tiles (the count depends on logical_rows only; per-row arithmetic does not
  // depend on it at all)
  const int64_t chunk_tiles = (logical_rows + kTile - 1) / kTile;
  const int clusters = (int)(chunk_tiles < max_clusters ? chunk_tiles : max_clusters);

  return launch_pdl(pre_stats_kernel<NM>, dim3((unsigned)(clusters * kCl)), dim3(kThreads),
                    Cfg<NM>::kSmemBytes, s, kCl, use_pdl(logical_rows), map, a);
}

}  // namespace

// ---- prepared weights: fn's B-tile image of every cluster rank ---------------------
namespace {
constexpr int kImgRankBytes = kKb * Cfg<kMix>::kFnBlkBytes;      // 122880
constexpr int kImgItemsPerRank = kMix * kKb * 8;                  // 3840 items of 8 k

__global__ void __launch_bounds__(256) fn_img_prep_kernel(const float *__restrict__ fn,
                                                          uint8_t *__restrict__ img) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 256 + threadIdx.x;
  if (t >= kCl * kImgItemsPerRank) return;
  const int rank = t / kImgItemsPerRank, item = t % kImgItemsPerRank;
  const int q = item & 7, j = (item >> 3) % kKb, c = item / (8 * kKb);
  const int k0 = (j & 3) * kH + rank * kHs + (j >> 2) * kBk + 8 * q;
  const float4 f0 = __ldg(reinterpret_cast<const float4 *>(fn + (int64_t)c * kK + k0));
  const float4 f1 = __ldg(reinterpret_cast<const float4 *>(fn + (int64_t)c * kK + k0 + 4));
  fn_item_to_tile<kMix>(f0, f1, c, q,
                        img + (size_t)rank * kImgRankBytes + j * Cfg<kMix>::kFnBlkBytes);
}
}  // namespace

size_t fn_img_bytes() { return (size_t)kCl * kImgRankBytes; }

cudaError_t launch_fn_img_prep(const float *fn, uint8_t *img, cudaStream_t s) {
  constexpr int kItems = kCl * kImgItemsPerRank;
  return launch_pdl(fn_img_prep_kernel, dim3((kItems + 255) / 256), dim3(256), 0, s, 1, false,
                    fn, img);
}

cudaError_t launch_pre_stats(const uint16_t *R, const float *fn, const uint8_t *fn_img,
                             const float *scale, const float *base, int64_t rows,
                             int64_t logical_rows, const mhc_params &p, float *pre_ws,
                             float *logit_ws, float *post, float *pre_out, float *mix_out,
                             cudaStream_t s) {
  StatsArgs a;
  a.fn = fn; a.fn_img = fn_img; a.scale = scale; a.base = base; a.pre_ws = pre_ws;
  a.post = post; a.logit_ws = logit_ws; a.pre_out = pre_out; a.mix_out = mix_out;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTile - 1) / kTile);
  a.rms_eps = p.rms_eps; a.pre_eps = p.hc_pre_eps; a.sink_eps = p.hc_sinkhorn_eps;
  a.post_mult = p.post_mult; a.iters = p.sinkhorn_iters;
  return launch_stats<kMix>(R, a, logical_rows, s);
}

cudaError_t launch_head_stats(const uint16_t *R, const float *fn, const float *scale,
                              const float *base, int64_t rows, int64_t logical_rows,
                              float norm_eps, float hc_eps, float *pre_ws, float *pre_out,
                              float *mix_out, cudaStream_t s) {
  StatsArgs a;
  a.fn = fn; a.fn_img = nullptr; a.scale = scale; a.base = base; a.pre_ws = pre_ws;
  a.post = nullptr; a.logit_ws = nullptr; a.pre_out = pre_out; a.mix_out = mix_out;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTile - 1) / kTile);
  a.rms_eps = norm_eps; a.pre_eps = hc_eps; a.sink_eps = 0.f; a.post_mult = 0.f; a.iters = 0;
  return launch_stats<kHeadMix>(R, a, logical_rows, s);
}

cudaError_t fused_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fused_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_fused_error, &z, sizeof z);
  }
  return e;
}

cudaError_t fused_error_where(unsigned int *out64) {
  cudaError_t e = cudaMemcpyFromSymbol(out64, g_fused_where, 32 * sizeof(unsigned int));
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbol(out64 + 32, g_fused_where_aborted, 32 * sizeof(unsigned int));
  return e;
}

}  // namespace mhc
