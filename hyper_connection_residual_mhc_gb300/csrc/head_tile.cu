// head_tile.cu -- mhc_hc_head in one launch that reads R from HBM once and
// combines every row from shared memory: the model's final collapse of the 4
// residual streams into one hidden vector per row, for chunks above the size
// that head_onepass.cu serves.
//
// Definition: deepseek_v4.py (sglang), hc_head_torch: mixes = (x @ fn^T) *
// rsqrt(mean(x^2) + norm_eps) on the flattened row x (4 x 5120,
// stream-major), pre_i = sigmoid(mix_i * scale + base_i) + hc_eps,
// y = sum_i pre_i R_i, cast once to bf16.
//
// With 4 mixes fn's operand tiles take 40 KB of shared memory per CTA, so
// the rest holds a ring deep enough to keep each tile until its gates have
// come back: the combine reads the tile from shared memory, not again from
// L2 or HBM.
//
// Decomposition.  A cluster of 8 CTAs owns a 16-row tile at a time; CTA s
// owns hidden columns [640 s, 640 s + 640) of all four streams.
//   * warp 0 streams the tile through an 11-stage ring with TMA: a stage is
//     two 64-column blocks (2 p, 2 p + 1), each a 3-D box (columns, streams,
//     rows) of 8 KB, landing as lines 64 h + 4 r + i (block 2 p + h, stream i
//     of tile row r), 128-byte swizzled;
//   * one thread of warp 1 issues tcgen05.mma with the stage as A (M = 128)
//     and fn's bf16 hi and lo for both blocks as B (N = 64: for block half h
//     and stream j, the hi and lo rows of mix c at 32 h + 8 j + 2 c and
//     32 h + 8 j + 2 c + 1), resident in shared memory; D[64 h + 4 r + i]
//     [32 h' + 8 j + n] accumulates over the tile's five stages in tensor
//     memory, and only the h' = h, j = i blocks are used;
//   * four sum-of-squares warps (one thread per line) add the squares of
//     each stage's lines in packed fp32 pairs;
//   * four readout warps (lane quarter q: half q / 2, rows 8 (q % 2) ..)
//     take each line's own block of the accumulator, add hi + lo, sum the
//     four streams of a row in a fixed order, and send each row's 4 dots and
//     sum of squares over that half's columns to the CTA that finalises the
//     row (CTA s owns tile rows 2 s, 2 s + 1): 16 records a row;
//   * the owner warp sums the 16 records in (CTA, half) order, forms rsqrt,
//     the mixes and the 4 gates, and sends the gates to all 8 CTAs;
//   * eight combine warps, once a tile's gates are in, form y from the
//     tile's stages in shared memory stage by stage, freeing each stage as
//     soon as its values are in registers, and write y.
// The exchanges are asynchronous remote stores (st.async) counted in bytes on
// the receiver's mbarrier.  The pushes of tile t wait until this CTA's
// combine has read the gates of tile t - 2 (every owner has then consumed
// the receive buffer tile t reuses, and this CTA's gate buffer for tile t is
// free).
//
// Every row is reduced in one fixed order that depends only on its own data,
// so any row range gives the whole-chunk bits.  Every wait is bounded (~2 s);
// on expiry a CTA raises an abort flag, records the site in its error word,
// drains its copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>

#include <mutex>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

__device__ unsigned int g_htile_error;
__device__ unsigned int g_htile_where[32];
__device__ unsigned int g_htile_where_aborted[32];

namespace {
using namespace ptx;

// ---- geometry -------------------------------------------------------------
constexpr int kCl = 8;                         // CTAs per cluster (K split)
constexpr int kHs = kH / kCl;                  // 640 hidden columns per CTA
constexpr int kBk = 64;                        // hidden columns per box (128-byte rows)
constexpr int kHb = kHs / kBk;                 // 10 blocks per tile
constexpr int kHalves = 2;                     // blocks per stage: lines 64 h + 4 r + i
constexpr int kSt = kHb / kHalves;             // 5 stages per tile
constexpr int kTR = 16;                        // rows per tile
constexpr int kM = kHalves * kHC * kTR;        // 128: MMA M
constexpr int kOwn = kTR / kCl;                // 2 rows finalised per CTA per tile
constexpr int kHalfBytes = kHC * kTR * kBk * 2;     // 8192: one block of a tile
constexpr int kStageBytes = kHalves * kHalfBytes;   // 16384
constexpr int kStages = 11;
constexpr int kMixes = kHC;                    // hc_head: one mix per stream
constexpr int kFnRowsPerStream = 2 * kMixes;   // 8: hi and lo of 4 mixes, interleaved
constexpr int kNh = kHC * kFnRowsPerStream;    // 32: fn rows of one half
constexpr int kN = kHalves * kNh;              // 64: MMA N (half h at 32 h)
constexpr int kFnBlkBytes = kN * kBk * 2;      // 8192: fn's B tile for one stage
constexpr int kDCols = kN;                     // accumulator columns per buffer
constexpr int kTmemCols = 128;
constexpr int kRec = 8;                        // pushed record: 4 dots, sum x^2, 3 pad
constexpr int kSrc = kCl * kHalves;            // records per row: one per CTA and half
constexpr int kNR = 2, kNG = 2;                // receive and gate buffers

static_assert(kHb % kHalves == 0 && kTR % kCl == 0 && kOwn == 2 && kM == 128, "");
static_assert(2 * kDCols <= kTmemCols, "two accumulators fit in tensor memory");
static_assert(kStages >= 2 * kSt, "the ring holds the tile being combined and the next one");

// ---- warp roles -------------------------------------------------------------
constexpr int kProducerWarp = 0, kMmaWarp = 1, kOwnerWarp = 2;
constexpr int kRead0 = 4, kReadN = 4;          // warp & 3 = lane quarter
constexpr int kSq0 = 8, kSqN = 4;              // line 32 (warp - 8) + lane
// combine warps: 3 and 12..18
__device__ __forceinline__ int comb_index(int w) { return w == 3 ? 0 : w - 11; }
constexpr int kCombN = 8, kComb0 = 3;          // kComb0 re-arms the gate barrier
constexpr int kWarps = 19;
constexpr int kThreads = kWarps * 32;          // 608
constexpr int kCombT = kCombN * 32;            // 256
static_assert(kRead0 % 4 == 0 && kCombT == kHalves * kTR * (kBk / 8), "one (half, row, chunk) of a stage per combine thread");

// 96 registers a thread: warp w runs on SM sub-partition w % 4, whose 16 K
// registers are allocated to a warp in units of 512; 5 warps x 3072 fit
constexpr int kMaxRegs = 96;
static_assert((kWarps + 3) / 4 * ((kMaxRegs * 32 + 511) / 512 * 512) <= 16384,
              "register budget of each SM sub-partition with one block per SM");

enum Bar : int {
  B_FULL = 0,                     // [kStages] TMA landed
  B_EMPTY = B_FULL + kStages,     // [kStages] MMA, squares and combine done with the stage
  B_DFULL = B_EMPTY + kStages,    // [2] dot accumulator complete
  B_DEMPTY = B_DFULL + 2,         // [2] dot accumulator read out
  B_SFULL = B_DEMPTY + 2,         // [2] a tile's sums of squares written
  B_SEMPTY = B_SFULL + 2,         // [2] a tile's sums of squares read
  B_RX = B_SEMPTY + 2,            // [kNR] the 16 records of each owned row landed (bytes)
  B_GIN = B_RX + kNR,             // [kNG] the 8 owners' gates landed (bytes)
  B_GREAD = B_GIN + kNG,          // [kNG] the combine warps have read the tile's gates
  B_FNREADY = B_GREAD + kNG,      // fn's B tiles written
  B_DRAIN = B_FNREADY + 1,        // final MMA drain
  B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT == 2 * kStages + 8 + kNR + 2 * kNG + 2, "barrier slots overlap");

struct Cfg {
  static constexpr int kOffFn = 0;                                    // [5 stages][64][64] bf16
  static constexpr int kOffStage = kOffFn + kSt * kFnBlkBytes;        // [11][128][64] bf16
  static constexpr int kOffRx = kOffStage + kStages * kStageBytes;    // [kNR][16 src][2 rows][8]
  static constexpr int kRxBytes = kSrc * kOwn * kRec * 4;
  static constexpr int kOffGin = kOffRx + kNR * kRxBytes;             // [kNG][16 rows][4]
  static constexpr int kGinBytes = kTR * kHC * 4;
  static constexpr int kOffSs = kOffGin + kNG * kGinBytes;            // [2][2 halves][16 rows] sum x^2
  static constexpr int kOffBar = kOffSs + 2 * kHalves * kTR * 4;
  static constexpr int kOffMisc = kOffBar + B_COUNT * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;             // slack to align the base
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
  static_assert(kOffStage % 1024 == 0 && kFnBlkBytes % 1024 == 0, "SW128 tiles need 1024-B alignment");
  static_assert(kOffRx % 16 == 0 && kOffGin % 16 == 0 && kOffBar % 8 == 0, "alignment");
};

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// M = 128, N = 64
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kM >> 4) << 24);

// byte offset of 16-byte chunk c of line l in a [lines][64] bf16 SW128 tile
__device__ __forceinline__ int sw128_off(int l, int c) {
  return (l >> 3) * 1024 + (l & 7) * 128 + ((c ^ (l & 7)) << 4);
}

struct HeadTileArgs {
  const uint16_t *R;
  const float *fn, *scale, *base;
  uint16_t *y;
  float *pre_out, *mix_out;
  int64_t rows;
  int num_tiles;
  float norm_eps, hc_eps;
};

__global__ void __maxnreg__(kMaxRegs)
head_tile_kernel(const __grid_constant__ CUtensorMap tmap, const HeadTileArgs a) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;   // our tiles
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)i; };
  auto stage_addr = [&](int s) -> uint32_t { return sb + C::kOffStage + (uint32_t)(s * kStageBytes); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kOffMisc);
  Abort ab{reinterpret_cast<volatile int *>(sm + C::kOffMisc + 4), crank, &g_htile_error,
           g_htile_where, g_htile_where_aborted};
  // a push of tile t waits until this CTA's combine has read the gates of
  // tile t - 2
  auto push_ready = [&](int t, int site) -> bool {
    if (t < kNG) return true;
    const int tr = t - kNG;
    return waitw(bar(B_GREAD + tr % kNG), (uint32_t)((tr / kNG) & 1), false, ab, site, t);
  };

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *ab.flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1 + kSqN + kCombN);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_DFULL + b), 1);
      mbar_init(bar(B_DEMPTY + b), kReadN);
      mbar_init(bar(B_SFULL + b), kSqN);
      mbar_init(bar(B_SEMPTY + b), kReadN);
    }
    for (int b = 0; b < kNG; ++b) {
      mbar_init(bar(B_GIN + b), 1);
      mbar_init(bar(B_GREAD + b), kCombN);
    }
    for (int b = 0; b < kNR; ++b) mbar_init(bar(B_RX + b), 1);
    mbar_init(bar(B_FNREADY), kCombN);
    mbar_init(bar(B_DRAIN), 1);
    for (int b = 0; b < kNR; ++b) mbar_expect_tx(bar(B_RX + b), C::kRxBytes);
    for (int b = 0; b < kNG; ++b) mbar_expect_tx(bar(B_GIN + b), C::kGinBytes);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  const bool is_comb = warp == 3 || (warp >= 12 && warp < kWarps);
  if (is_comb) {
    // fn's B tiles for this CTA's columns: 8 k of mix c, stream j, block b ->
    // bf16 hi into row 8 j + 2 c, lo = bf16(f - hi) into row 8 j + 2 c + 1
    const int t = comb_index(warp) * 32 + lane;
    for (int item = t; item < kHb * kHC * kMixes * 8; item += kCombT) {
      const int q = item & 7, c = (item >> 3) % kMixes, j = (item / (8 * kMixes)) % kHC,
                b = item / (8 * kMixes * kHC);          // block b = 2 stage + half
      const float4 *src = reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + j * kH +
                                                           (int)crank * kHs + b * kBk + 8 * q);
      const float4 f0 = __ldg(src), f1 = __ldg(src + 1);
      const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float h0 = __bfloat162float(__float2bfloat16_rn(f[2 * e]));
        const float h1 = __bfloat162float(__float2bfloat16_rn(f[2 * e + 1]));
        hw[e] = pack2_rn(h0, h1);
        lw[e] = pack2_rn(f[2 * e] - h0, f[2 * e + 1] - h1);
      }
      uint8_t *tile = sm + C::kOffFn + (b / kHalves) * kFnBlkBytes;
      const int nh = kNh * (b % kHalves) + kFnRowsPerStream * j + 2 * c;
      *reinterpret_cast<uint4 *>(tile + sw128_off(nh, q)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(tile + sw128_off(nh + 1, q)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    // generic-proxy writes -> visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_FNREADY));
  }

  if (warp == kProducerWarp) {
    // ---- producer ---------------------------------------------------------------
    int g = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int y = (cid + it * ncl) * kTR;
      for (int b = 0; b < kSt; ++b, ++g) {
        const int s = g % kStages;
        if (!waitw(bar(B_EMPTY + s), (uint32_t)((g / kStages) & 1) ^ 1, false, ab, 1, it)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(bar(B_FULL + s), kStageBytes);
          tma_load_3d(stage_addr(s), &tmap, (int)crank * kHs + 2 * b * kBk, 0, y, bar(B_FULL + s));
          tma_load_3d(stage_addr(s) + kHalfBytes, &tmap, (int)crank * kHs + (2 * b + 1) * kBk, 0, y,
                      bar(B_FULL + s));
        }
        __syncwarp();
      }
    }
    // every copy issued must have landed before the CTA may exit
    for (int s = 0; s < kStages && s < g; ++s) {
      const int g_last = s + ((g - 1 - s) / kStages) * kStages;
      drain1(bar(B_FULL + s), (uint32_t)((g_last / kStages) & 1));
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer -------------------------------------------------------------
    int g = 0;
    bool ok = waitw(bar(B_FNREADY), 0, false, ab, 2, 0);
    tc_fence_after();
    for (int it = 0; it < T && ok; ++it) {
      const int buf = it & 1;
      if (!waitw(bar(B_DEMPTY + buf), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 3, it)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * kDCols);
      for (int b = 0; b < kSt; ++b, ++g) {
        const int s = g % kStages;
        if (!waitw(bar(B_FULL + s), (uint32_t)((g / kStages) & 1), false, ab, 4, it)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t ad = sw128_desc(stage_addr(s));
          const uint64_t bd = sw128_desc(sb + C::kOffFn + b * kFnBlkBytes);
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk)
            tc_mma(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (b | kk) != 0);
          tc_commit(bar(B_EMPTY + s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(B_DFULL + buf));
      __syncwarp();
    }
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp >= kSq0 && warp < kSq0 + kSqN) {
    // ---- sum-of-squares warps: line l = 32 (warp - 8) + lane = 64 h + 4 r + i --
    const int l = 32 * (warp - kSq0) + lane;
    float *ss = reinterpret_cast<float *>(sm + C::kOffSs);
    int g = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      uint64_t acc = 0ull;
      for (int b = 0; b < kSt; ++b, ++g) {
        const int s = g % kStages;
        if (!waitw(bar(B_FULL + s), (uint32_t)((g / kStages) & 1), false, ab, 5, it)) {
          ok = false;
          break;
        }
        const uint8_t *st = sm + C::kOffStage + s * kStageBytes;
        uint4 x[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = *reinterpret_cast<const uint4 *>(st + sw128_off(l, c));
        // the values are in registers once these loads have returned: only
        // then may this warp count itself out of the stage
        uint32_t sink = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) sink |= x[c].x;
        asm volatile("" ::"r"(sink));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + s));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t w4[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t v = f2_of_bf2(w4[k]);
            fma2(acc, v, v);
          }
        }
      }
      if (!ok) break;
      // the row's sum over its four lines, the same bits in all four lanes
      float v = f2_sum(acc);
      v = v + __shfl_xor_sync(0xffffffffu, v, 1);
      v = v + __shfl_xor_sync(0xffffffffu, v, 2);
      const int buf = it & 1;
      if (!waitw(bar(B_SEMPTY + buf), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 6, it)) break;
      if ((l & 3) == 0) ss[(buf * kHalves + (l >> 6)) * kTR + ((l & 63) >> 2)] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFULL + buf));
    }
  } else if (warp >= kRead0 && warp < kRead0 + kReadN) {
    // ---- readout warps: the row's 4 dots and sum of squares to its owner -------
    // lane l of quarter q holds line 32 q + l = 64 h + 4 r + i (h = q / 2);
    // its useful columns are 32 h + 8 i .. 32 h + 8 i + 7
    const int quarter = warp & 3, hq = quarter >> 1;   // half of the stage
    const int i_s = lane & 3, r = 8 * (quarter & 1) + (lane >> 2);
    const float *ss = reinterpret_cast<const float *>(sm + C::kOffSs);
    const unsigned full = 0xffffffffu;
    for (int it = 0; it < T; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!waitw(bar(B_DFULL + buf), use & 1, false, ab, 7, it)) break;
      tc_fence_after();
      float v[32];
      tc_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * kDCols + kNh * hq), v);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DEMPTY + buf));
      float m[kMixes];
#pragma unroll
      for (int c = 0; c < kMixes; ++c) m[c] = 0.f;
#pragma unroll
      for (int j = 0; j < kHC; ++j)
        if (i_s == j) {
#pragma unroll
          for (int c = 0; c < kMixes; ++c)
            m[c] = v[kFnRowsPerStream * j + 2 * c] + v[kFnRowsPerStream * j + 2 * c + 1];
        }
      // the four streams of row r, in lanes 4 (l / 4) .. + 3: (s0 + s1) + (s2 + s3)
#pragma unroll
      for (int c = 0; c < kMixes; ++c) {
        float x = m[c];
        x = x + __shfl_xor_sync(full, x, 1);
        x = x + __shfl_xor_sync(full, x, 2);
        m[c] = x;
      }
      if (!waitw(bar(B_SFULL + buf), use & 1, false, ab, 8, it)) break;
      const float sq = ss[(buf * kHalves + hq) * kTR + r];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SEMPTY + buf));
      if (!push_ready(it, 9)) break;
      if (i_s == 0) {
        const int rb = it % kNR;
        const uint32_t owner = (uint32_t)(r / kOwn);
        const uint32_t dst = mapa(sb + C::kOffRx + (uint32_t)(rb * C::kRxBytes +
                                                              (((int)crank * kHalves + hq) * kOwn + (r % kOwn)) * kRec * 4),
                                  owner);
        const uint32_t rbar = mapa(bar(B_RX + rb), owner);
        st_async_v4(dst, m[0], m[1], m[2], m[3], rbar);
        st_async_v4(dst + 16, sq, 0.f, 0.f, 0.f, rbar);
      }
      __syncwarp();
    }
  } else if (warp == kOwnerWarp) {
    // ---- owner warp: rows 2 crank, 2 crank + 1 of every tile -----------------
    // lane = 16 n + e: row n; lanes e < 5 sum value e of the record
    const int n = lane >> 4, e = lane & 15;
    const int hb = lane & 16;
    const float *rx = reinterpret_cast<const float *>(sm + C::kOffRx);
    const float sc = __ldg(a.scale);
    const float bs = e < kMixes ? __ldg(a.base + e) : 0.f;
    const unsigned full = 0xffffffffu;
    for (int it = 0; it < T; ++it) {
      const int rb = it % kNR;
      const uint32_t use = (uint32_t)(it / kNR);
      const int64_t grow = (int64_t)(cid + it * ncl) * kTR + (int)crank * kOwn + n;
      if (!waitw(bar(B_RX + rb), use & 1, true, ab, 10, it)) break;
      float v = 0.f;
      if (e < kRec) {
#pragma unroll
        for (int src = 0; src < kSrc; ++src)
          v += rx[rb * (C::kRxBytes / 4) + (src * kOwn + n) * kRec + e];
      }
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(B_RX + rb), C::kRxBytes);
      const float sq = __shfl_sync(full, v, hb + kMixes);
      const float rsq = rsqrt_nr(fmaf(sq, 1.0f / (float)kK, a.norm_eps));
      const float mx = v * rsq;
      const float sg = rcp_nr(1.0f + expf(-fmaf(mx, sc, bs)));
      const float gate = sg + a.hc_eps;
      float pg[kHC];
#pragma unroll
      for (int i = 0; i < kHC; ++i) pg[i] = __shfl_sync(full, gate, hb + i);
      // the row's 4 gates to CTA e < kCl (16 bytes counted on its gate barrier)
      if (e < kCl) {
        const uint32_t gbuf = (uint32_t)(it % kNG);
        const uint32_t dst = mapa(sb + C::kOffGin + gbuf * C::kGinBytes +
                                  (uint32_t)(((int)crank * kOwn + n) * kHC * 4),
                                  (uint32_t)e);
        const uint32_t gbar = mapa(bar(B_GIN) + 8u * gbuf, (uint32_t)e);
        st_async_v4(dst, pg[0], pg[1], pg[2], pg[3], gbar);
      }
      if (grow < a.rows && e < kMixes) {
        if (a.pre_out) a.pre_out[grow * kHC + e] = gate;
        if (a.mix_out) a.mix_out[grow * kMixes + e] = mx;
      }
    }
  } else if (is_comb) {
    // ---- combine warps: y of the CTA's columns from the tile's stages --------
    // stage by stage, so each stage is handed back as soon as it is combined:
    // thread t takes half t / 128 (block 2 p + half of stage p), row
    // (t / 8) % 16, chunk t % 8 of that block's 64 columns
    const int t = comb_index(warp) * 32 + lane;
    const int hh = t >> 7, rr = (t >> 3) & (kTR - 1), c8 = t & 7;
    const float *gin = reinterpret_cast<const float *>(sm + C::kOffGin);
    for (int it = 0; it < T; ++it) {
      const int buf = it % kNG;
      if (!waitw(bar(B_GIN + buf), (uint32_t)((it / kNG) & 1), true, ab, 12, it)) break;
      const int g0 = it * kSt;                    // the tile's first stage
      const int64_t grow = (int64_t)(cid + it * ncl) * kTR + rr;
      const float4 pq = *reinterpret_cast<const float4 *>(gin + buf * (kTR * kHC) + rr * kHC);
      const float pv[kHC] = {pq.x, pq.y, pq.z, pq.w};
      // every lane has its gates: the gate buffer is free for tile it + kNG
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_GREAD + buf));
        if (warp == kComb0) mbar_expect_tx(bar(B_GIN + buf), C::kGinBytes);
      }
#pragma unroll 1
      for (int b = 0; b < kSt; ++b) {
        const int s = (g0 + b) % kStages;
        const uint8_t *st = sm + C::kOffStage + s * kStageBytes;
        uint4 rv[kHC];
#pragma unroll
        for (int i = 0; i < kHC; ++i)
          rv[i] = *reinterpret_cast<const uint4 *>(st + sw128_off(64 * hh + 4 * rr + i, c8));
        // the block's values are in registers: hand the stage back
        uint32_t sink = 0;
#pragma unroll
        for (int i = 0; i < kHC; ++i) sink |= rv[i].x;
        asm volatile("" ::"r"(sink));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + s));
        float yv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t sh = (e & 1) ? 0u : 16u;   // bf16 e of the chunk: low half first
          float acc = pv[0] * __uint_as_float(((&rv[0].x)[e >> 1] << sh) & 0xFFFF0000u);
#pragma unroll
          for (int i = 1; i < kHC; ++i)
            acc = fmaf(pv[i], __uint_as_float(((&rv[i].x)[e >> 1] << sh) & 0xFFFF0000u), acc);
          yv[e] = acc;
        }
        if (grow < a.rows)
          st_stream(reinterpret_cast<uint4 *>(a.y + grow * kH + (int64_t)crank * kHs +
                                              (2 * b + hh) * kBk + 8 * c8),
                    pack8_rn(yv));
      }
    }
  }

  pdl_trigger();

  // ---- teardown: no CTA leaves while its shared memory may still be addressed
  tc_fence_before();
  __syncthreads();
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
int g_max_clusters[kMaxDev];   // 0: not yet configured on that device

cudaError_t configure(int dev, int *max_clusters) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_max_clusters[dev] > 0) {
    *max_clusters = g_max_clusters[dev];
    return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(head_tile_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(head_tile_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  cfg.gridDim = dim3(kCl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, head_tile_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_max_clusters[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_head_tile(const uint16_t *R, const float *fn, const float *scale,
                             const float *base, int64_t rows, int64_t logical_rows,
                             float norm_eps, float hc_eps, uint16_t *y, float *pre_out,
                             float *mix_out, cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  int max_clusters = 0;
  e = configure(dev, &max_clusters);
  if (e != cudaSuccess) return e;

  // R as a 3-D tensor (hidden column, stream, row): a box of 64 columns x
  // 4 streams x 16 rows lands with the four streams of a row adjacent
  CUtensorMap map;
  const cuuint64_t gdim[3] = {(cuuint64_t)kH, (cuuint64_t)kHC, (cuuint64_t)rows};
  const cuuint64_t gstride[2] = {(cuuint64_t)kH * 2, (cuuint64_t)kK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBk, (cuuint32_t)kHC, (cuuint32_t)kTR};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(R), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  HeadTileArgs a;
  a.R = R; a.fn = fn; a.scale = scale; a.base = base; a.y = y;
  a.pre_out = pre_out; a.mix_out = mix_out; a.rows = rows;
  a.num_tiles = (int)((rows + kTR - 1) / kTR);
  a.norm_eps = norm_eps; a.hc_eps = hc_eps;
  // grid from the chunk's row count only
  const int64_t chunk_tiles = (logical_rows + kTR - 1) / kTR;
  const int clusters = (int)(chunk_tiles < max_clusters ? chunk_tiles : max_clusters);
  return launch_pdl(head_tile_kernel, dim3((unsigned)(clusters * kCl)), dim3(kThreads),
                    Cfg::kSmemBytes, s, kCl, use_pdl(logical_rows), map, a);
}

cudaError_t head_tile_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_htile_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_htile_error, &z, sizeof z);
  }
  return e;
}

}  // namespace mhc
