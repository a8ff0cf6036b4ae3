// pre_onepass.cu -- all of mhc_pre (stats, gates, Sinkhorn, combine + RMSNorm)
// in one launch that reads the residual R from HBM once.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre:
// hc_pre_torch_impl (rsqrt of mean(x^2) + rms_eps; mixes = (x @ fn^T) * rsqrt),
// hc_split_sinkhorn (pre = sigmoid + hc_pre_eps, post = post_mult * sigmoid,
// the 4x4 Sinkhorn with eps in its denominators) and the combine
// y = sum_i pre_i R_i; the RMSNorm of y fused as prefill_sp.py's
// _combine_norm_fused does it (y kept in fp32, the weight applied before the
// single cast).
//
// Decomposition.  A cluster owns a 32-row tile at a time; CTA s of the
// cluster owns a contiguous range of hidden columns of all four streams.
// Builds (kCl, kS): 16 CTAs of 320 columns (1280 of a row's 20480 k) with
// fn's operand tiles resident in shared memory (no image: converted in the
// kernel); the same with fn's tile of each block streamed from the image into
// the ring stage beside the block of R (an image given, fewer than
// kStreamMinRows rows: no 120 KB copy before the first MMA); and, for chunks
// of kStreamMinRows rows and more with the image, 8 CTAs of 640 columns,
// streamed (the 120 KB of resident fn no longer fill shared memory; 15 such
// clusters fit, 120 SMs, where 7 of 16 hold 112).  All builds of one cluster
// size do the same arithmetic on the same operand bytes: the same bits.
//   * warp 0 streams the tile's R through a 5-stage ring with TMA: a stage is
//     one 64-column block of all four streams, a single 3-D box (columns,
//     streams, rows) that lands as a [128, 64] bf16 tile with the four
//     streams of a row adjacent (tile line 4 r + i is stream i of tile row r),
//     128-byte swizzled.  (Prefetching boxes into L2 one to four ring depths
//     ahead changed nothing measurable and is not done.)
//   * one thread of warp 1 issues tcgen05.mma with that stage as A (M = 128)
//     and fn's bf16 hi/lo for the block as B (N = 192: for each stream j, the
//     hi and lo rows of mix c at 48 j + 2 c and 48 j + 2 c + 1), resident in
//     shared memory or in the stage; D[4 r + i][48 j + n] accumulates over
//     the CTA's blocks in tensor memory, and only the j = i blocks are used.
//   * the same thread issues a second MMA with the stage as both operands
//     (N = 128): D2[4 r + i][4 r' + j] = sum_h R_i[r][h] R_j[r'][h], whose
//     diagonal 4x4 blocks are each row's stream Gram matrix
//     G_ij = sum_h R_i[h] R_j[h] over the CTA's columns.  Its trace is
//     sum x^2, and sum_h y[h]^2 = p^T G p for any gates p, so one cluster
//     exchange carries everything the combine needs.
//   * readout warps (one per tensor-memory lane quarter: 8 tile rows) keep
//     each lane's own stream block of the accumulator, add hi + lo, sum the
//     four streams of a row across its four adjacent lanes in a fixed order,
//     and send each row's 24 partial dots and 10 Gram entries to the CTA
//     that finalises the row (CTA s owns kOwn = 32 / kCl tile rows).
//   * owner warps (one per receive buffer, alternating tiles) sum the
//     cluster's partials in CTA order, form rsqrt, the mixes, the gates, the
//     comb logits and 1/rms(y) = 1/sqrt(p^T G p / 5120 + norm_eps), two rows
//     a pass, broadcast the 4 pre gates and 1/rms(y) of their rows to every
//     CTA of the cluster, write post, and queue the comb logits for the
//     Sinkhorn warp.
//   * both exchanges are asynchronous remote stores (st.async) counted in
//     bytes on the receiver's mbarrier, so neither side fences or signals.
//   * the Sinkhorn warp runs the 4x4 Sinkhorn of 32 queued rows at a time,
//     one row per lane, and writes comb.
//   * combine warps, once a tile's gates are in, read the tile's columns
//     back (from L2: the stats pass read them a few microseconds earlier;
//     non-coherent loads that allocate no L1 line),
//     form y = sum_i pre_i R_i, x_norm = bf16(y / rms(y) * w) (and, in the
//     MXFP8 build, its E4M3 codes and block scales) and store them.
// A stage is freed as soon as its MMAs have completed, so the
// ring only has to cover the copy latency; the combine's second read of R is
// served by L2.  The pushes of tile t wait until the gates of tile t - 2 have
// arrived here (so every owner has consumed that tile's receive buffer) and
// until this CTA's combine has finished with the gates of tile t - 4 (so
// every CTA's gate buffer for tile t is free once all pushes of it are in);
// this also bounds how far the stats run ahead of the combine.
//
// Every row is reduced in one fixed order that depends only on its own data
// (the same MMA sequence for every row, the same lanes, CTA-ordered cross-CTA
// sums), so any row range gives the whole-chunk bits.
//
// Every wait is bounded (~2 s of wall time); on expiry a CTA raises an abort
// flag, records which wait expired, drains its in-flight MMAs and copies,
// frees its tensor memory and returns.
#include <cuda.h>

#include <mutex>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

// Bit s set: a bounded wait at site s expired (g_onepass_where[s] holds
// (tile << 8) | cluster rank of the last one).  Bit 16 + s: a wait at site s
// gave up because its CTA had already aborted.
__device__ unsigned int g_onepass_error;
__device__ unsigned int g_onepass_where[32];
__device__ unsigned int g_onepass_where_aborted[32];

namespace {
using namespace ptx;

// ---- geometry -------------------------------------------------------------
// kCl = 16: a CTA takes 1280 k (320 hidden columns of all four streams);
// fn's operand tiles for them stay resident in shared memory (120 KB) or,
// with kS, stream beside each block of R; 7 such clusters fit, 112 SMs.
// kCl = 8 (always streamed): a CTA takes 2560 k; 15 clusters fit, 120 SMs.
constexpr int kBk = 64;                        // hidden columns per box (128-byte rows)
constexpr int kTR = 32;                        // rows per tile
constexpr int kSlotBytes = kTR * kBk * 2;      // 4096: one stream's box
constexpr int kStageBytes = kHC * kSlotBytes;  // 16384: the four streams of a block
constexpr int kStages = 5;
constexpr int kM = kHC * kTR;                  // 128: MMA M (line 4 r + i)
constexpr int kFnRowsPerStream = 2 * kMix;     // 48: hi and lo of 24 mixes, interleaved
constexpr int kN = kHC * kFnRowsPerStream;     // 192: MMA N
constexpr int kFnBlkBytes = kN * kBk * 2;      // 24576: fn's B tile for one block
constexpr int kDCols = kN;                     // accumulator columns per buffer
constexpr int kD2Col = 2 * kDCols;             // the Gram accumulator (128 columns, one buffer)
constexpr int kTmemCols = 512;
constexpr int kRec = 36;                       // pushed record: 24 dots, 10 Gram, 2 pad
constexpr int kNGram = 10;                     // Gram entries (i <= j)
// the prepared image is laid out for 16 ranks of 5 blocks; rank s of the
// 8-CTA build reads ranks 2 s and 2 s + 1, i.e. blocks 10 s .. 10 s + 9
constexpr int kImgRanks = 16, kImgHs = kH / kImgRanks, kImgHb = kImgHs / kBk;

static_assert(kD2Col + kM <= kTmemCols, "two dot accumulators and the Gram fit in tensor memory");
static_assert(kN % 16 == 0 && kN <= 256, "MMA N for M = 128");

// ---- warp roles -------------------------------------------------------------
constexpr int kProducerWarp = 0, kMmaWarp = 1;
constexpr int kOwner0 = 2, kOwnerN = 2;        // owner warp o takes tiles t = o (mod 2)
constexpr int kRead0 = 4, kReadN = 4;          // warp & 3 = lane quarter = tile rows 8q..8q+7
constexpr int kComb0 = 8, kCombN = 10;         // also convert fn into its B tiles
constexpr int kSinkWarp = kComb0 + kCombN;     // 18
constexpr int kWarps = kSinkWarp + 1;          // 19
constexpr int kThreads = kWarps * 32;          // 608
constexpr int kCombT = kCombN * 32;            // 320 combine threads
constexpr int kNR = kOwnerN;                   // receive buffers (one per owner warp)
constexpr int kNG = 4;                         // gate buffers (tiles the combine may lag)
constexpr int kSkRows = 32;                    // rows per Sinkhorn batch (one per lane)
static_assert(kRead0 % 4 == 0, "lane quarters follow warp & 3");

template <int kCl_, bool kS_ = (kCl_ == 8)>
struct Geo {
  static constexpr int kCl = kCl_;                 // CTAs per cluster (K split)
  static constexpr bool kStream = kS_;             // fn streamed beside each R box
  static constexpr int kHs = kH / kCl;             // hidden columns per CTA
  static constexpr int kHb = kHs / kBk;            // blocks (stages) per tile
  static constexpr int kOwn = kTR / kCl;           // rows finalised per CTA per tile
  static constexpr int kPairs = kOwn / 2;          // owner passes, two rows each
  static constexpr int kSkTiles = kSkRows / kOwn;  // tiles per Sinkhorn batch
  static constexpr int kChunks = kHs / 8;          // 16-byte chunks of a row per stream
  static constexpr int kCombItems = kTR * kChunks / kCombT;   // rows per combine thread
  static constexpr int kCombRowStep = kCombT / kChunks;
  static constexpr int kRing = kStageBytes + (kStream ? kN * kBk * 2 : 0);   // a ring stage
  static constexpr int kFnItems = kHb * kHC * kMix * 8;   // 8-k items of a CTA's fn slice
  static_assert(kCl == 16 || kCl == 8, "the two builds");
  static_assert(kHs % kBk == 0 && kTR % kCl == 0 && kOwn % 2 == 0, "");
  static_assert(kCombT % kChunks == 0 && (kTR * kChunks) % kCombT == 0, "combine items tile evenly");
  static_assert(kCl <= 16, "one owner lane per destination CTA");
};

// mbarrier slots (arrays are given explicit, non-overlapping ranges)
enum Bar : int {
  B_FULL = 0,                     // [kStages] TMA landed
  B_EMPTY = B_FULL + kStages,     // [kStages] the stage's MMAs completed
  B_DFULL = B_EMPTY + kStages,    // [2] dot accumulators (and the Gram) complete
  B_DEMPTY = B_DFULL + 2,         // [2] dot accumulators read out
  B_D2EMPTY = B_DEMPTY + 2,       // the Gram accumulator read out
  B_RX = B_D2EMPTY + 1,           // [kNR] the 16 CTAs' partials landed (bytes, remote st.async)
  B_GIN = B_RX + kNR,             // [kNG] the 16 owners' gates landed (bytes, remote st.async)
  B_GREAD = B_GIN + kNG,          // [kNG] the combine warps are done with this buffer's gates
  B_SKFULL = B_GREAD + kNG,       // [2] a Sinkhorn batch's comb logits queued
  B_SKFREE = B_SKFULL + 2,        // [2] the Sinkhorn warp read the batch
  B_FNREADY = B_SKFREE + 2,       // fn's B tiles written
  B_DRAIN = B_FNREADY + 1,        // final MMA drain
  B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT == 2 * kStages + 5 + kNR + 2 * kNG + 6, "barrier slots overlap");

template <bool kMx, int kCl, bool kS>
struct Cfg {
  using G = Geo<kCl, kS>;
  static constexpr int kOffFn = 0;                                    // resident build: [5 blocks][192][64] bf16
  static constexpr int kOffStage = G::kStream ? 0 : G::kHb * kFnBlkBytes;   // [5 stages][128 (+ 192 streamed)][64] bf16
  static constexpr int kOffRx = kOffStage + kStages * G::kRing;       // [kNR][kCl src][kOwn rows][36]
  static constexpr int kRxBytes = kCl * G::kOwn * kRec * 4;
  static constexpr int kOffGin = kOffRx + kNR * kRxBytes;             // [kNG][32 rows][8]
  static constexpr int kGinBytes = kTR * 8 * 4;
  static constexpr int kOffSk = kOffGin + kNG * kGinBytes;            // [2][32 rows][16] logits
  static constexpr int kSkBytes = kSkRows * 16 * 4;
  static constexpr int kOffBar = kOffSk + 2 * kSkBytes;
  static constexpr int kOffMisc = kOffBar + B_COUNT * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;             // slack to align the base
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
  static_assert(kOffStage % 1024 == 0 && G::kRing % 1024 == 0 && kFnBlkBytes % 1024 == 0,
                "SW128 tiles need 1024-byte alignment");
  static_assert(kOffRx % 16 == 0 && kOffGin % 16 == 0 && kOffSk % 16 == 0 && kOffBar % 8 == 0,
                "vector and barrier alignment");
};

// instruction descriptors, kind::f16: D fp32, A and B bf16, both K-major,
// M = 128; N = 192 (dots) and N = 128 (Gram)
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kM >> 4) << 24);
constexpr uint32_t kIdescG = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kM >> 3) << 17) |
                             ((uint32_t)(kM >> 4) << 24);

// fn's 8 consecutive k (16-byte chunk q of hidden block b, stream j, mix c)
// of image rank `rank` (16 ranks of 320 columns) -> bf16 hi = bf16(f) into B row 48 j + 2 c and lo =
// bf16(f - hi) into row 48 j + 2 c + 1 of the block's tile (K-major,
// 128-byte swizzle).  The in-kernel conversion and the prepared-weights image both use
// this routine, so they give the same bits.
__device__ __forceinline__ void fn_b_item(const float *__restrict__ fn, int rank, int b, int j,
                                          int c, int q, uint8_t *tile) {
  const float4 *src = reinterpret_cast<const float4 *>(fn + (int64_t)c * kK + j * kH +
                                                       rank * kImgHs + b * kBk + 8 * q);
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
  const int nh = kFnRowsPerStream * j + 2 * c, nl = nh + 1;
  *reinterpret_cast<uint4 *>(tile + (nh >> 3) * 1024 + (nh & 7) * 128 + ((q ^ (nh & 7)) << 4)) =
      make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4 *>(tile + (nl >> 3) * 1024 + (nl & 7) * 128 + ((q ^ (nl & 7)) << 4)) =
      make_uint4(lw[0], lw[1], lw[2], lw[3]);
}
constexpr int kImgItems = kImgHb * kHC * kMix * 8;   // 3840 items of 8 k per image rank

struct OnePassArgs {
  const uint16_t *R;
  const float *fn;
  const uint8_t *fn_img;    // NULL, or fn's B tiles of every cluster rank (prepared weights)
  const float *scale;
  const float *base;
  const uint16_t *norm_w;
  uint16_t *x_norm;
  float *post;
  float *comb;
  float *pre_out;
  float *mix_out;
  uint8_t *mx_q;            // MXFP8 build: codes [rows, 5120]
  uint8_t *mx_s;            // MXFP8 build: linear scales [rows, 160]
  int64_t rows;
  int num_tiles;
  float rms_eps, pre_eps, sink_eps, post_mult, norm_eps;
  int iters;
};

// 96 registers a thread (a warp's registers are allocated in units of 512,
// so 19 warps x 3072 fit the 64 K-register file with one block per SM)
constexpr int kMaxRegs = 96;
static_assert(kWarps * ((kMaxRegs * 32 + 511) / 512 * 512) <= 65536, "register budget of one block per SM");
template <bool kMx, int kCl, bool kS>
__global__ void __maxnreg__(kMaxRegs)
pre_onepass_kernel(const __grid_constant__ CUtensorMap tmap, const OnePassArgs a) {
  using G = Geo<kCl, kS>;
  using C = Cfg<kMx, kCl, kS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;   // our tiles
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)i; };
  auto stage_addr = [&](int s) -> uint32_t { return sb + C::kOffStage + (uint32_t)(s * G::kRing); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::kOffMisc);
  Abort ab{reinterpret_cast<volatile int *>(sm + C::kOffMisc + 4), crank, &g_onepass_error,
           g_onepass_where, g_onepass_where_aborted};
  // A push of tile t may go out once the gates of tile t - 2 have arrived
  // here (every owner has consumed that tile's receive buffer, which tile t
  // reuses) and this CTA's combine is done with the gates of tile t - kNG
  // (so that, once all pushes of tile t are in, every CTA's gate buffer for
  // it is free).  Whole warp; false if a wait gave up.
  auto push_ready = [&](int t, int site) -> bool {
    if (t >= 2) {
      const int tg = t - 2;
      if (!waitw(bar(B_GIN + tg % kNG), (uint32_t)((tg / kNG) & 1), true, ab, site, t)) return false;
    }
    if (t >= kNG) {
      const int tr = t - kNG;
      if (!waitw(bar(B_GREAD + tr % kNG), (uint32_t)((tr / kNG) & 1), false, ab, site, t))
        return false;
    }
    return true;
  };

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *ab.flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_DFULL + b), 1);
      mbar_init(bar(B_DEMPTY + b), kReadN);
      mbar_init(bar(B_SKFULL + b), G::kSkTiles);
      mbar_init(bar(B_SKFREE + b), 1);
    }
    for (int b = 0; b < kNG; ++b) {
      mbar_init(bar(B_GIN + b), 1);
      mbar_init(bar(B_GREAD + b), kCombN);
    }
    for (int b = 0; b < kNR; ++b) mbar_init(bar(B_RX + b), 1);
    mbar_init(bar(B_D2EMPTY), kReadN);
    // (streamed: no resident tiles to wait for, the phase completes at once)
    mbar_init(bar(B_FNREADY), G::kStream ? 1 : kCombN);
    if (G::kStream) mbar_arrive(bar(B_FNREADY));
    mbar_init(bar(B_DRAIN), 1);
    // the byte-counted barriers are armed for their first phase here; each
    // later phase is armed by the side that consumed the previous one
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

  // fn's B tiles for this CTA's columns (resident build, which runs only
  // without an image): converted by the combine warps
  if (!G::kStream && warp >= kComb0 && warp < kComb0 + kCombN) {
    const int t = (warp - kComb0) * 32 + lane;
    for (int item = t; item < G::kFnItems; item += kCombT) {
      const int q = item & 7, c = (item >> 3) % kMix, j = (item / (8 * kMix)) % kHC,
                b = item / (8 * kMix * kHC);
      fn_b_item(a.fn, (int)crank, b, j, c, q, sm + C::kOffFn + b * kFnBlkBytes);
    }
    // generic-proxy writes -> visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_FNREADY));
  }

  // ---- roles -------------------------------------------------------------------
  if (warp == kProducerWarp) {
    // the whole warp walks the loop (waits are warp-collective); lane 0 issues
    int g = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int y = (cid + it * ncl) * kTR;
      for (int b = 0; b < G::kHb; ++b, ++g) {
        const int s = g % kStages;
        if (!waitw(bar(B_EMPTY + s), (uint32_t)((g / kStages) & 1) ^ 1, false, ab, 1, it)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(bar(B_FULL + s), G::kRing);
          tma_load_3d(stage_addr(s), &tmap, (int)crank * G::kHs + b * kBk, 0, y, bar(B_FULL + s));
          // streamed build: the block's fn tile lands in the same stage (image
          // blocks 10 crank + b: this CTA's 2560 k)
          if (G::kStream)
            bulk_load(stage_addr(s) + kStageBytes,
                      a.fn_img + ((size_t)crank * G::kHb + b) * kFnBlkBytes, kFnBlkBytes,
                      bar(B_FULL + s));
        }
        __syncwarp();
      }
    }
    // every copy issued must have landed before the CTA may exit: the last
    // use of stage s is group g_last with g_last % kStages == s
    for (int s = 0; s < kStages && s < g; ++s) {
      const int g_last = s + ((g - 1 - s) / kStages) * kStages;
      drain1(bar(B_FULL + s), (uint32_t)((g_last / kStages) & 1));
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    int g = 0;
    bool ok = waitw(bar(B_FNREADY), 0, false, ab, 0, 0);
    tc_fence_after();
    for (int it = 0; it < T && ok; ++it) {
      const int buf = it & 1;
      if (!waitw(bar(B_DEMPTY + buf), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 2, it)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * kDCols);
      for (int b = 0; b < G::kHb; ++b, ++g) {
        const int s = g % kStages;
        if (!waitw(bar(B_FULL + s), (uint32_t)((g / kStages) & 1), false, ab, 3, it)) {
          ok = false;
          break;
        }
        // the Gram accumulator has one buffer: the previous tile's must have
        // been read out before this tile's first Gram MMA
        if (b == 0 && it > 0 &&
            !waitw(bar(B_D2EMPTY), (uint32_t)((it - 1) & 1), false, ab, 4, it)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t ad = sw128_desc(stage_addr(s));
          const uint64_t bd = sw128_desc(G::kStream ? stage_addr(s) + kStageBytes
                                                    : sb + C::kOffFn + b * kFnBlkBytes);
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk)
            tc_mma(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (b | kk) != 0);
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk)
            tc_mma(tmem + kD2Col, ad + 2 * kk, ad + 2 * kk, kIdescG, (b | kk) != 0);
          tc_commit(bar(B_EMPTY + s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(B_DFULL + buf));
      __syncwarp();
    }
    // all issued MMAs complete before tensor memory is freed
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp >= kRead0 && warp < kRead0 + kReadN) {
    // ---- readout warps: accumulators -> owners' receive buffers -------------
    // lane l of quarter q holds accumulator line 32 q + l = 4 r + i: tile row
    // r = 8 q + l / 4, stream i = l % 4; its useful columns are 48 i .. + 47
    const int quarter = warp & 3;
    const int i_s = lane & 3, r = 8 * quarter + (lane >> 2);
    const unsigned full = 0xffffffffu;
    for (int it = 0; it < T; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!waitw(bar(B_DFULL + buf), use & 1, false, ab, 6, it)) break;
      tc_fence_after();
      // the Gram first (its single buffer holds up the next tile's MMAs):
      // lane 4 r' + i of the quarter takes columns 32 q + 4 r' .. + 3, i.e.
      // row i of row r's 4x4 Gram matrix
      float gi[kHC];
      {
        float v[32];
        tc_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kD2Col + 32 * quarter), v);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_D2EMPTY));
#pragma unroll
        for (int j = 0; j < kHC; ++j) gi[j] = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if ((lane >> 2) == k) {
#pragma unroll
            for (int j = 0; j < kHC; ++j) gi[j] = v[4 * k + j];
          }
      }
      // Three groups of 8 mixes.  For each stream block j the warp loads the
      // 16 columns of the group (a load reads the same columns in all lanes:
      // hi, lo of mix 8 g + c at 2 c, 2 c + 1); lanes of stream j keep
      // hi + lo.  Then the four streams of row r, in lanes 4 (l / 4) .. + 3,
      // are summed as (s0 + s1) + (s2 + s3), the same bits in all four.
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * kDCols);
      float m[kMix];
#pragma unroll
      for (int g8 = 0; g8 < 3; ++g8) {
        float mg[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mg[c] = 0.f;
#pragma unroll
        for (int j = 0; j < kHC; ++j) {
          float v[16];
          tc_ld16(ta + kFnRowsPerStream * j + 16 * g8, v);
          tc_wait_ld();
          if (i_s == j) {
#pragma unroll
            for (int c = 0; c < 8; ++c) mg[c] = v[2 * c] + v[2 * c + 1];
          }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float x = mg[c];
          x = x + __shfl_xor_sync(full, x, 1);
          x = x + __shfl_xor_sync(full, x, 2);
          m[8 * g8 + c] = x;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DEMPTY + buf));
      if (!push_ready(it, 7)) break;
      const int rb = it % kNR;
      const uint32_t owner = (uint32_t)(r / G::kOwn);
      const uint32_t dst = mapa(sb + C::kOffRx + (uint32_t)(rb * C::kRxBytes +
                                                            ((int)crank * G::kOwn + r % G::kOwn) *
                                                                kRec * 4),
                                owner);
      const uint32_t rbar = mapa(bar(B_RX + rb), owner);
      // the row's Gram entries from the quad: diagonal, then i < j
      const int qb = lane & ~3;
      float diag = gi[0];
#pragma unroll
      for (int j = 1; j < kHC; ++j)
        if (i_s == j) diag = gi[j];
      const float g00 = __shfl_sync(full, diag, qb), g11 = __shfl_sync(full, diag, qb + 1);
      const float g22 = __shfl_sync(full, diag, qb + 2), g33 = __shfl_sync(full, diag, qb + 3);
      const float g01 = __shfl_sync(full, gi[1], qb), g02 = __shfl_sync(full, gi[2], qb);
      const float g03 = __shfl_sync(full, gi[3], qb), g12 = __shfl_sync(full, gi[2], qb + 1);
      const float g13 = __shfl_sync(full, gi[3], qb + 1), g23 = __shfl_sync(full, gi[3], qb + 2);
      // record chunks: dots 4 ch .. 4 ch + 3 at ch = 0..5, Gram at 6..8 (every
      // lane of the quad holds all the sums; compile-time indices only)
      if (i_s == 0) {
        st_async_v4(dst, m[0], m[1], m[2], m[3], rbar);
        st_async_v4(dst + 64, m[16], m[17], m[18], m[19], rbar);
        st_async_v4(dst + 96, g00, g11, g22, g33, rbar);
      } else if (i_s == 1) {
        st_async_v4(dst + 16, m[4], m[5], m[6], m[7], rbar);
        st_async_v4(dst + 80, m[20], m[21], m[22], m[23], rbar);
        st_async_v4(dst + 112, g01, g02, g03, g12, rbar);
      } else if (i_s == 2) {
        st_async_v4(dst + 32, m[8], m[9], m[10], m[11], rbar);
        st_async_v4(dst + 128, g13, g23, 0.f, 0.f, rbar);
      } else {
        st_async_v4(dst + 48, m[12], m[13], m[14], m[15], rbar);
      }
      __syncwarp();
    }
  } else if (warp >= kOwner0 && warp < kOwner0 + kOwnerN) {
    // ---- owner warps: finalise rows kOwn crank .. + kOwn - 1 of every other
    // tile, two rows a pass (16 lanes a row)
    const int ow = warp - kOwner0;
    const int sub = lane >> 4, e = lane & 15;    // row of the pair, lane of 16
    const float *rx = reinterpret_cast<const float *>(sm + C::kOffRx + ow * C::kRxBytes);
    float *sk = reinterpret_cast<float *>(sm + C::kOffSk);
    const float sc0 = __ldg(a.scale), sc1 = __ldg(a.scale + 1), sc2 = __ldg(a.scale + 2);
    const float bcomb = __ldg(a.base + 8 + e);
    const float bgate = e < 8 ? __ldg(a.base + e) : 0.f;
    const unsigned full = 0xffffffffu;
    for (int it = ow; it < T; it += kOwnerN) {
      const uint32_t use = (uint32_t)(it / kNR);
      if (!waitw(bar(B_RX + ow), use & 1, true, ab, 10, it)) break;
      const int bt = it / G::kSkTiles, skb = bt & 1;
      bool ok = true;
      for (int pp = 0; pp < G::kPairs; ++pp) {
        const int own = 2 * pp + sub;               // row among this CTA's kOwn
        const int n = (int)crank * G::kOwn + own;    // tile row
        const int64_t grow = (int64_t)(cid + it * ncl) * kTR + n;
        // this row's 34 partials from the kCl CTAs, summed in CTA order: lane
        // e holds values e, e + 16 and (e < 2) e + 32 of the record
        float v0 = 0.f, v1 = 0.f, v2 = 0.f;
#pragma unroll
        for (int src = 0; src < kCl; ++src) {
          const float *rec = rx + (src * G::kOwn + own) * kRec;
          v0 += rec[e];
          v1 += rec[e + 16];
          if (e < 2) v2 += rec[e + 32];
        }
        // once every row is read, arm the buffer's next phase (tile it + kNR,
        // whose stores can only come after this tile's gates, which depend on
        // the sums just read)
        __syncwarp();
        if (pp == G::kPairs - 1 && lane == 0) mbar_expect_tx(bar(B_RX + ow), C::kRxBytes);
        // record: dots 0..23 at 0..23, Gram entries 0..9 at 24..33
        const int hb = lane & 16;                   // first lane of this row's half
        auto val = [&](int idx) -> float {          // record value idx of this row
          const float a0 = __shfl_sync(full, v0, hb + (idx & 15));
          const float a1 = __shfl_sync(full, v1, hb + ((idx - 16) & 15));
          const float a2 = __shfl_sync(full, v2, hb + ((idx - 32) & 15));
          return idx < 16 ? a0 : (idx < 32 ? a1 : a2);
        };
        float G2[kNGram];
#pragma unroll
        for (int q = 0; q < kNGram; ++q) G2[q] = val(24 + q);
        const float ssx = (G2[0] + G2[1]) + (G2[2] + G2[3]);
        const float rsq = rsqrt_nr(fmaf(ssx, 1.0f / (float)kK, a.rms_eps));
        const float dg = e < 8 ? v0 : 0.f;          // dot e (gates)
        const float dc = val(8 + e);                // dot 8 + e (comb logit e)
        float gate = 0.f;
        if (e < 8) {
          const float l = fmaf(dg * rsq, e < 4 ? sc0 : sc1, bgate);
          const float sg = rcp_nr(1.0f + expf(-l));
          gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
        }
        const float lc = fmaf(dc * rsq, sc2, bcomb);
        float p[kHC];
#pragma unroll
        for (int i = 0; i < kHC; ++i) p[i] = __shfl_sync(full, gate, hb + i);
        // sum_h y^2 = p^T G p in a fixed order, clamped at 0 against rounding
        const float diag = fmaf(p[3] * p[3], G2[3], fmaf(p[2] * p[2], G2[2],
                                fmaf(p[1] * p[1], G2[1], (p[0] * p[0]) * G2[0])));
        float off = (p[0] * p[1]) * G2[4];
        off = fmaf(p[0] * p[2], G2[5], off);
        off = fmaf(p[0] * p[3], G2[6], off);
        off = fmaf(p[1] * p[2], G2[7], off);
        off = fmaf(p[1] * p[3], G2[8], off);
        off = fmaf(p[2] * p[3], G2[9], off);
        const float ssy = fmaxf(fmaf(2.0f, off, diag), 0.f);
        const float rn = rsqrt_nr(fmaf(ssy, 1.0f / (float)kH, a.norm_eps));
        // broadcast this row's pre gates and 1/rms(y): lane e -> CTA e, 32
        // bytes counted on that CTA's gate barrier
        if (e < kCl) {
          const uint32_t gbuf = (uint32_t)(it % kNG);
          const uint32_t dst = mapa(sb + C::kOffGin + gbuf * C::kGinBytes + (uint32_t)(n * 32),
                                    (uint32_t)e);
          const uint32_t gbar = mapa(bar(B_GIN) + 8u * gbuf, (uint32_t)e);
          st_async_v4(dst, p[0], p[1], p[2], p[3], gbar);
          st_async_v4(dst + 16, rn, 0.f, 0.f, 0.f, gbar);
        }
        // outputs of the row: post, optional pre and mixes
        if (grow < a.rows) {
          if (e >= 4 && e < 8) a.post[grow * kHC + (e - 4)] = gate;
          if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
          if (a.mix_out) {
            a.mix_out[grow * kMix + e] = v0 * rsq;
            if (e < 8) a.mix_out[grow * kMix + 16 + e] = v1 * rsq;
          }
        }
        // queue the comb logits for the Sinkhorn warp (row kOwn (it %
        // kSkTiles) + own of batch it / kSkTiles)
        if (pp == 0 &&
            !waitw(bar(B_SKFREE + skb), (uint32_t)((bt >> 1) & 1) ^ 1, false, ab, 8, it)) {
          ok = false;
          break;
        }
        sk[skb * (kSkRows * 16) + ((it % G::kSkTiles) * G::kOwn + own) * 16 + e] = lc;
        __syncwarp();
      }
      if (!ok) break;
      // the tile's rows are queued; the last tile completes its batch's count
      if (lane == 0) {
        mbar_arrive(bar(B_SKFULL + skb));
        if (it == T - 1)
          for (int k = it % G::kSkTiles + 1; k < G::kSkTiles; ++k) mbar_arrive(bar(B_SKFULL + skb));
      }
    }
  } else if (warp == kSinkWarp) {
    // ---- Sinkhorn warp: hc_split_sinkhorn's 4x4 Sinkhorn, one row per lane --
    // Row sums pair (c0 + c1) + (c2 + c3), likewise the column sums; eps is
    // added to every sum, and each entry is multiplied by its reciprocal
    // (rcp_nr: no branch, so a step's four reciprocals overlap; an IEEE
    // division or reciprocal per sum serialised them, 8 us a batch).
    const float *sk = reinterpret_cast<const float *>(sm + C::kOffSk);
    const int nb = (T + G::kSkTiles - 1) / G::kSkTiles;
    const int r = lane & (kSkRows - 1);
    const int tl = r / G::kOwn, sub = r % G::kOwn;   // tile within the batch, row of the CTA's
    for (int bt = 0; bt < nb; ++bt) {
      const int skb = bt & 1;
      if (!waitw(bar(B_SKFULL + skb), (uint32_t)((bt >> 1) & 1), false, ab, 9, bt)) break;
      const int tile = bt * G::kSkTiles + tl;
      const bool valid = lane < kSkRows && tile < T;
      // lanes without a row run on ones: a zero matrix would send every
      // division down its slow path (0 / d)
      float c[kHC][kHC];
#pragma unroll
      for (int j = 0; j < kHC; ++j)
#pragma unroll
        for (int i = 0; i < kHC; ++i)
          c[j][i] = valid ? expf(sk[skb * (kSkRows * 16) + r * 16 + 4 * j + i]) : 1.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SKFREE + skb));
      for (int k = 0; k < a.iters; ++k) {
#pragma unroll
        for (int j = 0; j < kHC; ++j) {
          const float d = rcp_nr(((c[j][0] + c[j][1]) + (c[j][2] + c[j][3])) + a.sink_eps);
#pragma unroll
          for (int i = 0; i < kHC; ++i) c[j][i] = c[j][i] * d;
        }
#pragma unroll
        for (int i = 0; i < kHC; ++i) {
          const float d = rcp_nr(((c[0][i] + c[1][i]) + (c[2][i] + c[3][i])) + a.sink_eps);
#pragma unroll
          for (int j = 0; j < kHC; ++j) c[j][i] = c[j][i] * d;
        }
      }
      const int64_t grow = (int64_t)(cid + tile * ncl) * kTR + (int)crank * G::kOwn + sub;
      if (valid && grow < a.rows) {
        float4 *o = reinterpret_cast<float4 *>(a.comb + grow * 16);
#pragma unroll
        for (int j = 0; j < kHC; ++j) o[j] = make_float4(c[j][0], c[j][1], c[j][2], c[j][3]);
      }
    }
  } else {
    // ---- combine warps: x_norm of the CTA's columns, read back from L2 ------
    // thread t: 16-byte chunk cq = t % kChunks of the CTA's kHs columns, tile
    // rows t / kChunks + kCombRowStep u
    const int t = (warp - kComb0) * 32 + lane;
    const int cq = t % G::kChunks, r0 = t / G::kChunks;
    const float *gin = reinterpret_cast<const float *>(sm + C::kOffGin);
    const int64_t col = (int64_t)crank * G::kHs + 8 * cq;
    float wf[8];
    unpack8(__ldg(reinterpret_cast<const uint4 *>(a.norm_w + col)), wf);
    for (int it = 0; it < T; ++it) {
      const int buf = it % kNG;
      if (!waitw(bar(B_GIN + buf), (uint32_t)((it / kNG) & 1), true, ab, 12, it)) break;
      const int64_t row0 = (int64_t)(cid + it * ncl) * kTR;
      // one row's loads at a time in the resident build (more in flight only
      // added to the load on the shared-memory / L1 data path the MMAs and TMA
      // also use); two in the streamed build, whose combine walks twice the
      // columns a tile, unless it also quantizes (MXFP8), where one is faster
      uint4 rv[2][kHC];
      auto load = [&](int u, uint4 (&dst)[kHC]) {
        const int64_t grow = row0 + r0 + G::kCombRowStep * u;
        if (grow < a.rows) {
          const uint4 *src = reinterpret_cast<const uint4 *>(a.R + grow * kK + col);
#pragma unroll
          for (int i = 0; i < kHC; ++i) dst[i] = ld_nc_noalloc(src + i * (kH / 8));
        } else {
#pragma unroll
          for (int i = 0; i < kHC; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      };
      // the streamed build: the next row's loads in flight while this one is
      // combined
      if (G::kStream && !kMx) load(0, rv[0]);
#pragma unroll
      for (int u = 0; u < G::kCombItems; ++u) {
        if (G::kStream && !kMx) {
          if (u + 1 < G::kCombItems) load(u + 1, rv[(u + 1) & 1]);
        } else {
          load(u, rv[u & 1]);
        }
        const float *gr = gin + buf * (kTR * 8) + (r0 + G::kCombRowStep * u) * 8;
        const float4 pq = *reinterpret_cast<const float4 *>(gr);
        const float pv[kHC] = {pq.x, pq.y, pq.z, pq.w};
        const float rn = gr[4];
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t sh = (e & 1) ? 0u : 16u;   // bf16 e of the chunk: low half first
          float acc = pv[0] * __uint_as_float(((&rv[u & 1][0].x)[e >> 1] << sh) & 0xFFFF0000u);
#pragma unroll
          for (int i = 1; i < kHC; ++i)
            acc = fmaf(pv[i], __uint_as_float(((&rv[u & 1][i].x)[e >> 1] << sh) & 0xFFFF0000u), acc);
          v[e] = (acc * rn) * wf[e];
        }
        const uint4 xb = pack8_rn(v);
        const int64_t grow = row0 + r0 + G::kCombRowStep * u;
        const bool live = grow < a.rows;
        if (live) st_stream(reinterpret_cast<uint4 *>(a.x_norm + grow * kH + col), xb);
        if constexpr (kMx) {
          float vb[8];
          unpack8(xb, vb);                 // the bf16 values, as stored
          uint32_t sc;
          const uint2 codes = mx_block8(vb, sc);
          if (live) {
            __stcs(reinterpret_cast<uint2 *>(a.mx_q + grow * kH + col), codes);
            if ((cq & 3) == 0) a.mx_s[grow * (kH / kMxBlock) + (col >> 5)] = (uint8_t)sc;
          }
        }
      }
      // every lane is done with this buffer's gates: count this warp out of
      // it, and arm its next phase (tile it + kNG, whose gates need this
      // CTA's pushes of that tile, which wait for this barrier)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_GREAD + buf));
        if (warp == kComb0) mbar_expect_tx(bar(B_GIN + buf), C::kGinBytes);
      }
    }
  }

  // this CTA's work is done: the next launch may start scheduling
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
template <bool kMx, int kCl, bool kS>
int g_max_clusters[kMaxDev];   // 0: not yet configured on that device

template <bool kMx, int kCl, bool kS>
cudaError_t configure(int dev, int *max_clusters) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_max_clusters<kMx, kCl, kS>[dev] > 0) {
    *max_clusters = g_max_clusters<kMx, kCl, kS>[dev];
    return cudaSuccess;
  }
  constexpr int kSmemBytes = Cfg<kMx, kCl, kS>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(pre_onepass_kernel<kMx, kCl, kS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  // a cluster of 16 is a non-portable size
  if (e == cudaSuccess && kCl > 8)
    e = cudaFuncSetAttribute(pre_onepass_kernel<kMx, kCl, kS>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  e = cudaOccupancyMaxActiveClusters(&n, pre_onepass_kernel<kMx, kCl, kS>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_max_clusters<kMx, kCl, kS>[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

template <bool kMx, int kCl, bool kS>
cudaError_t launch(const OnePassArgs &a, int64_t logical_rows, cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  int max_clusters = 0;
  e = configure<kMx, kCl, kS>(dev, &max_clusters);
  if (e != cudaSuccess) return e;

  // R as a 3-D tensor (hidden column, stream, row): a box of 64 columns x
  // 4 streams x 32 rows lands with the four streams of a row adjacent
  CUtensorMap map;
  const cuuint64_t gdim[3] = {(cuuint64_t)kH, (cuuint64_t)kHC, (cuuint64_t)a.rows};
  const cuuint64_t gstride[2] = {(cuuint64_t)kH * 2, (cuuint64_t)kK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBk, (cuuint32_t)kHC, (cuuint32_t)kTR};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(a.R), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // grid: as many clusters as fit at once, never more than the whole chunk's
  // tiles (the count depends on logical_rows only; per-row arithmetic does not
  // depend on it at all)
  const int64_t chunk_tiles = (logical_rows + kTR - 1) / kTR;
  const int clusters = (int)(chunk_tiles < max_clusters ? chunk_tiles : max_clusters);
  return launch_pdl(pre_onepass_kernel<kMx, kCl, kS>, dim3((unsigned)(clusters * kCl)),
                    dim3(kThreads), Cfg<kMx, kCl, kS>::kSmemBytes, s, kCl, use_pdl(logical_rows),
                    map, a);
}

// ---- prepared weights: fn's B tiles of every image rank ------------------------
// [16 ranks][5 blocks][192 rows][64 k] bf16 in the kernel's shared-memory
// layout, written once by mhc_prepare_weights (or into mhc_pre's workspace)
__global__ void __launch_bounds__(256) fn_b_img_kernel(const float *__restrict__ fn,
                                                       uint8_t *__restrict__ img) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 256 + threadIdx.x;
  if (t >= kImgRanks * kImgItems) return;
  const int rank = t / kImgItems, item = t % kImgItems;
  const int q = item & 7, c = (item >> 3) % kMix, j = (item / (8 * kMix)) % kHC,
            b = item / (8 * kMix * kHC);
  fn_b_item(fn, rank, b, j, c, q, img + ((size_t)rank * kImgHb + b) * kFnBlkBytes);
}

}  // namespace

size_t fn_b_img_bytes() { return (size_t)kImgRanks * kImgHb * kFnBlkBytes; }

cudaError_t launch_fn_b_img(const float *fn, uint8_t *img, cudaStream_t s) {
  constexpr int kItems = kImgRanks * kImgItems;
  return launch_pdl(fn_b_img_kernel, dim3((kItems + 255) / 256), dim3(256), 0, s, 1, false, fn,
                    img);
}

cudaError_t launch_pre_onepass(const uint16_t *R, const float *fn, const uint8_t *fn_img,
                               const float *scale, const float *base, const uint16_t *norm_w,
                               int64_t rows, int64_t logical_rows, const mhc_params &p,
                               uint16_t *x_norm, float *post, float *comb, float *pre_out,
                               float *mix_out, cudaStream_t s, uint8_t *mx_q, uint8_t *mx_s) {
  OnePassArgs a;
  a.R = R; a.fn = fn; a.fn_img = fn_img; a.scale = scale; a.base = base; a.norm_w = norm_w;
  a.x_norm = x_norm; a.post = post; a.comb = comb; a.pre_out = pre_out; a.mix_out = mix_out;
  a.mx_q = mx_q; a.mx_s = mx_s;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTR - 1) / kTR);
  a.rms_eps = p.rms_eps; a.pre_eps = p.hc_pre_eps; a.sink_eps = p.hc_sinkhorn_eps;
  a.post_mult = p.post_mult; a.norm_eps = p.norm_eps; a.iters = p.sinkhorn_iters;
  // with fn's image at hand: chunks of kStreamMinRows rows and more take the
  // 8-CTA build, smaller ones the 16-CTA build streaming fn (the choice
  // depends on logical_rows, so every shard of a chunk takes the same build,
  // and fn's source does not change the bits)
  if (fn_img && logical_rows >= kStreamMinRows) {
    if (mx_q) return launch<true, 8, true>(a, logical_rows, s);
    return launch<false, 8, true>(a, logical_rows, s);
  }
  if (fn_img) {
    if (mx_q) return launch<true, 16, true>(a, logical_rows, s);
    return launch<false, 16, true>(a, logical_rows, s);
  }
  // the resident build: fn converted inside the kernel, no image
  if (mx_q) return launch<true, 16, false>(a, logical_rows, s);
  return launch<false, 16, false>(a, logical_rows, s);
}

cudaError_t onepass_error_where(unsigned int *out64) {
  cudaError_t e = cudaMemcpyFromSymbol(out64, g_onepass_where, 32 * sizeof(unsigned int));
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbol(out64 + 32, g_onepass_where_aborted, 32 * sizeof(unsigned int));
  return e;
}

cudaError_t onepass_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_onepass_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_onepass_error, &z, sizeof z);
  }
  return e;
}

}  // namespace mhc
