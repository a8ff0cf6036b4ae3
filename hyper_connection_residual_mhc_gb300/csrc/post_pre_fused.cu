// post_pre_fused.cu -- hc_post of one sublayer fused with the stats half of
// the next sublayer's hc_pre, on GB300.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_post
// (hc_post_torch_impl: R'_i = post_i * y + sum_j comb[j][i] * R_j, one bf16
// rounding) followed by DeepseekV4DecoderLayer.hc_pre on R' (rsqrt of
// mean(x^2) + rms_eps, mixes = (x @ fn^T) * rsqrt, hc_split_sinkhorn); the
// pages run the pair as one call (mhc_fused_post_pre) between sublayers.
//
// Unfused, R' is written by hc_post and read back by the stats; here the
// stats take R' from shared memory where it was just formed, so for them R'
// costs one write and no read.  A cluster owns a 128-row tile at a time and
// CTA s owns a contiguous range of hidden columns of all four streams: 320
// columns in 16-CTA clusters, or, for chunks of 2048 rows and more, 640 in
// 8-CTA clusters (15 of those fit, 120 SMs, against 7 of 16, 112 SMs).  Per
// tile and CTA the columns go through in "half-sets" of 32 columns, four in
// flight:
//   * a producer thread loads a half-set -- R_0..3 and y, 128 rows x 32
//     columns each, 64-byte swizzle, 40 KB, by TMA, and the four streams' fn
//     blocks for those columns (bf16 hi + lo, 12 KB) by bulk copy from an
//     image of fn in the operand layout that fn_prep_sw64_kernel writes
//     once per call -- into a free buffer (fn is not held in shared memory,
//     which leaves room for four 52 KB buffers);
//   * eight converter warps form R' in place (the same arithmetic as
//     mhc_post, so R' has mhc_post's bits) and add its squares to the rows'
//     sums of squares;
//   * the converters also write R' to R_out from their registers (the TMA
//     unit carries only the loads);
//   * one thread issues tcgen05.mma (M=128 rows, N=48, K=16) on the four R'
//     stages; the buffer is refilled once those MMAs have completed;
//   * four readout warps load the accumulator, push each row's 24 partials
//     and sum of squares to the row's owner CTA, then, as owners, reduce the
//     cluster's partials in CTA order and write the gates and comb logits.
// The combine + RMSNorm and the Sinkhorn of the next pre then run as the
// pre pass's streaming launch (pre_simt.cu) on R_out.
//
// Every wait is bounded (~2 s); on expiry a CTA raises an abort flag, records
// the site in this kernel's error word, drains its copies and MMAs, frees its
// tensor memory and returns.
#include <type_traits>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

__device__ unsigned int g_fpp_error;
__device__ unsigned int g_fpp_where[32];
__device__ unsigned int g_fpp_where_aborted[32];

namespace {
using namespace ptx;

constexpr int kTile = 128;                    // rows per tile = UMMA M
constexpr int kBh = 32;                       // columns per half-set (64-byte rows)
constexpr int kN = 2 * kMix;                  // fn hi (24) + lo (24)
constexpr int kStageBytes = kTile * kBh * 2;  // 8192: one stream (or y), 128 rows x 32
constexpr int kFnBlkBytes = kN * kBh * 2;     // 3072: fn hi/lo for 32 k (64-byte rows)
constexpr int kSetBytes = (kHC + 1) * kStageBytes + kHC * kFnBlkBytes;  // R_0..3, y, 4 fn blocks
constexpr int kBufs = 4;                      // half-sets in flight
constexpr int kFnBlocks = kK / kBh;           // 640 fn blocks of 32 k
constexpr int kRw = 28;                       // receive words per row
constexpr int kTmemCols = 128;

// warps: 0 TMA producer; 1 MMA; 2..9 converters; 10..13 readout, then owners
// (14 warps: at most 4 on a sub-partition, 128 registers each)
constexpr int kProdWarp = 0, kMmaWarp = 1;
constexpr int kConv0 = 2, kConvN = 8;
constexpr int kRead0 = 10, kReadN = 4;
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;         // 448
constexpr int kItems = 2;                     // (row, 8 columns) items per converter thread
static_assert(kConvN * 32 * kItems == kTile * (kBh / 8), "one item per (row, 8 columns)");

// shared memory (from a 1024-byte aligned base)
constexpr int kOffBuf = 0;                                    // [kBufs][R_0..3, y, fn x 4]
constexpr int kOffRecv = kOffBuf + kBufs * kSetBytes;         // [kCl src][kOwn rows][kRw]
enum Bar : int {
  B_FULL = 0,                    // [kBufs] a half-set landed (copy bytes)
  B_CONV = B_FULL + kBufs,       // [kBufs] converted to R' (8 converter warps)
  B_FREE = B_CONV + kBufs,       // [kBufs] the MMAs on it completed (commit)
  B_TFULL = B_FREE + kBufs,      // [2] accumulator complete
  B_TEMPTY = B_TFULL + 2,        // [2] accumulator and sum x^2 read out
  B_SSREADY = B_TEMPTY + 2,      // [2] the converters wrote a tile's sum x^2
  B_PREADY = B_SSREADY + 2,      // all 16 CTAs pushed partials to us (remote)
  B_PFREE = B_PREADY + 1,        // all 16 owners pulled our previous push (remote)
  B_GALL = B_PFREE + 1,          // the readout warps pushed
  B_OPULL = B_GALL + 1,          // the owner warps read the receive buffer
  B_DRAIN = B_OPULL + 1,         // final MMA drain
  B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT == 3 * kBufs + 3 * 2 + 5, "barrier slots overlap");

// Two builds: kCl = 16 CTAs a cluster, 320 columns (10 half-sets) and 8 owned
// rows a CTA; kCl = 8 (chunks of kStreamMinRows rows and more), 640 columns
// (20 half-sets) and 16 owned rows: 15 such clusters fit, 120 SMs, where 7
// 16-CTA clusters hold 112.
template <int kCl_>
struct FGeo {
  static constexpr int kCl = kCl_;                          // CTAs per cluster (K split)
  static constexpr int kHs = kH / kCl;                      // columns per CTA
  static constexpr int kNh = kHs / kBh;                     // half-sets per tile
  static constexpr int kOwn = kTile / kCl;                  // rows finalised per CTA
  static constexpr int kOwnPasses = kOwn / 8;               // the 128 owner threads take 8 rows a pass
  static constexpr int kOffRed = kOffRecv + kCl * kOwn * kRw * 4;   // [kOwn rows][kRw]
  static constexpr int kOffSs = kOffRed + kOwn * kRw * 4;           // [2][128] sum x^2
  static constexpr int kOffBar = kOffSs + 2 * kTile * 4;
  static constexpr int kOffMisc = kOffBar + B_COUNT * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kCl == 16 || kCl == 8, "the two builds");
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
};
static_assert(kOffBuf % 1024 == 0 && kStageBytes % 1024 == 0 && kFnBlkBytes % 1024 == 0 &&
                  kSetBytes % 1024 == 0, "64-byte swizzle tiles need 512-byte alignment");
static_assert(kOffRecv % 16 == 0, "");

constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kTile >> 4) << 24);

struct FusedArgs {
  const uint8_t *fnp;      // fn as bf16 hi/lo 32-k blocks in their shared-memory image
  const float *post_in;    // [rows, 4]
  const float *comb_in;    // [rows, 4, 4]
  uint4 *R_out;            // [rows, 4, 640] 16-byte chunks
  const float *scale;
  const float *base;
  float *pre_ws;           // [rows, 4] pre gates of R'
  float *logit_ws;         // [rows, 16] comb logits of R'
  float *post_out;         // [rows, 4]
  float *pre_out;
  float *mix_out;
  int64_t rows;
  int num_tiles;
  float rms_eps, pre_eps, post_mult;
};

template <int kCl>
__global__ void __launch_bounds__(kThreads, 1)
post_pre_fused_kernel(const __grid_constant__ CUtensorMap map_r,
                      const __grid_constant__ CUtensorMap map_y, const FusedArgs a) {
  using F = FGeo<kCl>;
  constexpr int kHs = F::kHs, kNh = F::kNh, kOwn = F::kOwn;
  constexpr int kOffRed = F::kOffRed, kOffSs = F::kOffSs, kOffBar = F::kOffBar,
                kOffMisc = F::kOffMisc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  Abort ab{reinterpret_cast<volatile int *>(sm + kOffMisc + 4), crank, &g_fpp_error, g_fpp_where,
           g_fpp_where_aborted};

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *ab.flag = 0;
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(bar(B_FULL + b), 1);
      mbar_init(bar(B_CONV + b), kConvN);
      mbar_init(bar(B_FREE + b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_TFULL + b), 1);
      mbar_init(bar(B_TEMPTY + b), kReadN);
      mbar_init(bar(B_SSREADY + b), kConvN);
    }
    mbar_init(bar(B_PREADY), kCl);
    mbar_init(bar(B_PFREE), kCl);
    mbar_init(bar(B_GALL), kReadN);
    mbar_init(bar(B_OPULL), kReadN);
    mbar_init(bar(B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  // ---- roles -------------------------------------------------------------------
  if (warp == kProdWarp) {
    // whole warp walks the loop (warp-collective waits); lane 0 issues
    uint32_t g = 0;
    int last[kBufs];
#pragma unroll
    for (int b = 0; b < kBufs; ++b) last[b] = -1;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int y0 = (cid + it * ncl) * kTile;
      for (int hh = 0; hh < kNh; ++hh, ++g) {
        const int b = (int)(g % kBufs);
        const uint32_t use = g / kBufs;
        if (!waitw(bar(B_FREE + b), (use & 1) ^ 1, false, ab, 1, it)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t dst = sb + kOffBuf + b * kSetBytes;
          const int xc = (int)crank * kHs + hh * kBh;
          mbar_expect_tx(bar(B_FULL + b), kSetBytes);
#pragma unroll
          for (int i = 0; i < kHC; ++i)
            tma_load_2d(dst + i * kStageBytes, &map_r, i * kH + xc, y0, bar(B_FULL + b));
          tma_load_2d(dst + kHC * kStageBytes, &map_y, xc, y0, bar(B_FULL + b));
          // the 4 streams' fn blocks of these 32 columns: block i * 160 + xc / 32
#pragma unroll
          for (int i = 0; i < kHC; ++i)
            bulk_load(dst + (kHC + 1) * kStageBytes + i * kFnBlkBytes,
                      a.fnp + (size_t)(i * (kH / kBh) + xc / kBh) * kFnBlkBytes, kFnBlkBytes,
                      bar(B_FULL + b));
        }
        __syncwarp();
        last[b] = (int)(use & 1);
      }
    }
    // every copy issued must have landed before the CTA may exit
    for (int b = 0; b < kBufs; ++b)
      if (last[b] >= 0) drain1(bar(B_FULL + b), (uint32_t)last[b]);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    uint32_t g = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int y0 = (cid + it * ncl) * kTile;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!waitw(bar(B_TEMPTY + buf), (use & 1) ^ 1, false, ab, 2, it)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * 64);
      for (int hh = 0; hh < kNh; ++hh, ++g) {
        const int b = (int)(g % kBufs);
        if (!waitw(bar(B_CONV + b), (g / kBufs) & 1, false, ab, 3, it)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t src = sb + kOffBuf + b * kSetBytes;
#pragma unroll 1
          for (int i = 0; i < kHC; ++i) {
            const uint64_t ad = sw64_desc(src + i * kStageBytes);
            const uint64_t bd = sw64_desc(src + (kHC + 1) * kStageBytes + i * kFnBlkBytes);
#pragma unroll
            for (int kk = 0; kk < kBh / 16; ++kk)
              tc_mma(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (hh | i | kk) != 0);
          }
          tc_commit(bar(B_FREE + b));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(B_TFULL + buf));
      __syncwarp();
    }
    if (lane == 0) tc_commit(bar(B_DRAIN));   // all issued MMAs complete before TMEM is freed
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp >= kConv0 && warp < kConv0 + kConvN) {
    // ---- converters: R' = post(R, y) in place, and the rows' sums of squares
    const int cw = warp - kConv0, c = lane & 3, rs = lane >> 2;
    float *ssbuf = reinterpret_cast<float *>(sm + kOffSs);
    uint32_t g = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      const int64_t row0 = (int64_t)(cid + it * ncl) * kTile;
      // post and comb of this thread's two rows (zeros past the last row)
      float pv[kItems][kHC], cb[kItems][kHC][kHC];
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        const int64_t gr = row0 + cw * 16 + 8 * k + rs;
        const bool in = gr < a.rows;
        const float4 p4 = in ? __ldg(reinterpret_cast<const float4 *>(a.post_in + gr * kHC))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        pv[k][0] = p4.x; pv[k][1] = p4.y; pv[k][2] = p4.z; pv[k][3] = p4.w;
#pragma unroll
        for (int j = 0; j < kHC; ++j) {
          const float4 c4 = in ? __ldg(reinterpret_cast<const float4 *>(a.comb_in + gr * 16 + 4 * j))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          cb[k][j][0] = c4.x; cb[k][j][1] = c4.y; cb[k][j][2] = c4.z; cb[k][j][3] = c4.w;
        }
      }
      float ssq[kItems] = {0.f, 0.f};
      for (int hh = 0; hh < kNh; ++hh, ++g) {
        const int b = (int)(g % kBufs);
        const int h8c = (int)crank * (kHs / 8) + hh * (kBh / 8);   // first 16-byte column
        if (!waitw(bar(B_FULL + b), (g / kBufs) & 1, false, ab, 4, it)) { ok = false; break; }
        uint8_t *buf = sm + kOffBuf + b * kSetBytes;
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
          const int r = cw * 16 + 8 * k + rs;
          const int off = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);   // 64-byte swizzle
          uint4 rv[kHC];
#pragma unroll
          for (int i = 0; i < kHC; ++i) rv[i] = *reinterpret_cast<const uint4 *>(buf + i * kStageBytes + off);
          const uint4 yv = *reinterpret_cast<const uint4 *>(buf + kHC * kStageBytes + off);
          uint4 ov[kHC];
          post_chunk(rv, yv, pv[k], cb[k], ov);
          float si[kHC];                        // per stream: 8 squares
#pragma unroll
          for (int i = 0; i < kHC; ++i) {
            *reinterpret_cast<uint4 *>(buf + i * kStageBytes + off) = ov[i];
            if (row0 + r < a.rows)
              st_stream(a.R_out + ((row0 + r) * kHC + i) * kChunksPerStream + h8c + c, ov[i]);
            float of[8];
            unpack8(ov[i], of);
            si[i] = of[0] * of[0];
#pragma unroll
            for (int e = 1; e < 8; ++e) si[i] = fmaf(of[e], of[e], si[i]);
          }
          ssq[k] += (si[0] + si[1]) + (si[2] + si[3]);
        }
        // generic-proxy writes -> visible to the tensor core
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_CONV + b));
      }
      if (!ok) break;
      // the rows' sums of squares: the 4 lanes of a row (c = 0..3), fixed tree
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        ssq[k] += __shfl_xor_sync(0xffffffffu, ssq[k], 1);
        ssq[k] += __shfl_xor_sync(0xffffffffu, ssq[k], 2);
      }
      const int tb = it & 1;
      if (!waitw(bar(B_TEMPTY + tb), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 10, it)) break;
      if (c == 0) {
#pragma unroll
        for (int k = 0; k < kItems; ++k) ssbuf[tb * kTile + cw * 16 + 8 * k + rs] = ssq[k];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SSREADY + tb));
    }
  } else {
    // ---- readout (one thread per tile row), then owners of kOwn rows --------
    const int quarter = warp & 3;               // a warp reads TMEM lanes 32*(warp%4) .. +31
    const int row = 32 * quarter + lane;
    const float *ssbuf = reinterpret_cast<const float *>(sm + kOffSs);
    const int o = (warp - kRead0) * 32 + lane; // owner thread 0..127
    const int oq = o >> 4, e = o & 15;          // owned row (of 8 a pass), lane of 16
    const float *recv = reinterpret_cast<const float *>(sm + kOffRecv);
    float *red = reinterpret_cast<float *>(sm + kOffRed);
    const float sc0 = __ldg(a.scale), sc1 = __ldg(a.scale + 1), sc2 = __ldg(a.scale + 2);
    const float bcomb = __ldg(a.base + 8 + e);
    const float bgate = e < 8 ? __ldg(a.base + e) : 0.f;
    for (int t = 0; t < T; ++t) {
      const int buf = t & 1;
      const uint32_t use = (uint32_t)(t >> 1);
      if (!waitw(bar(B_TFULL + buf), use & 1, false, ab, 5, t)) break;
      if (!waitw(bar(B_SSREADY + buf), use & 1, false, ab, 11, t)) break;
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * 64);
      float a0[16], a1[16], a2[16];             // columns 0..47: hi 0..23, lo 24..47
      tc_ld16(ta + 0, a0);
      tc_ld16(ta + 16, a1);
      tc_ld16(ta + 32, a2);
      tc_wait_ld();
      const float ss = ssbuf[buf * kTile + row];
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TEMPTY + buf));
      float mix[kMix];
#pragma unroll
      for (int c = 0; c < 8; ++c) mix[c] = a0[c] + a1[c + 8];
#pragma unroll
      for (int c = 8; c < 16; ++c) mix[c] = a0[c] + a2[c - 8];
#pragma unroll
      for (int c = 16; c < 24; ++c) mix[c] = a1[c - 16] + a2[c - 8];
      if (!waitw(bar(B_PFREE), (uint32_t)(t & 1) ^ 1, true, ab, 6, t)) break;
      const uint32_t dm = mapa(sb + kOffRecv + (uint32_t)(((crank * kOwn + (row % kOwn)) * kRw) * 4),
                               (uint32_t)(row / kOwn));
#pragma unroll
      for (int v = 0; v < 6; ++v)
        st_cluster_v4(dm + 16 * v, mix[4 * v], mix[4 * v + 1], mix[4 * v + 2], mix[4 * v + 3]);
      st_cluster_f32(dm + 4 * kMix, ss);
      fence_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_GALL));
      if (warp == kRead0) {
        if (!waitw(bar(B_GALL), (uint32_t)(t & 1), false, ab, 7, t)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PREADY), kCl);
        __syncwarp();
      }
      // ---- as owners: the kCl CTAs' partials of rows oq + 8 h, in CTA order ---
      if (!waitw(bar(B_PREADY), (uint32_t)(t & 1), true, ab, 8, t)) break;
      float acc0[F::kOwnPasses], acc1[F::kOwnPasses];
#pragma unroll
      for (int h = 0; h < F::kOwnPasses; ++h) {
        const int oq2 = oq + 8 * h;
        acc0[h] = 0.f;
        acc1[h] = 0.f;
#pragma unroll
        for (int src = 0; src < kCl; ++src) acc0[h] += recv[(src * kOwn + oq2) * kRw + e];
        if (e + 16 <= kMix) {
#pragma unroll
          for (int src = 0; src < kCl; ++src) acc1[h] += recv[(src * kOwn + oq2) * kRw + e + 16];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OPULL));
      if (warp == kRead0) {
        if (!waitw(bar(B_OPULL), (uint32_t)(t & 1), false, ab, 9, t)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PFREE), kCl);
        __syncwarp();
      }
#pragma unroll
      for (int h = 0; h < F::kOwnPasses; ++h) {
      const int oq2 = oq + 8 * h;
      const int64_t grow = (int64_t)(cid + t * ncl) * kTile + (int)crank * kOwn + oq2;
      float *rq = red + oq2 * kRw;
      rq[e] = acc0[h];
      if (e + 16 <= kMix) rq[e + 16] = acc1[h];
      __syncwarp();
      const float rsq = rsqrt_nr(fmaf(rq[kMix], 1.0f / (float)kK, a.rms_eps));
      float gate = 0.f;
      if (e < 8) {
        const float l = fmaf(rq[e] * rsq, e < 4 ? sc0 : sc1, bgate);
        const float sg = rcp_nr(1.0f + expf(-l));
        gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
      }
      const float lc = fmaf(rq[8 + e] * rsq, sc2, bcomb);
      if (grow < a.rows) {
        a.logit_ws[grow * 16 + e] = lc;
        if (e < 4) a.pre_ws[grow * kHC + e] = gate;
        if (e >= 4 && e < 8) a.post_out[grow * kHC + (e - 4)] = gate;
        if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
        if (a.mix_out) {
          a.mix_out[grow * kMix + e] = rq[e] * rsq;
          if (e < 8) a.mix_out[grow * kMix + 16 + e] = rq[16 + e] * rsq;
        }
      }
      __syncwarp();
      }
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

// fn [24, 20480] -> 640 blocks of 32 k (block i * 160 + h/32 for stream i):
// a 48 x 32 bf16 tile in 64-byte-swizzled K-major layout, row c = bf16(fn[c])
// (hi), row 24 + c = bf16(fn[c] - hi) (lo)
__global__ void __launch_bounds__(256) fn_prep_sw64_kernel(const float *__restrict__ fn,
                                                            uint8_t *__restrict__ fnp) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 256 + threadIdx.x;
  if (t >= kFnBlocks * kMix * 4) return;
  const int q = t & 3, c = (t >> 2) % kMix, kb = t / (4 * kMix);
  const int k0 = (kb / (kH / kBh)) * kH + (kb % (kH / kBh)) * kBh + 8 * q;
  const float4 f0 = __ldg(reinterpret_cast<const float4 *>(fn + (int64_t)c * kK + k0));
  const float4 f1 = __ldg(reinterpret_cast<const float4 *>(fn + (int64_t)c * kK + k0 + 4));
  const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * e]);
    const __nv_bfloat16 h1 = __float2bfloat16_rn(f[2 * e + 1]);
    hw[e] = pack2_rn(__bfloat162float(h0), __bfloat162float(h1));
    lw[e] = pack2_rn(f[2 * e] - __bfloat162float(h0), f[2 * e + 1] - __bfloat162float(h1));
  }
  uint8_t *blk = fnp + (size_t)kb * kFnBlkBytes;
  const int rh = c, rl = c + kMix;
  *reinterpret_cast<uint4 *>(blk + (rh >> 3) * 512 + (rh & 7) * 64 + ((q ^ ((rh >> 1) & 3)) << 4)) =
      make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4 *>(blk + (rl >> 3) * 512 + (rl & 7) * 64 + ((q ^ ((rl >> 1) & 3)) << 4)) =
      make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

std::mutex g_fpp_mu;
template <int kCl>
int g_fpp_clusters[64];   // per device: co-resident clusters (0: not configured)

template <int kCl>
cudaError_t fpp_configure(int dev, int *max_clusters) {
  std::lock_guard<std::mutex> lock(g_fpp_mu);
  if (g_fpp_clusters<kCl>[dev] > 0) {
    *max_clusters = g_fpp_clusters<kCl>[dev];
    return cudaSuccess;
  }
  constexpr int kSmemBytes = FGeo<kCl>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(post_pre_fused_kernel<kCl>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  // a cluster of 16 is a non-portable size
  if (e == cudaSuccess && kCl > 8)
    e = cudaFuncSetAttribute(post_pre_fused_kernel<kCl>,
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
  e = cudaOccupancyMaxActiveClusters(&n, post_pre_fused_kernel<kCl>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_fpp_clusters<kCl>[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

}  // namespace

namespace {
// 2D bf16 tensor map over [rows, cols] (row-major), 128-row x 32-column
// boxes, 64-byte swizzle
bool encode_rows(CUtensorMap *map, const uint16_t *base, int64_t cols, int64_t rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBh, (cuuint32_t)kTile};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), gdim, gstride,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t fused_fn_bytes() { return (size_t)kFnBlocks * kFnBlkBytes; }

cudaError_t launch_fn_prep_sw64(const float *fn, uint8_t *fnp, cudaStream_t s, bool pdl) {
  constexpr int kPrepItems = kFnBlocks * kMix * 4;
  return launch_pdl(fn_prep_sw64_kernel, dim3((kPrepItems + 255) / 256), dim3(256), 0, s, 1, pdl,
                    fn, fnp);
}

cudaError_t launch_post_pre_fused(const uint16_t *R, const uint16_t *y, const float *post,
                                  const float *comb, const float *fn, const float *scale,
                                  const float *base, int64_t rows, int64_t logical_rows,
                                  const mhc_params &p, float *pre_ws, float *logit_ws,
                                  const uint8_t *fnp, uint16_t *R_out, float *post_out,
                                  float *pre_out, float *mix_out, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  CUtensorMap map_r, map_y;
  if (!encode_rows(&map_r, R, kK, rows) || !encode_rows(&map_y, y, kH, rows))
    return cudaErrorInvalidValue;
  // fn == NULL: fnp already holds the image (prepared weights)
  if (fn) {
    e = launch_fn_prep_sw64(fn, const_cast<uint8_t *>(fnp), s, use_pdl(logical_rows));
    if (e != cudaSuccess) return e;
  }
  FusedArgs a;
  a.post_in = post;
  a.comb_in = comb;
  a.R_out = reinterpret_cast<uint4 *>(R_out);
  a.fnp = fnp; a.scale = scale; a.base = base;
  a.pre_ws = pre_ws; a.logit_ws = logit_ws; a.post_out = post_out;
  a.pre_out = pre_out; a.mix_out = mix_out;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTile - 1) / kTile);
  a.rms_eps = p.rms_eps; a.pre_eps = p.hc_pre_eps; a.post_mult = p.post_mult;
  // build and grid from the chunk's row count only (per-row arithmetic never
  // depends on the grid; the build fixes the order of the cross-CTA sums)
  auto go = [&](auto cl) -> cudaError_t {
    constexpr int kCl = decltype(cl)::value;
    int max_clusters = 0;
    cudaError_t e2 = fpp_configure<kCl>(dev, &max_clusters);
    if (e2 != cudaSuccess) return e2;
    const int64_t chunk_tiles = (logical_rows + kTile - 1) / kTile;
    const int clusters = (int)(chunk_tiles < max_clusters ? chunk_tiles : max_clusters);
    return launch_pdl(post_pre_fused_kernel<kCl>, dim3((unsigned)(clusters * kCl)),
                      dim3(kThreads), FGeo<kCl>::kSmemBytes, s, kCl, use_pdl(logical_rows),
                      map_r, map_y, a);
  };
  if (logical_rows >= kStreamMinRows) return go(std::integral_constant<int, 8>());
  return go(std::integral_constant<int, 16>());
}

cudaError_t fused_post_pre_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fpp_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_fpp_error, &z, sizeof z);
  }
  return e;
}

}  // namespace mhc
