// pre_fused.cu -- mhc_pre in one launch on GB300: stats on the 5th-generation
// tensor cores, split/Sinkhorn, combine + RMSNorm, reading R from HBM once.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre
// (hc_pre_torch_impl, hc_split_sinkhorn, the combine) with RMSNorm fused as in
// prefill_sp.py, hc_combine_norm_rows.
//
// Decomposition.  A cluster of 16 CTAs owns a 128-row tile at a time; CTA s
// owns hidden columns [320 s, 320 s + 320) of all four streams, i.e. 1280 of a
// row's 20480 k.  Per tile and CTA:
//   * TMA streams R[128 rows, 64 k] boxes (128B swizzle) through a 5-stage ring;
//   * one thread issues tcgen05.mma (M=128 rows, N=48, K=16, bf16 -> fp32 in
//     TMEM) against fn split into bf16 hi (rows 0..23) and lo (rows 24..47)
//     halves, resident in shared memory for the whole kernel (120 KB), so the
//     24 dot products carry ~2^-17 relative error per term;
//   * 16 "Gram" warps read the same stages and accumulate, per row, the ten
//     products G_ij = sum_h R_i[h] R_j[h] of the CTA's columns.  sum_k x_k^2 is
//     the trace of G, and the RMSNorm of y = sum_i pre_i R_i needs only
//     sum_h y_h^2 = pre^T G pre, so the norm is known before y is formed;
//   * the 34 partial sums per row go to the CTA that finalises the row (CTA s
//     owns tile rows 8s..8s+7), which pulls all 16 partials over DSMEM,
//     reduces them in CTA order, computes rsqrt, mix, gates and the 4x4
//     Sinkhorn (16 lanes per row), writes post/comb, and broadcasts
//     (pre, 1/rms(y)) back to the 16 CTAs' tables;
//   * 8 combine warps re-read the tile's own columns of R (still L2-resident:
//     the cluster's live tile is ~5 MB) and write x_norm.
// Roles run concurrently on consecutive tiles (two TMEM accumulators, two
// (pre, rnorm) tables), so HBM keeps streaming while a tile is finalised.
//
// Every row is reduced in one fixed order that depends only on its own data
// (same MMA sequence, same Gram lanes, CTA-ordered cross-CTA sums), so any
// row range gives the whole-chunk bits.
//
// Every wait is bounded (~2 s of wall time); on expiry a CTA raises an abort
// flag, records an error word, drains its in-flight MMAs and copies, frees
// its TMEM and returns.
#include <cuda.h>

#include <mutex>

#include "mhc_common.cuh"

namespace mhc {

// Bit s set: a bounded wait at site s expired (sites are numbered in the
// kernel); g_fused_where[s] holds (tile << 8) | cluster rank of the last one.
__device__ unsigned int g_fused_error;
__device__ unsigned int g_fused_where[32];
// Bit 16 + s: a wait at site s gave up because its CTA had already aborted.
__device__ unsigned int g_fused_where_aborted[32];

namespace {

// ---- geometry -------------------------------------------------------------
constexpr int kCl = 16;                       // CTAs per cluster (K split)
constexpr int kTile = 128;                    // rows per tile = UMMA M
constexpr int kHs = kH / kCl;                 // 320 hidden columns per CTA
constexpr int kBk = 64;                       // k per stage: 128-byte rows
constexpr int kHb = kHs / kBk;                // 5 column blocks per stream
constexpr int kKb = kHC * kHb;                // 20 k-blocks per tile per CTA
constexpr int kStages = 5;
constexpr int kN = 2 * kMix;                  // 48 = fn hi (24) + fn lo (24)
constexpr int kStageBytes = kTile * kBk * 2;  // 16384
constexpr int kFnBlkBytes = kN * kBk * 2;     // 6144
constexpr int kPw = 34;                       // partial words per row: 24 dots + 10 Gram
constexpr int kOwn = kTile / kCl;             // 8 rows finalised per CTA
constexpr int kPreW = 5;                      // table words per row: pre0..3, rnorm
constexpr int kChunks = kHs / 8;              // 40 16-byte chunks per stream and row
constexpr int kTmemCols = 128;                // two 48-column accumulators at 0 and 64

static_assert(kHs % kBk == 0 && kTile % kCl == 0, "");

// ---- warp roles -------------------------------------------------------------
constexpr int kProducerWarp = 0, kMmaWarp = 1;
constexpr int kGram0 = 2, kGramN = 16;
constexpr int kOwner0 = kGram0 + kGramN, kOwnerN = 4;
constexpr int kComb0 = kOwner0 + kOwnerN, kCombN = 8;
constexpr int kWarps = kComb0 + kCombN;       // 30
constexpr int kThreads = kWarps * 32;         // 960

// ---- shared memory (offsets from a 1024-byte aligned base) -----------------
constexpr int kOffFn = 0;
constexpr int kOffStage = kOffFn + kKb * kFnBlkBytes;
constexpr int kOffPart = kOffStage + kStages * kStageBytes;
constexpr int kOffTab = kOffPart + kTile * kPw * 4;
constexpr int kOffRed = kOffTab + 2 * kTile * kPreW * 4;
constexpr int kOffW = kOffRed + kOwn * kPw * 4;
constexpr int kOffBar = kOffW + kHs * 2;
// mbarrier slots (arrays are given explicit, non-overlapping ranges)
enum Bar : int {
  B_FULL = 0,                    // [kStages] TMA landed
  B_EMPTY = B_FULL + kStages,    // [kStages] MMA commit + 16 Gram warps done
  B_TFULL = B_EMPTY + kStages,   // [2] accumulator complete
  B_TEMPTY = B_TFULL + 2,        // [2] accumulator read by the 16 Gram warps
  B_PREADY = B_TEMPTY + 2,       // partials of all 16 CTAs published (remote)
  B_PFREE = B_PREADY + 1,        // our partials pulled by all 16 owners (remote)
  B_QREADY = B_PFREE + 1,        // [2] (pre, rnorm) table filled by 16 owners (remote)
  B_QFREE = B_QREADY + 2,        // [2] table consumed by all 16 CTAs (remote)
  B_GALL = B_QFREE + 2,          // 16 Gram warps wrote their partials
  B_OPULL = B_GALL + 1,          // 4 owner warps pulled
  B_OTAB = B_OPULL + 1,          // 4 owner warps wrote the tables
  B_CDONE = B_OTAB + 1,          // 8 combine warps done with a table
  B_DRAIN = B_CDONE + 1,         // final MMA drain
  B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT == 2 * kStages + 2 + 2 + 1 + 1 + 2 + 2 + 5, "barrier slots overlap");
constexpr int kOffMisc = kOffBar + B_COUNT * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
static_assert(kOffStage % 1024 == 0 && kFnBlkBytes % 1024 == 0, "SW128 tiles need 1024-B alignment");

constexpr uint64_t kTimeoutNs = 2000000000ull;

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
  return r;
}
__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
// arrive on the barrier at the same offset in CTA `cta` of this cluster
__device__ __forceinline__ void mbar_arrive_remote(uint32_t b, uint32_t cta) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa(b, cta))
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
// acquire at cluster scope: for barriers completed by other CTAs' arrivals
__device__ __forceinline__ bool mbar_test_cluster(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(b), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// tcgen05 (5th-generation tensor core, accumulator in tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_ld2(uint32_t taddr, float &v0, float &v1) {
  uint32_t r0, r1;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1) : "r"(taddr));
  v0 = __uint_as_float(r0);
  v1 = __uint_as_float(r1);
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // LBO (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // SBO
  d |= (uint64_t)1 << 46;                 // version
  d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, N = 48, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kTile >> 4) << 24);

// ---- bounded waits ------------------------------------------------------------
struct Abort {
  volatile int *flag;
  uint32_t rank;
  // a wait at `site` expired on tile `it`: stop the CTA, record where
  __device__ bool raise(int site, int it) const {
    *flag = 1;
    atomicOr(&g_fused_error, 1u << site);
    g_fused_where[site] = ((uint32_t)it << 8) | rank;
    return false;
  }
  // a wait at `site` gave up because the CTA aborted elsewhere
  __device__ bool follow(int site, int it) const {
    atomicOr(&g_fused_error, 1u << (16 + site));
    g_fused_where_aborted[site] = ((uint32_t)it << 8) | rank;
    return false;
  }
};

// one thread
__device__ __forceinline__ bool wait1(uint32_t b, uint32_t parity, bool cl, const Abort &ab,
                                      int site, int it) {
  if (cl ? mbar_test_cluster(b, parity) : mbar_test(b, parity)) return true;
  const uint64_t t0 = now_ns();
  for (;;) {
    if (cl ? mbar_test_cluster(b, parity) : mbar_test(b, parity)) return true;
    if (*ab.flag) return ab.follow(site, it);
    if (now_ns() - t0 > kTimeoutNs) return ab.raise(site, it);
  }
}
// whole warp; the outcome is warp-uniform
__device__ __forceinline__ bool waitw(uint32_t b, uint32_t parity, bool cl, const Abort &ab,
                                      int site, int it) {
  const uint64_t t0 = now_ns();
  for (;;) {
    const bool done = cl ? mbar_test_cluster(b, parity) : mbar_test(b, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    const bool expired = now_ns() - t0 > kTimeoutNs;
    if (__any_sync(0xffffffffu, expired || *ab.flag)) {
      const bool any_expired = __any_sync(0xffffffffu, expired);
      if ((threadIdx.x & 31) == 0) {
        if (any_expired) ab.raise(site, it);
        else ab.follow(site, it);
      }
      return false;
    }
  }
}

// bounded wait that ignores the abort flag: drains copies/MMAs already issued
__device__ __forceinline__ void drain1(uint32_t b, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (!mbar_test(b, parity) && now_ns() - t0 <= kTimeoutNs) {
  }
}

__device__ __forceinline__ float lo_bf(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

struct FusedArgs {
  const float *fn;
  const float *scale;
  const float *base;
  const uint16_t *norm_w;
  const uint16_t *R;
  uint16_t *x_norm;
  float *post;
  float *comb;
  float *pre_out;
  float *mix_out;
  int64_t rows;
  int num_tiles;
  float rms_eps, pre_eps, sink_eps, norm_eps, post_mult;
  int iters;
};

__global__ void __launch_bounds__(kThreads, 1)
pre_fused_kernel(const __grid_constant__ CUtensorMap tmap, const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int my_tiles = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  Abort ab{reinterpret_cast<volatile int *>(sm + kOffMisc + 4), crank};

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *ab.flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1 + kGramN);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_TFULL + b), 1);
      mbar_init(bar(B_TEMPTY + b), kGramN);
      mbar_init(bar(B_QREADY + b), kCl);
      mbar_init(bar(B_QFREE + b), kCl);
    }
    mbar_init(bar(B_PREADY), kCl);
    mbar_init(bar(B_PFREE), kCl);
    mbar_init(bar(B_GALL), kGramN);
    mbar_init(bar(B_OPULL), kOwnerN);
    mbar_init(bar(B_OTAB), kOwnerN);
    mbar_init(bar(B_CDONE), kCombN);
    mbar_init(bar(B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);

  // fn columns of this CTA -> bf16 hi/lo B tiles (K-major, 128-byte swizzle):
  // k-block j covers k = (j%4)*5120 + 320*crank + 64*(j/4) + [0, 64)
  for (int item = threadIdx.x; item < kMix * kKb * 8; item += kThreads) {
    const int q = item & 7, j = (item >> 3) % kKb, c = item / (8 * kKb);
    const int k0 = (j & 3) * kH + (int)crank * kHs + (j >> 2) * kBk + 8 * q;
    const float4 f0 = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + k0));
    const float4 f1 = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + k0 + 4));
    const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * e]);
      const __nv_bfloat16 h1 = __float2bfloat16_rn(f[2 * e + 1]);
      hw[e] = pack2_rn(__bfloat162float(h0), __bfloat162float(h1));
      lw[e] = pack2_rn(f[2 * e] - __bfloat162float(h0), f[2 * e + 1] - __bfloat162float(h1));
    }
    uint8_t *tile = sm + kOffFn + j * kFnBlkBytes;
    const int nh = c, nl = c + kMix;
    *reinterpret_cast<uint4 *>(tile + (nh >> 3) * 1024 + (nh & 7) * 128 + ((q ^ (nh & 7)) << 4)) =
        make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(tile + (nl >> 3) * 1024 + (nl & 7) * 128 + ((q ^ (nl & 7)) << 4)) =
        make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  if (threadIdx.x < kChunks)
    reinterpret_cast<uint4 *>(sm + kOffW)[threadIdx.x] =
        __ldg(reinterpret_cast<const uint4 *>(a.norm_w + crank * kHs) + threadIdx.x);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *tmem_slot;

  // ---- roles -------------------------------------------------------------------
  if (warp == kProducerWarp) {
    // the whole warp walks the loop (waits are warp-collective); lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    int last[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last[s] = -1;
    bool ok = true;
    for (int it = 0; it < my_tiles && ok; ++it) {
      const int y = (cid + it * ncl) * kTile;
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_EMPTY + stage), phase ^ 1, false, ab, 1, it)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(bar(B_FULL + stage), kStageBytes);
          const int x = (j & 3) * kH + (int)crank * kHs + (j >> 2) * kBk;
          tma_load_2d(sb + kOffStage + stage * kStageBytes, &tmap, x, y, bar(B_FULL + stage));
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
    bool ok = true;
    for (int it = 0; it < my_tiles && ok; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!waitw(bar(B_TEMPTY + buf), (use & 1) ^ 1, false, ab, 2, it)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * 64);
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_FULL + stage), phase, false, ab, 3, it)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t ad = sw128_desc(sb + kOffStage + stage * kStageBytes);
          const uint64_t bd = sw128_desc(sb + kOffFn + j * kFnBlkBytes);
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk)
            tc_mma(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (j | kk) != 0);
          tc_commit(bar(B_EMPTY + stage));
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (ok && lane == 0) tc_commit(bar(B_TFULL + buf));
      __syncwarp();
    }
    // all issued MMAs complete before TMEM is freed
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp < kOwner0) {
    // ---- Gram warps: per-row stream Gram matrix + TMEM readout ---------------
    const int gw = warp - kGram0;
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int part = gw >> 2;                   // 0..3
    const int grow = 32 * quarter + 8 * part + (lane >> 2);
    const int hq = lane & 3;                    // 16 columns of a 64-column block
    const int trow = 32 * quarter + lane;       // row of this lane in TMEM
    const int sw = grow & 7;
    float *P = reinterpret_cast<float *>(sm + kOffPart);
    int stage = 0;
    uint32_t phase = 0;
    for (int it = 0; it < my_tiles; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      float g00 = 0.f, g01 = 0.f, g02 = 0.f, g03 = 0.f, g11 = 0.f, g12 = 0.f, g13 = 0.f,
            g22 = 0.f, g23 = 0.f, g33 = 0.f;
      uint32_t v0[8], v1[8], v2[8];
      bool ok = true;
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_FULL + stage), phase, false, ab, 4, it)) { ok = false; break; }
        const uint8_t *st = sm + kOffStage + stage * kStageBytes + grow * 128;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(st + (((2 * hq) ^ sw) << 4));
        const uint4 c1 = *reinterpret_cast<const uint4 *>(st + (((2 * hq + 1) ^ sw) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + stage));
        if (++stage == kStages) { stage = 0; phase ^= 1; }
        const uint32_t cur[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        switch (j & 3) {
          case 0:
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a0 = lo_bf(cur[e]), a1 = hi_bf(cur[e]);
              g00 = fmaf(a0, a0, g00); g00 = fmaf(a1, a1, g00);
              v0[e] = cur[e];
            }
            break;
          case 1:
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a0 = lo_bf(cur[e]), a1 = hi_bf(cur[e]);
              const float p0 = lo_bf(v0[e]), p1 = hi_bf(v0[e]);
              g11 = fmaf(a0, a0, g11); g11 = fmaf(a1, a1, g11);
              g01 = fmaf(p0, a0, g01); g01 = fmaf(p1, a1, g01);
              v1[e] = cur[e];
            }
            break;
          case 2:
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a0 = lo_bf(cur[e]), a1 = hi_bf(cur[e]);
              const float p0 = lo_bf(v0[e]), p1 = hi_bf(v0[e]);
              const float q0 = lo_bf(v1[e]), q1 = hi_bf(v1[e]);
              g22 = fmaf(a0, a0, g22); g22 = fmaf(a1, a1, g22);
              g02 = fmaf(p0, a0, g02); g02 = fmaf(p1, a1, g02);
              g12 = fmaf(q0, a0, g12); g12 = fmaf(q1, a1, g12);
              v2[e] = cur[e];
            }
            break;
          default:
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a0 = lo_bf(cur[e]), a1 = hi_bf(cur[e]);
              const float p0 = lo_bf(v0[e]), p1 = hi_bf(v0[e]);
              const float q0 = lo_bf(v1[e]), q1 = hi_bf(v1[e]);
              const float r0 = lo_bf(v2[e]), r1 = hi_bf(v2[e]);
              g33 = fmaf(a0, a0, g33); g33 = fmaf(a1, a1, g33);
              g03 = fmaf(p0, a0, g03); g03 = fmaf(p1, a1, g03);
              g13 = fmaf(q0, a0, g13); g13 = fmaf(q1, a1, g13);
              g23 = fmaf(r0, a0, g23); g23 = fmaf(r1, a1, g23);
            }
            break;
        }
      }
      if (!ok) break;
      // this tile's accumulator: hi and lo halves of 6 of the 24 mixes
      if (!waitw(bar(B_TFULL + buf), use & 1, false, ab, 5, it)) break;
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * 64 + 6 * part);
      float hv[6], lv[6];   // columns 6p..6p+5 (hi) and 24+6p.. (lo), even-aligned pairs
      tc_ld2(ta + 0, hv[0], hv[1]);
      tc_ld2(ta + 2, hv[2], hv[3]);
      tc_ld2(ta + 4, hv[4], hv[5]);
      tc_ld2(ta + kMix + 0, lv[0], lv[1]);
      tc_ld2(ta + kMix + 2, lv[2], lv[3]);
      tc_ld2(ta + kMix + 4, lv[4], lv[5]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TEMPTY + buf));
      // Gram partials of the row: lanes 4r'..4r'+3 hold its four column quarters
      float gg[10] = {g00, g01, g02, g03, g11, g12, g13, g22, g23, g33};
#pragma unroll
      for (int t = 0; t < 10; ++t) {
        gg[t] += __shfl_xor_sync(0xffffffffu, gg[t], 1);
        gg[t] += __shfl_xor_sync(0xffffffffu, gg[t], 2);
      }
      if (!waitw(bar(B_PFREE), (uint32_t)(it & 1) ^ 1, true, ab, 6, it)) break;
      float *pr = P + trow * kPw + 6 * part;
#pragma unroll
      for (int t = 0; t < 6; ++t) pr[t] = hv[t] + lv[t];
      if (hq == 0) {
#pragma unroll
        for (int t = 0; t < 10; ++t) P[grow * kPw + kMix + t] = gg[t];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_GALL));
      if (warp == kGram0) {
        if (!waitw(bar(B_GALL), (uint32_t)(it & 1), false, ab, 7, it)) break;
        if (lane == 0) {
          fence_cluster();
          for (uint32_t dst = 0; dst < kCl; ++dst) mbar_arrive_remote(bar(B_PREADY), dst);
        }
        __syncwarp();
      }
    }
  } else if (warp < kComb0) {
    // ---- owner warps: finalise 8 rows of each tile --------------------------
    const int o = threadIdx.x - kOwner0 * 32;   // 0..127
    const int q = o >> 4, e = o & 15;           // row of 8, lane of 16
    const int row_t = (int)crank * kOwn + q;
    float *red = reinterpret_cast<float *>(sm + kOffRed);
    const float sc0 = __ldg(a.scale), sc1 = __ldg(a.scale + 1), sc2 = __ldg(a.scale + 2);
    const float bcomb = __ldg(a.base + 8 + e);
    const float bgate = e < 8 ? __ldg(a.base + e) : 0.f;
    // a row's 16 lanes are one half of the warp; xor 1/2/4/8 stay inside it
    const unsigned gmask = 0xffffffffu;
    for (int it = 0; it < my_tiles; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      const int64_t grow = (int64_t)(cid + it * ncl) * kTile + row_t;
      if (!waitw(bar(B_PREADY), (uint32_t)(it & 1), true, ab, 8, it)) break;
      // pull this row's 34 partials from the 16 CTAs, summed in CTA order
      const uint32_t pa = sb + kOffPart + (uint32_t)(row_t * kPw) * 4u;
      float acc[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int w3 = 0; w3 < 3; ++w3) {
        const int v = e + 16 * w3;
        if (v < kPw) {
          float tv[kCl];
#pragma unroll
          for (int src = 0; src < kCl; ++src) {
            asm volatile("ld.shared::cluster.f32 %0, [%1];"
                         : "=f"(tv[src]) : "r"(mapa(pa + 4u * (uint32_t)v, (uint32_t)src)));
          }
          float s = 0.f;
#pragma unroll
          for (int src = 0; src < kCl; ++src) s += tv[src];
          acc[w3] = s;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OPULL));
      if (warp == kOwner0) {
        if (!waitw(bar(B_OPULL), (uint32_t)(it & 1), false, ab, 9, it)) break;
        if (lane == 0) {
          fence_cluster();
          for (uint32_t dst = 0; dst < kCl; ++dst) mbar_arrive_remote(bar(B_PFREE), dst);
        }
        __syncwarp();
      }
      float *rq = red + q * kPw;
      rq[e] = acc[0];
      rq[e + 16] = acc[1];
      if (e < 2) rq[e + 32] = acc[2];
      __syncwarp();
      const float G00 = rq[24], G01 = rq[25], G02 = rq[26], G03 = rq[27], G11 = rq[28];
      const float G12 = rq[29], G13 = rq[30], G22 = rq[31], G23 = rq[32], G33 = rq[33];
      const float ss = ((G00 + G11) + G22) + G33;
      const float rsq = 1.0f / sqrtf(ss / (float)kK + a.rms_eps);
      // Sinkhorn on exp(logits): lane e holds comb[e/4][e%4]
      float C = expf(fmaf(rq[8 + e] * rsq, sc2, bcomb));
      for (int t = 0; t < a.iters; ++t) {
        float rs = C + __shfl_xor_sync(gmask, C, 1);
        rs = rs + __shfl_xor_sync(gmask, rs, 2);
        C = C / (rs + a.sink_eps);
        float cs = C + __shfl_xor_sync(gmask, C, 4);
        cs = cs + __shfl_xor_sync(gmask, cs, 8);
        C = C / (cs + a.sink_eps);
      }
      // gates: lanes 0..3 pre, 4..7 post
      float gate = 0.f;
      if (e < 8) {
        const float l = fmaf(rq[e] * rsq, e < 4 ? sc0 : sc1, bgate);
        const float sg = 1.0f / (1.0f + expf(-l));
        gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
      }
      const int gb = lane & 16;
      const float p0 = __shfl_sync(gmask, gate, gb + 0), p1 = __shfl_sync(gmask, gate, gb + 1);
      const float p2 = __shfl_sync(gmask, gate, gb + 2), p3 = __shfl_sync(gmask, gate, gb + 3);
      // sum_h y_h^2 = pre^T G pre
      float yy = p0 * p0 * G00 + p1 * p1 * G11 + p2 * p2 * G22 + p3 * p3 * G33;
      yy += 2.0f * (p0 * p1 * G01 + p0 * p2 * G02 + p0 * p3 * G03 + p1 * p2 * G12 +
                    p1 * p3 * G13 + p2 * p3 * G23);
      yy = fmaxf(yy, 0.f);
      const float rn = 1.0f / sqrtf(yy / (float)kH + a.norm_eps);
      if (grow < a.rows) {
        a.comb[grow * 16 + e] = C;
        if (e >= 4 && e < 8) a.post[grow * kHC + (e - 4)] = gate;
        if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
        if (a.mix_out) {
          a.mix_out[grow * kMix + e] = rq[e] * rsq;
          if (e < 8) a.mix_out[grow * kMix + 16 + e] = rq[16 + e] * rsq;
        }
      }
      // (pre, rnorm) of this row into table `buf` of CTA e
      if (!waitw(bar(B_QFREE + buf), (use & 1) ^ 1, true, ab, 10, it)) break;
      const uint32_t ta = mapa(sb + kOffTab + (uint32_t)((buf * kTile + row_t) * kPreW) * 4u, (uint32_t)e);
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ta), "f"(p0) : "memory");
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ta + 4), "f"(p1) : "memory");
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ta + 8), "f"(p2) : "memory");
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ta + 12), "f"(p3) : "memory");
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ta + 16), "f"(rn) : "memory");
      fence_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OTAB));
      if (warp == kOwner0) {
        if (!waitw(bar(B_OTAB), (uint32_t)(it & 1), false, ab, 11, it)) break;
        if (lane == 0) {
          fence_cluster();
          for (uint32_t dst = 0; dst < kCl; ++dst) mbar_arrive_remote(bar(B_QREADY + buf), dst);
        }
        __syncwarp();
      }
    }
  } else {
    // ---- combine warps: x_norm of this CTA's 320 columns ---------------------
    const int ct = threadIdx.x - kComb0 * 32;    // 0..255
    const float *tabs = reinterpret_cast<const float *>(sm + kOffTab);
    const uint4 *wv = reinterpret_cast<const uint4 *>(sm + kOffW);
    for (int it = 0; it < my_tiles; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      const int64_t row0 = (int64_t)(cid + it * ncl) * kTile;
      if (!waitw(bar(B_QREADY + buf), use & 1, true, ab, 12, it)) break;
      const float *tab = tabs + buf * kTile * kPreW;
      constexpr int kItems = kTile * kChunks;          // 5120
      constexpr int kPer = kItems / (kCombN * 32);     // 20
#pragma unroll 1
      for (int n = 0; n < kPer; n += 2) {
        uint4 rv[2][kHC];
        int rt[2], cc[2];
        bool live[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int item = ct + (kCombN * 32) * (n + u);
          rt[u] = item / kChunks;
          cc[u] = item - rt[u] * kChunks;
          live[u] = row0 + rt[u] < a.rows;
          if (live[u]) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                a.R + (row0 + rt[u]) * kK + (int64_t)crank * kHs + 8 * cc[u]);
#pragma unroll
            for (int i = 0; i < kHC; ++i) rv[u][i] = ld_stream(src + i * (kH / 8));
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (!live[u]) continue;
          const float *tr = tab + rt[u] * kPreW;
          const float q0 = tr[0], q1 = tr[1], q2 = tr[2], q3 = tr[3], rn = tr[4];
          const uint4 wq = wv[cc[u]];
          const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w};
          const uint32_t s0[4] = {rv[u][0].x, rv[u][0].y, rv[u][0].z, rv[u][0].w};
          const uint32_t s1[4] = {rv[u][1].x, rv[u][1].y, rv[u][1].z, rv[u][1].w};
          const uint32_t s2[4] = {rv[u][2].x, rv[u][2].y, rv[u][2].z, rv[u][2].w};
          const uint32_t s3[4] = {rv[u][3].x, rv[u][3].y, rv[u][3].z, rv[u][3].w};
          uint32_t ow[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            float ya = q0 * lo_bf(s0[x]);
            ya = fmaf(q1, lo_bf(s1[x]), ya);
            ya = fmaf(q2, lo_bf(s2[x]), ya);
            ya = fmaf(q3, lo_bf(s3[x]), ya);
            float yb = q0 * hi_bf(s0[x]);
            yb = fmaf(q1, hi_bf(s1[x]), yb);
            yb = fmaf(q2, hi_bf(s2[x]), yb);
            yb = fmaf(q3, hi_bf(s3[x]), yb);
            ow[x] = pack2_rn((ya * rn) * lo_bf(ww[x]), (yb * rn) * hi_bf(ww[x]));
          }
          st_stream(reinterpret_cast<uint4 *>(a.x_norm + (row0 + rt[u]) * kH +
                                              (int64_t)crank * kHs + 8 * cc[u]),
                    make_uint4(ow[0], ow[1], ow[2], ow[3]));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_CDONE));
      if (warp == kComb0) {
        if (!waitw(bar(B_CDONE), (uint32_t)(it & 1), false, ab, 13, it)) break;
        if (lane == 0) {
          fence_cluster();
          for (uint32_t dst = 0; dst < kCl; ++dst) mbar_arrive_remote(bar(B_QFREE + buf), dst);
        }
        __syncwarp();
      }
    }
  }

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
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

constexpr int kMaxDev = 64;
std::mutex g_dev_mu;
int g_max_clusters[kMaxDev];   // 0: not yet configured on that device

cudaError_t configure(int dev, int *max_clusters) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_max_clusters[dev] > 0) {
    *max_clusters = g_max_clusters[dev];
    return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(pre_fused_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pre_fused_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  e = cudaOccupancyMaxActiveClusters(&n, pre_fused_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_max_clusters[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_pre_fused(const uint16_t *R, const float *fn, const float *scale,
                             const float *base, const uint16_t *norm_w, int64_t rows,
                             int64_t logical_rows, const mhc_params &p, uint16_t *x_norm,
                             float *post, float *comb, float *pre_out, float *mix_out,
                             cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  int max_clusters = 0;
  e = configure(dev, &max_clusters);
  if (e != cudaSuccess) return e;

  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)kK, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)kK * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBk, (cuuint32_t)kTile};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(R), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  FusedArgs a;
  a.fn = fn; a.scale = scale; a.base = base; a.norm_w = norm_w; a.R = R;
  a.x_norm = x_norm; a.post = post; a.comb = comb; a.pre_out = pre_out; a.mix_out = mix_out;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTile - 1) / kTile);
  a.rms_eps = p.rms_eps; a.pre_eps = p.hc_pre_eps; a.sink_eps = p.hc_sinkhorn_eps;
  a.norm_eps = p.norm_eps; a.post_mult = p.post_mult; a.iters = p.sinkhorn_iters;

  // grid: as many clusters as fit at once, never more than the whole chunk's
  // tiles (the count depends on logical_rows only; per-row arithmetic does not
  // depend on it at all)
  const int64_t chunk_tiles = (logical_rows + kTile - 1) / kTile;
  const int clusters = (int)(chunk_tiles < max_clusters ? chunk_tiles : max_clusters);

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  cfg.gridDim = dim3((unsigned)(clusters * kCl));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pre_fused_kernel, map, a);
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
