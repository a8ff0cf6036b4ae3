// pre_fused.cu -- mhc_pre in one launch on GB300: stats on the 5th-generation
// tensor cores, split/Sinkhorn, combine + RMSNorm, reading R from HBM once.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre
// (hc_pre_torch_impl, hc_split_sinkhorn, the combine) with RMSNorm fused as in
// prefill_sp.py, hc_combine_norm_rows.
//
// Decomposition.  A cluster of 16 CTAs owns a 128-row tile at a time; CTA s
// owns hidden columns [320 s, 320 s + 320) of all four streams, i.e. 1280 of a
// row's 20480 k.  fn's 24 x 1280 slice of the CTA, split into bf16 hi (B rows
// 0..23) and lo (rows 24..47) halves, stays in shared memory (120 KB) for the
// whole kernel, so each of the 24 dot products carries ~2^-17 relative error
// per term.  One TMA ring (5 x 16 KB stages of R[128 rows, 64 k], 128-byte
// swizzle) carries, per CTA, the sequence
//     stats(0), stats(1), combine(0), stats(2), combine(1), ...
// where stats(t) reads tile t from HBM and combine(t) reads it again one tile
// later, while it is still resident in L2.
//   * stats blocks: one thread issues tcgen05.mma (M=128 rows, N=48, K=16,
//     bf16 -> fp32 in TMEM, two accumulators); 16 row warps (4 lanes per row,
//     16 columns each) accumulate the ten per-row stream products
//     G_ij = sum_h R_i[h] R_j[h].  sum_k x_k^2 is the trace of G and the
//     RMSNorm of y = sum_i pre_i R_i needs only sum_h y_h^2 = pre^T G pre,
//     so the norm is known before y is formed;
//   * end of stats(t): the row warps read the accumulator and push each row's
//     34 partial sums into the receive buffer of the CTA that finalises it
//     (CTA s owns tile rows 8s..8s+7).  The owner reduces the 16 partials in
//     CTA order, computes rsqrt, mix and the gates, pushes (pre, 1/rms(y)) to
//     all 16 CTAs, and only then runs the 4x4 Sinkhorn (16 lanes per row) and
//     writes post/comb;
//   * combine blocks: the row warps form y from the four stream blocks of a
//     64-column block and write x_norm.
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

namespace mhc {

// Bit s set: a bounded wait at site s expired (sites are numbered in the
// kernel); g_fused_where[s] holds (tile << 8) | cluster rank of the last one.
__device__ unsigned int g_fused_error;
__device__ unsigned int g_fused_where[32];
// Bit 16 + s: a wait at site s gave up because its CTA had already aborted.
__device__ unsigned int g_fused_where_aborted[32];

#ifdef MHC_TRACE
// Diagnostic builds only: per-CTA timestamps of pipeline events.
constexpr int kTraceTiles = 32, kTraceEv = 16, kTraceSlots = kTraceTiles * kTraceEv;
__device__ unsigned long long *g_trace;
#define MHC_TRACE_AT(tile, ev)                                                         \
  do {                                                                                 \
    if (g_trace && (tile) < kTraceTiles)                                               \
      g_trace[(size_t)blockIdx.x * kTraceSlots + (tile) * kTraceEv + (ev)] = now_ns(); \
  } while (0)
#else
#define MHC_TRACE_AT(tile, ev) \
  do {                         \
  } while (0)
#endif

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
constexpr int kRow0 = 2, kRowN = 16;          // row warps: Gram, readout, combine
constexpr int kOwner0 = kRow0 + kRowN, kOwnerN = 4;
constexpr int kWarps = kOwner0 + kOwnerN;     // 22
constexpr int kThreads = kWarps * 32;         // 704

// ---- shared memory (offsets from a 1024-byte aligned base) -----------------
constexpr int kOffFn = 0;
constexpr int kOffStage = kOffFn + kKb * kFnBlkBytes;
constexpr int kOffRecv = kOffStage + kStages * kStageBytes;   // [16 src][8 rows][34]
constexpr int kOffTab = kOffRecv + kCl * kOwn * kPw * 4;      // [2][128 rows][5]
constexpr int kOffRed = kOffTab + 2 * kTile * kPreW * 4;      // [8 rows][34]
constexpr int kOffW = kOffRed + kOwn * kPw * 4;
constexpr int kOffBar = kOffW + kHs * 2;
// mbarrier slots (arrays are given explicit, non-overlapping ranges)
enum Bar : int {
  B_FULL = 0,                    // [kStages] TMA landed
  B_EMPTY = B_FULL + kStages,    // [kStages] MMA role + 16 row warps done with the stage
  B_TFULL = B_EMPTY + kStages,   // [2] accumulator complete
  B_TEMPTY = B_TFULL + 2,        // [2] accumulator read by the 16 row warps
  B_PREADY = B_TEMPTY + 2,       // all 16 CTAs pushed partials to us (remote)
  B_PFREE = B_PREADY + 1,        // all 16 owners consumed our previous push (remote)
  B_QREADY = B_PFREE + 1,        // [2] (pre, rnorm) table filled by 16 owners (remote)
  B_QFREE = B_QREADY + 2,        // [2] table consumed by all 16 CTAs (remote)
  B_GALL = B_QFREE + 2,          // 16 row warps pushed their partials
  B_OPULL = B_GALL + 1,          // 4 owner warps read the receive buffer
  B_OTAB = B_OPULL + 1,          // 4 owner warps pushed the tables
  B_CDONE = B_OTAB + 1,          // 16 row warps done with a combine
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
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Arrive on the barrier at the same offset in every CTA of the cluster: one
// cluster-scope fence orders this thread's earlier writes (and those it has
// observed) before the arrivals, which are then relaxed.  (A release arrive
// per CTA would fence 16 times.)
__device__ __forceinline__ void arrive_all_ctas(uint32_t b, uint32_t n_cta) {
  fence_cluster();
  for (uint32_t dst = 0; dst < n_cta; ++dst)
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa(b, dst))
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
      mbar_init(bar(B_EMPTY + s), 1 + kRowN);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_TFULL + b), 1);
      mbar_init(bar(B_TEMPTY + b), kRowN);
      mbar_init(bar(B_QREADY + b), kCl);
      mbar_init(bar(B_QFREE + b), kCl);
    }
    mbar_init(bar(B_PREADY), kCl);
    mbar_init(bar(B_PFREE), kCl);
    mbar_init(bar(B_GALL), kRowN);
    mbar_init(bar(B_OPULL), kOwnerN);
    mbar_init(bar(B_OTAB), kOwnerN);
    mbar_init(bar(B_CDONE), kRowN);
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
  // Per CTA the block sequence is stats(0); then for t >= 1: stats(t),
  // combine(t-1); and combine(T-1) last.  Every ring role walks it in order.
  const int T = my_tiles;
  if (warp == kProducerWarp) {
    // the whole warp walks the sequence (waits are warp-collective); lane 0 issues
    int stage = 0;
    uint32_t phase = 0;
    int last[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last[s] = -1;
    bool ok = true;
    for (int it = 0; it <= T && ok; ++it) {
      for (int kind = 0; kind < 2 && ok; ++kind) {
        const int t = kind == 0 ? it : it - 1;       // stats(it), then combine(it-1)
        if (t < 0 || t >= T) continue;
        if (kind == 1 && lane == 0) MHC_TRACE_AT(t, 2);
        if (kind == 1 &&
            !waitw(bar(B_QREADY + (t & 1)), (uint32_t)(t >> 1) & 1, true, ab, 12, t)) {
          ok = false;
          break;
        }
        const int y = (cid + t * ncl) * kTile;
        if (lane == 0) MHC_TRACE_AT(t, kind == 0 ? 0 : 3);
        for (int j = 0; j < kKb; ++j) {
          if (!waitw(bar(B_EMPTY + stage), phase ^ 1, false, ab, 1, t)) { ok = false; break; }
          if (lane == 0) {
            mbar_expect_tx(bar(B_FULL + stage), kStageBytes);
            const int x = (j & 3) * kH + (int)crank * kHs + (j >> 2) * kBk;
            tma_load_2d(sb + kOffStage + stage * kStageBytes, &tmap, x, y, bar(B_FULL + stage));
          }
          __syncwarp();
          last[stage] = (int)phase;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (lane == 0) MHC_TRACE_AT(t, kind == 0 ? 1 : 4);
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
    for (int it = 0; it <= T && ok; ++it) {
      if (it < T) {                                   // stats(it): 20 k-blocks into TMEM
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!waitw(bar(B_TEMPTY + buf), (use & 1) ^ 1, false, ab, 2, it)) break;
        tc_fence_after();
        if (lane == 0) MHC_TRACE_AT(it, 5);
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
        if (!ok) break;
        if (lane == 0) tc_commit(bar(B_TFULL + buf));
        if (lane == 0) MHC_TRACE_AT(it, 6);
        __syncwarp();
      }
      if (it >= 1) {                                  // combine(it-1): not ours, release
        for (int j = 0; j < kKb; ++j) {
          if (!waitw(bar(B_FULL + stage), phase, false, ab, 3, it - 1)) { ok = false; break; }
          if (lane == 0) mbar_arrive(bar(B_EMPTY + stage));
          __syncwarp();
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
    // all issued MMAs complete before TMEM is freed
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp < kOwner0) {
    // ---- row warps: Gram + accumulator readout (stats), x_norm (combine) -----
    const int rw = warp - kRow0;
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int part = rw >> 2;                   // 0..3
    const int grow = 32 * quarter + 8 * part + (lane >> 2);   // row of the stage work
    const int hq = lane & 3;                    // 16 columns of a 64-column block
    const int trow = 32 * quarter + lane;       // row of this lane in TMEM
    const int sw = grow & 7;
    const float *tabs = reinterpret_cast<const float *>(sm + kOffTab);
    const uint4 *wsm = reinterpret_cast<const uint4 *>(sm + kOffW);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // 16 bf16 of this lane's row in the current stage -> fp32
    auto load16 = [&](float (&x)[16]) {
      const uint8_t *st = sm + kOffStage + stage * kStageBytes + grow * 128;
      const uint4 c0 = *reinterpret_cast<const uint4 *>(st + (((2 * hq) ^ sw) << 4));
      const uint4 c1 = *reinterpret_cast<const uint4 *>(st + (((2 * hq + 1) ^ sw) << 4));
      const uint32_t w8[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[2 * e] = lo_bf(w8[e]);
        x[2 * e + 1] = hi_bf(w8[e]);
      }
    };
    // every lane's reads of the stage are complete (their values were used)
    // before the warp's arrival lets the producer refill it
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EMPTY + stage));
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    };
    for (int it = 0; it <= T && ok; ++it) {
      if (it < T) {
        // ---- stats(it)
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        float g00 = 0.f, g01 = 0.f, g02 = 0.f, g03 = 0.f, g11 = 0.f, g12 = 0.f, g13 = 0.f,
              g22 = 0.f, g23 = 0.f, g33 = 0.f;
        float s0[16], s1[16], s2[16];
        for (int hb = 0; hb < kHb && ok; ++hb) {
#pragma unroll
          for (int i = 0; i < kHC; ++i) {
            if (!waitw(bar(B_FULL + stage), phase, false, ab, 4, it)) { ok = false; break; }
            if (hb == 0 && i == 0 && warp == kRow0 && lane == 0) MHC_TRACE_AT(it, 7);
            float x[16];
            load16(x);
            if (i == 0) {
#pragma unroll
              for (int e = 0; e < 16; ++e) { g00 = fmaf(x[e], x[e], g00); s0[e] = x[e]; }
            } else if (i == 1) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                g11 = fmaf(x[e], x[e], g11); g01 = fmaf(s0[e], x[e], g01); s1[e] = x[e];
              }
            } else if (i == 2) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                g22 = fmaf(x[e], x[e], g22); g02 = fmaf(s0[e], x[e], g02);
                g12 = fmaf(s1[e], x[e], g12); s2[e] = x[e];
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                g33 = fmaf(x[e], x[e], g33); g03 = fmaf(s0[e], x[e], g03);
                g13 = fmaf(s1[e], x[e], g13); g23 = fmaf(s2[e], x[e], g23);
              }
            }
            // the stage is released only after every lane has used its data
            release();
          }
        }
        if (!ok) break;
        if (warp == kRow0 && lane == 0) MHC_TRACE_AT(it, 8);
        // accumulator: hi and lo halves of mixes 6*part .. 6*part+5 of row trow
        if (!waitw(bar(B_TFULL + buf), use & 1, false, ab, 5, it)) break;
        if (warp == kRow0 && lane == 0) MHC_TRACE_AT(it, 9);
        tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * 64 + 6 * part);
        float hv[6], lv[6];
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
        // Gram of the row: lanes 4r'..4r'+3 hold its four column quarters
        float gg[10] = {g00, g01, g02, g03, g11, g12, g13, g22, g23, g33};
#pragma unroll
        for (int q = 0; q < 10; ++q) {
          gg[q] += __shfl_xor_sync(0xffffffffu, gg[q], 1);
          gg[q] += __shfl_xor_sync(0xffffffffu, gg[q], 2);
        }
        // push the partials into the owners' receive buffers
        if (!waitw(bar(B_PFREE), (uint32_t)(it & 1) ^ 1, true, ab, 6, it)) break;
        {
          const uint32_t dst = mapa(sb + kOffRecv +
                                        (uint32_t)(((crank * kOwn + (trow & 7)) * kPw + 6 * part) * 4),
                                    (uint32_t)(trow >> 3));
#pragma unroll
          for (int q = 0; q < 6; ++q)
            asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + 4 * q), "f"(hv[q] + lv[q])
                         : "memory");
          if (hq == 0) {
            const uint32_t dg = mapa(sb + kOffRecv +
                                         (uint32_t)(((crank * kOwn + (grow & 7)) * kPw + kMix) * 4),
                                     (uint32_t)(grow >> 3));
#pragma unroll
            for (int q = 0; q < 10; ++q)
              asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dg + 4 * q), "f"(gg[q])
                           : "memory");
          }
        }
        fence_cluster();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_GALL));
        if (warp == kRow0) {
          if (!waitw(bar(B_GALL), (uint32_t)(it & 1), false, ab, 7, it)) break;
          if (lane == 0)
            arrive_all_ctas(bar(B_PREADY), kCl);
          if (lane == 0) MHC_TRACE_AT(it, 10);
          __syncwarp();
        }
      }
      if (it >= 1) {
        // ---- combine(t): y = sum_i pre_i R_i, x_norm = bf16(y * rnorm * w)
        const int t = it - 1;
        if (!waitw(bar(B_QREADY + (t & 1)), (uint32_t)(t >> 1) & 1, true, ab, 12, t)) break;
        if (warp == kRow0 && lane == 0) MHC_TRACE_AT(t, 11);
        const float *tr = tabs + ((t & 1) * kTile + grow) * kPreW;
        const float p0 = tr[0], p1 = tr[1], p2 = tr[2], p3 = tr[3], rn = tr[4];
        const int64_t grow_g = (int64_t)(cid + t * ncl) * kTile + grow;
        const bool live = grow_g < a.rows;
        for (int hb = 0; hb < kHb && ok; ++hb) {
          float yv[16];
#pragma unroll
          for (int i = 0; i < kHC; ++i) {
            if (!waitw(bar(B_FULL + stage), phase, false, ab, 4, t)) { ok = false; break; }
            float x[16];
            load16(x);
            const float pi = i == 0 ? p0 : (i == 1 ? p1 : (i == 2 ? p2 : p3));
#pragma unroll
            for (int e = 0; e < 16; ++e) yv[e] = i == 0 ? pi * x[e] : fmaf(pi, x[e], yv[e]);
            release();
          }
          if (!ok) break;
          if (live) {
            const uint4 wa = wsm[(kBk * hb + 16 * hq) / 8], wb = wsm[(kBk * hb + 16 * hq) / 8 + 1];
            const uint32_t ww[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            uint32_t ow[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              ow[e] = pack2_rn((yv[2 * e] * rn) * lo_bf(ww[e]), (yv[2 * e + 1] * rn) * hi_bf(ww[e]));
            uint4 *dst = reinterpret_cast<uint4 *>(a.x_norm + grow_g * kH + (int64_t)crank * kHs +
                                                   kBk * hb + 16 * hq);
            st_stream(dst, make_uint4(ow[0], ow[1], ow[2], ow[3]));
            st_stream(dst + 1, make_uint4(ow[4], ow[5], ow[6], ow[7]));
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_CDONE));
        if (warp == kRow0) {
          if (!waitw(bar(B_CDONE), (uint32_t)(t & 1), false, ab, 13, t)) break;
          if (lane == 0)
            arrive_all_ctas(bar(B_QFREE + (t & 1)), kCl);
          if (lane == 0) MHC_TRACE_AT(t, 12);
          __syncwarp();
        }
      }
    }
  } else {
    // ---- owner warps: finalise 8 rows of each tile --------------------------
    const int o = threadIdx.x - kOwner0 * 32;   // 0..127
    const int q = o >> 4, e = o & 15;           // row of 8, lane of 16
    const int row_t = (int)crank * kOwn + q;
    const float *recv = reinterpret_cast<const float *>(sm + kOffRecv);
    float *red = reinterpret_cast<float *>(sm + kOffRed);
    const float sc0 = __ldg(a.scale), sc1 = __ldg(a.scale + 1), sc2 = __ldg(a.scale + 2);
    const float bcomb = __ldg(a.base + 8 + e);
    const float bgate = e < 8 ? __ldg(a.base + e) : 0.f;
    const unsigned full = 0xffffffffu;          // a row's 16 lanes are half the warp
    const int gb = lane & 16;
    for (int it = 0; it < T; ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      const int64_t grow = (int64_t)(cid + it * ncl) * kTile + row_t;
      if (!waitw(bar(B_PREADY), (uint32_t)(it & 1), true, ab, 8, it)) break;
      if (warp == kOwner0 && lane == 0) MHC_TRACE_AT(it, 13);
      // this row's 34 partials from the 16 CTAs, summed in CTA order
      float acc[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int w3 = 0; w3 < 3; ++w3) {
        const int v = e + 16 * w3;
        if (v < kPw) {
          float sacc = 0.f;
#pragma unroll
          for (int src = 0; src < kCl; ++src) sacc += recv[(src * kOwn + q) * kPw + v];
          acc[w3] = sacc;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OPULL));
      if (warp == kOwner0) {
        if (!waitw(bar(B_OPULL), (uint32_t)(it & 1), false, ab, 9, it)) break;
        if (lane == 0)
          arrive_all_ctas(bar(B_PFREE), kCl);
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
      // gates: lanes 0..3 pre, 4..7 post
      float gate = 0.f;
      if (e < 8) {
        const float l = fmaf(rq[e] * rsq, e < 4 ? sc0 : sc1, bgate);
        const float sg = 1.0f / (1.0f + expf(-l));
        gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
      }
      const float p0 = __shfl_sync(full, gate, gb + 0), p1 = __shfl_sync(full, gate, gb + 1);
      const float p2 = __shfl_sync(full, gate, gb + 2), p3 = __shfl_sync(full, gate, gb + 3);
      // sum_h y_h^2 = pre^T G pre
      float yy = p0 * p0 * G00 + p1 * p1 * G11 + p2 * p2 * G22 + p3 * p3 * G33;
      yy += 2.0f * (p0 * p1 * G01 + p0 * p2 * G02 + p0 * p3 * G03 + p1 * p2 * G12 +
                    p1 * p3 * G13 + p2 * p3 * G23);
      yy = fmaxf(yy, 0.f);
      const float rn = 1.0f / sqrtf(yy / (float)kH + a.norm_eps);
      // (pre, rnorm) of this row into table `buf` of CTA e: the combines wait on it
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
        if (lane == 0)
          arrive_all_ctas(bar(B_QREADY + buf), kCl);
        if (lane == 0) MHC_TRACE_AT(it, 14);
        __syncwarp();
      }
      // Sinkhorn on exp(logits), off the combine's critical path: lane e holds comb[e/4][e%4]
      float C = expf(fmaf(rq[8 + e] * rsq, sc2, bcomb));
      for (int k = 0; k < a.iters; ++k) {
        float rs = C + __shfl_xor_sync(full, C, 1);
        rs = rs + __shfl_xor_sync(full, rs, 2);
        C = C / (rs + a.sink_eps);
        float cs = C + __shfl_xor_sync(full, C, 4);
        cs = cs + __shfl_xor_sync(full, cs, 8);
        C = C / (cs + a.sink_eps);
      }
      if (warp == kOwner0 && lane == 0) MHC_TRACE_AT(it, 15);
      if (grow < a.rows) {
        a.comb[grow * 16 + e] = C;
        if (e >= 4 && e < 8) a.post[grow * kHC + (e - 4)] = gate;
        if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
        if (a.mix_out) {
          a.mix_out[grow * kMix + e] = rq[e] * rsq;
          if (e < 8) a.mix_out[grow * kMix + 16 + e] = rq[16 + e] * rsq;
        }
      }
      __syncwarp();
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

#ifdef MHC_TRACE
extern "C" int mhc_trace_set(void *buf) {
  return (int)cudaMemcpyToSymbol(g_trace, &buf, sizeof buf);
}
#endif

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
