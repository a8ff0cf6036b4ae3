// pre_stats.cu -- the stats half of mhc_pre on GB300: per row, the 24
// projections of the flattened residual on the 5th-generation tensor cores,
// the row's sum of squares, and the split into gates and the Sinkhorn mix.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre:
// hc_pre_torch_impl (rsqrt of mean(x^2) + rms_eps; mixes = (x @ fn^T) * rsqrt)
// and hc_split_sinkhorn (gates and the 4x4 Sinkhorn).
//
// Decomposition.  A cluster of 16 CTAs owns a 128-row tile at a time; CTA s
// owns hidden columns [320 s, 320 s + 320) of all four streams, i.e. 1280 of a
// row's 20480 k.  fn's 24 x 1280 slice of the CTA, split into bf16 hi (B rows
// 0..23) and lo (rows 24..47) halves, stays in shared memory (120 KB) for the
// whole kernel, so each product is exact and the dot products carry ~2^-17
// relative error per term.  Per tile and CTA:
//   * TMA streams R[128 rows, 64 k] boxes (128-byte swizzle) through a
//     5-stage ring -- R is read from HBM exactly once;
//   * one thread issues tcgen05.mma (M=128 rows, N=48, K=16, bf16 -> fp32,
//     two accumulators in tensor memory);
//   * 16 row warps (4 lanes per row, 16 columns each) accumulate sum x^2 from
//     the same stages, then read the accumulator and push each row's 24 mix
//     partials and its sum of squares into the receive buffer of the CTA
//     that finalises the row (CTA s owns tile rows 8s..8s+7);
//   * 4 owner warps reduce the 16 partials of a row in CTA order, compute
//     rsqrt, mix, the gates and the 4x4 Sinkhorn (16 lanes per row) and write
//     pre, post and comb.
// The combine + RMSNorm (x_norm) runs as a second, streaming launch
// (pre_simt.cu, combine_norm_kernel) that reads the pre gates this kernel
// writes.
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

namespace mhc {

// Bit s set: a bounded wait at site s expired; g_fused_where[s] holds
// (tile << 8) | cluster rank of the last one.  Bit 16 + s: a wait at site s
// gave up because its CTA had already aborted (g_fused_where_aborted[s]).
__device__ unsigned int g_fused_error;
__device__ unsigned int g_fused_where[32];
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
constexpr int kRw = 28;                       // receive words per row: 24 dots, sum x^2, pad
constexpr int kOwn = kTile / kCl;             // 8 rows finalised per CTA
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

// ---- shared memory (offsets from a 1024-byte aligned base) -----------------
constexpr int kOffFn = 0;
constexpr int kOffStage = kOffFn + kKb * kFnBlkBytes;
constexpr int kOffRecv = kOffStage + kStages * kStageBytes;   // [16 src][8 rows][kRw]
constexpr int kOffRed = kOffRecv + kCl * kOwn * kRw * 4;      // [8 rows][kRw]
constexpr int kOffSs = kOffRed + kOwn * kRw * 4;              // [2][128 rows] sum x^2
constexpr int kOffBar = kOffSs + 2 * kTile * 4;
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
constexpr int kOffMisc = kOffBar + B_COUNT * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block limit");
static_assert(kOffStage % 1024 == 0 && kFnBlkBytes % 1024 == 0, "SW128 tiles need 1024-B alignment");
static_assert(kOffRecv % 16 == 0 && (kRw * 4) % 16 == 0, "receive rows must take 16-byte stores");

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
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
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

struct StatsArgs {
  const float *fn;
  const float *scale;
  const float *base;
  float *pre_ws;     // [rows, 4] pre gates for the combine launch
  float *post;
  float *comb;
  float *pre_out;
  float *mix_out;
  int64_t rows;
  int num_tiles;
  float rms_eps, pre_eps, sink_eps, post_mult;
  int iters;
};

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float a) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
pre_stats_kernel(const __grid_constant__ CUtensorMap tmap, const StatsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;   // our tiles
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
      mbar_init(bar(B_TEMPTY + b), kReadN);
      mbar_init(bar(B_SSREADY + b), kRowN);
    }
    mbar_init(bar(B_PREADY), kCl);
    mbar_init(bar(B_PFREE), kCl);
    mbar_init(bar(B_GALL), kReadN);
    mbar_init(bar(B_OPULL), kOwnerN);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_FNREADY), kWarps - 1 - kRowN);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem = *tmem_slot;

  // fn columns of this CTA -> bf16 hi/lo B tiles (K-major, 128-byte swizzle),
  // written by the MMA, readout and owner warps while the producer starts
  // streaming R and the row warps wait for it:
  // k-block j covers k = (j%4)*5120 + 320*crank + 64*(j/4) + [0, 64)
  if (warp != kProducerWarp && !(warp >= kRow0 && warp < kRow0 + kRowN)) {
    // 10 loader warps; loads of 8 items are issued before any is converted
    const int loader = warp == kMmaWarp ? 0 : (warp < kRow0 ? warp - 1 : warp - kRowN - 1);
    const int lt = loader * 32 + lane, nl = (kWarps - 1 - kRowN) * 32;
    constexpr int kItems = kMix * kKb * 8;     // 3840 items of 8 consecutive k
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
        const float f[8] = {f0[u].x, f0[u].y, f0[u].z, f0[u].w, f1[u].x, f1[u].y, f1[u].z, f1[u].w};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * e]);
          const __nv_bfloat16 h1 = __float2bfloat16_rn(f[2 * e + 1]);
          hw[e] = pack2_rn(__bfloat162float(h0), __bfloat162float(h1));
          lw[e] = pack2_rn(f[2 * e] - __bfloat162float(h0), f[2 * e + 1] - __bfloat162float(h1));
        }
        uint8_t *tile = sm + kOffFn + j * kFnBlkBytes;
        const int nh = c, nlo = c + kMix;
        *reinterpret_cast<uint4 *>(tile + (nh >> 3) * 1024 + (nh & 7) * 128 + ((q ^ (nh & 7)) << 4)) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(tile + (nlo >> 3) * 1024 + (nlo & 7) * 128 +
                                   ((q ^ (nlo & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
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
      if (lane == 0) MHC_TRACE_AT(it, 0);
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
      if (lane == 0) MHC_TRACE_AT(it, 1);
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
      __syncwarp();
    }
    // all issued MMAs complete before TMEM is freed
    if (lane == 0) tc_commit(bar(B_DRAIN));
    __syncwarp();
    drain1(bar(B_DRAIN), 0);
    __syncwarp();
  } else if (warp >= kRow0 && warp < kRow0 + kRowN) {
    // ---- row warps: one thread per tile row; sum x^2 from every stage -------
    const int row = 32 * (warp & 3) + lane;     // tile row
    const int sw = row & 7;
    float *ssbuf = reinterpret_cast<float *>(sm + kOffSs);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; it < T && ok; ++it) {
      float ss = 0.f;
      for (int j = 0; j < kKb; ++j) {
        if (!waitw(bar(B_FULL + stage), phase, false, ab, 4, it)) { ok = false; break; }
        if (j == 0 && warp == kRow0 && lane == 0) MHC_TRACE_AT(it, 2);
        const uint8_t *st = sm + kOffStage + stage * kStageBytes + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 c = *reinterpret_cast<const uint4 *>(st + ((q ^ sw) << 4));
          const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = lo_bf(w4[e]), x1 = hi_bf(w4[e]);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
          }
        }
        // the stage is released only after every lane has used its data
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + stage));
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (warp == kRow0 && lane == 0) MHC_TRACE_AT(it, 3);
      // hand the row's sum x^2 to the readout warps (slot free once tile it-2
      // was read out)
      const int buf = it & 1;
      if (!waitw(bar(B_TEMPTY + buf), (uint32_t)((it >> 1) & 1) ^ 1, false, ab, 10, it)) break;
      ssbuf[buf * kTile + row] = ss;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SSREADY + buf));
    }
  } else if (warp >= kRead0 && warp < kRead0 + kReadN) {
    // ---- readout warps: one thread per tile row (= TMEM lane) ---------------
    // accumulator + sum x^2 of tile t -> the owner CTA's receive buffer
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = 32 * quarter + lane;
    const float *ssbuf = reinterpret_cast<const float *>(sm + kOffSs);
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
      float mix[kMix];                          // hi + lo of the 24 dots
#pragma unroll
      for (int c = 0; c < 8; ++c) mix[c] = a0[c] + a1[c + 8];
#pragma unroll
      for (int c = 8; c < 16; ++c) mix[c] = a0[c] + a2[c - 8];
#pragma unroll
      for (int c = 16; c < 24; ++c) mix[c] = a1[c - 16] + a2[c - 8];
      // slot [our rank][row % 8] of the owner CTA (row / 8)
      if (!waitw(bar(B_PFREE), (uint32_t)(t & 1) ^ 1, true, ab, 6, t)) break;
      const uint32_t dm = mapa(sb + kOffRecv + (uint32_t)(((crank * kOwn + (row & 7)) * kRw) * 4),
                               (uint32_t)(row >> 3));
#pragma unroll
      for (int v = 0; v < 6; ++v)
        st_cluster_v4(dm + 16 * v, mix[4 * v], mix[4 * v + 1], mix[4 * v + 2], mix[4 * v + 3]);
      st_cluster_f32(dm + 4 * kMix, ss);
      // make the stores visible cluster-wide, then count this warp in
      fence_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_GALL));
      if (warp == kRead0) {
        // all readout warps pushed tile t: tell all 16 owners
        if (!waitw(bar(B_GALL), (uint32_t)(t & 1), false, ab, 7, t)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PREADY), kCl);
        if (lane == 0) MHC_TRACE_AT(t, 4);
        __syncwarp();
      }
    }
  } else {
    // ---- owner warps: finalise 8 rows of each tile --------------------------
    const int o = owner_index(warp) * 32 + lane;   // 0..127
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
      const int64_t grow = (int64_t)(cid + it * ncl) * kTile + row_t;
      if (!waitw(bar(B_PREADY), (uint32_t)(it & 1), true, ab, 8, it)) break;
      if (warp == kOwnerLead && lane == 0) MHC_TRACE_AT(it, 5);
      // this row's 25 partials from the 16 CTAs, summed in CTA order
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int src = 0; src < kCl; ++src) acc0 += recv[(src * kOwn + q) * kRw + e];
      if (e + 16 <= kMix) {
#pragma unroll
        for (int src = 0; src < kCl; ++src) acc1 += recv[(src * kOwn + q) * kRw + e + 16];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OPULL));
      if (warp == kOwnerLead) {
        if (!waitw(bar(B_OPULL), (uint32_t)(it & 1), false, ab, 9, it)) break;
        if (lane == 0) arrive_all_ctas(bar(B_PFREE), kCl);
        __syncwarp();
      }
      float *rq = red + q * kRw;
      rq[e] = acc0;
      if (e + 16 <= kMix) rq[e + 16] = acc1;
      __syncwarp();
      const float rsq = 1.0f / sqrtf(rq[kMix] / (float)kK + a.rms_eps);
      // gates: lanes 0..3 pre, 4..7 post
      float gate = 0.f;
      if (e < 8) {
        const float l = fmaf(rq[e] * rsq, e < 4 ? sc0 : sc1, bgate);
        const float sg = 1.0f / (1.0f + expf(-l));
        gate = e < 4 ? sg + a.pre_eps : a.post_mult * sg;
      }
      // Sinkhorn on exp(logits): lane e holds comb[e/4][e%4]
      float C = expf(fmaf(rq[8 + e] * rsq, sc2, bcomb));
      for (int k = 0; k < a.iters; ++k) {
        float rs = C + __shfl_xor_sync(full, C, 1);
        rs = rs + __shfl_xor_sync(full, rs, 2);
        C = C / (rs + a.sink_eps);
        float cs = C + __shfl_xor_sync(full, C, 4);
        cs = cs + __shfl_xor_sync(full, cs, 8);
        C = C / (cs + a.sink_eps);
      }
      if (grow < a.rows) {
        a.comb[grow * 16 + e] = C;
        if (e < 4) a.pre_ws[grow * kHC + e] = gate;
        if (e >= 4 && e < 8) a.post[grow * kHC + (e - 4)] = gate;
        if (a.pre_out && e < 4) a.pre_out[grow * kHC + e] = gate;
        if (a.mix_out) {
          a.mix_out[grow * kMix + e] = rq[e] * rsq;
          if (e < 8) a.mix_out[grow * kMix + 16 + e] = rq[16 + e] * rsq;
        }
      }
      if (warp == kOwnerLead && lane == 0) MHC_TRACE_AT(it, 6);
      (void)gb;
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
  cudaError_t e = cudaFuncSetAttribute(pre_stats_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pre_stats_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  e = cudaOccupancyMaxActiveClusters(&n, pre_stats_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_max_clusters[dev] = n;
  *max_clusters = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_pre_stats(const uint16_t *R, const float *fn, const float *scale,
                             const float *base, int64_t rows, int64_t logical_rows,
                             const mhc_params &p, float *pre_ws, float *post, float *comb,
                             float *pre_out, float *mix_out, cudaStream_t s) {
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

  StatsArgs a;
  a.fn = fn; a.scale = scale; a.base = base; a.pre_ws = pre_ws;
  a.post = post; a.comb = comb; a.pre_out = pre_out; a.mix_out = mix_out;
  a.rows = rows;
  a.num_tiles = (int)((rows + kTile - 1) / kTile);
  a.rms_eps = p.rms_eps; a.pre_eps = p.hc_pre_eps; a.sink_eps = p.hc_sinkhorn_eps;
  a.post_mult = p.post_mult; a.iters = p.sinkhorn_iters;

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
  return cudaLaunchKernelEx(&cfg, pre_stats_kernel, map, a);
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
