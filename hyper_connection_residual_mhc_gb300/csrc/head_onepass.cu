// head_onepass.cu -- mhc_hc_head in one pass over R on GB300: the model's
// final collapse of the 4 residual streams into one hidden vector per row.
//
// Definition: deepseek_v4.py (sglang), hc_head_torch: mixes = (x @ fn^T) *
// rsqrt(mean(x^2) + norm_eps) on the flattened row x (4 x 5120, stream-major),
// pre_i = sigmoid(mix_i * scale + base_i) + hc_eps, y = sum_i pre_i R_i, cast
// once to bf16.
//
// With 4 mixes the projections are 0.16 MFLOP a row, which the CUDA cores do
// in fp32 well inside the time it takes to stream the row, so R can be read
// once and combined from shared memory.
//
// Decomposition.  A cluster of 4 CTAs takes 4-row tiles in turn; CTA s owns
// hidden columns [1280 s, 1280 s + 1280) of all four streams.  Thread t
// (640 per CTA) owns stream t / 160 and 8 columns, and keeps its 4 x 8 fn
// values in registers for the whole kernel.  Per tile:
//   * bulk copies bring the tile's 16 (row, stream) segments of 2560 B into
//     one of five 40 KB buffers;
//   * every thread forms its 5 partials per row (4 dots, sum of squares) in
//     fp32, summed over the warp by a fixed transpose tree and over the 20
//     warps in warp order;
//   * the CTA's 20 sums go to all 4 CTAs of the cluster, which each sum the
//     four in rank order -- every CTA forms the same gates;
//   * every thread then combines one (row, 8 columns) item of the tile two
//     iterations back from shared memory and writes it, so that a tile's
//     exchange has a whole iteration to complete.
// Receive slots: a CTA pushing tile t has combined tile t - 3, which needed
// every peer's partials of tile t - 3, so no peer still has a tile older than
// t - 5 to consume; eight slots never overrun.
//
// The phases are separated by CTA barriers, and with one 640-thread CTA per
// SM a tile costs ~3.9 us per cluster in latency rather than bytes (about 550
// instructions per warp at ~14 cycles each, half of it waiting at barriers),
// so the library uses this kernel for chunks of up to 256 rows and the tiled
// kernel (head_tile.cu) above.
//
// Every row is reduced in one fixed order that depends only on its own data,
// so any row range gives the whole-chunk bits.  Every wait is bounded (~2 s);
// on expiry the CTA raises an abort flag, records the site in its error word,
// lets its copies land and returns.
#include <mutex>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

__device__ unsigned int g_head_error;
__device__ unsigned int g_head_where[32];
__device__ unsigned int g_head_where_aborted[32];

namespace {
using namespace ptx;

constexpr int kHeadMixes = kHC;               // hc_head: one mix per stream
constexpr int kHCl = 4;                       // CTAs per cluster
constexpr int kHCols = kH / kHCl;             // 1280 columns per CTA
constexpr int kHGroups = kHCols / 8;          // 160 8-column groups
constexpr int kHThreads = kHC * kHGroups;     // 640: (stream, group)
constexpr int kHWarps = kHThreads / 32;       // 20
constexpr int kTR = 4;                        // rows per tile
constexpr int kDepth = 2;                     // a tile is combined kDepth iterations after its partials
constexpr int kNB = 5;                        // tile buffers: kDepth + 1 in use, the rest in flight
constexpr int kNS = 8;                        // receive slots (a peer is at most 6 tiles behind)
constexpr int kNP = kHeadMixes + 1;           // 4 dots + sum of squares
constexpr int kTV = kTR * kNP;                // 20 values per tile
constexpr int kSegBytes = kHCols * 2;         // 2560: one (row, stream) segment
constexpr int kBufBytes = kTR * kHC * kSegBytes;   // 40960
static_assert(kHThreads == kTR * kHGroups, "one combine item per thread");
static_assert(kTV <= 32, "the tile's partials fit one transpose");

// shared memory from a 128-byte aligned base
constexpr int kOffBuf = 0;                                   // [kNB][kTR][4][1280] bf16
constexpr int kOffRed = kOffBuf + kNB * kBufBytes;           // [20 warps][20]
constexpr int kOffRecv = kOffRed + kHWarps * kTV * 4;        // [kNS][4 src][20]
constexpr int kOffGate = kOffRecv + kNS * kHCl * kTV * 4;    // [kTR][4] pre gates
constexpr int kOffBar = kOffGate + kTR * kHC * 4;            // FULL[kNB], RREADY[kNS]
constexpr int kOffMisc = kOffBar + (kNB + kNS) * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 128;
static_assert(kOffBar % 8 == 0 && kSmemBytes <= 232448, "");

struct HeadArgs {
  const uint16_t *R;
  const float *fn, *scale, *base;
  uint16_t *y;
  float *pre_out, *mix_out;
  int64_t rows;
  int num_tiles;
  float norm_eps, hc_eps;
};

// lane l ends with the warp's sum of v[l] (a fixed pairing tree: halves at
// distance 16, 8, 4, 2, 1)
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = up ? v[j] : v[j + w];
      const float keep = up ? v[j + w] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

__global__ void __cluster_dims__(kHCl, 1, 1) __launch_bounds__(kHThreads, 1)
head_onepass_kernel(const HeadArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                            ~static_cast<uintptr_t>(127));
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int cid = (int)cluster_id(), ncl = (int)cluster_count();
  const int T = cid < a.num_tiles ? (a.num_tiles - 1 - cid) / ncl + 1 : 0;   // our tiles
  auto full = [&](int b) -> uint32_t { return sb + kOffBar + 8u * (uint32_t)b; };
  auto rready = [&](int s) -> uint32_t { return sb + kOffBar + 8u * (uint32_t)(kNB + s); };
  float *red = reinterpret_cast<float *>(sm + kOffRed);
  float *recv = reinterpret_cast<float *>(sm + kOffRecv);
  float *gate = reinterpret_cast<float *>(sm + kOffGate);
  Abort ab{reinterpret_cast<volatile int *>(sm + kOffMisc), rank, &g_head_error, g_head_where,
           g_head_where_aborted};

  if (tid == 0) {
    *ab.flag = 0;
    for (int b = 0; b < kNB; ++b) mbar_init(full(b), 1);
    for (int s = 0; s < kNS; ++s) mbar_init(rready(s), kHCl);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();
  pdl_wait();

  // the thread's dot item: stream si, columns [1280 rank + 8 g, +8)
  const int si = tid / kHGroups, g = tid % kHGroups;
  const int h0 = (int)rank * kHCols + 8 * g;
  float f[kHeadMixes][8];
#pragma unroll
  for (int c = 0; c < kHeadMixes; ++c) {
    const float4 u = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + si * kH + h0));
    const float4 v = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + si * kH + h0 + 4));
    f[c][0] = u.x; f[c][1] = u.y; f[c][2] = u.z; f[c][3] = u.w;
    f[c][4] = v.x; f[c][5] = v.y; f[c][6] = v.z; f[c][7] = v.w;
  }
  const float sc = __ldg(a.scale);

  // thread 0 keeps the copies going: tile j of this cluster into buffer j % kNB
  auto issue = [&](int j) {
    const int64_t r0 = (int64_t)(cid + j * ncl) * kTR;
    const int nr = (int)min((int64_t)kTR, a.rows - r0);
    const int b = j % kNB;
    mbar_expect_tx(full(b), (uint32_t)(nr * kHC * kSegBytes));
    for (int r = 0; r < nr; ++r)
      for (int i = 0; i < kHC; ++i)
        bulk_load(sb + kOffBuf + b * kBufBytes + (r * kHC + i) * kSegBytes,
                  a.R + ((r0 + r) * kHC + i) * kH + (int)rank * kHCols, kSegBytes, full(b));
  };
  if (tid == 0)
    for (int j = 0; j < kNB && j < T; ++j) issue(j);
  int issued = T < kNB ? T : kNB;

  bool ok = true;
  for (int t = 0; t < T + kDepth && ok; ++t) {
    if (t < T) {
      // ---- partials of tile t --------------------------------------------------
      const int b = t % kNB;
      // every wait's outcome is agreed by the whole CTA, so that no warp leaves
      // the loop while the others wait at a CTA barrier
      const bool got = waitw(full(b), (uint32_t)((t / kNB) & 1), false, ab, 0, t);
      if (!__syncthreads_and(got)) { ok = false; break; }
      const uint8_t *buf = sm + kOffBuf + b * kBufBytes;
      float v[32];
#pragma unroll
      for (int r = 0; r < kTR; ++r) {
        const uint4 q = *reinterpret_cast<const uint4 *>(buf + (r * kHC + si) * kSegBytes + 16 * g);
        float x[8];
        unpack8(q, x);
#pragma unroll
        for (int c = 0; c < kHeadMixes; ++c) {
          float s = x[0] * f[c][0];
#pragma unroll
          for (int e = 1; e < 8; ++e) s = fmaf(x[e], f[c][e], s);
          v[r * kNP + c] = s;
        }
        float ss = x[0] * x[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
        v[r * kNP + kHeadMixes] = ss;
      }
#pragma unroll
      for (int j = kTV; j < 32; ++j) v[j] = 0.f;
      const float ws = transpose_sum32(v, lane);
      if (lane < kTV) red[warp * kTV + lane] = ws;
      __syncthreads();
      // warp 0: the CTA's 20 sums (warps in order) to every CTA's slot
      if (warp == 0) {
        const int s = t % kNS;
        if (lane < kTV) {
          float tot = 0.f;
#pragma unroll
          for (int w = 0; w < kHWarps; ++w) tot += red[w * kTV + lane];
          const uint32_t dst = sb + kOffRecv + (uint32_t)(((s * kHCl + (int)rank) * kTV + lane) * 4);
#pragma unroll
          for (int c = 0; c < kHCl; ++c) st_cluster_f32(mapa(dst, (uint32_t)c), tot);
          fence_cluster();
        }
        __syncwarp();
        if (lane == 0) arrive_all_ctas(rready(s), kHCl);
        __syncwarp();
      }
      __syncthreads();   // warp 0 has read red: the next tile may overwrite it
    }
    if (t >= kDepth) {
      // ---- gates and combine of tile t - kDepth -----------------------------------
      const int tp = t - kDepth, b = tp % kNB, s = tp % kNS;
      const bool got = waitw(rready(s), (uint32_t)((tp / kNS) & 1), true, ab, 1, tp);
      if (!__syncthreads_and(got)) { ok = false; break; }
      const int64_t r0 = (int64_t)(cid + tp * ncl) * kTR;
      if (tid < kTR) {
        const int r = tid;
        float d[kNP];
#pragma unroll
        for (int j = 0; j < kNP; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int src = 0; src < kHCl; ++src) acc += recv[(s * kHCl + src) * kTV + r * kNP + j];
          d[j] = acc;
        }
        const float rsq = rsqrt_nr(fmaf(d[kHeadMixes], 1.0f / (float)kK, a.norm_eps));
        const bool mine = r0 + r < a.rows && rank == 0;
#pragma unroll
        for (int c = 0; c < kHeadMixes; ++c) {
          const float mx = d[c] * rsq;
          const float sg = rcp_nr(1.0f + expf(-fmaf(mx, sc, __ldg(a.base + c))));
          gate[r * kHC + c] = sg + a.hc_eps;
          if (mine && a.pre_out) a.pre_out[(r0 + r) * kHC + c] = sg + a.hc_eps;
          if (mine && a.mix_out) a.mix_out[(r0 + r) * kHeadMixes + c] = mx;
        }
      }
      __syncthreads();
      // thread -> (row tid / 160, columns 8 g'): y = sum_i pre_i R_i, one rounding
      {
        const int r = tid / kHGroups, gg = tid % kHGroups;
        if (r0 + r < a.rows) {
          const uint8_t *buf = sm + kOffBuf + b * kBufBytes + r * kHC * kSegBytes + 16 * gg;
          float rf[kHC][8];
#pragma unroll
          for (int i = 0; i < kHC; ++i)
            unpack8(*reinterpret_cast<const uint4 *>(buf + i * kSegBytes), rf[i]);
          const float pv[kHC] = {gate[r * kHC + 0], gate[r * kHC + 1], gate[r * kHC + 2],
                                 gate[r * kHC + 3]};
          float yv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float acc = pv[0] * rf[0][e];
#pragma unroll
            for (int i = 1; i < kHC; ++i) acc = fmaf(pv[i], rf[i][e], acc);
            yv[e] = acc;
          }
          st_stream(reinterpret_cast<uint4 *>(a.y + (r0 + r) * kH + (int)rank * kHCols + 8 * gg),
                    pack8_rn(yv));
        }
      }
      // buffer b and the gates are free: refill b with the tile kNB further on
      __syncthreads();
      if (tid == 0 && issued < T) issue(issued);
      ++issued;
    }
  }

  // no copy may still be landing when the CTA leaves (a wait that gave up
  // leaves it to these bounded drains)
  if (tid == 0) {
    const int last = issued < T ? issued : T;
    for (int j = last - kNB < 0 ? 0 : last - kNB; j < last; ++j) drain1(full(j % kNB), (uint32_t)((j / kNB) & 1));
  }
  pdl_trigger();
  __syncthreads();
  // no CTA leaves while a peer may still write into its shared memory
  cluster_sync_all();
}

std::mutex g_head_mu;
int g_head_clusters[64];

cudaError_t head_configure(int dev, int *ncl) {
  std::lock_guard<std::mutex> lock(g_head_mu);
  if (g_head_clusters[dev] > 0) {
    *ncl = g_head_clusters[dev];
    return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(head_onepass_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kHCl);
  cfg.blockDim = dim3(kHThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, head_onepass_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_head_clusters[dev] = n;
  *ncl = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_head_onepass(const uint16_t *R, const float *fn, const float *scale,
                                const float *base, int64_t rows, int64_t logical_rows,
                                float norm_eps, float hc_eps, uint16_t *y, float *pre_out,
                                float *mix_out, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int ncl_max = 0;
  e = head_configure(dev, &ncl_max);
  if (e != cudaSuccess) return e;
  HeadArgs a;
  a.R = R; a.fn = fn; a.scale = scale; a.base = base; a.y = y;
  a.pre_out = pre_out; a.mix_out = mix_out; a.rows = rows;
  a.num_tiles = (int)((rows + kTR - 1) / kTR);
  a.norm_eps = norm_eps; a.hc_eps = hc_eps;
  // grid from the chunk's row count only (the per-row arithmetic does not
  // depend on which cluster takes a tile)
  const int64_t chunk_tiles = (logical_rows + kTR - 1) / kTR;
  const int clusters = (int)(chunk_tiles < ncl_max ? chunk_tiles : ncl_max);
  return launch_pdl(head_onepass_kernel, dim3((unsigned)(clusters * kHCl)), dim3(kHThreads),
                    kSmemBytes, s, 1, use_pdl(logical_rows), a);
}

cudaError_t head_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_head_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_head_error, &z, sizeof z);
  }
  return e;
}

}  // namespace mhc
