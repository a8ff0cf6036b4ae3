// pre_decode.cu -- mhc_pre (and mhc_fused_post_pre) for decode-size chunks
// (up to 48 rows) in a single launch.
//
// Definitions: deepseek_v4.py (sglang), DeepseekV4DecoderLayer.hc_pre
// (hc_pre_torch_impl: rsqrt of mean(x^2) + rms_eps, mixes = (x @ fn^T) *
// rsqrt; hc_split_sinkhorn: gates and the 4x4 Sinkhorn; the combine
// y = sum_i pre_i x_i) with the RMSNorm fused as in prefill_sp.py,
// _combine_norm_fused.
//
// At these sizes the work is a few MFLOP and a few MB, so time is latency:
// launches, round trips to L2, and the serial Sinkhorn.  One cluster of 16
// CTAs takes up to 8 rows; CTA s owns hidden columns [320 s, 320 s + 320) of
// all four streams (1280 of the 20480 k).  Thread t handles stream t / 80 and
// four consecutive columns, and keeps its 4 x 24 fn values and its rows' x in
// registers for the whole kernel:
//   1. per row, the thread's 25 partials (24 dots, sum of squares), summed
//      over the warp by a fixed transpose tree and over the CTA's 10 warps in
//      warp order, go to the row's owner CTA (rank = row in the group);
//   -- cluster barrier --
//   2. the owner (warp 9 of that CTA) sums the 16 CTAs' partials in rank
//      order, computes rsqrt and the gates, and sends the 4 pre gates to
//      every CTA;
//   -- cluster barrier --
//   3. each CTA forms y on its 320 columns, sends its partial sum of y^2 to
//      every CTA -- meanwhile the owner warp runs the Sinkhorn (16 lanes) and
//      writes post, comb and the exports: nothing downstream in this kernel
//      needs comb, so the owner arrives at the next barrier before it starts;
//   -- cluster barrier --
//   4. each CTA sums the 16 partials in rank order and writes its 320
//      columns of x_norm.
// A cluster takes groups of up to 8 rows, as many as spread the chunk over
// the co-resident clusters.  The barriers are the hardware cluster barrier;
// every thread of every CTA arrives at each of them (no early exit), so each
// completes.
//
// Built twice: kPost = false is mhc_pre; kPost = true is mhc_fused_post_pre
// at these sizes (deepseek_v4.py, the use_fused_mhc_post_pre path): each
// thread first forms its 4 columns of R' = hc_post(R, y, post, comb) from the
// four streams and y at those columns, writes them to R_out, and runs the
// pre on R' -- one launch, and R' is never read back.
#include <mutex>

#include "mhc_common.cuh"

namespace mhc {

namespace {

constexpr int kDCl = 16;                      // CTAs per cluster
constexpr int kDThreads = 320;                // 10 warps
constexpr int kDWarps = kDThreads / 32;
constexpr int kDRows = 8;                     // rows per cluster
constexpr int kDHs = kH / kDCl;               // 320 columns per CTA
constexpr int kDQ = kDHs / 4;                 // 80 threads per stream
constexpr int kDPart = kMix + 1;              // 24 dots + sum of squares
static_assert(kDQ * kHC == kDThreads, "one thread per (stream, 4 columns)");

__device__ __forceinline__ uint32_t d_smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t d_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t d_mapa(uint32_t addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
  return r;
}
__device__ __forceinline__ void d_st_remote(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void d_cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void d_cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void d_cluster_sync() {
  d_cluster_arrive();
  d_cluster_wait();
}

// v[0..31] of every lane -> lane l holds the warp's sum of index l (a fixed
// pairing tree: halves at distance 16, 8, 4, 2, 1)
__device__ __forceinline__ float d_transpose_sum32(float (&v)[32], int lane) {
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

struct DecArgs {
  const uint16_t *R;
  const float *fn, *scale, *base;
  const uint16_t *norm_w;
  uint16_t *x_norm;
  float *post, *comb, *pre_out, *mix_out;
  // kPost: hc_post of the previous sublayer first, x = R_out
  const uint16_t *y;
  const float *post_in, *comb_in;
  uint16_t *R_out;
  int64_t rows;
  int group;          // rows per cluster pass (1..8)
  int fn_stable;      // fn is a prepared handle's copy: no earlier launch writes it
  mhc_params p;
};

// kPost: the thread's 4 columns of stream si of R' = hc_post(R, y, post,
// comb) for row `row`, written to R_out and returned as the pre's x.  Per
// element: post_si * y, then one fma per stream j in order, one rounding --
// the arithmetic of post_chunk, so R_out has mhc_post's bits.
__device__ __forceinline__ uint2 post_cols(const DecArgs &a, int64_t row, int si, int k0, int h0) {
  const uint16_t *rr = a.R + row * kK + h0;
  uint2 rv[kHC];
#pragma unroll
  for (int j = 0; j < kHC; ++j) rv[j] = __ldg(reinterpret_cast<const uint2 *>(rr + j * kH));
  const uint2 yv = __ldg(reinterpret_cast<const uint2 *>(a.y + row * kH + h0));
  const float pv = __ldg(a.post_in + row * kHC + si);
  float cb[kHC];
#pragma unroll
  for (int j = 0; j < kHC; ++j) cb[j] = __ldg(a.comb_in + row * kHC * kHC + j * kHC + si);
  const float yf[4] = {__uint_as_float(yv.x << 16), __uint_as_float(yv.x & 0xFFFF0000u),
                       __uint_as_float(yv.y << 16), __uint_as_float(yv.y & 0xFFFF0000u)};
  float acc[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float s = pv * yf[e];
#pragma unroll
    for (int j = 0; j < kHC; ++j) {
      const uint32_t w = (e < 2) ? rv[j].x : rv[j].y;
      const float rf = (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
      s = fmaf(cb[j], rf, s);
    }
    acc[e] = s;
  }
  const uint2 o = make_uint2(pack2_rn(acc[0], acc[1]), pack2_rn(acc[2], acc[3]));
  *reinterpret_cast<uint2 *>(a.R_out + row * kK + k0) = o;
  return o;
}

template <bool kPost>
__global__ void __cluster_dims__(kDCl, 1, 1) __launch_bounds__(kDThreads, 1)
pre_decode_kernel(const DecArgs a) {
  __shared__ float red[kDWarps][kDRows][32];        // per-warp row partials
  __shared__ float recv[kDCl][kDRows][kDPart];      // owner: partials from each CTA
  __shared__ float pre_all[kDRows][kHC];            // gates of the group's rows
  __shared__ float sq[kDCl][kDRows];                // partial sums of y^2 from each CTA
  __shared__ uint2 xs[kDRows][kHC][kDQ];            // the CTA's x, for the combine
  __shared__ float dot[kDRows][kDPart];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = d_rank();
  const int cl = (int)(blockIdx.x / kDCl), ncl = (int)(gridDim.x / kDCl);
  const int si = tid / kDQ, q = tid % kDQ;          // stream, 4-column group
  const int k0 = si * kH + (int)rank * kDHs + 4 * q;
  const int h0 = (int)rank * kDHs + 4 * q;          // threads tid < 80: their columns
  // A prepared handle's fn copy is never written after preparation, so its
  // loads may overlap the previous launch's tail; anything else waits first.
  float f[kMix][4];
  auto load_fn = [&]() {
#pragma unroll
    for (int c = 0; c < kMix; ++c) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(a.fn + (int64_t)c * kK + k0));
      f[c][0] = v.x; f[c][1] = v.y; f[c][2] = v.z; f[c][3] = v.w;
    }
  };
  if (a.fn_stable) load_fn();
  pdl_wait();
  if (!a.fn_stable) load_fn();
  float wf[4] = {0.f, 0.f, 0.f, 0.f};
  if (tid < kDQ) {
    const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(a.norm_w + h0));
    wf[0] = __uint_as_float(wv.x << 16); wf[1] = __uint_as_float(wv.x & 0xFFFF0000u);
    wf[2] = __uint_as_float(wv.y << 16); wf[3] = __uint_as_float(wv.y & 0xFFFF0000u);
  }
  const int G = a.group;
  const int64_t ngroups = (a.rows + G - 1) / G;

  for (int64_t g = cl; g < ngroups; g += ncl) {    // uniform across the cluster
    const int64_t row0 = g * G;
    const int nr = (int)(a.rows - row0 < G ? a.rows - row0 : G);
    uint2 xr[kDRows];
#pragma unroll
    for (int r = 0; r < kDRows; ++r) {
      if constexpr (kPost)
        xr[r] = r < nr ? post_cols(a, row0 + r, si, k0, h0) : make_uint2(0u, 0u);
      else
        xr[r] = r < nr ? __ldg(reinterpret_cast<const uint2 *>(a.R + (row0 + r) * kK + k0))
                       : make_uint2(0u, 0u);
    }

    // ---- 1. partials (row loops unrolled with a uniform guard, so the
    // per-row arrays stay in registers) --------------------------------------
#pragma unroll
    for (int r = 0; r < kDRows; ++r) {
      if (r >= nr) break;
      const float x[4] = {__uint_as_float(xr[r].x << 16), __uint_as_float(xr[r].x & 0xFFFF0000u),
                          __uint_as_float(xr[r].y << 16), __uint_as_float(xr[r].y & 0xFFFF0000u)};
      float v[32];
#pragma unroll
      for (int c = 0; c < kMix; ++c) {
        float s = x[0] * f[c][0];
#pragma unroll
        for (int e = 1; e < 4; ++e) s = fmaf(x[e], f[c][e], s);
        v[c] = s;
      }
      float ss = x[0] * x[0];
#pragma unroll
      for (int e = 1; e < 4; ++e) ss = fmaf(x[e], x[e], ss);
      v[kMix] = ss;
#pragma unroll
      for (int c = kDPart; c < 32; ++c) v[c] = 0.f;
      red[warp][r][lane] = d_transpose_sum32(v, lane);
      xs[r][si][q] = xr[r];
    }
    __syncthreads();
    for (int t = tid; t < nr * kDPart; t += kDThreads) {
      const int r = t / kDPart, c = t % kDPart;
      float s = red[0][r][c];
#pragma unroll
      for (int w = 1; w < kDWarps; ++w) s += red[w][r][c];
      d_st_remote(d_mapa(d_smem_addr(&recv[rank][r][c]), (uint32_t)r), s);
    }
    d_cluster_sync();

    // ---- 2. owner of group row `rank` (warp 9, which has no combine work):
    // the gates go to every CTA first; the Sinkhorn then runs while the other
    // warps do the combine and the norm (it feeds only comb, an output)
    constexpr int kOwnerWarp = kDWarps - 1;
    static_assert(kOwnerWarp * 32 >= kDQ, "the owner warp must not own combine columns");
    if (warp == kOwnerWarp) {
      const bool own = (int)rank < nr;
      const int r = own ? (int)rank : 0;
      const int64_t row = row0 + r;
      const int e = lane & 15;                // lanes 16..31 mirror 0..15
      const unsigned full = 0xffffffffu;
      float rsq = 0.f, gate = 0.f;
      if (own) {
        if (lane < kDPart) {
          float s = 0.f;
#pragma unroll
          for (int src = 0; src < kDCl; ++src) s += recv[src][r][lane];
          dot[r][lane] = s;
        }
        __syncwarp();
        rsq = 1.0f / sqrtf(dot[r][kMix] / (float)kK + a.p.rms_eps);
        if (e < 8) {
          const float l = fmaf(dot[r][e] * rsq, __ldg(a.scale + (e < 4 ? 0 : 1)), __ldg(a.base + e));
          const float sg = 1.0f / (1.0f + expf(-l));
          gate = e < 4 ? sg + a.p.hc_pre_eps : a.p.post_mult * sg;
        }
        // the 4 pre gates to every CTA of the cluster (lanes 0..3 x 16 CTAs)
        for (int t = lane; t < kHC * kDCl; t += 32) {
          const float gv = __shfl_sync(full, gate, t & 3);
          d_st_remote(d_mapa(d_smem_addr(&pre_all[r][t & 3]), (uint32_t)(t >> 2)), gv);
        }
      }
      d_cluster_arrive();        // barrier 2: the gates are out
      d_cluster_wait();
      d_cluster_arrive();        // barrier 3: this warp sends no partial sums
      if (own) {
        // Sinkhorn on exp(logits): lane e holds comb[e/4][e%4]
        float cm = expf(fmaf(dot[r][8 + e] * rsq, __ldg(a.scale + 2), __ldg(a.base + 8 + e)));
        for (int k = 0; k < a.p.sinkhorn_iters; ++k) {
          float rs = cm + __shfl_xor_sync(full, cm, 1);
          rs = rs + __shfl_xor_sync(full, rs, 2);
          cm = cm / (rs + a.p.hc_sinkhorn_eps);
          float cs = cm + __shfl_xor_sync(full, cm, 4);
          cs = cs + __shfl_xor_sync(full, cs, 8);
          cm = cm / (cs + a.p.hc_sinkhorn_eps);
        }
        if (lane < 16) {
          a.comb[row * 16 + e] = cm;
          if (e >= 4 && e < 8) a.post[row * kHC + (e - 4)] = gate;
          if (e < 4 && a.pre_out) a.pre_out[row * kHC + e] = gate;
          if (a.mix_out) {
            a.mix_out[row * kMix + e] = dot[r][e] * rsq;
            if (e < 8) a.mix_out[row * kMix + 16 + e] = dot[r][16 + e] * rsq;
          }
        }
      }
      d_cluster_wait();
      continue;                  // nothing of steps 3 and 4 is this warp's
    }
    d_cluster_sync();            // barrier 2

    // ---- 3. y on this CTA's columns; partial sums of y^2 to every CTA --------
    float y[kDRows][4];
    float sy[kDRows];
#pragma unroll
    for (int r = 0; r < kDRows; ++r) {
      sy[r] = 0.f;
      if (tid < kDQ && r < nr) {
        float xf[kHC][4];
#pragma unroll
        for (int i = 0; i < kHC; ++i) {
          const uint2 w2 = xs[r][i][tid];
          xf[i][0] = __uint_as_float(w2.x << 16);
          xf[i][1] = __uint_as_float(w2.x & 0xFFFF0000u);
          xf[i][2] = __uint_as_float(w2.y << 16);
          xf[i][3] = __uint_as_float(w2.y & 0xFFFF0000u);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float s = pre_all[r][0] * xf[0][e];
#pragma unroll
          for (int i = 1; i < kHC; ++i) s = fmaf(pre_all[r][i], xf[i][e], s);
          y[r][e] = s;
        }
        float s2 = y[r][0] * y[r][0];
#pragma unroll
        for (int e = 1; e < 4; ++e) s2 = fmaf(y[r][e], y[r][e], s2);
        sy[r] = s2;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) y[r][e] = 0.f;
      }
    }
    // warps 0..2 (the 80 threads, zeros elsewhere): lane l < 8 gets the
    // warp's sum for row l -- a fixed tree (halves 4, 2, 1, then 8, 16)
    if (warp < 3) {
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int jj = 0; jj < w; ++jj) {
          const float send = up ? sy[jj] : sy[jj + w];
          const float keep = up ? sy[jj + w] : sy[jj];
          sy[jj] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
      }
      float s = sy[0];
      s += __shfl_xor_sync(0xffffffffu, s, 8);
      s += __shfl_xor_sync(0xffffffffu, s, 16);
      if (lane < kDRows) red[warp][lane][0] = s;
    }
    // warps 0..8 only: the owner warp has left for its Sinkhorn
    asm volatile("bar.sync 1, %0;" ::"n"(kOwnerWarp * 32) : "memory");
    if (tid < nr * kDCl) {
      const int r = tid / kDCl, dst = tid % kDCl;
      const float s = (red[0][r][0] + red[1][r][0]) + red[2][r][0];
      d_st_remote(d_mapa(d_smem_addr(&sq[rank][r]), (uint32_t)dst), s);
    }
    d_cluster_sync();

    // ---- 4. x_norm on this CTA's columns ---------------------------------------
    if (tid < kDQ) {
#pragma unroll
      for (int r = 0; r < kDRows; ++r) {
        if (r >= nr) break;
        float tot = 0.f;
#pragma unroll
        for (int src = 0; src < kDCl; ++src) tot += sq[src][r];
        const float rn = 1.0f / sqrtf(tot / (float)kH + a.p.norm_eps);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = (y[r][e] * rn) * wf[e];
        uint2 o;
        o.x = pack2_rn(v[0], v[1]);
        o.y = pack2_rn(v[2], v[3]);
        *reinterpret_cast<uint2 *>(a.x_norm + (row0 + r) * kH + h0) = o;
      }
    }
  }
  // the next launch may start scheduling once every CTA got here
  pdl_trigger();
}

std::mutex g_dec_mu;
int g_dec_clusters[2][64];   // [kPost][device]: co-resident clusters (0: not configured)

template <bool kPost>
cudaError_t dec_configure(int dev, int *ncl) {
  std::lock_guard<std::mutex> lock(g_dec_mu);
  if (g_dec_clusters[kPost][dev] > 0) {
    *ncl = g_dec_clusters[kPost][dev];
    return cudaSuccess;
  }
  // a cluster of 16 is a non-portable size
  cudaError_t e = cudaFuncSetAttribute(pre_decode_kernel<kPost>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  cfg.gridDim = dim3(kDCl);
  cfg.blockDim = dim3(kDThreads);
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kDCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, pre_decode_kernel<kPost>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  g_dec_clusters[kPost][dev] = n;
  *ncl = n;
  return cudaSuccess;
}

template <bool kPost>
cudaError_t launch_decode(DecArgs a, int64_t logical_rows, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int ncl_max = 0;
  e = dec_configure<kPost>(dev, &ncl_max);
  if (e != cudaSuccess) return e;
  // rows per cluster pass from the chunk's row count: spread the chunk over
  // all co-resident clusters, at most 8 rows a pass (the per-row arithmetic
  // does not depend on the grouping)
  int64_t grp = (logical_rows + ncl_max - 1) / ncl_max;
  grp = grp < 1 ? 1 : (grp > kDRows ? kDRows : grp);
  const int64_t groups = (a.rows + grp - 1) / grp;
  const int clusters = (int)(groups < ncl_max ? groups : ncl_max);
  a.group = (int)grp;
  // (the cluster shape is the kernel's compile-time __cluster_dims__)
  return launch_pdl(pre_decode_kernel<kPost>, dim3((unsigned)(clusters * kDCl)), dim3(kDThreads),
                    0, s, 1, use_pdl(logical_rows), a);
}

}  // namespace

cudaError_t launch_pre_decode(const uint16_t *R, const float *fn, const float *scale,
                              const float *base, const uint16_t *norm_w, int64_t rows,
                              int64_t logical_rows, const mhc_params &p, uint16_t *x_norm,
                              float *post, float *comb, float *pre_out, float *mix_out,
                              cudaStream_t s, bool fn_stable) {
  DecArgs a = {};
  a.fn_stable = fn_stable ? 1 : 0;
  a.R = R; a.fn = fn; a.scale = scale; a.base = base; a.norm_w = norm_w; a.x_norm = x_norm;
  a.post = post; a.comb = comb; a.pre_out = pre_out; a.mix_out = mix_out; a.rows = rows;
  a.p = p;
  return launch_decode<false>(a, logical_rows, s);
}

cudaError_t launch_post_pre_decode(const uint16_t *R, const uint16_t *y, const float *post_in,
                                   const float *comb_in, const float *fn, const float *scale,
                                   const float *base, const uint16_t *norm_w, int64_t rows,
                                   int64_t logical_rows, const mhc_params &p, uint16_t *R_out,
                                   uint16_t *x_norm, float *post, float *comb, float *pre_out,
                                   float *mix_out, cudaStream_t s, bool fn_stable) {
  DecArgs a = {};
  a.fn_stable = fn_stable ? 1 : 0;
  a.R = R; a.fn = fn; a.scale = scale; a.base = base; a.norm_w = norm_w; a.x_norm = x_norm;
  a.post = post; a.comb = comb; a.pre_out = pre_out; a.mix_out = mix_out; a.rows = rows;
  a.y = y; a.post_in = post_in; a.comb_in = comb_in; a.R_out = R_out;
  a.p = p;
  return launch_decode<true>(a, logical_rows, s);
}

}  // namespace mhc
