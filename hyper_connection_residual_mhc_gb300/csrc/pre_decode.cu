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
// launches, round trips to L2 and between CTAs, and the serial Sinkhorn.
// One cluster of 16 CTAs takes a group of up to 8 rows; CTA s owns hidden
// columns [320 s, 320 s + 320) of all four streams (1280 of the 20480 k).
// Thread t handles stream t / 80 and four consecutive columns, and keeps its
// 4 x 24 fn values and its rows' x in registers for the whole kernel:
//   1. per row, the thread's 25 partials (24 dots, sum of squares), summed
//      over the warp by a fixed transpose tree and over the CTA's 10 warps in
//      warp order, go to the row's owner CTA (rank = row in the group);
//   2. in the owner CTA, warp 9 sums the 16 CTAs' partials in rank order,
//      computes rsqrt and the gates, and sends the 4 pre gates to every CTA;
//      beside it warp 8 forms the same sums of the comb logits and runs the
//      Sinkhorn (nothing in this kernel waits on comb, an output);
//   3. warps 0..2 of each CTA form y on its 320 columns and send each warp's
//      partial sums of y^2 to every CTA;
//   4. each CTA sums the 48 partials (CTA by CTA, warps in order) and writes
//      its 320 columns of x_norm.
// Every exchange is a set of 16-byte st.async stores into the receiving
// CTA's shared memory, counted as transaction bytes on one of its three
// mbarriers (partials, gates, y^2), each armed once with the bytes it will
// receive; a receiver's bounded wait ends when they have landed.  Two
// hardware cluster barriers remain: one before the first remote store (every
// CTA's mbarriers exist), its wait overlapping the loads, and one before
// exit (every CTA has issued its last store), arrived at as each warp
// finishes sending.
//
// Built twice: kPost = false is mhc_pre; kPost = true is mhc_fused_post_pre
// at these sizes (deepseek_v4.py, the use_fused_mhc_post_pre path): each
// thread first forms its 4 columns of R' = hc_post(R, y, post, comb) from the
// four streams and y at those columns, writes them to R_out, and runs the
// pre on R' -- one launch, and R' is never read back.
#include <mutex>

#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

namespace {

constexpr int kDCl = 16;                      // CTAs per cluster
constexpr int kDThreads = 320;                // 10 warps
constexpr int kDWarps = kDThreads / 32;
constexpr int kDRows = 8;                     // rows per cluster
constexpr int kDHs = kH / kDCl;               // 320 columns per CTA
constexpr int kDQ = kDHs / 4;                 // 80 threads per stream
constexpr int kDPart = kMix + 1;              // 24 dots + sum of squares
constexpr int kDPartV4 = (kDPart + 3) / 4;    // 16-byte stores per row (7)
constexpr int kDPartV = 4 * kDPartV4;         // the partials padded to 28
static_assert(kDQ * kHC == kDThreads, "one thread per (stream, 4 columns)");

__device__ unsigned int g_dec_error;   // bit s: a wait at site s expired

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

// Bounded wait, whole warp, on a barrier that other CTAs' st.async bytes
// complete (acquire at cluster scope; each barrier has one phase).  Expiry
// sets bit `site` of the error word and returns false: the warp then carries
// on with what has landed, so every thread still reaches the final cluster
// barrier.
__device__ __forceinline__ bool d_wait(uint32_t b, int site) {
  if (__all_sync(0xffffffffu, ptx::mbar_test_cluster(b, 0))) return true;
  const uint64_t t0 = ptx::now_ns();
  for (;;) {
    if (__all_sync(0xffffffffu, ptx::mbar_test_cluster(b, 0))) return true;
    if (__any_sync(0xffffffffu, ptx::now_ns() - t0 > ptx::kTimeoutNs)) {
      if ((threadIdx.x & 31) == 0) atomicOr(&g_dec_error, 1u << site);
      return false;
    }
  }
}

constexpr int kOwnerWarp = kDWarps - 1;        // the row owner's gates
constexpr int kSinkWarp = kDWarps - 2;         // the row owner's Sinkhorn
static_assert(kSinkWarp * 32 >= kDQ, "the owner warps must not own combine columns");
static_assert(kDPartV4 * kDRows <= 3 * 32, "the partial stores are warps 0..2's");

template <bool kPost>
__global__ void __cluster_dims__(kDCl, 1, 1) __launch_bounds__(kDThreads, 1)
pre_decode_kernel(const DecArgs a) {
  __shared__ __align__(16) float red[kDWarps][kDRows][32];   // per-warp row partials
  __shared__ __align__(16) float recv[kDCl][kDPartV];        // owner: its row's partials, per CTA
  __shared__ __align__(16) float pre_all[kDRows][kHC];       // the group rows' pre gates
  __shared__ __align__(16) float sq[kDCl][3][kDRows];        // y^2 partials, per CTA and warp
  __shared__ __align__(16) uint2 xs[kDRows][kHC][kDQ];       // the CTA's x, for the combine
  __shared__ float dot[kDPartV];                             // owner: 24 dots + sum of x^2
  __shared__ __align__(8) uint64_t bars[3];                  // partials, gates, y^2 landed

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = d_rank();
  const int si = tid / kDQ, q = tid % kDQ;          // stream, 4-column group
  const int k0 = si * kH + (int)rank * kDHs + 4 * q;
  const int h0 = (int)rank * kDHs + 4 * q;          // threads tid < 80: their columns
  const int G = a.group;
  const int64_t row0 = (int64_t)(blockIdx.x / kDCl) * G;
  const int nr = (int)(a.rows - row0 < G ? a.rows - row0 : G);
  const int ymsg = nr > 4 ? 2 : 1;                  // float4s of y^2 partials per warp pair
  const uint32_t b_part = d_smem_addr(&bars[0]), b_gate = d_smem_addr(&bars[1]),
                 b_sq = d_smem_addr(&bars[2]);
  if (tid == 0) {
    ptx::mbar_init(b_part, 1);
    ptx::mbar_init(b_gate, 1);
    ptx::mbar_init(b_sq, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // each phase completes once the bytes armed here have landed (bytes that
    // land first count down from zero)
    if ((int)rank < nr) ptx::mbar_expect_tx(b_part, kDCl * kDPartV * 4);
    ptx::mbar_expect_tx(b_gate, nr * kHC * 4);
    ptx::mbar_expect_tx(b_sq, kDCl * 3 * ymsg * 16);
  }
  // no CTA may store into another before that one's barriers exist: arrive
  // now, wait before the first remote store
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

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
  // the gate weights of the owner warp (pre and post) and the Sinkhorn warp
  // (comb), in flight while the partials form
  float w_sc = 0.f, w_base = 0.f;
  if (warp == kOwnerWarp && (lane & 15) < 8) {
    w_sc = __ldg(a.scale + ((lane & 15) < 4 ? 0 : 1));
    w_base = __ldg(a.base + (lane & 15));
  } else if (warp == kSinkWarp) {
    w_sc = __ldg(a.scale + 2);
    w_base = __ldg(a.base + 8 + (lane & 15));
  }
  if (!a.fn_stable) load_fn();
  float wf[4] = {0.f, 0.f, 0.f, 0.f};
  if (tid < kDQ) {
    const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(a.norm_w + h0));
    wf[0] = __uint_as_float(wv.x << 16); wf[1] = __uint_as_float(wv.x & 0xFFFF0000u);
    wf[2] = __uint_as_float(wv.y << 16); wf[3] = __uint_as_float(wv.y & 0xFFFF0000u);
  }
  // the cluster wait while loads are in flight (post_cols uses its loads at
  // once, so the fused build waits before them)
  if constexpr (kPost) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  uint2 xr[kDRows];
#pragma unroll
  for (int r = 0; r < kDRows; ++r) {
    if constexpr (kPost)
      xr[r] = r < nr ? post_cols(a, row0 + r, si, k0, h0) : make_uint2(0u, 0u);
    else
      xr[r] = r < nr ? __ldg(reinterpret_cast<const uint2 *>(a.R + (row0 + r) * kK + k0))
                     : make_uint2(0u, 0u);
  }
  if constexpr (!kPost) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

  // ---- 1. partials (row loops unrolled with a uniform guard, so the per-row
  // arrays stay in registers) ---------------------------------------------------
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
  // row r's 25 sums (in warp order; padded with zeros to 28) to CTA r, as
  // seven 16-byte stores that count on its partials barrier
  if (tid < nr * kDPartV4) {
    const int r = tid / kDPartV4, c0 = 4 * (tid % kDPartV4);
    float4 s = *reinterpret_cast<const float4 *>(&red[0][r][c0]);
#pragma unroll
    for (int w = 1; w < kDWarps; ++w) {
      const float4 t = *reinterpret_cast<const float4 *>(&red[w][r][c0]);
      s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
    }
    ptx::st_async_v4(d_mapa(d_smem_addr(&recv[rank][c0]), (uint32_t)r), s.x, s.y, s.z, s.w,
                     d_mapa(b_part, (uint32_t)r));
  }

  const unsigned full = 0xffffffffu;
  const bool own = (int)rank < nr;
  if (warp == kOwnerWarp && own) {
    // ---- 2. owner of group row `rank`: the pre and post gates, the mixes -----
    const int64_t row = row0 + rank;
    d_wait(b_part, 0);
    if (lane < kDPart) {
      float s = 0.f;
#pragma unroll
      for (int src = 0; src < kDCl; ++src) s += recv[src][lane];
      dot[lane] = s;
    }
    __syncwarp();
    const float rsq = rsqrt_nr(fmaf(dot[kMix], 1.0f / (float)kK, a.p.rms_eps));
    const int e = lane & 15;                  // lanes 16..31 mirror 0..15
    float gate = 0.f;
    if (e < 8) {
      const float l = fmaf(dot[e] * rsq, w_sc, w_base);
      const float sg = rcp_nr(1.0f + expf(-l));
      gate = e < 4 ? sg + a.p.hc_pre_eps : a.p.post_mult * sg;
    }
    // the 4 pre gates: lane d < 16 sends them to CTA d as one 16-byte store
    const float g0 = __shfl_sync(full, gate, 0), g1 = __shfl_sync(full, gate, 1);
    const float g2 = __shfl_sync(full, gate, 2), g3 = __shfl_sync(full, gate, 3);
    if (lane < kDCl)
      ptx::st_async_v4(d_mapa(d_smem_addr(&pre_all[rank][0]), (uint32_t)lane), g0, g1, g2, g3,
                       d_mapa(b_gate, (uint32_t)lane));
    __syncwarp();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (lane < 16) {
      if (e >= 4 && e < 8) a.post[row * kHC + (e - 4)] = gate;
      if (e < 4 && a.pre_out) a.pre_out[row * kHC + e] = gate;
      if (a.mix_out) {
        a.mix_out[row * kMix + e] = dot[e] * rsq;
        if (e < 8) a.mix_out[row * kMix + 16 + e] = dot[16 + e] * rsq;
      }
    }
  } else if (warp == kSinkWarp && own) {
    // ---- 2'. the same row's Sinkhorn, beside the owner warp: it feeds only
    // comb, an output, so nothing else waits on it --------------------------
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const int64_t row = row0 + rank;
    d_wait(b_part, 0);
    // lane e < 16 sums comb dot e, lanes 16.. the sum of squares: the owner
    // warp's sums, in the same order
    const int idx = lane < 16 ? 8 + lane : kMix;
    float s = 0.f;
#pragma unroll
    for (int src = 0; src < kDCl; ++src) s += recv[src][idx];
    const float ssq = __shfl_sync(full, s, 16);
    const float rsq = rsqrt_nr(fmaf(ssq, 1.0f / (float)kK, a.p.rms_eps));
    // exp(logits), then the whole 4x4 in every lane: rows then columns, each
    // sum paired (c0 + c1) + (c2 + c3) plus eps, each entry times the
    // reciprocal of its sum
    const float lg = expf(fmaf(s * rsq, w_sc, w_base));
    float c[kHC][kHC];
#pragma unroll
    for (int j = 0; j < kHC; ++j)
#pragma unroll
      for (int i = 0; i < kHC; ++i) c[j][i] = __shfl_sync(full, lg, 4 * j + i);
    for (int k = 0; k < a.p.sinkhorn_iters; ++k) {
#pragma unroll
      for (int j = 0; j < kHC; ++j) {
        const float d = rcp_nr(((c[j][0] + c[j][1]) + (c[j][2] + c[j][3])) + a.p.hc_sinkhorn_eps);
#pragma unroll
        for (int i = 0; i < kHC; ++i) c[j][i] = c[j][i] * d;
      }
#pragma unroll
      for (int i = 0; i < kHC; ++i) {
        const float d = rcp_nr(((c[0][i] + c[1][i]) + (c[2][i] + c[3][i])) + a.p.hc_sinkhorn_eps);
#pragma unroll
        for (int j = 0; j < kHC; ++j) c[j][i] = c[j][i] * d;
      }
    }
    if (lane < kHC) {
      float4 *o = reinterpret_cast<float4 *>(a.comb + row * 16);
#pragma unroll
      for (int j = 0; j < kHC; ++j)
        if (j == lane) o[j] = make_float4(c[j][0], c[j][1], c[j][2], c[j][3]);
    }
  } else if (warp >= 3) {
    // warps 3..9 without an owner's work: nothing of steps 3 and 4 is theirs
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  } else {
    // ---- 3. y on this CTA's columns (threads tid < 80); each warp's partial
    // sums of y^2 to every CTA ------------------------------------------------
    d_wait(b_gate, 1);
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
    // lane l < 8 gets the warp's sum for row l -- a fixed tree (halves 4, 2,
    // 1, then 8, 16)
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
      const bool up = (lane & w) != 0;
#pragma unroll
      for (int jj = 0; jj < w; ++jj) {
        const float send = up ? sy[jj] : sy[jj + w];
        const float keep = up ? sy[jj + w] : sy[jj];
        sy[jj] = keep + __shfl_xor_sync(full, send, w);
      }
    }
    float s = sy[0];
    s += __shfl_xor_sync(full, s, 8);
    s += __shfl_xor_sync(full, s, 16);
    // lane l: this warp's rows 4 (l / 16) .. + 3 to CTA l % 16, one 16-byte
    // store
    {
      const int dst = lane & 15, hf = lane >> 4;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float t = __shfl_sync(full, s, 4 * hf + e);
        v[e] = 4 * hf + e < nr ? t : 0.f;
      }
      if (hf < ymsg)
        ptx::st_async_v4(d_mapa(d_smem_addr(&sq[rank][warp][4 * hf]), (uint32_t)dst), v[0], v[1],
                         v[2], v[3], d_mapa(b_sq, (uint32_t)dst));
    }
    __syncwarp();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- 4. x_norm on this CTA's columns ---------------------------------------
    d_wait(b_sq, 2);
    if (tid < kDQ) {
#pragma unroll
      for (int r = 0; r < kDRows; ++r) {
        if (r >= nr) break;
        float tot = 0.f;
#pragma unroll
        for (int src = 0; src < kDCl; ++src) tot += (sq[src][0][r] + sq[src][1][r]) + sq[src][2][r];
        const float rn = rsqrt_nr(fmaf(tot, 1.0f / (float)kH, a.p.norm_eps));
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
  // the next launch may start scheduling once every CTA got here; no CTA
  // leaves before every CTA of the cluster has issued its last store
  pdl_trigger();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
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
  // one group per cluster (a chunk of up to 48 rows needs at most 8
  // clusters; more would queue behind the co-resident ones)
  const int64_t groups = (a.rows + grp - 1) / grp;
  if (groups > kDecodeMaxRows) return cudaErrorInvalidValue;
  const int clusters = (int)groups;
  a.group = (int)grp;
  // (the cluster shape is the kernel's compile-time __cluster_dims__)
  return launch_pdl(pre_decode_kernel<kPost>, dim3((unsigned)(clusters * kDCl)), dim3(kDThreads),
                    0, s, 1, use_pdl(logical_rows), a);
}

}  // namespace

cudaError_t decode_error_word(unsigned int *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dec_error, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_dec_error, &z, sizeof z);
  }
  return e;
}

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
